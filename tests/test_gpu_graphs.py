"""The forward and the recurrent call inside CUDA graphs: both are captured
once into a torch.cuda.CUDAGraph on static buffers (workspace included) and
replayed after new inputs are copied in.  Every replay must match the FP64
oracle on that replay's inputs (the calls do host work only at capture: the
tensor maps and launch parameters are baked into the graph, so replays must
not depend on anything but the buffers' contents).

Bar: max|x - x_ref| / max|x_ref| <= 1e-2 for o and for the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import gdn2 as gdn2_mod
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
KEYS = ("q", "k", "v", "g", "beta", "w", "h0")


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def captured(fn, wl, **kw):
    """Static device buffers for wl's inputs, the call captured on them."""
    d0 = inputs.generate(wl)
    st = {k: (d0[k].cuda() if torch.is_tensor(d0[k]) else d0[k]) for k in d0}
    dims = gdn2_mod.make_dims(st["q"], st["k"], st["v"], st["g"], st["beta"], st["w"], st["v"], st["cu_seqlens"])
    dims.state_segments = kw.get("state_segments", 0)
    nbytes = gdn2_mod.workspace_bytes(dims) if fn is gdn2_mod.chunk_gdn2_fwd else 256
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.T_tot, wl.HV, wl.V), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((wl.N, wl.HV, wl.K, wl.V), dtype=torch.float32, device="cuda")

    def call():
        fn(st["q"], st["k"], st["v"], st["g"], st["beta"], st["w"], scale=st["scale"], initial_state=st["h0"],
           cu_seqlens=st["cu_seqlens"], out=out, final_state=fs, workspace=ws, **kw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside the graph (library load, kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    return graph, st, out, fs


def replay_and_check(graph, st, out, fs, wl, seeds):
    for seed in seeds:
        d = inputs.generate(inputs.with_seed(wl, seed))
        for k in KEYS:
            if torch.is_tensor(d[k]):
                st[k].copy_(d[k])
        graph.replay()
        torch.cuda.synchronize()
        o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                           initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
        eo = rel_max(out.float().cpu().numpy(), o_ref)
        eh = rel_max(fs.cpu().numpy(), h_ref)
        assert eo <= TOL and eh <= TOL, "seed %d: o err %.3e, state err %.3e" % (seed, eo, eh)


def test_chunk_forward_in_a_graph(cuda_lib):
    wl = inputs.small("graph", [200, 64, 1, 333], H=2, HV=4, K=128, V=128, g_max=1.0, beta_max=2.0,
                      h0_std=0.05, seed=81)
    replay_and_check(*captured(cuda_lib.chunk_gdn2_fwd, wl), wl, seeds=(82, 83, 84))


def test_chunk_forward_with_segments_in_a_graph(cuda_lib):
    """The chunk-parallel state pass (five launches) captured."""
    wl = inputs.small("graphscan", [2000], H=1, HV=2, K=128, V=128, g_max=0.02, beta_max=1.0, h0_std=0.05,
                      seed=85)
    replay_and_check(*captured(cuda_lib.chunk_gdn2_fwd, wl, state_segments=4), wl, seeds=(86, 87))


def test_decode_step_in_a_graph(cuda_lib):
    wl = inputs.small("graphdec", [1] * 16, H=2, HV=4, K=128, V=128, g_max=0.5, beta_max=2.0, h0_std=0.05,
                      seed=88)
    replay_and_check(*captured(cuda_lib.recurrent_gdn2_fwd, wl), wl, seeds=(89, 90, 91))


def test_exact_pass_in_a_graph(cuda_lib):
    """The intra kernel's exact pass (a programmatic dependent launch) inside a
    graph: captured on slow decays (an empty exact list), then replayed with
    decays of up to 30 nats per token (most items listed) and slow ones again.
    The list is rebuilt on the device at every replay."""
    wl = inputs.small("graphwide", [130, 64, 1, 200], H=2, HV=4, K=128, V=128, g_max=0.5, beta_max=2.0,
                      h0_std=0.05, seed=92)
    graph, st, out, fs = captured(cuda_lib.chunk_gdn2_fwd, wl)
    for seed, wide in ((93, True), (94, False), (95, True)):
        d = inputs.generate(inputs.with_seed(wl, seed))
        if wide:
            gen = torch.Generator().manual_seed(seed)
            d["g"] = torch.rand(d["g"].shape, generator=gen).mul_(-30.0)
        for k in KEYS:
            if torch.is_tensor(d[k]):
                st[k].copy_(d[k])
        graph.replay()
        torch.cuda.synchronize()
        o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                           initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
        eo = rel_max(out.float().cpu().numpy(), o_ref)
        eh = rel_max(fs.cpu().numpy(), h_ref)
        assert eo <= TOL and eh <= TOL, "seed %d (wide %s): o err %.3e, state err %.3e" % (seed, wide, eo, eh)
