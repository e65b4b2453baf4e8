"""GPU parity of the chunk-parallel state pass (tensor-core path, K = V =
128): each sequence's chunks in P segments; segment 0 replayed from the
initial state beside the transitions [M | B] of S_out = M S_in + B of
segments 1 .. P - 2, a combine over those, then segments 1 .. P - 1 replayed
from their incoming states.  The transitions and the replay run on the
lookahead state kernels (on the plain one with GDN2_STATE_LOOKAHEAD=0).
Checked against the FP64 oracle and against the sequential pass.

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


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def run(gdn2, d, segments, **kw):
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    o, hT = gdn2.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], state_segments=segments, **kw)
    torch.cuda.synchronize()
    return o, hT


@pytest.mark.parametrize("segments", [2, 3, 5, 16])
def test_forced_segments_match_oracle(cuda_lib, segments):
    """Ragged sequences (one shorter than the segment count: empty segments),
    grouped value heads, decay stress, an initial state."""
    wl = inputs.small("scan", [700, 1, 129, 2000], H=2, HV=4, K=128, V=128, g_max=2.0, beta_max=2.0,
                      h0_std=0.05, seed=71)
    d = inputs.generate(wl)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    o, hT = run(cuda_lib, d, segments)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL
    o1, h1 = run(cuda_lib, d, 1)  # sequential pass
    assert rel_max(o.float().cpu().numpy(), o1.float().cpu().numpy()) <= TOL
    assert rel_max(hT.cpu().numpy(), h1.cpu().numpy()) <= TOL


@pytest.mark.parametrize("segments", [2, 3, 6])
def test_forced_segments_plain_kernel(cuda_lib, monkeypatch, segments):
    """The same with the transitions and the replay on the plain state kernel
    (GDN2_STATE_LOOKAHEAD=0); the default runs them on the lookahead kernels.
    The replay of P - 1 segments takes 64-column tiles at P = 2 and 3 (16
    (sequence, head) pairs), 128-column ones at P = 6; P = 2 has no combine."""
    monkeypatch.setenv("GDN2_STATE_LOOKAHEAD", "0")
    wl = inputs.small("scanplain", [700, 1, 129, 2000], H=2, HV=4, K=128, V=128, g_max=2.0, beta_max=2.0,
                      h0_std=0.05, seed=73)
    d = inputs.generate(wl)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    o, hT = run(cuda_lib, d, segments)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("combine", ["cuda", "tc"])
def test_combine_kernels(cuda_lib, monkeypatch, combine):
    """Both combine kernels (the tensor-core one by default, the CUDA-core
    one with GDN2_SCAN_COMBINE=cuda) at 9 segments (7 dependent steps from
    segment 1's incoming state), with slow decay so that every step's M S_in
    term matters, and a bf16 V-major initial state read by segment 0's
    replay."""
    if combine == "cuda":
        monkeypatch.setenv("GDN2_SCAN_COMBINE", "cuda")
    wl = inputs.small("comb", [1500, 700], H=2, HV=2, K=128, V=128, g_max=0.02, beta_max=1.0, h0_std=0.5,
                      seed=74)
    d = inputs.generate(wl)
    d["h0"] = d["h0"].to(torch.bfloat16)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = dict(d)
    dd["h0"] = d["h0"].transpose(-1, -2).contiguous()  # V-major
    o, hT = run(cuda_lib, dd, 9, state_v_major=True)
    hT = hT.float().transpose(-1, -2)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("segments", [3, 5])
def test_segments_with_head_counts_fp16_l2norm(cuda_lib, segments):
    """The chunk-parallel pass with more query than value heads and fewer key
    heads (H = 4, HK = HV = 2: four state heads), fp16 q/k/v/w/beta, the
    fused L2 norm and an initial state; 64-column replay tiles at P = 3,
    128-column ones at P = 5."""
    wl = inputs.small("scanheads", [900, 2000, 1], H=4, HV=4, K=128, V=128, g_max=0.3, beta_max=2.0,
                      h0_std=0.05, seed=75)
    d = inputs.generate(wl)
    d["k"] = d["k"][:, :2].contiguous()
    d["v"] = d["v"][:, :2].contiguous()
    for key in ("q", "k", "v", "beta", "w"):
        d[key] = (d[key].float() * (2.0 if key == "q" else 1.0)).to(torch.float16)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], use_qk_l2norm=True)
    o, hT = run(cuda_lib, d, segments, use_qk_l2norm=True)
    assert o.shape == o_ref.shape and hT.shape == h_ref.shape
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


def test_automatic_segments(cuda_lib):
    """A few long heads: the library picks P > 1 (visible in the launch
    count) and the result matches the oracle."""
    wl = inputs.small("autoscan", [4096], H=2, HV=2, K=128, V=128, g_max=0.5, h0_std=0.05, seed=72)
    d = inputs.generate(wl)
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    dims = gdn2_mod.make_dims(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], dd["v"], dd["cu_seqlens"])
    assert gdn2_mod.launch_count(dims) == 6  # map, intra (2 passes), transitions, combine, replay
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    o, hT = run(cuda_lib, d, 0)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("state,v_major", [(torch.float32, False), (torch.bfloat16, True)])
def test_segments_with_state_variants_and_fp16(cuda_lib, state, v_major):
    wl = inputs.small("scanvar", [1500, 300], H=1, HV=2, K=128, V=128, g_max=1.0, beta_max=2.0, h0_std=0.05,
                      seed=73)
    d = inputs.generate(wl)
    for key in ("q", "k", "v", "beta", "w"):
        d[key] = d[key].float().to(torch.float16)
    d["h0"] = d["h0"].to(state)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = dict(d)
    if v_major:
        dd["h0"] = d["h0"].transpose(-1, -2).contiguous()
    o, hT = run(cuda_lib, dd, 4, state_v_major=v_major)
    hT = hT.float()
    if v_major:
        hT = hT.transpose(-1, -2)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("segments", [4, 16])
def test_slow_decay_segments(cuda_lib, segments):
    """Slow decay (about 0.88 per 64-token chunk): each segment's transition M
    keeps most of the incoming state, so a wrong or missing M S_in term in the
    combine, or a replay that ignores its incoming state, shows in o and in the
    final state.  One sequence without an initial state next to one with."""
    for h0_std in (None, 0.05):
        wl = inputs.small("scanslow", [3000, 1100], H=2, HV=2, K=128, V=128, g_max=0.004, beta_max=1.0,
                          h0_std=h0_std, seed=74)
        d = inputs.generate(wl)
        o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                           initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
        o, hT = run(cuda_lib, d, segments)
        assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
        assert rel_max(hT.cpu().numpy(), h_ref) <= TOL
