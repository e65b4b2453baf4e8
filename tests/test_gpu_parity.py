"""GPU parity: the CUDA library against the FP64 oracle on the same inputs.

Bar (GDN-2 prefill forward): max|o - o_ref| / max|o_ref| <= 1e-2, and the
same bound on the final state, per compared set of outputs.  Small cases are
compared element by element; the full-size workloads on every
(sequence, value head) unit, which the oracle computes one by one, in the
launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
IMPLS = ["simt", "tc"]


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def to_dev(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


def run_gpu(gdn2, d, impl, **kw):
    o, hT = gdn2.chunk_gdn2_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], impl=impl, **kw)
    torch.cuda.synchronize()
    return o, hT


def run_oracle(d, **kw):
    return oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                               initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], **kw)


def check_full(gdn2, wl, impl, tol=TOL, **kw):
    d = inputs.generate(wl)
    o_ref, h_ref = run_oracle(d, use_qk_l2norm=kw.get("use_qk_l2norm", False))
    o, hT = run_gpu(gdn2, to_dev(d), impl, **kw)
    eo = rel_max(o.float().cpu().numpy(), o_ref) if wl.T_tot else 0.0
    eh = rel_max(hT.cpu().numpy(), h_ref)
    assert eo <= tol and eh <= tol, "%s/%s: o err %.3e, state err %.3e" % (wl.name, impl, eo, eh)
    return eo, eh


@pytest.mark.parametrize("impl", IMPLS)
def test_tiny_workload(cuda_lib, impl):
    check_full(cuda_lib, inputs.workload(1), impl)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_varlen_gva(cuda_lib, impl, D):
    """Partial chunks (1, 63, 65, ...), an empty sequence, several tiles per
    sequence, grouped value heads and an initial state."""
    wl = inputs.small("ragged", [1, 63, 64, 65, 0, 200, 130], H=2, HV=4, K=D, V=D, g_max=0.5,
                      beta_max=2.0, h0_std=0.05, seed=31)
    check_full(cuda_lib, wl, impl)


@pytest.mark.parametrize("impl", IMPLS)
def test_strong_decay(cuda_lib, impl):
    """g = -U(0,3), beta in [0,2]: the decay-stress regime at small size."""
    wl = inputs.small("decay", [300, 77], H=2, HV=2, K=128, V=128, g_max=3.0, beta_max=2.0,
                      h0_std=0.05, seed=32)
    check_full(cuda_lib, wl, impl)


@pytest.mark.parametrize("impl", IMPLS)
def test_missing_gates(cuda_lib, impl):
    wl = inputs.small("nogates", [129, 40], H=1, HV=2, K=64, V=64, seed=33)
    d = inputs.generate(wl)
    d["g"] = d["beta"] = d["w"] = None
    o_ref, h_ref = run_oracle(d)
    o, hT = run_gpu(cuda_lib, to_dev(d), impl)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("case", ["linear_attention", "no_write", "scalar_gated_delta"])
def test_degenerate_gates(cuda_lib, impl, case):
    """Gates present but degenerate, where the method reduces to a simpler one
    (the oracle pins check the same reductions on the host): g = 0, beta = 0,
    w = 1 is cumulative linear attention (A = 0, T = I); w = 0 writes nothing,
    so the output reads the decayed and erased initial state; g and beta
    constant over the channels with w = beta is the scalar gated delta rule."""
    wl = inputs.small("degen_" + case, [0, 1, 63, 64, 200], H=2, HV=4, K=128, V=128, g_max=0.5, beta_max=1.0,
                      h0_std=0.05, seed=41)
    d = inputs.generate(wl)
    if case == "linear_attention":
        d["g"] = torch.zeros_like(d["g"])
        d["beta"] = torch.zeros_like(d["beta"])
        d["w"] = torch.ones_like(d["w"])
    elif case == "no_write":
        d["w"] = torch.zeros_like(d["w"])
    else:
        d["g"] = d["g"][..., :1].expand_as(d["g"]).contiguous()
        d["beta"] = d["beta"][..., :1].expand_as(d["beta"]).contiguous()
        d["w"] = d["beta"].clone()
    o_ref, h_ref = run_oracle(d)
    o, hT = run_gpu(cuda_lib, to_dev(d), impl)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
def test_l2norm_in_kernel(cuda_lib, impl):
    wl = inputs.small("l2", [150], H=2, HV=2, K=128, V=128, seed=34)
    d = inputs.generate(wl)
    d["q"] = (d["q"].float() * 3.0).to(torch.bfloat16)
    d["k"] = (d["k"].float() * 0.25).to(torch.bfloat16)
    o_ref, h_ref = run_oracle(d, use_qk_l2norm=True)
    o, hT = run_gpu(cuda_lib, to_dev(d), impl, use_qk_l2norm=True)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
def test_strided_inputs_and_int64_cu(cuda_lib, impl):
    """Token/head strides other than packed (only the channel dim contiguous)
    and int64 cu_seqlens."""
    wl = inputs.small("strided", [100, 37], H=2, HV=2, K=64, V=64, h0_std=0.05, seed=35)
    d = inputs.generate(wl)
    o_ref, h_ref = run_oracle(d)
    dd = to_dev(d)
    for key in ("q", "k", "v", "beta", "w", "g"):
        x = dd[key]
        big = torch.zeros(x.shape[0], x.shape[1], 2 * x.shape[2], dtype=x.dtype, device=x.device)
        big[..., :x.shape[2]] = x
        dd[key] = big[..., :x.shape[2]]
        assert not dd[key].is_contiguous()
    dd["cu_seqlens"] = dd["cu_seqlens"].long()
    out_big = torch.zeros(wl.T_tot, wl.HV, 2 * wl.V, dtype=torch.bfloat16, device="cuda")
    o, hT = run_gpu(cuda_lib, dd, impl, out=out_big[..., :wl.V])
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert float(out_big[..., wl.V:].abs().max()) == 0.0, "wrote outside the strided output"
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
def test_head_major_layout(cuda_lib, impl):
    """Tensors stored head-major ([heads, T, D] memory, viewed as [T, heads,
    D]): the head stride exceeds the token stride."""
    wl = inputs.small("headmajor", [90, 64, 3], H=2, HV=4, K=128, V=128, g_max=0.5, beta_max=2.0,
                      h0_std=0.05, seed=36)
    d = inputs.generate(wl)
    o_ref, h_ref = run_oracle(d)
    dd = to_dev(d)
    for key in ("q", "k", "v", "beta", "w", "g"):
        x = dd[key]
        dd[key] = x.transpose(0, 1).contiguous().transpose(0, 1)
        assert dd[key].stride(1) > dd[key].stride(0)
    o, hT = run_gpu(cuda_lib, dd, impl)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("D", [64, 128])
def test_tc_row_copies(cuda_lib, monkeypatch, D):
    """The tensor-core intra kernel's row-by-row copies of g, v, w (used when
    the tensor maps cannot be encoded; GDN2_ROW_COPIES=1 forces them), with
    ragged chunks and no w."""
    monkeypatch.setenv("GDN2_ROW_COPIES", "1")
    wl = inputs.small("rows", [1, 70, 129], H=1, HV=2, K=D, V=D, g_max=1.0, beta_max=2.0, h0_std=0.05,
                      seed=37)
    check_full(cuda_lib, wl, "tc")
    d = inputs.generate(wl)
    d["w"] = None
    o_ref, h_ref = run_oracle(d)
    o, hT = run_gpu(cuda_lib, to_dev(d), "tc")
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("segments", [1, 4])
def test_plain_launches_match_chained(cuda_lib, monkeypatch, segments):
    """Every launch after the first of a call is chained to its predecessor
    (programmatic dependent launches); GDN2_PDL=0 launches them plainly.  The
    kernels and their arithmetic are the same, so the two give bit-identical
    results, here with the exact pass active (decays past its threshold in
    some channels) and both state passes, and both match the oracle."""
    wl = inputs.small("pdl", [700, 1, 129, 2000], H=2, HV=4, K=128, V=128, g_max=1.0, beta_max=2.0,
                      h0_std=0.05, seed=38)
    d = inputs.generate(wl)
    g = d["g"].clone()
    g[:, :, :8] *= 40.0  # 8 channels decaying up to 40 nats per token
    d["g"] = g
    o_ref, h_ref = run_oracle(d)
    dd = to_dev(d)
    o1, h1 = run_gpu(cuda_lib, dd, "tc", state_segments=segments)
    monkeypatch.setenv("GDN2_PDL", "0")
    o0, h0 = run_gpu(cuda_lib, dd, "tc", state_segments=segments)
    assert torch.equal(o1, o0) and torch.equal(h1, h0)
    assert rel_max(o1.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(h1.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
def test_split_sequence_matches_one_pass(cuda_lib, impl):
    """Prefill in two calls carrying the final state equals one call
    (FlashGDN-2 quick start: prefill, then continue from the state)."""
    wl = inputs.small("split", [257], H=2, HV=2, K=128, V=128, h0_std=0.05, seed=36)
    d = to_dev(inputs.generate(wl))
    o, hT = run_gpu(cuda_lib, d, impl)
    t = 100
    a = {**d, **{x: d[x][:t] for x in ("q", "k", "v", "g", "beta", "w")},
         "cu_seqlens": torch.tensor([0, t], dtype=torch.int32, device="cuda")}
    o1, h1 = run_gpu(cuda_lib, a, impl)
    b = {**d, **{x: d[x][t:] for x in ("q", "k", "v", "g", "beta", "w")}, "h0": h1,
         "cu_seqlens": torch.tensor([0, 257 - t], dtype=torch.int32, device="cuda")}
    o2, h2 = run_gpu(cuda_lib, b, impl)
    assert rel_max(torch.cat([o1, o2]).float().cpu().numpy(), o.float().cpu().numpy()) <= TOL
    assert rel_max(h2.cpu().numpy(), hT.cpu().numpy()) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
def test_empty_tokens_keep_state(cuda_lib, impl):
    """T_tot = 0 with N = 2 sequences: final_state = initial_state."""
    h0 = torch.randn(2, 2, 64, 64, device="cuda")
    z = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(0, 2, 64, device="cuda")
    cu = torch.tensor([0, 0, 0], dtype=torch.int32, device="cuda")
    o, hT = cuda_lib.chunk_gdn2_fwd(z, z, z, g, z, z, initial_state=h0, cu_seqlens=cu, impl=impl)
    torch.cuda.synchronize()
    assert torch.equal(hT, h0)


@pytest.mark.parametrize("impl", IMPLS)
def test_bad_cu_seqlens_reported_on_device(cuda_lib, impl):
    wl = inputs.small("badcu", [64, 64], H=1, HV=1, K=64, V=64, seed=37)
    d = to_dev(inputs.generate(wl))
    d["cu_seqlens"] = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")  # decreasing
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    run_gpu(cuda_lib, d, impl, workspace=ws)
    assert cuda_lib.device_status(ws) == 9
    d["cu_seqlens"] = torch.tensor([0, 64, 128], dtype=torch.int32, device="cuda")
    run_gpu(cuda_lib, d, impl, workspace=ws)
    assert cuda_lib.device_status(ws) == 0


# ---------------------------------------------------------------------------
# Full-size workloads: run the whole launch, compare every unit.
# ---------------------------------------------------------------------------
def unit_problem(d, wl, n, hv):
    """Inputs of one (sequence, value head) unit as a stand-alone problem."""
    cu = d["cu_seqlens"].tolist()
    a, b = cu[n], cu[n + 1]
    h = hv // (wl.HV // wl.H)
    sl = lambda x, head: None if x is None else x[a:b, head:head + 1].cpu()
    return dict(q=sl(d["q"], h), k=sl(d["k"], h), v=sl(d["v"], hv), g=sl(d["g"], hv),
                beta=sl(d["beta"], hv), w=sl(d["w"], hv),
                h0=None if d["h0"] is None else d["h0"][n:n + 1, hv:hv + 1].cpu(),
                cu_seqlens=[0, b - a], scale=d["scale"]), (a, b)


@pytest.mark.parametrize("index", [2, 3, 4, 5])
def test_full_size_every_unit(cuda_lib, index):
    """Each D = 128 workload at full size, in the launch configuration the
    benchmark times, through both GPU paths; every (sequence, value head)
    unit's output rows and final state against the FP64 oracle (one oracle
    call per unit, units in parallel).  The bar is the global one,
    max|x - x_ref| / max|x_ref| <= 1e-2 over all units; the achieved errors
    are printed, and the worst units on failure."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    wl = inputs.workload(index)
    d = inputs.generate(wl, device="cuda")
    outs = {}
    for impl in IMPLS:
        o, hT = run_gpu(cuda_lib, d, impl)
        outs[impl] = (o.float().cpu().numpy(), hT.float().cpu().numpy())
        del o, hT
    units = [(n, hv) for n in range(wl.N) for hv in range(wl.HV)]

    def one(u):
        n, hv = u
        pd, (a, b) = unit_problem(d, wl, n, hv)
        o_ref, h_ref = oracle.gdn2_forward(pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], pd["w"],
                                           scale=pd["scale"], initial_state=pd["h0"],
                                           cu_seqlens=pd["cu_seqlens"], threads=1)
        res = {"ref": (float(np.abs(o_ref).max(initial=0.0)), float(np.abs(h_ref).max()))}
        for impl, (o, hT) in outs.items():
            res[impl] = (float(np.abs(o[a:b, hv] - o_ref[:, 0]).max(initial=0.0)),
                         float(np.abs(hT[n, hv] - h_ref[0, 0]).max()))
        return u, res

    with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
        per_unit = dict(ex.map(one, units))
    ref_o = max(r["ref"][0] for r in per_unit.values())
    ref_h = max(r["ref"][1] for r in per_unit.values())
    bad = []
    for impl in IMPLS:
        eo = max(r[impl][0] for r in per_unit.values()) / ref_o
        eh = max(r[impl][1] for r in per_unit.values()) / ref_h
        print("full size %s, %d units, %s: o err %.3e, final-state err %.3e"
              % (wl.name, len(units), impl, eo, eh))
        if eo > TOL or eh > TOL:
            worst = sorted(per_unit.items(), key=lambda kv: -max(kv[1][impl][0] / ref_o, kv[1][impl][1] / ref_h))
            bad.append("%s: o %.3e state %.3e; worst units %s" % (
                impl, eo, eh, ["(n=%d, hv=%d): o %.3e state %.3e" % (u[0], u[1], r[impl][0] / ref_o,
                                                                       r[impl][1] / ref_h)
                                for u, r in worst[:5]]))
    assert not bad, "; ".join(bad)


@pytest.mark.parametrize("groups,slices", [(1, 0), (3, 0), (4, 4), (4, 8)])
def test_host_runner_matches_device_call(cuda_lib, groups, slices):
    """HostRunner (pinned host buffers, pieces pipelined over three streams)
    matches the oracle.  Sequence groups (slices = 0) return exactly what one
    device call returns; time slices (every sequence cut into pieces of whole
    chunks, the state carried from piece to piece) differ from it by rounding
    only."""
    wl = inputs.small("host", [100, 1, 0, 64, 250, 33, 700], H=2, HV=4, K=128, V=128, g_max=1.0, beta_max=2.0,
                      h0_std=0.05, seed=38)
    d = inputs.generate(wl)
    host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in d.items()}
    runner = cuda_lib.HostRunner(host, groups=groups, slices=slices)
    assert (type(runner).__name__ == "_SlicedRunner") == (slices > 0)
    for _ in range(2):  # twice in a row: buffers are reused
        o_h, h_h = runner()
    torch.cuda.synchronize()
    o_d, h_d = run_gpu(cuda_lib, to_dev(d), "tc")
    tol_dev = 1e-6 if slices == 0 else TOL
    assert rel_max(o_h.float().numpy(), o_d.float().cpu().numpy()) <= tol_dev
    assert rel_max(h_h.numpy(), h_d.cpu().numpy()) <= tol_dev
    o_ref, h_ref = run_oracle(d)
    assert rel_max(o_h.float().numpy(), o_ref) <= TOL
    assert rel_max(h_h.numpy(), h_ref) <= TOL


@pytest.mark.parametrize("lookahead", ["1", "0"])
def test_state_kernels_64_column_tiles(cuda_lib, monkeypatch, lookahead):
    """Both state kernels of the 64-column tile (few (sequence, head) pairs):
    the one-chunk lookahead kernel (default) and the plain one; ragged
    sequences of 0 to 15 chunks (every count up to one past the three record
    stages, then several wraps), decay stress, initial state."""
    monkeypatch.setenv("GDN2_STATE_LOOKAHEAD", lookahead)
    wl = inputs.small("vt64_%s" % lookahead, [0, 1, 64, 65, 129, 192, 200, 900], H=2, HV=4, K=128, V=128, g_max=2.0,
                      beta_max=2.0, h0_std=0.05, seed=95)
    d = inputs.generate(wl)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    o, hT = cuda_lib.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                    initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], state_segments=1)
    torch.cuda.synchronize()
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("lookahead,variant", [("1", False), ("64", False), ("1", True)])
def test_state_kernels_128_column_tiles(cuda_lib, monkeypatch, lookahead, variant):
    """Both state kernels of the 128-column tile (more (sequence, head) pairs
    than half the SMs): the lookahead kernel (default) and the plain one
    (GDN2_STATE_LOOKAHEAD=64); ragged sequences of 0 to 15 chunks, grouped
    value heads, decay stress, initial state.  The variant case runs the
    lookahead kernel on fp16 inputs, fp16 g, a bf16 V-major state, the fused
    q/k L2 norm and no w gate."""
    monkeypatch.setenv("GDN2_STATE_LOOKAHEAD", lookahead)
    lens = [0, 1, 64, 65, 129, 192, 200, 900, 333, 64]
    wl = inputs.small("vt128_%s_%d" % (lookahead, variant), lens, H=4, HV=8, K=128, V=128, g_max=2.0,
                      beta_max=2.0, h0_std=0.05, seed=96)
    assert 2 * len(lens) * 8 > 152  # the host picks 128-column tiles
    d = inputs.generate(wl)
    kw = {}
    if variant:
        d["w"] = None
        for k in ("q", "k", "v", "beta"):
            d[k] = d[k].float().to(torch.float16)
        d["g"] = d["g"].to(torch.float16)
        d["h0"] = d["h0"].to(torch.bfloat16)
        kw = dict(use_qk_l2norm=True, state_v_major=True, state_dtype=torch.bfloat16)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                                       use_qk_l2norm=variant)
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    h0 = dd["h0"].transpose(-1, -2).contiguous() if variant else dd["h0"]
    o, hT = cuda_lib.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                    initial_state=h0, cu_seqlens=dd["cu_seqlens"], state_segments=1, **kw)
    torch.cuda.synchronize()
    hT = hT.float()
    if variant:
        hT = hT.transpose(-1, -2)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("n_seq", [2500, 5000])
def test_many_short_sequences(cuda_lib, n_seq):
    """2,500 or 5,000 ragged sequences of 0-130 tokens (more than the chunk
    map's 1024 threads: its scans and its longest-first counting sort loop;
    5,000 is past the 4,095 sequences whose chunk offsets it keeps in shared
    memory), grouped value heads, an initial state; every output row and
    final state against the oracle."""
    rng = np.random.default_rng(99)
    lens = [int(x) for x in rng.integers(0, 131, size=n_seq)]
    lens[::97] = [0] * len(lens[::97])  # some empty sequences
    wl = inputs.small("many", lens, H=1, HV=2, K=64, V=64, g_max=1.0, beta_max=2.0, h0_std=0.05, seed=98)
    d = inputs.generate(wl)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    o, hT = cuda_lib.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                    initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"])
    torch.cuda.synchronize()
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL
