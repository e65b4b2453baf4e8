"""GPU parity for the head counts of the FlashInfer docs' parameter list:
num_k_heads equal to num_q_heads or num_v_heads, query and value head counts
equal or one a multiple of the other, one state per state head
HS = max(H, HV).  Both chunked paths and the token-by-token call against the
FP64 oracle, which takes the same head counts.

Bar: max|x - x_ref| / max|x_ref| <= 1e-2 for o and for the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2

CASES = [(4, 2, 2), (4, 4, 2), (2, 4, 4), (2, 2, 4), (3, 6, 6), (6, 2, 2)]  # (H, HK, HV)


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def problem(H, HK, HV, D, lens, seed, g_max=1.0):
    """Inputs with H query, HK key and HV value heads: drawn for HS state
    heads, then q, k, v keep their first H, HK, HV heads."""
    HS = max(H, HV)
    wl = inputs.small("heads_%d_%d_%d" % (H, HK, HV), lens, H=HS, HV=HS, K=D, V=D, g_max=g_max, beta_max=2.0,
                      h0_std=0.05, seed=seed)
    d = inputs.generate(wl)
    d["q"] = d["q"][:, :H].contiguous()
    d["k"] = d["k"][:, :HK].contiguous()
    d["v"] = d["v"][:, :HV].contiguous()
    return d


def run(cuda_lib, d, fn="chunk", **kw):
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                                       use_qk_l2norm=kw.get("use_qk_l2norm", False))
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    call = cuda_lib.chunk_gdn2_fwd if fn == "chunk" else cuda_lib.recurrent_gdn2_fwd
    o, hT = call(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                 initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    assert o.shape == o_ref.shape and hT.shape == h_ref.shape
    return rel_max(o.float().cpu().numpy(), o_ref), rel_max(hT.float().cpu().numpy(), h_ref)


@pytest.mark.parametrize("impl", ["simt", "tc"])
@pytest.mark.parametrize("heads", CASES, ids=["H%d_HK%d_HV%d" % c for c in CASES])
def test_head_counts(cuda_lib, impl, heads):
    H, HK, HV = heads
    d = problem(H, HK, HV, 128, [1, 63, 130, 200], seed=71)
    eo, eh = run(cuda_lib, d, impl=impl)
    assert eo <= TOL and eh <= TOL, (heads, impl, eo, eh)


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_head_counts_l2norm_d64(cuda_lib, impl):
    """Key heads differing from query heads through the fused L2 norm (the
    SIMT path normalises q and k into separate packed copies) at D = 64."""
    d = problem(4, 2, 2, 64, [70, 129], seed=72)
    d["q"] = (d["q"].float() * 3.0).to(torch.bfloat16)
    d["k"] = (d["k"].float() * 0.5).to(torch.bfloat16)
    eo, eh = run(cuda_lib, d, impl=impl, use_qk_l2norm=True)
    assert eo <= TOL and eh <= TOL, (eo, eh)


def test_head_counts_tc_lookahead_tiles(cuda_lib, monkeypatch):
    """More query heads than value heads with enough (sequence, head) pairs
    for the 128-column lookahead state kernel (the 64-column one runs in the
    cases above)."""
    d = problem(8, 4, 4, 128, [65, 200, 129, 64, 300, 1, 90, 77, 150, 33], seed=73)
    assert 2 * 10 * 8 > 152  # 128-column tiles
    eo, eh = run(cuda_lib, d, impl="tc", state_segments=1)
    assert eo <= TOL and eh <= TOL, (eo, eh)


@pytest.mark.parametrize("heads", [(4, 2, 2), (2, 4, 4), (4, 4, 2)], ids=["H4_HK2_HV2", "H2_HK4_HV4", "H4_HK4_HV2"])
def test_head_counts_recurrent(cuda_lib, heads):
    H, HK, HV = heads
    d = problem(H, HK, HV, 128, [1, 20, 33], seed=74)
    eo, eh = run(cuda_lib, d, fn="recurrent")
    assert eo <= TOL and eh <= TOL, (heads, eo, eh)


def test_head_counts_host_runner(cuda_lib):
    """HostRunner (pinned host buffers, pieces pipelined over three streams)
    with more query than value heads and fewer key heads: outputs and states
    are allocated per state head and match the oracle."""
    d = problem(4, 2, 2, 128, [100, 1, 0, 257, 64], seed=75)
    host = {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in d.items()}
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    for slices in (0, 4):
        runner = cuda_lib.HostRunner(host, groups=2, slices=slices)
        o, hT = runner()
        torch.cuda.synchronize()
        assert o.shape == o_ref.shape and hT.shape == h_ref.shape
        assert rel_max(o.float().numpy(), o_ref) <= TOL, slices
        assert rel_max(hT.float().numpy(), h_ref) <= TOL, slices
