"""GPU parity at the edges of the input domain.

The FlashInfer docs give g as a natural-log decay, elementwise <= 0, with no
floor, and q/k/v as bf16 or fp16 of any magnitude.  These tests take the
chunked forward to those edges against the FP64 oracle:

* decays of up to 80 nats per token, where a 16-token sub-chunk reference
  alone would need factors of e^{1280} (burn-gdn2 README, "Numerical
  stability": every weight e^{G_p - G_q} must stay <= 1), mixed within one
  chunk with channels of slow decay;
* values and initial states three orders of magnitude above the workloads';
* values past the range of the tensor-core path's fp16 intermediates, which
  must come back as GDN2_ERR_RANGE in the device status, never as a silent
  wrong answer with status OK.

Bar: max|x - x_ref| / max|x_ref| <= 1e-2 for o and for the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
IMPLS = ["simt", "tc"]
ERR_RANGE = 14


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def run_both(gdn2, d, impl, ws=None):
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    if ws is None:
        ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    o, hT = gdn2.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], impl=impl, workspace=ws)
    status = gdn2.device_status(ws)
    return o.float().cpu().numpy(), hT.float().cpu().numpy(), o_ref, h_ref, status


def wide_decay_g(T, HV, K, seed, g_max=30.0, fast=(0, 5, 17, 40, 63), fast_g=-80.0):
    """g = -U(0, g_max) per token and channel; the channels in `fast` decay by
    `fast_g` nats at every token."""
    gen = torch.Generator().manual_seed(seed)
    g = torch.rand((T, HV, K), generator=gen).mul_(-g_max)
    g[:, :, [c for c in fast if c < K]] = fast_g
    return g


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("D", [64, 128])
def test_wide_decay(cuda_lib, impl, D):
    """g = -U(0,30), several channels at -80 per token, beta in [0,2], an
    initial state, ragged sequences over several chunks."""
    wl = inputs.small("wide%d" % D, [1, 63, 200, 130, 17], H=2, HV=4, K=D, V=D, g_max=3.0, beta_max=2.0,
                      h0_std=0.05, seed=51)
    d = inputs.generate(wl)
    d["g"] = wide_decay_g(wl.T_tot, wl.HV, wl.K, seed=52)
    o, hT, o_ref, h_ref, status = run_both(cuda_lib, d, impl)
    assert status == 0
    eo, eh = rel_max(o, o_ref), rel_max(hT, h_ref)
    print("wide decay D=%d %s: o %.3e, state %.3e" % (D, impl, eo, eh))
    assert eo <= TOL and eh <= TOL, (eo, eh)


@pytest.mark.parametrize("impl", IMPLS)
def test_wide_decay_some_items(cuda_lib, impl):
    """Wide decays in some (chunk, head) items only: one sequence's heads
    decay at up to 30 nats per token, the other sequence and every second
    head of the first stay at the workloads' slow decay, so the tensor-core
    path's exact pass rewrites some records and leaves the others."""
    wl = inputs.small("somewide", [300, 190], H=2, HV=4, K=128, V=128, g_max=0.1, beta_max=2.0, h0_std=0.05,
                      seed=61)
    d = inputs.generate(wl)
    gw = wide_decay_g(wl.T_tot, wl.HV, wl.K, seed=62)
    d["g"][:300, 0::2] = gw[:300, 0::2]
    o, hT, o_ref, h_ref, status = run_both(cuda_lib, d, impl)
    assert status == 0
    eo, eh = rel_max(o, o_ref), rel_max(hT, h_ref)
    print("some wide items %s: o %.3e, state %.3e" % (impl, eo, eh))
    assert eo <= TOL and eh <= TOL, (eo, eh)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("g_max", [6.0, 8.0, 12.0])
def test_decay_across_the_exact_path_threshold(cuda_lib, impl, g_max):
    """g = -U(0, g_max): the decay of a 16-token sub-chunk straddles the
    tensor-core kernel's 63.8-nat switch between the factorised diagonal
    block and the per-pair path, so one chunk mixes channels of both kinds
    (and sub-chunks of both kinds within a channel)."""
    wl = inputs.small("thr%g" % g_max, [256, 100], H=2, HV=2, K=128, V=128, g_max=g_max, beta_max=2.0,
                      h0_std=0.05, seed=53)
    d = inputs.generate(wl)
    o, hT, o_ref, h_ref, status = run_both(cuda_lib, d, impl)
    assert status == 0
    eo, eh = rel_max(o, o_ref), rel_max(hT, h_ref)
    print("g_max %g %s: o %.3e, state %.3e" % (g_max, impl, eo, eh))
    assert eo <= TOL and eh <= TOL, (eo, eh)


def test_wide_decay_fp16_inputs_l2norm(cuda_lib):
    """The tensor-core exact path with fp16 q/k/v, the fused L2 norm (q, k
    given at 3x and 0.25x unit length) and no beta (beta = 1)."""
    wl = inputs.small("wide16", [150, 64], H=2, HV=2, K=128, V=128, g_max=3.0, h0_std=0.05, seed=54)
    d = inputs.generate(wl)
    d["g"] = wide_decay_g(wl.T_tot, wl.HV, wl.K, seed=55, g_max=20.0)
    d["beta"] = None
    d["q"] = (d["q"].float() * 3.0).to(torch.float16)
    d["k"] = (d["k"].float() * 0.25).to(torch.float16)
    d["v"] = d["v"].float().to(torch.float16)
    d["w"] = d["w"].float().to(torch.float16)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], use_qk_l2norm=True)
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    o, hT = cuda_lib.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                    initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], use_qk_l2norm=True,
                                    workspace=ws)
    assert cuda_lib.device_status(ws) == 0
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.float().cpu().numpy(), h_ref) <= TOL


@pytest.mark.parametrize("impl", IMPLS)
def test_large_values_and_state(cuda_lib, impl):
    """g = -U(0,3), v scaled by 1000 and an initial state of std 100: inside
    the fp16 range of the intermediates, so the result matches the oracle and
    the status is OK."""
    wl = inputs.small("big", [300, 77, 64], H=2, HV=2, K=128, V=128, g_max=3.0, beta_max=2.0, h0_std=100.0,
                      seed=56)
    d = inputs.generate(wl)
    d["v"] = (d["v"].float() * 1000.0).to(torch.bfloat16)
    o, hT, o_ref, h_ref, status = run_both(cuda_lib, d, impl)
    assert status == 0
    eo, eh = rel_max(o, o_ref), rel_max(hT, h_ref)
    print("large values %s: o %.3e, state %.3e, max|o| %.3e" % (impl, eo, eh, np.abs(o_ref).max()))
    assert eo <= TOL and eh <= TOL, (eo, eh)


@pytest.mark.parametrize("scale_v,h0_std", [(1.0e6, 0.05), (1.0, 1.0e6)])
def test_out_of_range_is_reported(cuda_lib, scale_v, h0_std):
    """Values (or an initial state) past the fp16 range of the tensor-core
    path's intermediates: the call reports GDN2_ERR_RANGE through the device
    status; the next call on the same workspace with in-range inputs reports
    OK and matches the oracle."""
    wl = inputs.small("huge", [200, 64], H=2, HV=2, K=128, V=128, g_max=0.5, beta_max=1.0, h0_std=h0_std,
                      seed=57)
    d = inputs.generate(wl)
    d["v"] = (d["v"].float() * scale_v).to(torch.bfloat16)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    *_, status = run_both(cuda_lib, d, "tc", ws=ws)
    assert status == ERR_RANGE
    d = inputs.generate(inputs.small("huge_ok", [200, 64], H=2, HV=2, K=128, V=128, g_max=0.5, h0_std=0.05,
                                     seed=58))
    o, hT, o_ref, h_ref, status = run_both(cuda_lib, d, "tc", ws=ws)
    assert status == 0
    assert rel_max(o, o_ref) <= TOL and rel_max(hT, h_ref) <= TOL


def test_wide_decay_recurrent(cuda_lib):
    """The token-by-token call with the same wide decays."""
    wl = inputs.small("rwide", [1, 30, 40], H=2, HV=4, K=128, V=128, beta_max=2.0, h0_std=0.05, seed=59)
    d = inputs.generate(wl)
    d["g"] = wide_decay_g(wl.T_tot, wl.HV, wl.K, seed=60)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    o, hT = cuda_lib.recurrent_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"],
                                        scale=dd["scale"], initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"])
    torch.cuda.synchronize()
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.float().cpu().numpy(), h_ref) <= TOL
