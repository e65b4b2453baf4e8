"""GPU parity of the token-by-token recurrence (gdn2_recurrent_fwd) against
the FP64 oracle: decode steps, ragged short continuations, a prefill followed
by decode, in-place state updates, the optional gates and the L2 norm.

Bar: max|x - x_ref| / max|x_ref| <= 1e-2 for o and for the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def to_dev(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


def run_oracle(d, **kw):
    return oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                               initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], **kw)


def run_rec(gdn2, d, **kw):
    o, hT = gdn2.recurrent_gdn2_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                    initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o, hT


def check(gdn2, wl, **kw):
    d = inputs.generate(wl)
    o_ref, h_ref = run_oracle(d, use_qk_l2norm=kw.get("use_qk_l2norm", False))
    o, hT = run_rec(gdn2, to_dev(d), **kw)
    eo = rel_max(o.float().cpu().numpy(), o_ref) if wl.T_tot else 0.0
    eh = rel_max(hT.cpu().numpy(), h_ref)
    assert eo <= TOL and eh <= TOL, "%s: o err %.3e, state err %.3e" % (wl.name, eo, eh)


@pytest.mark.parametrize("D", [64, 128])
def test_decode_one_token(cuda_lib, D):
    """One token per sequence from a non-zero state (a decode step)."""
    wl = inputs.small("decode1", [1] * 12, H=2, HV=4, K=D, V=D, g_max=1.0, beta_max=2.0, h0_std=0.05, seed=51)
    check(cuda_lib, wl)


def test_plain_launches_match_chained(cuda_lib, monkeypatch):
    """The step kernel is chained to the check kernel (a programmatic
    dependent launch); GDN2_PDL=0 launches it plainly, with bit-identical
    results."""
    wl = inputs.small("decpdl", [1] * 6 + [9, 40], H=2, HV=4, K=128, V=128, g_max=1.0, beta_max=2.0,
                      h0_std=0.05, seed=53)
    d = to_dev(inputs.generate(wl))
    o1, h1 = run_rec(cuda_lib, d)
    monkeypatch.setenv("GDN2_PDL", "0")
    o0, h0 = run_rec(cuda_lib, d)
    assert torch.equal(o1, o0) and torch.equal(h1, h0)
    check(cuda_lib, wl)


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_continuations(cuda_lib, D):
    """Sequences of 0 .. 70 tokens, grouped value heads, decay stress."""
    wl = inputs.small("cont", [1, 5, 0, 17, 64, 3, 70], H=2, HV=4, K=D, V=D, g_max=3.0, beta_max=2.0,
                      h0_std=0.05, seed=52)
    check(cuda_lib, wl)


def test_missing_gates_and_l2norm(cuda_lib):
    wl = inputs.small("rec_opts", [9, 4], H=1, HV=2, K=128, V=128, h0_std=0.05, seed=53)
    d = inputs.generate(wl)
    d["g"] = d["beta"] = d["w"] = None
    o_ref, h_ref = run_oracle(d)
    o, hT = run_rec(cuda_lib, to_dev(d))
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL
    d = inputs.generate(wl)
    d["q"] = (d["q"].float() * 3.0).to(torch.bfloat16)
    d["k"] = (d["k"].float() * 0.25).to(torch.bfloat16)
    o_ref, h_ref = run_oracle(d, use_qk_l2norm=True)
    o, hT = run_rec(cuda_lib, to_dev(d), use_qk_l2norm=True)
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


def test_in_place_state_and_strided_inputs(cuda_lib):
    """final_state is the initial_state buffer; inputs are strided views."""
    wl = inputs.small("inplace", [3, 8, 1], H=2, HV=2, K=64, V=64, g_max=1.0, h0_std=0.05, seed=54)
    d = inputs.generate(wl)
    o_ref, h_ref = run_oracle(d)
    dd = to_dev(d)
    for key in ("q", "k", "v", "beta", "w", "g"):
        x = dd[key]
        big = torch.zeros(x.shape[0], x.shape[1], 2 * x.shape[2], dtype=x.dtype, device=x.device)
        big[..., :x.shape[2]] = x
        dd[key] = big[..., :x.shape[2]]
    state = dd["h0"].clone()
    o, hT = cuda_lib.recurrent_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"],
                                        scale=dd["scale"], initial_state=state, final_state=state,
                                        cu_seqlens=dd["cu_seqlens"])
    torch.cuda.synchronize()
    assert hT.data_ptr() == state.data_ptr()
    assert rel_max(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_max(state.cpu().numpy(), h_ref) <= TOL


def test_prefill_then_decode_matches_one_pass(cuda_lib):
    """Chunked prefill of the first T - m tokens, then m recurrent steps from
    its final state, equals the oracle over all T tokens (FlashGDN-2 README
    quick start: prefill, then decode)."""
    T, m = 200, 7
    wl = inputs.small("pd", [T], H=2, HV=2, K=128, V=128, g_max=1.0, beta_max=2.0, h0_std=0.05, seed=55)
    d = inputs.generate(wl)
    o_ref, h_ref = run_oracle(d)
    dd = to_dev(d)
    pre = {k: (v[:T - m] if torch.is_tensor(v) and k in ("q", "k", "v", "g", "beta", "w") else v)
           for k, v in dd.items()}
    pre["cu_seqlens"] = torch.tensor([0, T - m], dtype=torch.int32, device="cuda")
    _, h_mid = cuda_lib.chunk_gdn2_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], pre["w"],
                                       scale=pre["scale"], initial_state=pre["h0"],
                                       cu_seqlens=pre["cu_seqlens"])
    dec = {k: (v[T - m:] if torch.is_tensor(v) and k in ("q", "k", "v", "g", "beta", "w") else v)
           for k, v in dd.items()}
    dec["cu_seqlens"] = torch.tensor([0, m], dtype=torch.int32, device="cuda")
    dec["h0"] = h_mid
    o, hT = run_rec(cuda_lib, dec)
    assert rel_max(o.float().cpu().numpy(), o_ref[T - m:]) <= TOL
    assert rel_max(hT.cpu().numpy(), h_ref) <= TOL


def test_bad_cu_seqlens_is_a_no_op(cuda_lib):
    wl = inputs.small("badcu", [4, 4], H=1, HV=1, K=64, V=64, h0_std=0.05, seed=56)
    d = to_dev(inputs.generate(wl))
    d["cu_seqlens"] = torch.tensor([0, 6, 5], dtype=torch.int32, device="cuda")  # decreasing
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = torch.full((wl.T_tot, 1, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    cuda_lib.recurrent_gdn2_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], out=out, workspace=ws)
    assert cuda_lib.device_status(ws) == 9  # GDN2_ERR_CU_SEQLENS
    assert float(out.float().sub(7.0).abs().max()) == 0.0


def test_decode_batch_full_size_sampled(cuda_lib):
    """The decode benchmark's shape (128 sequences x 1 token, H = HV = 32,
    D = 128) on sampled (sequence, value head) units."""
    wl = inputs.decode_workload()
    d = inputs.generate(wl)
    o, hT = run_rec(cuda_lib, to_dev(d))
    rng = np.random.default_rng(7)
    flat = sorted(int(x) for x in rng.choice(wl.N * wl.HV, size=64, replace=False))
    units = [divmod(u, wl.HV) for u in flat]  # (sequence, value head)
    o_ref, h_ref = run_oracle(d, units=units)
    o = o.float().cpu().numpy()
    hT = hT.cpu().numpy()
    cu = d["cu_seqlens"].numpy()
    for n, hv in units:
        a, b = cu[n], cu[n + 1]
        assert rel_max(o[a:b, hv], o_ref[a:b, hv]) <= TOL
        assert rel_max(hT[n, hv], h_ref[n, hv]) <= TOL
