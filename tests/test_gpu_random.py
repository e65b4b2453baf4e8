"""A seeded random sweep of the chunked forward against the FP64 oracle:
ragged sequence sets (empty sequences included), D = 64 or 128, grouped value
heads, decays up to 20 nats per token, absent gates, the fused L2 norm,
initial states, fp16 inputs, 16-bit g, bf16 and V-major states, and the state
pass forced sequential or chunk-parallel where the shape allows (a second
draw covers the chunk-parallel pass on sequences of up to 25 chunks with 2 to
8 segments).  Each case is drawn from its own seed
and printed on failure.

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


def draw(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.choice([64, 128]))
    H = int(rng.choice([1, 2]))
    HV = H * int(rng.choice([1, 2]))
    n = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(0, 400, size=n)]
    if rng.random() < 0.3:
        lens[int(rng.integers(0, n))] = 0
    if sum(lens) == 0:
        lens[0] = 1
    case = dict(D=D, H=H, HV=HV, lens=lens, g_max=float(rng.choice([0.05, 0.5, 2.0, 8.0, 20.0])),
                beta_max=float(rng.choice([1.0, 2.0])), h0=bool(rng.random() < 0.6),
                drop=[k for k in ("g", "beta", "w") if rng.random() < 0.15], l2=bool(rng.random() < 0.3),
                qkv=[torch.bfloat16, torch.float16][int(rng.integers(0, 2))],
                gdt=[torch.float32, torch.bfloat16, torch.float16][int(rng.integers(0, 3))],
                sdt=[torch.float32, torch.bfloat16][int(rng.integers(0, 2))], vmajor=bool(rng.random() < 0.3),
                segments=int(rng.choice([0, 1, 3])) if D == 128 else 0)
    return case


def draw_segmented(seed):
    """The chunk-parallel state pass: D = 128, sequences up to 1600 tokens (25
    chunks), segment counts forced to 2 .. 8 or chosen by the library."""
    rng = np.random.default_rng(seed)
    H = int(rng.choice([1, 2]))
    HV = H * int(rng.choice([1, 2]))
    n = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(0, 1600, size=n)]
    if rng.random() < 0.3:
        lens[int(rng.integers(0, n))] = int(rng.integers(0, 70))
    if sum(lens) == 0:
        lens[0] = 1
    return dict(D=128, H=H, HV=HV, lens=lens, g_max=float(rng.choice([0.005, 0.05, 0.5, 2.0, 8.0, 20.0])),
                beta_max=float(rng.choice([1.0, 2.0])), h0=bool(rng.random() < 0.6),
                drop=[k for k in ("g", "beta", "w") if rng.random() < 0.15], l2=bool(rng.random() < 0.3),
                qkv=[torch.bfloat16, torch.float16][int(rng.integers(0, 2))],
                gdt=[torch.float32, torch.bfloat16, torch.float16][int(rng.integers(0, 3))],
                sdt=[torch.float32, torch.bfloat16][int(rng.integers(0, 2))], vmajor=bool(rng.random() < 0.3),
                segments=int(rng.choice([0, 2, 3, 4, 5, 8])))


@pytest.mark.parametrize("seed", list(range(1000, 1020)))
def test_random_case(cuda_lib, seed):
    run_case(cuda_lib, draw(seed), "rand%d" % seed, seed)


@pytest.mark.parametrize("seed", list(range(3000, 3020)))
def test_random_segmented_case(cuda_lib, seed):
    run_case(cuda_lib, draw_segmented(seed), "srand%d" % seed, seed)


def run_case(cuda_lib, c, name, seed):
    wl = inputs.small(name, c["lens"], H=c["H"], HV=c["HV"], K=c["D"], V=c["D"], g_max=c["g_max"],
                      beta_max=c["beta_max"], h0_std=0.05 if c["h0"] else None, seed=seed)
    d = inputs.generate(wl)
    for k in c["drop"]:
        d[k] = None
    for k in ("q", "k", "v", "beta", "w"):
        if d[k] is not None:
            d[k] = d[k].float().to(c["qkv"])
    if d["g"] is not None:
        d["g"] = d["g"].to(c["gdt"])
    if d["h0"] is not None:
        d["h0"] = d["h0"].to(c["sdt"])
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                                       use_qk_l2norm=c["l2"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    h0 = dd["h0"]
    if h0 is not None and c["vmajor"]:
        h0 = h0.transpose(-1, -2).contiguous()
    o, hT = cuda_lib.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                    initial_state=h0, cu_seqlens=dd["cu_seqlens"], use_qk_l2norm=c["l2"],
                                    state_v_major=c["vmajor"], state_dtype=c["sdt"],
                                    state_segments=c["segments"])
    torch.cuda.synchronize()
    hT = hT.float()
    if c["vmajor"]:
        hT = hT.transpose(-1, -2)
    eo = rel_max(o.float().cpu().numpy(), o_ref)
    eh = rel_max(hT.cpu().numpy(), h_ref)
    assert eo <= TOL and eh <= TOL, "case %r: o err %.3e, state err %.3e" % (c, eo, eh)


@pytest.mark.parametrize("seed", list(range(2000, 2008)))
def test_random_case_recurrent(cuda_lib, seed):
    """The same draws through the token-by-token call (short sequences)."""
    c = draw(seed)
    c["lens"] = [min(x, 40) for x in c["lens"]]
    wl = inputs.small("rrand%d" % seed, c["lens"], H=c["H"], HV=c["HV"], K=c["D"], V=c["D"], g_max=c["g_max"],
                      beta_max=c["beta_max"], h0_std=0.05 if c["h0"] else None, seed=seed)
    d = inputs.generate(wl)
    for k in c["drop"]:
        d[k] = None
    for k in ("q", "k", "v", "beta", "w"):
        if d[k] is not None:
            d[k] = d[k].float().to(c["qkv"])
    if d["g"] is not None:
        d["g"] = d["g"].to(c["gdt"])
    if d["h0"] is not None:
        d["h0"] = d["h0"].to(c["sdt"])
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                                       use_qk_l2norm=c["l2"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    h0 = dd["h0"]
    if h0 is not None and c["vmajor"]:
        h0 = h0.transpose(-1, -2).contiguous()
    o, hT = cuda_lib.recurrent_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"],
                                        scale=dd["scale"], initial_state=h0, cu_seqlens=dd["cu_seqlens"],
                                        use_qk_l2norm=c["l2"], state_v_major=c["vmajor"], state_dtype=c["sdt"])
    torch.cuda.synchronize()
    hT = hT.float()
    if c["vmajor"]:
        hT = hT.transpose(-1, -2)
    eo = rel_max(o.float().cpu().numpy(), o_ref) if wl.T_tot else 0.0
    eh = rel_max(hT.cpu().numpy(), h_ref)
    assert eo <= TOL and eh <= TOL, "case %r: o err %.3e, state err %.3e" % (c, eo, eh)
