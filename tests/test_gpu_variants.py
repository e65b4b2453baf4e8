"""GPU parity of the interface variants the FlashInfer docs list for
chunk_gated_delta_rule2: fp16 q/k/v (beta, w and the output at q's dtype),
g in bf16 or fp16, states in bf16 and in the V-major [N, HV, V, K] layout.
Both the chunked prefill (tensor-core path) and the recurrent call are
checked against the FP64 oracle on the same (converted) input values.

Bar: max|x - x_ref| / max|x_ref| <= 1e-2 for o and for the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
CALLS = ["chunk", "recurrent"]


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all(), "non-finite output"
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def variant(d, qkv=None, g=None, state=None):
    """Cast the inputs: qkv dtype for q, k, v, beta, w; g dtype; state dtype."""
    d = dict(d)
    if qkv is not None:
        for key in ("q", "k", "v", "beta", "w"):
            if d[key] is not None:
                d[key] = d[key].float().to(qkv)
    if g is not None and d["g"] is not None:
        d["g"] = d["g"].to(g)
    if state is not None and d["h0"] is not None:
        d["h0"] = d["h0"].to(state)
    return d


def run(gdn2, call, d, v_major=False, state_dtype=None):
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    h0 = dd["h0"]
    if h0 is not None and v_major:
        h0 = h0.transpose(-1, -2).contiguous()
    fn = gdn2.chunk_gdn2_fwd if call == "chunk" else gdn2.recurrent_gdn2_fwd
    o, hT = fn(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"], initial_state=h0,
               cu_seqlens=dd["cu_seqlens"], state_v_major=v_major, state_dtype=state_dtype)
    torch.cuda.synchronize()
    hT = hT.float()
    if v_major:
        hT = hT.transpose(-1, -2)
    return o, hT


def check(gdn2, call, wl, qkv=None, g=None, state=None, v_major=False):
    d = variant(inputs.generate(wl), qkv, g, state)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    o, hT = run(gdn2, call, d, v_major, state)
    assert o.dtype == (qkv or torch.bfloat16)
    eo = rel_max(o.float().cpu().numpy(), o_ref)
    eh = rel_max(hT.cpu().numpy(), h_ref)
    assert eo <= TOL and eh <= TOL, "%s/%s: o err %.3e, state err %.3e" % (wl.name, call, eo, eh)


def ragged(D, seed, g_max=1.0):
    return inputs.small("var%d" % D, [1, 63, 65, 130, 7], H=2, HV=4, K=D, V=D, g_max=g_max, beta_max=2.0,
                        h0_std=0.05, seed=seed)


@pytest.mark.parametrize("call", CALLS)
@pytest.mark.parametrize("D", [64, 128])
def test_fp16_inputs(cuda_lib, call, D):
    check(cuda_lib, call, ragged(D, 61), qkv=torch.float16)


@pytest.mark.parametrize("call", CALLS)
@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128])
def test_16bit_g(cuda_lib, call, gdt, D):
    """g rounded to 16 bits (both sides see the same values), decay stress."""
    check(cuda_lib, call, ragged(D, 62, g_max=3.0), g=gdt)


@pytest.mark.parametrize("call", CALLS)
@pytest.mark.parametrize("state,v_major", [(torch.bfloat16, False), (torch.float32, True), (torch.bfloat16, True)])
def test_state_layouts(cuda_lib, call, state, v_major):
    check(cuda_lib, call, ragged(128, 63), state=state, v_major=v_major)


@pytest.mark.parametrize("call", CALLS)
def test_all_variants_together(cuda_lib, call):
    check(cuda_lib, call, ragged(128, 64, g_max=2.0), qkv=torch.float16, g=torch.float16, state=torch.bfloat16,
          v_major=True)


def test_16bit_g_row_copies(cuda_lib, monkeypatch):
    """The intra kernel's row-by-row copies (no tensor maps) with 16-bit g."""
    monkeypatch.setenv("GDN2_ROW_COPIES", "1")
    check(cuda_lib, "chunk", ragged(128, 65, g_max=2.0), g=torch.bfloat16)
    check(cuda_lib, "chunk", ragged(64, 66, g_max=2.0), qkv=torch.float16, g=torch.float16)
