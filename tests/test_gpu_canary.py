"""Memory-safety checks without a sanitizer: every buffer the library is
given sits inside a larger allocation filled with a canary byte pattern.
After the call, the bytes around the outputs and the workspace, and every
byte of the inputs, must be unchanged: the kernels write only inside the
outputs and the workspace they were given, and never write their inputs.
The outputs themselves are checked against the FP64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import gdn2, inputs

pytestmark = pytest.mark.gpu
PAD = 4096  # bytes of canary on each side (a multiple of 256: payloads stay aligned)
CANARY = 0xA5


class Padded:
    """A device tensor of `shape`/`dtype` inside a canary-filled byte buffer."""

    def __init__(self, shape, dtype, fill=None):
        es = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) if shape else 1
        self.nbytes = n * es
        self.raw = torch.full((PAD + self.nbytes + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[PAD:PAD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def pads_intact(self):
        return bool((self.raw[:PAD] == CANARY).all()) and bool((self.raw[PAD + self.nbytes:] == CANARY).all())


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all()
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.mark.parametrize("impl,D", [("tc", 128), ("tc", 64), ("simt", 128), ("recurrent", 128)])
def test_writes_stay_inside_outputs_and_workspace(cuda_lib, impl, D):
    lens = [1, 63, 200, 0, 129] if impl != "recurrent" else [1, 17, 0, 40]
    wl = inputs.small("canary_%s_%d" % (impl, D), lens, H=2, HV=4, K=D, V=D, g_max=1.0, beta_max=2.0,
                      h0_std=0.05, seed=81)
    d = inputs.generate(wl)
    ins = {k: Padded(tuple(v.shape), v.dtype, v.cuda()) for k, v in d.items() if torch.is_tensor(v)}
    before = {k: p.raw.clone() for k, p in ins.items()}
    out = Padded((wl.T_tot, wl.HV, wl.V), torch.bfloat16)
    fs = Padded((wl.N, wl.HV, wl.K, wl.V), torch.float32)
    args = [ins[k].t for k in ("q", "k", "v", "g", "beta", "w")]
    if impl == "recurrent":
        ws = Padded((64,), torch.uint8)
        cuda_lib.recurrent_gdn2_fwd(*args, scale=d["scale"], initial_state=ins["h0"].t,
                                    cu_seqlens=ins["cu_seqlens"].t, out=out.t, final_state=fs.t, workspace=ws.t)
    else:
        dims = gdn2.make_dims(*args, out.t, ins["cu_seqlens"].t, False, impl)
        ws = Padded((gdn2.workspace_bytes(dims),), torch.uint8)
        cuda_lib.chunk_gdn2_fwd(*args, scale=d["scale"], initial_state=ins["h0"].t, cu_seqlens=ins["cu_seqlens"].t,
                                out=out.t, final_state=fs.t, workspace=ws.t, impl=impl)
    torch.cuda.synchronize()
    assert cuda_lib.device_status(ws.t) == 0
    for k, p in ins.items():
        assert torch.equal(p.raw, before[k]), "input %s was written" % k
    for name, p in (("out", out), ("final_state", fs), ("workspace", ws)):
        assert p.pads_intact(), "a write landed outside %s" % name
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    assert rel_max(out.t.float().cpu().numpy(), o_ref) <= 1e-2
    assert rel_max(fs.t.cpu().numpy(), h_ref) <= 1e-2


def test_chunk_parallel_writes_stay_inside(cuda_lib):
    """The same check for the chunk-parallel state pass (transitions with
    their M operand images, the tensor-core combine, the replay), 4
    segments."""
    wl = inputs.small("canary_scan", [900, 1, 700], H=2, HV=2, K=128, V=128, g_max=0.3, beta_max=2.0,
                      h0_std=0.05, seed=84)
    d = inputs.generate(wl)
    ins = {k: Padded(tuple(v.shape), v.dtype, v.cuda()) for k, v in d.items() if torch.is_tensor(v)}
    before = {k: p.raw.clone() for k, p in ins.items()}
    out = Padded((wl.T_tot, wl.HV, wl.V), torch.bfloat16)
    fs = Padded((wl.N, wl.HV, wl.K, wl.V), torch.float32)
    args = [ins[k].t for k in ("q", "k", "v", "g", "beta", "w")]
    dims = gdn2.make_dims(*args, out.t, ins["cu_seqlens"].t)
    dims.state_segments = 4
    ws = Padded((gdn2.workspace_bytes(dims),), torch.uint8)
    cuda_lib.chunk_gdn2_fwd(*args, scale=d["scale"], initial_state=ins["h0"].t, cu_seqlens=ins["cu_seqlens"].t,
                            out=out.t, final_state=fs.t, workspace=ws.t, state_segments=4)
    torch.cuda.synchronize()
    assert cuda_lib.device_status(ws.t) == 0
    for k, p in ins.items():
        assert torch.equal(p.raw, before[k]), "input %s was written" % k
    for name, p in (("out", out), ("final_state", fs), ("workspace", ws)):
        assert p.pads_intact(), "a write landed outside %s" % name
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    assert rel_max(out.t.float().cpu().numpy(), o_ref) <= 1e-2
    assert rel_max(fs.t.cpu().numpy(), h_ref) <= 1e-2


def test_exact_pass_writes_stay_inside(cuda_lib):
    """The same check with decays of up to 30 nats per token, so that the
    intra kernel's exact pass rewrites records."""
    wl = inputs.small("canary_wide", [70, 130], H=1, HV=2, K=128, V=128, beta_max=2.0, h0_std=0.05, seed=82)
    d = inputs.generate(wl)
    gen = torch.Generator().manual_seed(83)
    d["g"] = torch.rand(d["g"].shape, generator=gen).mul_(-30.0)
    ins = {k: Padded(tuple(v.shape), v.dtype, v.cuda()) for k, v in d.items() if torch.is_tensor(v)}
    out = Padded((wl.T_tot, wl.HV, wl.V), torch.bfloat16)
    fs = Padded((wl.N, wl.HV, wl.K, wl.V), torch.float32)
    args = [ins[k].t for k in ("q", "k", "v", "g", "beta", "w")]
    dims = gdn2.make_dims(*args, out.t, ins["cu_seqlens"].t)
    ws = Padded((gdn2.workspace_bytes(dims),), torch.uint8)
    cuda_lib.chunk_gdn2_fwd(*args, scale=d["scale"], initial_state=ins["h0"].t, cu_seqlens=ins["cu_seqlens"].t,
                            out=out.t, final_state=fs.t, workspace=ws.t)
    torch.cuda.synchronize()
    assert cuda_lib.device_status(ws.t) == 0
    for name, p in (("out", out), ("final_state", fs), ("workspace", ws)):
        assert p.pads_intact(), "a write landed outside %s" % name
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    assert rel_max(out.t.float().cpu().numpy(), o_ref) <= 1e-2
    assert rel_max(fs.t.cpu().numpy(), h_ref) <= 1e-2
