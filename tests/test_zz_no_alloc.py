"""The allocation-free entry point, gdn2_chunk_fwd_noalloc.

It serves callers that cannot allocate device memory: it takes no workspace
and runs on a fixed device array inside the library.  These tests call it
through the C ABI (the binding is a ctypes pass-through) and compare its
results with gdn2_chunk_fwd on the same inputs and with the FP64 oracle.  The
file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_prefill_gb300 import build as gbuild
from gated_deltanet_prefill_gb300 import gdn2, inputs

TOL = 1e-2  # same bound as the parity tests


def _rel(x, ref):
    x = x.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(x).all()
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def test_limit_is_checked_before_the_device():
    """A problem whose workspace exceeds the fixed scratch is refused with
    GDN2_ERR_NOALLOC_LIMIT before any CUDA call (runs without a GPU)."""
    gbuild.build()
    lib = gdn2.load()
    big = gdn2.Dims()
    assert lib.gdn2_dims_init(ctypes.byref(big), 1 << 20, 1, 32, 32, 128, 128) == 0
    assert lib.gdn2_workspace_bytes(ctypes.byref(big)) > gdn2.NOALLOC_SCRATCH_BYTES
    fake = 1 << 40
    st = lib.gdn2_chunk_fwd_noalloc(fake, fake, fake, None, None, None, ctypes.c_float(0.0), None, fake,
                                    fake + (1 << 36), None, ctypes.byref(big), None)
    assert st == 13
    # the sizes the header quotes fit
    for T, N, H, HV, D in ((2048, 1, 16, 16, 128), (256, 1, 2, 2, 64)):
        d = gdn2.Dims()
        assert lib.gdn2_dims_init(ctypes.byref(d), T, N, H, HV, D, D) == 0
        assert 0 < lib.gdn2_workspace_bytes(ctypes.byref(d)) <= gdn2.NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point(cuda_lib):
    """Two calls in a row (different problems, so a stale scratch would show)
    match gdn2_chunk_fwd with a caller-allocated workspace and the FP64
    oracle, and the device-side status of each call (read back through
    gdn2_noalloc_device_status, since the caller holds no workspace) is OK."""
    import oracle

    cases = [
        inputs.small("noalloc_a", [100, 64, 37], H=2, HV=4, K=128, V=128, g_max=0.5, beta_max=2.0,
                     h0_std=0.05, seed=41),
        inputs.small("noalloc_b", [300, 5], H=1, HV=2, K=64, V=64, g_max=3.0, beta_max=2.0, seed=42),
    ]
    for wl in cases:
        host = inputs.generate(wl)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in host.items()}
        args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"])
        kw = dict(scale=d["scale"], initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
        o_ref, h_ref = cuda_lib.chunk_gdn2_fwd(*args, **kw)
        o, h = cuda_lib.chunk_gdn2_fwd_noalloc(*args, **kw)
        assert cuda_lib.noalloc_device_status() == 0, wl.name
        torch.cuda.synchronize()
        eo, eh = _rel(o, o_ref), _rel(h, h_ref)
        assert eo <= TOL and eh <= TOL, (wl.name, eo, eh)
        oo, ho = oracle.gdn2_forward(host["q"], host["k"], host["v"], host["g"], host["beta"], host["w"],
                                     scale=host["scale"], initial_state=host["h0"],
                                     cu_seqlens=host["cu_seqlens"])
        eo = float(np.abs(o.float().cpu().numpy() - oo).max() / np.abs(oo).max())
        eh = float(np.abs(h.float().cpu().numpy() - ho).max() / np.abs(ho).max())
        assert eo <= TOL and eh <= TOL, (wl.name, "oracle", eo, eh)


@pytest.mark.gpu
def test_noalloc_reports_bad_cu_seqlens(cuda_lib):
    """A decreasing cu_seqlens is found on the device; the caller of the
    allocation-free entry point reads it with gdn2_noalloc_device_status, and
    the next good call clears it."""
    wl = inputs.small("noalloc_bad", [64, 64], H=1, HV=1, K=64, V=64, seed=43)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inputs.generate(wl).items()}
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"])
    bad = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")
    cuda_lib.chunk_gdn2_fwd_noalloc(*args, scale=d["scale"], cu_seqlens=bad)
    assert cuda_lib.noalloc_device_status() == 9
    cuda_lib.chunk_gdn2_fwd_noalloc(*args, scale=d["scale"], cu_seqlens=d["cu_seqlens"])
    assert cuda_lib.noalloc_device_status() == 0
