"""The checked build: the library compiled with the device-side index checks
(-DGDN2_CHECK_BOUNDS; build.py's libgdn2_checked.so).  Each check guards an
index read from the device-built chunk map, the exact list or the sequence
order before it addresses a record, a chunk or a sequence; a failure is
recorded in the status and reported as GDN2_ERR_BOUNDS.  These cases run
every kernel of both chunked paths and the recurrent call through the
checked library; the status must be OK and the results must match the FP64
oracle.  The checks stand in for a sanitizer, which this GPU pool does not
offer.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import build as gbuild
from gated_deltanet_prefill_gb300 import gdn2, inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def checked():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = gdn2.load(gbuild.build(checked=True))
    saved = gdn2._lib
    gdn2._lib = lib
    yield gdn2
    gdn2._lib = saved


def rel_max(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(x).all()
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


def run(g, d, fn="chunk", **kw):
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    call = g.chunk_gdn2_fwd if fn == "chunk" else g.recurrent_gdn2_fwd
    o, hT = call(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                 initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], workspace=ws, **kw)
    status = g.device_status(ws)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    return status, rel_max(o.float().cpu().numpy(), o_ref), rel_max(hT.float().cpu().numpy(), h_ref)


def test_the_checked_library_is_loaded(checked):
    assert checked._lib._name.endswith("libgdn2_checked.so")


CASES = {
    # name: (lens, H, HV, D, g_max, call kwargs)
    "ragged_gva_128": ([1, 63, 64, 65, 0, 200, 130], 2, 4, 128, 0.5, {}),
    "ragged_64": ([1, 70, 129, 0, 33], 2, 2, 64, 0.5, {}),
    "simt": ([1, 63, 200, 130], 2, 4, 128, 0.5, {"impl": "simt"}),
    "segments": ([900, 333, 64, 0], 2, 2, 128, 0.1, {"state_segments": 3}),
    "vt64_lookahead": ([0, 1, 64, 65, 129, 192, 200, 900], 2, 4, 128, 2.0, {"state_segments": 1}),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_checked_build_cases(checked, name):
    lens, H, HV, D, g_max, kw = CASES[name]
    wl = inputs.small("chk_" + name, lens, H=H, HV=HV, K=D, V=D, g_max=g_max, beta_max=2.0, h0_std=0.05, seed=91)
    status, eo, eh = run(checked, inputs.generate(wl), **kw)
    assert status == 0, "status %d (%s)" % (status, gdn2.STATUS_NAMES.get(status))
    assert eo <= TOL and eh <= TOL, (eo, eh)


def test_checked_build_vt128_and_exact_pass(checked):
    """128-column lookahead tiles (more (sequence, head) pairs than half the
    SMs) with decays to 30 nats per token, so the intra kernel's exact pass
    reads its list."""
    lens = [65, 200, 129, 64, 300, 1, 90, 77, 150, 33]
    wl = inputs.small("chk_wide", lens, H=4, HV=8, K=128, V=128, beta_max=2.0, h0_std=0.05, seed=92)
    d = inputs.generate(wl)
    gen = torch.Generator().manual_seed(93)
    d["g"] = torch.rand(d["g"].shape, generator=gen).mul_(-30.0)
    status, eo, eh = run(checked, d, state_segments=1)
    assert status == 0
    assert eo <= TOL and eh <= TOL, (eo, eh)


def test_checked_build_recurrent(checked):
    wl = inputs.small("chk_rec", [1, 20, 0, 33], H=2, HV=4, K=128, V=128, g_max=1.0, beta_max=2.0, h0_std=0.05,
                      seed=94)
    status, eo, eh = run(checked, inputs.generate(wl), fn="recurrent")
    assert status == 0
    assert eo <= TOL and eh <= TOL, (eo, eh)
