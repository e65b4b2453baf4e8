"""Device-side failure detection, exercised without a GPU fault.  Every wait
in the tensor-core kernels is bounded in wall time; the self-test kernel
makes one such wait run out on a barrier that nothing completes (1 ms limit).
The kernel records GDN2_ERR_TIMEOUT in the workspace status word and returns:
the host reads the error, and the CUDA context stays usable for a forward
that still matches the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_prefill_gb300 import inputs

pytestmark = pytest.mark.gpu
TIMEOUT = 12  # GDN2_ERR_TIMEOUT


def test_wait_timeout_is_reported_and_context_survives(cuda_lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert cuda_lib.selftest_wait_timeout(ws, limit_ns=1_000_000) == 0
    assert cuda_lib.device_status(ws) == TIMEOUT
    assert cuda_lib.selftest_wait_timeout(ws, limit_ns=1_000_000) == 0  # repeatable
    assert cuda_lib.device_status(ws) == TIMEOUT
    wl = inputs.small("after_timeout", [100, 37], H=2, HV=2, K=128, V=128, g_max=1.0, h0_std=0.05, seed=97)
    d = inputs.generate(wl)
    o_ref, h_ref = oracle.gdn2_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                       initial_state=d["h0"], cu_seqlens=d["cu_seqlens"])
    dd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}
    dims = cuda_lib.make_dims(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], dd["v"], dd["cu_seqlens"])
    ws2 = torch.empty(cuda_lib.workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    o, hT = cuda_lib.chunk_gdn2_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["w"], scale=dd["scale"],
                                    initial_state=dd["h0"], cu_seqlens=dd["cu_seqlens"], workspace=ws2)
    torch.cuda.synchronize()
    assert cuda_lib.device_status(ws2) == 0
    err_o = np.abs(o.float().cpu().numpy() - o_ref).max() / np.abs(o_ref).max()
    err_h = np.abs(hT.cpu().numpy() - h_ref).max() / np.abs(h_ref).max()
    assert err_o <= 1e-2 and err_h <= 1e-2
