"""The seeded workload generator: shapes, dtypes, ranges and determinism."""
import numpy as np
import torch

from gated_deltanet_prefill_gb300 import inputs


def test_workload_shapes():
    for i in range(1, 6):
        wl = inputs.workload(i)
        assert wl.HV % wl.H == 0 and wl.K in (64, 128) and wl.V in (64, 128)
    assert inputs.workload(1).T_tot == 256
    assert inputs.workload(2).T_tot == 4096
    w3 = inputs.workload(3)
    assert w3.N == 8 and w3.T_tot == 32768 and min(w3.lens) >= 64 and max(w3.lens) <= 8192
    assert inputs.workload(4).T_tot == 32768 and inputs.workload(4).H == 16
    assert inputs.workload(5).T_tot == 4 * 32768


def test_generate_tiny():
    wl = inputs.workload(1)
    a = inputs.generate(wl)
    b = inputs.generate(wl)
    for k in ("q", "k", "v", "g", "beta", "w"):
        assert torch.equal(a[k], b[k]), k
    assert a["q"].dtype == torch.bfloat16 and a["g"].dtype == torch.float32
    assert a["q"].shape == (256, 2, 64) and a["v"].shape == (256, 2, 64)
    n = a["q"].float().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)
    assert float(a["g"].max()) <= 0.0 and float(a["g"].min()) >= -0.1
    assert float(a["beta"].min()) >= 0.0 and float(a["beta"].max()) <= 1.0
    assert a["h0"] is None
    assert a["cu_seqlens"].tolist() == [0, 256]


def test_generate_ranges_and_state():
    wl = inputs.small("x", [30, 70], H=2, HV=4, K=64, V=64, g_max=3.0, beta_max=2.0, h0_std=0.05, seed=7)
    a = inputs.generate(wl)
    assert a["h0"].shape == (2, 4, 64, 64)
    assert abs(float(a["h0"].std()) - 0.05) < 0.005
    assert float(a["beta"].max()) <= 2.0 and float(a["beta"].max()) > 1.0
    assert float(a["g"].min()) >= -3.0
    assert a["cu_seqlens"].tolist() == [0, 30, 100]


def test_varlen_lengths_seeded():
    a = inputs.varlen_lengths(8, 32768, 64, 8192, seed=3)
    b = inputs.varlen_lengths(8, 32768, 64, 8192, seed=3)
    assert a == b and sum(a) == 32768
