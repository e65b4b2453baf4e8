"""Seeded synthetic inputs for the GDN-2 prefill forward.

This module holds the workload recipes only: shapes, value distributions,
sequence-length mixes and seeds.  It contains none of the operator's
arithmetic and imports neither the CUDA library nor the oracle, so both sides
of every parity check consume the same bytes from here.

Recipe (FlashGDN-2 README quick start, which draws q, k ~ N(0, 1),
row-L2-normalises them in fp32 and casts to bf16, v ~ N(0, 1), a log-decay
g = -U(0, a) in fp32, and gates beta, w ~ U(0, 1)):

* q, k   [T_tot, H, K]  bf16, N(0,1) rows normalised in fp32 before the cast
* v      [T_tot, HV, V] bf16, N(0,1)
* g      [T_tot, HV, K] fp32, -g_max * U(0,1)
* beta   [T_tot, HV, K] bf16, beta_max * U(0,1)   (beta_max = 2 gives the
  negative-eigenvalue range of burn-gdn2's allow_neg_eigval)
* w      [T_tot, HV, V] bf16, U(0,1)
* h0     [N, HV, K, V]  fp32, N(0, h0_std^2) or absent
* cu_seqlens [N + 1] int32

Fixed-length batches are passed packed with cu_seqlens = [0, T, 2T, ...]
(the FlashInfer docs accept only packed input).  Draw order is q, k, v, g,
beta, w, h0 from one torch.Generator seeded per workload; on a CUDA device the
generator is a CUDA one (same recipe, different stream of numbers).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import List, Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    lens: tuple            # per-sequence token counts
    H: int
    HV: int
    K: int
    V: int
    g_max: float = 0.1     # g = -g_max * U(0,1)
    beta_max: float = 1.0  # beta = beta_max * U(0,1)
    h0_std: Optional[float] = None
    output_final_state: bool = True
    seed: int = 0
    scale: Optional[float] = None  # None -> 1/sqrt(K)
    use_qk_l2norm: bool = False
    description: str = ""

    @property
    def N(self) -> int:
        return len(self.lens)

    @property
    def T_tot(self) -> int:
        return int(sum(self.lens))

    def cu_seqlens(self) -> List[int]:
        return [0] + list(np.cumsum(self.lens).astype(int).tolist())


def varlen_lengths(n: int, total: int, lo: int, hi: int, seed: int) -> tuple:
    """n seeded lengths in [lo, hi] summing to ``total``: n-1 sorted integer
    cut points drawn uniformly in (0, total), redrawn until every gap lies in
    [lo, hi]."""
    rng = np.random.default_rng(seed)
    for _ in range(100000):
        cuts = np.sort(rng.integers(1, total, size=n - 1))
        lens = np.diff(np.concatenate([[0], cuts, [total]]))
        if lens.min() >= lo and lens.max() <= hi:
            return tuple(int(x) for x in lens)
    raise RuntimeError("no admissible length draw")


def workload(index: int) -> Workload:
    """The five benchmark workloads, 1-based."""
    if index == 1:
        return Workload("tiny_T256_H2_D64", (256,), 2, 2, 64, 64, g_max=0.1, seed=0,
                        scale=1.0 / 8.0, output_final_state=True,
                        description="B=1 T=256 H=HV=2 K=V=64, zero initial state")
    if index == 2:
        return Workload("fixed_T4096_H16_D128", (4096,), 16, 16, 128, 128, g_max=0.1, seed=2,
                        description="B=1 T=4096 H=HV=16 K=V=128, zero initial state")
    if index == 3:
        return Workload("varlen8_T32768_H32_D128", varlen_lengths(8, 32768, 64, 8192, seed=3),
                        32, 32, 128, 128, g_max=0.5, h0_std=0.05, seed=3,
                        description="8 packed sequences, lengths in [64,8192] summing to 32768, "
                                    "H=HV=32 K=V=128, initial state N(0,0.05)")
    if index == 4:
        return Workload("gva_B2_T16384_H16_HV32_D128", (16384, 16384), 16, 32, 128, 128,
                        g_max=0.1, seed=4, output_final_state=False,
                        description="B=2 T=16384, q/k heads H=16 shared by HV=32 value heads, "
                                    "K=V=128, zero initial state")
    if index == 5:
        return Workload("long_B4_T32768_H32_D128", (32768,) * 4, 32, 32, 128, 128, g_max=3.0,
                        beta_max=2.0, h0_std=0.05, seed=5,
                        description="B=4 T=32768 H=HV=32 K=V=128, g=-U(0,3), beta=U(0,2), "
                                    "initial state N(0,0.05)")
    raise ValueError(index)


def decode_workload(batch: int = 128, tokens: int = 1) -> Workload:
    """Decode steps from a carried state: ``batch`` sequences of ``tokens``
    tokens each, H = HV = 32, K = V = 128, initial state N(0, 0.05)."""
    return Workload("decode_B%d_T%d_H32_D128" % (batch, tokens), (tokens,) * batch, 32, 32, 128, 128,
                    g_max=0.5, beta_max=2.0, h0_std=0.05, seed=6,
                    description="%d sequences x %d token(s) from a carried state N(0,0.05), "
                                "H=HV=32 K=V=128, g=-U(0,0.5), beta=U(0,2)" % (batch, tokens))


def small(name: str, lens, H=2, HV=2, K=64, V=64, **kw) -> Workload:
    """A small ad-hoc workload for parity and edge-case tests."""
    return Workload(name, tuple(int(x) for x in lens), H, HV, K, V, **kw)


def generate(wl: Workload, device="cpu", cu_dtype=torch.int32) -> dict:
    """Draw one workload's inputs.  Returns a dict of tensors on ``device``:
    q, k, v, g, beta, w, h0 (or None), cu_seqlens, plus ``scale``."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(wl.seed))
    T, H, HV, K, V = wl.T_tot, wl.H, wl.HV, wl.K, wl.V

    def unit_rows(shape):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(torch.bfloat16)

    q = unit_rows((T, H, K))
    k = unit_rows((T, H, K))
    v = torch.randn((T, HV, V), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    g = torch.rand((T, HV, K), generator=gen, device=dev, dtype=torch.float32).mul_(-wl.g_max)
    beta = torch.rand((T, HV, K), generator=gen, device=dev, dtype=torch.float32).mul_(
        wl.beta_max).to(torch.bfloat16)
    w = torch.rand((T, HV, V), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    h0 = None
    if wl.h0_std is not None:
        h0 = torch.randn((wl.N, HV, K, V), generator=gen, device=dev,
                         dtype=torch.float32).mul_(wl.h0_std)
    cu = torch.tensor(wl.cu_seqlens(), dtype=cu_dtype, device=dev)
    scale = wl.scale if wl.scale is not None else 1.0 / float(K) ** 0.5
    return dict(q=q, k=k, v=v, g=g, beta=beta, w=w, h0=h0, cu_seqlens=cu, scale=scale)


def with_seed(wl: Workload, seed: int) -> Workload:
    return replace(wl, seed=seed)
