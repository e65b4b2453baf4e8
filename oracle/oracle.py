"""FP64 CPU oracle for the GDN-2 prefill forward: Python side.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this module.  The product
package never imports it and has no CPU fallback.

The arithmetic lives in ``gdn2_oracle.c`` (plain C, double precision, the
token-by-token recurrence of the FlashInfer docs page
"flashinfer.gdn2_prefill.chunk_gated_delta_rule2", op description).  This file
only builds that C file with gcc, converts inputs exactly to float64 and calls
it through ctypes.  Conversions bf16/fp32 -> fp64 are exact, so the oracle sees
the same values the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn2_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn2_oracle.so")
_lib = None
_lock = threading.Lock()


def compile_c(src: str, out: str) -> str:
    """gcc the oracle source ``src`` into the shared library ``out``.
    Portable flags only (x86_64 and aarch64 hosts); FP contraction is off so
    both hosts round identically."""
    tmp = out + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` (skipped when up to date)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_c(_SRC, _LIB_PATH)


def load_library(path: str):
    """Open a compiled oracle library and declare its one entry point."""
    lib = ctypes.CDLL(path)
    f = lib.gdn2_oracle_forward
    dp = ctypes.c_void_p
    f.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_double, dp, dp,
                  ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, ctypes.c_int,
                  dp, dp, ctypes.c_int]
    f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f64(x):
    """Exact conversion of a numpy array or a (CPU) torch tensor to a
    contiguous float64 numpy array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen in torch, bf16 -> fp64 is exact
        x = x.detach().cpu().double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def gdn2_forward(q, k, v, g=None, beta=None, w=None, scale=None, initial_state=None,
                 cu_seqlens=None, use_qk_l2norm=False, units=None, threads=None, lib=None):
    """Run the oracle.

    q: [T, H, K]; k: [T, HK, K]; v: [T, HV, V]; with HS = max(H, HV) state
    heads: g, beta [T, HS, K]; w [T, HS, V]; initial_state [N, HS, K, V];
    cu_seqlens [N + 1].  HK equals H or HV, and H, HV are equal or one a
    multiple of the other.  A leading batch dim of size B on q..w
    (fixed-length [B, T, ...] input) is folded into T when cu_seqlens is
    None.  ``units`` is an optional list of (n, hs) pairs to compute; rows of
    other units in the returned ``o`` are NaN and their final states NaN.
    ``lib`` selects another compiled copy of the oracle (see load_library).

    Returns (o [T, HS, V], final_state [N, HS, K, V]) as float64 arrays.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    g, beta, w, h0 = _f64(g), _f64(beta), _f64(w), _f64(initial_state)
    if q.ndim == 4:  # [B, T, H, K] fixed-length batch
        B, T = q.shape[:2]
        if cu_seqlens is None:
            cu_seqlens = np.arange(B + 1, dtype=np.int64) * T
        q, k, v = (x.reshape(B * T, *x.shape[2:]) for x in (q, k, v))
        g, beta, w = (None if x is None else x.reshape(B * T, *x.shape[2:]) for x in (g, beta, w))
    if cu_seqlens is None:
        cu_seqlens = [0, q.shape[0]]
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    T_tot, H, K = q.shape
    HK = k.shape[1]
    HV, V = v.shape[1], v.shape[2]
    HS = max(H, HV)
    N = cu.shape[0] - 1
    assert k.shape == (T_tot, HK, K) and v.shape == (T_tot, HV, V)
    for x, shp in ((g, (T_tot, HS, K)), (beta, (T_tot, HS, K)), (w, (T_tot, HS, V)),
                   (h0, (N, HS, K, V))):
        assert x is None or x.shape == shp, (None if x is None else x.shape, shp)
    o = np.full((T_tot, HS, V), np.nan)
    hT = np.full((N, HS, K, V), np.nan)
    if units is not None:
        u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        n_units = u.shape[0]
    else:
        u, n_units = None, N * HS
    if threads is None:
        threads = max(1, min(os.cpu_count() or 1, n_units))
    rc = (lib or _load()).gdn2_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w),
        0.0 if scale is None else float(scale), _ptr(h0), _ptr(cu),
        T_tot, N, H, HK, HV, K, V, int(bool(use_qk_l2norm)), _ptr(u), n_units,
        _ptr(o), _ptr(hT), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (code %d)" % rc)
    return o, hT
