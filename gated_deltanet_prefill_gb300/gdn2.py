"""ctypes binding of ``libgdn2.so`` (include/gdn2.h), argument marshalling only.

Every step of the forward runs in the library's CUDA kernels; this module
fills the ``gdn2_dims`` struct from torch tensors, allocates outputs and the
workspace with torch when the caller does not pass them (the library itself
never allocates), and passes raw device pointers and the current CUDA stream.
There is no CPU path: a missing library or a non-CUDA tensor is an error.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

GDN2_OK = 0
STATUS_NAMES = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_STRIDE", 4: "ERR_ALIAS",
                5: "ERR_WORKSPACE", 6: "ERR_ARCH", 7: "ERR_LAUNCH", 8: "ERR_DTYPE",
                9: "ERR_CU_SEQLENS", 10: "ERR_CUDA", 11: "ERR_IMPL", 12: "ERR_TIMEOUT",
                13: "ERR_NOALLOC_LIMIT", 14: "ERR_RANGE", 15: "ERR_BOUNDS"}
NOALLOC_SCRATCH_BYTES = 64 << 20
IMPL = {"tc": 0, "simt": 1}
DTYPE_BF16, DTYPE_F16, DTYPE_F32 = 0, 1, 2
_DTYPE_CODE = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16, torch.float32: DTYPE_F32}

EXPORTS = ("gdn2_workspace_bytes", "gdn2_dims_init", "gdn2_check_args", "gdn2_chunk_fwd",
           "gdn2_chunk_fwd_staged", "gdn2_num_stages", "gdn2_stage_name", "gdn2_launch_count",
           "gdn2_launch_plan",
           "gdn2_device_status", "gdn2_chunk_fwd_noalloc", "gdn2_noalloc_device_status",
           "gdn2_recurrent_workspace_bytes",
           "gdn2_recurrent_fwd", "gdn2_selftest_wait_timeout", "gdn2_status_string", "gdn2_version")


class Gdn2Error(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = "%s: %s (%s)" % (where or "gdn2", STATUS_NAMES.get(status, status), status_string(status))
        super().__init__(msg)


class Dims(ctypes.Structure):
    _fields_ = [("T_tot", ctypes.c_int64), ("N", ctypes.c_int32), ("H", ctypes.c_int32),
                ("HV", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
                ("q_stride", ctypes.c_int64 * 2), ("k_stride", ctypes.c_int64 * 2),
                ("v_stride", ctypes.c_int64 * 2), ("g_stride", ctypes.c_int64 * 2),
                ("beta_stride", ctypes.c_int64 * 2), ("w_stride", ctypes.c_int64 * 2),
                ("o_stride", ctypes.c_int64 * 2), ("dtype_qkv", ctypes.c_int32),
                ("dtype_g", ctypes.c_int32), ("cu_seqlens_i64", ctypes.c_int32),
                ("use_qk_l2norm", ctypes.c_int32), ("impl", ctypes.c_int32),
                ("state_v_major", ctypes.c_int32), ("dtype_state", ctypes.c_int32),
                ("state_segments", ctypes.c_int32), ("HK", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Open the library (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError("libgdn2.so is not built (%s); run __graft_entry__.build()" % p)
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.gdn2_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    lib.gdn2_workspace_bytes.restype = sz
    lib.gdn2_dims_init.argtypes = [ctypes.POINTER(Dims), i64, i32, i32, i32, i32, i32]
    lib.gdn2_dims_init.restype = ctypes.c_int
    lib.gdn2_check_args.argtypes = [vp] * 10 + [ctypes.POINTER(Dims), vp, sz]
    lib.gdn2_check_args.restype = ctypes.c_int
    lib.gdn2_chunk_fwd.argtypes = [vp] * 6 + [ctypes.c_float, vp, vp, vp, vp,
                                              ctypes.POINTER(Dims), vp, sz, vp]
    lib.gdn2_chunk_fwd.restype = ctypes.c_int
    lib.gdn2_chunk_fwd_staged.argtypes = [vp] * 6 + [ctypes.c_float, vp, vp, vp, vp,
                                                     ctypes.POINTER(Dims), vp, sz, vp,
                                                     ctypes.POINTER(vp), i32]
    lib.gdn2_chunk_fwd_staged.restype = ctypes.c_int
    lib.gdn2_num_stages.argtypes = [ctypes.POINTER(Dims)]
    lib.gdn2_num_stages.restype = i32
    lib.gdn2_stage_name.argtypes = [ctypes.POINTER(Dims), i32]
    lib.gdn2_stage_name.restype = ctypes.c_char_p
    lib.gdn2_launch_count.argtypes = [ctypes.POINTER(Dims)]
    lib.gdn2_launch_count.restype = i32
    lib.gdn2_launch_plan.argtypes = [ctypes.POINTER(Dims), i32, ctypes.c_char_p, sz]
    lib.gdn2_launch_plan.restype = i32
    lib.gdn2_chunk_fwd_noalloc.argtypes = [vp] * 6 + [ctypes.c_float, vp, vp, vp, vp,
                                                      ctypes.POINTER(Dims), vp]
    lib.gdn2_chunk_fwd_noalloc.restype = ctypes.c_int
    lib.gdn2_noalloc_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    lib.gdn2_noalloc_device_status.restype = ctypes.c_int
    lib.gdn2_recurrent_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    lib.gdn2_recurrent_workspace_bytes.restype = sz
    lib.gdn2_recurrent_fwd.argtypes = [vp] * 6 + [ctypes.c_float, vp, vp, vp, vp,
                                                  ctypes.POINTER(Dims), vp, sz, vp]
    lib.gdn2_recurrent_fwd.restype = ctypes.c_int
    lib.gdn2_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
    lib.gdn2_device_status.restype = ctypes.c_int
    lib.gdn2_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint64, vp]
    lib.gdn2_selftest_wait_timeout.restype = ctypes.c_int
    lib.gdn2_status_string.argtypes = [ctypes.c_int]
    lib.gdn2_status_string.restype = ctypes.c_char_p
    lib.gdn2_version.argtypes = []
    lib.gdn2_version.restype = i32
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().gdn2_status_string(int(status)).decode()
    except Exception:  # library not loadable: still give the name
        return STATUS_NAMES.get(status, "?")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _strides(t, name):
    if t is None:
        return (0, 0)
    if t.stride(-1) != 1:
        raise ValueError("%s: innermost dimension must be contiguous" % name)
    return (t.stride(0), t.stride(1))


def make_dims(q, k, v, g, beta, w, out, cu_seqlens, use_qk_l2norm=False, impl="tc", state_v_major=False,
              state_dtype=torch.float32) -> Dims:
    T, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    d = Dims()
    d.T_tot, d.N, d.H, d.HV, d.K, d.V = T, cu_seqlens.numel() - 1, H, HV, K, V
    d.HK = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("w", w), ("o", out)):
        s = _strides(t, name)
        getattr(d, name + "_stride")[0], getattr(d, name + "_stride")[1] = s
    # q, k, v, beta, w, out share one 16-bit dtype; anything else is refused
    d.dtype_qkv = _DTYPE_CODE.get(q.dtype, 99) if q.dtype != torch.float32 else 99
    for t in (k, v, beta, w, out):
        if t is not None and t.dtype != q.dtype:
            d.dtype_qkv = 99
    d.dtype_g = DTYPE_F32 if g is None else _DTYPE_CODE.get(g.dtype, 99)
    d.state_v_major = 1 if state_v_major else 0
    d.dtype_state = _DTYPE_CODE.get(state_dtype, 99) if state_dtype != torch.float16 else 99
    d.cu_seqlens_i64 = 1 if cu_seqlens.dtype == torch.int64 else 0
    d.use_qk_l2norm = 1 if use_qk_l2norm else 0
    d.impl = IMPL[impl]
    return d


def _state_dtype(initial_state, final_state, state_dtype):
    """dtype of the states: the one given, else that of the tensors passed, else fp32."""
    ts = [t.dtype for t in (initial_state, final_state) if t is not None]
    if state_dtype is None:
        state_dtype = ts[0] if ts else torch.float32
    if any(x != state_dtype for x in ts):
        raise ValueError("initial_state and final_state must have the same dtype (%s)" % state_dtype)
    return state_dtype


def workspace_bytes(dims: Dims) -> int:
    return int(load().gdn2_workspace_bytes(ctypes.byref(dims)))


def state_heads(q, v) -> int:
    """State (and output) heads: max(query heads, value heads) (the FlashInfer
    docs' num_sab_heads)."""
    return max(q.shape[1], v.shape[1])


def _check_inputs(q, k, v, cu_seqlens, initial_state):
    """The checks every wrapper makes before marshalling: packed input with
    cu_seqlens, CUDA tensors, and a contiguous initial state (the C ABI takes
    the state without strides)."""
    if cu_seqlens is None:
        raise ValueError("cu_seqlens is required (packed input only)")
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens", cu_seqlens), ("initial_state", initial_state)):
        if t is not None and not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
    if initial_state is not None and not initial_state.is_contiguous():
        raise ValueError("initial_state must be contiguous [N, HS, K, V]")


def chunk_gdn2_fwd(q, k, v, g=None, beta=None, w=None, scale=None, initial_state=None,
                   cu_seqlens=None, output_final_state=True, use_qk_l2norm=False, out=None,
                   final_state=None, workspace=None, impl="tc", stream=None, stage_events=None,
                   state_v_major=False, state_dtype=None, state_segments=0):
    """GDN-2 chunked prefill forward through ``gdn2_chunk_fwd``.

    Packed layout (FlashInfer docs, chunk_gated_delta_rule2): q [T, H, K],
    k [T, HK, K], v [T, HV, V] (HK equal to H or HV; H and HV equal or one a
    multiple of the other); with HS = max(H, HV) state heads: w [T, HS, V],
    g, beta [T, HS, K], initial_state [N, HS, K, V] fp32; cu_seqlens [N + 1]
    int32/int64.  Returns (out [T, HS, V] at q's dtype, final_state
    [N, HS, K, V] or None).
    """
    lib = load()
    _check_inputs(q, k, v, cu_seqlens, initial_state)
    T, H, K = q.shape
    V = v.shape[2]
    HS = state_heads(q, v)
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, HS, V), dtype=q.dtype, device=q.device)
    sdt = _state_dtype(initial_state, final_state, state_dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, HS, K, V), dtype=sdt, device=q.device)
    dims = make_dims(q, k, v, g, beta, w, out, cu_seqlens, use_qk_l2norm, impl, state_v_major, sdt)
    dims.state_segments = int(state_segments)  # 0: chosen by the library
    nbytes = workspace_bytes(dims)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w),
            ctypes.c_float(0.0 if scale is None else float(scale)),
            _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
            ctypes.byref(dims), _ptr(workspace), workspace.numel(), stream)
    if stage_events is None:
        st = lib.gdn2_chunk_fwd(*args)
    else:
        arr = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
        st = lib.gdn2_chunk_fwd_staged(*args, arr, len(stage_events))
    if st != GDN2_OK:
        raise Gdn2Error(st, "gdn2_chunk_fwd")
    return out, final_state


def chunk_gdn2_fwd_noalloc(q, k, v, g=None, beta=None, w=None, scale=None, initial_state=None,
                           cu_seqlens=None, output_final_state=True, use_qk_l2norm=False, out=None,
                           final_state=None, impl="tc", stream=None, state_v_major=False, state_dtype=None):
    """The forward through ``gdn2_chunk_fwd_noalloc``: no workspace argument;
    the library's fixed device scratch (NOALLOC_SCRATCH_BYTES) is used, so
    calls must not overlap on the GPU.  Outputs are allocated here only when
    the caller does not pass them; ``noalloc_device_status()`` reads the
    device-side status of the last call."""
    lib = load()
    _check_inputs(q, k, v, cu_seqlens, initial_state)
    T, H, K = q.shape
    V = v.shape[2]
    HS = state_heads(q, v)
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, HS, V), dtype=q.dtype, device=q.device)
    sdt = _state_dtype(initial_state, final_state, state_dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, HS, K, V), dtype=sdt, device=q.device)
    dims = make_dims(q, k, v, g, beta, w, out, cu_seqlens, use_qk_l2norm, impl, state_v_major, sdt)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    st = lib.gdn2_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w),
                                    ctypes.c_float(0.0 if scale is None else float(scale)),
                                    _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                    ctypes.byref(dims), stream)
    if st != GDN2_OK:
        raise Gdn2Error(st, "gdn2_chunk_fwd_noalloc")
    return out, final_state


def recurrent_gdn2_fwd(q, k, v, g=None, beta=None, w=None, scale=None, initial_state=None,
                       cu_seqlens=None, output_final_state=True, use_qk_l2norm=False, out=None,
                       final_state=None, workspace=None, stream=None, state_v_major=False, state_dtype=None):
    """Token-by-token recurrence from a carried state through
    ``gdn2_recurrent_fwd`` (decode steps, short continuations).  Same layouts
    as ``chunk_gdn2_fwd``; ``final_state`` may be ``initial_state`` itself
    (updated in place).  Returns (out, final_state)."""
    lib = load()
    _check_inputs(q, k, v, cu_seqlens, initial_state)
    T, H, K = q.shape
    V = v.shape[2]
    HS = state_heads(q, v)
    N = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, HS, V), dtype=q.dtype, device=q.device)
    sdt = _state_dtype(initial_state, final_state, state_dtype)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, HS, K, V), dtype=sdt, device=q.device)
    dims = make_dims(q, k, v, g, beta, w, out, cu_seqlens, use_qk_l2norm, "tc", state_v_major, sdt)
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    st = lib.gdn2_recurrent_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(w),
                                ctypes.c_float(0.0 if scale is None else float(scale)),
                                _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                ctypes.byref(dims), _ptr(workspace), workspace.numel(), stream)
    if st != GDN2_OK:
        raise Gdn2Error(st, "gdn2_recurrent_fwd")
    return out, final_state


def noalloc_device_status(device=None, stream=None) -> int:
    """Device-side status of the last ``chunk_gdn2_fwd_noalloc`` call on the
    current device (syncs the stream)."""
    if stream is None:
        stream = torch.cuda.current_stream(device).cuda_stream
    s = ctypes.c_int32(-1)
    st = load().gdn2_noalloc_device_status(stream, ctypes.byref(s))
    if st != GDN2_OK:
        raise Gdn2Error(st, "gdn2_noalloc_device_status")
    return int(s.value)


def device_status(workspace, stream=None) -> int:
    """Device-side status word of the last call on ``workspace`` (syncs the stream)."""
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device).cuda_stream
    s = ctypes.c_int32(-1)
    st = load().gdn2_device_status(_ptr(workspace), stream, ctypes.byref(s))
    if st != GDN2_OK:
        raise Gdn2Error(st, "gdn2_device_status")
    return int(s.value)


class _SlicedRunner:
    """HostRunner for few sequences: every sequence is cut in time into
    ``slices`` pieces of whole 64-token chunks (the last piece takes the
    remainder).  Piece j of all sequences is packed into a device staging
    buffer (two, alternating), run as one forward whose initial state is
    piece j - 1's final state (two state buffers, alternating), and its output
    rows are copied back into their places in the pinned host output."""

    def __init__(self, host, impl, use_qk_l2norm, output_final_state, slices, slice_weights=None):
        self.host, self.impl, self.l2, self.S = host, impl, use_qk_l2norm, slices
        # relative sizes of the pieces (integers).  By default the last two are
        # half and a quarter of the others: the copies in are the bottleneck,
        # and a small last piece shortens the forward and copy out that follow
        # the last copy in (long workload: 38.72 -> 38.01 ms per call)
        if slice_weights:
            self.weights = [int(x) for x in slice_weights]
        else:
            self.weights = [4] * (slices - 2) + [2, 1] if slices >= 3 else [1] * slices
        if len(self.weights) != slices or min(self.weights) <= 0:
            raise ValueError("slice_weights: one positive integer per slice")
        T, _, V = host["v"].shape
        HV = state_heads(host["q"], host["v"])  # output and state heads
        K = host["q"].shape[2]
        cu = [int(x) for x in host["cu_seqlens"].tolist()]
        self.N = N = len(cu) - 1
        sdt = host["h0"].dtype if host.get("h0") is not None else torch.float32
        self.keys = [k for k in ("q", "k", "v", "g", "beta", "w") if torch.is_tensor(host.get(k))]
        rows = max(self._plan(cu)[1])
        self.stage = [{k: torch.empty((max(rows, 1),) + tuple(host[k].shape[1:]), dtype=host[k].dtype,
                                      device="cuda") for k in self.keys} for _ in range(2)]
        self.out_stage = [torch.empty((max(rows, 1), HV, V), dtype=host["q"].dtype, device="cuda")
                          for _ in range(2)]
        self.state = [torch.empty((N, HV, K, V), dtype=sdt, device="cuda") for _ in range(2)]
        self.h0 = torch.empty_like(host["h0"], device="cuda") if torch.is_tensor(host.get("h0")) else None
        self.out_host = torch.empty((T, HV, V), dtype=host["q"].dtype).pin_memory()
        self.fs_host = torch.empty((N, HV, K, V), dtype=sdt).pin_memory() if output_final_state else None
        cu_dt = host["cu_seqlens"].dtype
        self.cu_host = [torch.empty(N + 1, dtype=cu_dt).pin_memory() for _ in range(slices)]
        self.cu_dev = [torch.empty(N + 1, dtype=cu_dt, device="cuda") for _ in range(slices)]
        self.cu_ev = [None] * slices
        dims = make_dims(self.stage[0]["q"], self.stage[0]["k"], self.stage[0]["v"], self.stage[0].get("g"),
                         self.stage[0].get("beta"), self.stage[0].get("w"), self.out_stage[0],
                         self.cu_dev[0], use_qk_l2norm, impl, False, sdt)
        self.ws = torch.empty(max(workspace_bytes(dims), 256), dtype=torch.uint8, device="cuda")
        self.streams = [torch.cuda.Stream() for _ in range(3)]
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in host.values() if torch.is_tensor(v))
        self.d2h_bytes = self.out_host.numel() * self.out_host.element_size() + (
            0 if self.fs_host is None else self.fs_host.numel() * self.fs_host.element_size())

    def _plan(self, cu):
        """Token bounds of every piece: b[n][j] = offset of piece j in sequence
        n (whole 64-token chunks, in proportion to the slice weights); returns
        (b, rows of each piece)."""
        S = self.S
        cw = [sum(self.weights[:j]) for j in range(S)]
        wt = sum(self.weights)
        b = []
        for n in range(self.N):
            L = cu[n + 1] - cu[n]
            b.append([64 * ((L * cw[j]) // (64 * wt)) for j in range(S)] + [L])
        rows = [sum(b[n][j + 1] - b[n][j] for n in range(self.N)) for j in range(S)]
        return b, rows

    def __call__(self):
        s_in, s_cmp, s_out = self.streams
        caller = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(caller)
        for st in self.streams:
            st.wait_event(start)
        h = self.host
        cu = [int(x) for x in h["cu_seqlens"].tolist()]
        b, _ = self._plan(cu)
        ev_c, ev_o = [None] * self.S, [None] * self.S
        if self.h0 is not None:
            with torch.cuda.stream(s_in):
                self.h0.copy_(h["h0"], non_blocking=True)
        for j in range(self.S):
            buf = j % 2
            # piece j's cu_seqlens (host arithmetic into a pinned buffer whose
            # previous copy to the device must be done)
            if self.cu_ev[j] is not None:
                self.cu_ev[j].synchronize()
            offs = [0]
            for n in range(self.N):
                offs.append(offs[-1] + b[n][j + 1] - b[n][j])
            self.cu_host[j].copy_(torch.tensor(offs, dtype=self.cu_host[j].dtype))
            with torch.cuda.stream(s_in):
                if j >= 2:
                    s_in.wait_event(ev_c[j - 2])  # the staging buffer was read by forward j - 2
                for n in range(self.N):
                    a, e = cu[n] + b[n][j], cu[n] + b[n][j + 1]
                    if e > a:
                        for k in self.keys:
                            self.stage[buf][k][offs[n]:offs[n + 1]].copy_(h[k][a:e], non_blocking=True)
                self.cu_dev[j].copy_(self.cu_host[j], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
                self.cu_ev[j] = ev_in
            s_cmp.wait_event(ev_in)
            if j >= 2:
                s_cmp.wait_event(ev_o[j - 2])  # the output staging was copied out
            with torch.cuda.stream(s_cmp):
                rows = offs[-1]
                st = self.stage[buf]
                sl = lambda k: st[k][:rows] if k in st else None
                init = self.h0 if j == 0 else self.state[(j - 1) % 2]
                chunk_gdn2_fwd(sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"), sl("w"), scale=h.get("scale"),
                               initial_state=init, cu_seqlens=self.cu_dev[j], use_qk_l2norm=self.l2,
                               out=self.out_stage[buf][:rows], final_state=self.state[j % 2], workspace=self.ws,
                               impl=self.impl, stream=s_cmp.cuda_stream)
                ev_c[j] = torch.cuda.Event()
                ev_c[j].record(s_cmp)
            s_out.wait_event(ev_c[j])
            with torch.cuda.stream(s_out):
                for n in range(self.N):
                    a, e = cu[n] + b[n][j], cu[n] + b[n][j + 1]
                    if e > a:
                        self.out_host[a:e].copy_(self.out_stage[buf][offs[n]:offs[n + 1]], non_blocking=True)
                if j == self.S - 1 and self.fs_host is not None:
                    self.fs_host.copy_(self.state[j % 2], non_blocking=True)
                ev_o[j] = torch.cuda.Event()
                ev_o[j].record(s_out)
        caller.wait_event(ev_o[-1])
        return self.out_host, self.fs_host


def selftest_wait_timeout(workspace, limit_ns=1_000_000, stream=None) -> int:
    """Run the bounded-wait self-test (``gdn2_selftest_wait_timeout``) on
    ``workspace``; returns the call's status (the timeout itself is then read
    with ``device_status``)."""
    if stream is None and workspace.is_cuda:
        stream = torch.cuda.current_stream(workspace.device).cuda_stream
    return int(load().gdn2_selftest_wait_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                                 int(limit_ns), stream))


def stage_names(dims: Dims):
    lib = load()
    return [lib.gdn2_stage_name(ctypes.byref(dims), i).decode()
            for i in range(lib.gdn2_num_stages(ctypes.byref(dims)))]


def launch_plan(dims: Dims, sm_count: int = 0) -> str:
    """The launch sequence of one call for ``dims`` as text (host only)."""
    lib = load()
    n = lib.gdn2_launch_plan(ctypes.byref(dims), sm_count, None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    lib.gdn2_launch_plan(ctypes.byref(dims), sm_count, buf, n + 1)
    return buf.value.decode()


def launch_count(dims: Dims) -> int:
    return int(load().gdn2_launch_count(ctypes.byref(dims)))


class HostRunner:
    """End-to-end call from HOST buffers: pinned host inputs are copied to
    preallocated device buffers, the forward runs, and the output and final
    state are copied back into pinned host buffers.  The work is cut into
    pieces whose host-to-device copy, forward and device-to-host copy run on
    three streams at once (piece i + 1 in, piece i computed, piece i - 1
    out), so the call is bounded by the host link rather than by the kernels.
    The caller's stream waits for the last copy.  Device buffers and the
    workspace are allocated once (torch) and reused.

    Pieces: with at most ``max_sliced_seqs`` sequences (each piece takes
    one copy per sequence and tensor) every sequence is cut in time into
    ``slices`` pieces of whole 64-token chunks (sizes in proportion to
    ``slice_weights``; by default the last two pieces are half and a quarter
    of the others), each forward starting from the previous piece's final
    state (_SlicedRunner); with more sequences,
    or slices <= 1, contiguous sequence groups (at most ``groups``, balanced
    by tokens)."""

    def __new__(cls, host: dict, impl="tc", use_qk_l2norm=False, output_final_state=True, groups=4,
                slices=8, max_sliced_seqs=8, slice_weights=None):
        n_seq = host["cu_seqlens"].numel() - 1
        if cls is HostRunner and slices and slices > 1 and 0 < n_seq <= max_sliced_seqs:
            return _SlicedRunner(host, impl, use_qk_l2norm, output_final_state, slices, slice_weights)
        return super().__new__(cls)

    def __init__(self, host: dict, impl="tc", use_qk_l2norm=False, output_final_state=True, groups=4,
                 slices=8, max_sliced_seqs=8, slice_weights=None):
        self.host = host
        self.impl = impl
        self.l2 = use_qk_l2norm
        self.dev = {k: (torch.empty_like(v, device="cuda") if torch.is_tensor(v) else v)
                    for k, v in host.items()}
        T, _, V = host["v"].shape
        HV = state_heads(host["q"], host["v"])  # output and state heads
        cu = [int(x) for x in host["cu_seqlens"].tolist()]
        N = len(cu) - 1
        K = host["q"].shape[2]
        sdt = host["h0"].dtype if host.get("h0") is not None else torch.float32
        self.out_host = torch.empty((T, HV, V), dtype=host["q"].dtype).pin_memory()
        self.fs_host = (torch.empty((N, HV, K, V), dtype=sdt).pin_memory() if output_final_state else None)
        self.out = torch.empty((T, HV, V), dtype=host["q"].dtype, device="cuda")
        self.fs = torch.empty((N, HV, K, V), dtype=sdt, device="cuda") if output_final_state else None
        dims = make_dims(self.dev["q"], self.dev["k"], self.dev["v"], self.dev["g"], self.dev["beta"],
                         self.dev["w"], self.out, self.dev["cu_seqlens"], use_qk_l2norm, impl, False, sdt)
        self.ws = torch.empty(max(workspace_bytes(dims), 256), dtype=torch.uint8, device="cuda")
        # contiguous sequence groups with about T / groups tokens each
        n_groups = max(1, min(groups, N))
        bounds, n = [0], 0
        for gi in range(1, n_groups):
            target = cu[-1] * gi / n_groups
            while n < N - (n_groups - gi) and cu[n + 1] <= target:
                n += 1
            n = max(n, bounds[-1] + 1)
            bounds.append(n)
        bounds.append(N)
        self.bounds = sorted(set(bounds))
        cu_dt = host["cu_seqlens"].dtype
        self.cu_host = [torch.empty(b - a + 1, dtype=cu_dt).pin_memory()
                        for a, b in zip(self.bounds[:-1], self.bounds[1:])]
        self.cu_dev = [torch.empty_like(c, device="cuda") for c in self.cu_host]
        self.cu_ev = [None] * len(self.cu_host)  # last copy out of each pinned cu buffer
        self.streams = [torch.cuda.Stream() for _ in range(3)]
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in host.values() if torch.is_tensor(v))
        self.d2h_bytes = self.out_host.numel() * self.out_host.element_size() + (
            0 if self.fs_host is None else self.fs_host.numel() * self.fs_host.element_size())

    def __call__(self):
        s_in, s_cmp, s_out = self.streams
        caller = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(caller)
        for st in self.streams:
            st.wait_event(start)
        h, d = self.host, self.dev
        cu = h["cu_seqlens"]
        for gi, (n0, n1) in enumerate(zip(self.bounds[:-1], self.bounds[1:])):
            t0, t1 = int(cu[n0]), int(cu[n1])
            # the group's cu_seqlens, rebased to its first token (host arithmetic);
            # the previous call's copy out of this pinned buffer must be done
            if self.cu_ev[gi] is not None:
                self.cu_ev[gi].synchronize()
            torch.sub(cu[n0:n1 + 1], cu[n0], out=self.cu_host[gi])
            with torch.cuda.stream(s_in):
                for key in ("q", "k", "v", "g", "beta", "w"):
                    if torch.is_tensor(h.get(key)):
                        d[key][t0:t1].copy_(h[key][t0:t1], non_blocking=True)
                if torch.is_tensor(h.get("h0")):
                    d["h0"][n0:n1].copy_(h["h0"][n0:n1], non_blocking=True)
                self.cu_dev[gi].copy_(self.cu_host[gi], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
                self.cu_ev[gi] = ev_in
            s_cmp.wait_event(ev_in)
            with torch.cuda.stream(s_cmp):
                sl = lambda key: d[key][t0:t1] if torch.is_tensor(d.get(key)) else None
                chunk_gdn2_fwd(sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"), sl("w"), scale=d.get("scale"),
                               initial_state=d["h0"][n0:n1] if torch.is_tensor(d.get("h0")) else None,
                               cu_seqlens=self.cu_dev[gi], use_qk_l2norm=self.l2, out=self.out[t0:t1],
                               final_state=None if self.fs is None else self.fs[n0:n1],
                               output_final_state=self.fs is not None, workspace=self.ws, impl=self.impl,
                               stream=s_cmp.cuda_stream)
                ev_c = torch.cuda.Event()
                ev_c.record(s_cmp)
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                self.out_host[t0:t1].copy_(self.out[t0:t1], non_blocking=True)
                if self.fs is not None:
                    self.fs_host[n0:n1].copy_(self.fs[n0:n1], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        caller.wait_event(done)
        return self.out_host, self.fs_host
