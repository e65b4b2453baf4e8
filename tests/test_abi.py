"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects bad arguments before touching a device.  No kernel is
launched here (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

from gated_deltanet_prefill_gb300 import build as gbuild
from gated_deltanet_prefill_gb300 import gdn2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn2.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "gdn2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"GDN2_API\s+[\w\s\*]+?\b(gdn2_\w+)\s*\(", src)))


def test_header_declares_entry_points():
    fns = header_functions()
    assert "gdn2_chunk_fwd" in fns and "gdn2_workspace_bytes" in fns
    assert set(fns) == set(gdn2.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for fn in header_functions():
        assert hasattr(lib, fn), fn


def test_version_and_strings(lib):
    assert lib.gdn2_version() >> 16 == 1
    for code in range(16):  # GDN2_OK .. GDN2_ERR_BOUNDS
        s = lib.gdn2_status_string(code).decode()
        assert s and s != "unknown status"
        assert code in gdn2.STATUS_NAMES
    assert lib.gdn2_status_string(999).decode() == "unknown status"


def _dims(lib, T=256, N=2, H=2, HV=4, K=64, V=64):
    d = gdn2.Dims()
    assert lib.gdn2_dims_init(ctypes.byref(d), T, N, H, HV, K, V) == 0
    return d


# Fake, well-separated, 256-byte aligned "device" addresses: the checks are
# host arithmetic only and never dereference them.
BASE = 1 << 40


def _ptrs(d, ws_bytes):
    MB = 1 << 26
    names = ["q", "k", "v", "g", "beta", "w", "h0", "cu", "out", "hT", "ws"]
    return {n: BASE + i * MB for i, n in enumerate(names)}


def _check(lib, d, p, ws_bytes=None, **over):
    p = {**p, **over}
    if ws_bytes is None:
        ws_bytes = lib.gdn2_workspace_bytes(ctypes.byref(d))
    return lib.gdn2_check_args(p["q"], p["k"], p["v"], p["g"], p["beta"], p["w"], p["h0"], p["cu"],
                               p["out"], p["hT"], ctypes.byref(d), p["ws"], ws_bytes)


def test_workspace_bytes(lib):
    d = _dims(lib)
    n = lib.gdn2_workspace_bytes(ctypes.byref(d))
    assert n > 0
    d2 = _dims(lib, T=512)
    assert lib.gdn2_workspace_bytes(ctypes.byref(d2)) > n
    bad = _dims(lib)
    bad.K = 96
    assert lib.gdn2_workspace_bytes(ctypes.byref(bad)) == 0


def test_check_args_ok(lib):
    d = _dims(lib)
    assert _check(lib, d, _ptrs(d, 0)) == 0


def test_check_args_errors(lib):
    d = _dims(lib)
    p = _ptrs(d, 0)
    assert _check(lib, d, p, q=None) == 1                 # ERR_NULL
    assert _check(lib, d, p, cu=None) == 1
    assert _check(lib, d, p, ws=None) == 1
    assert _check(lib, d, p, ws_bytes=100) == 5           # ERR_WORKSPACE
    assert _check(lib, d, p, q=p["q"] + 8) == 3           # ERR_STRIDE: base not 16B aligned
    assert _check(lib, d, p, out=p["v"]) == 4             # ERR_ALIAS: out == v
    assert _check(lib, d, p, hT=p["h0"]) == 4             # final_state == initial_state
    assert _check(lib, d, p, out=p["hT"]) == 4
    # optional gates may be NULL
    assert _check(lib, d, p, g=None, beta=None, w=None, h0=None, hT=None) == 0
    for field, val, code in (("K", 96, 2), ("HV", 3, 2), ("N", -1, 2), ("dtype_qkv", 2, 8),
                             ("dtype_qkv", 7, 8), ("dtype_g", 7, 8), ("dtype_state", 1, 8),
                             ("state_v_major", 2, 8), ("impl", 7, 11)):
        d2 = _dims(lib)
        setattr(d2, field, val)
        assert _check(lib, d2, p, ws_bytes=1 << 30) == code, field
    # the variants the FlashInfer docs list: fp16 inputs, bf16/fp16 g, bf16 and
    # V-major states (tensor-core path); the SIMT path keeps the defaults
    for field, val in (("dtype_qkv", 1), ("dtype_g", 0), ("dtype_g", 1), ("dtype_state", 0), ("state_v_major", 1)):
        d2 = _dims(lib)
        setattr(d2, field, val)
        assert _check(lib, d2, p, ws_bytes=1 << 30) == 0, field
        d2.impl = 1
        assert _check(lib, d2, p, ws_bytes=1 << 30) == 8, field
    d3 = _dims(lib)
    d3.q_stride[0] = 2 * 64 + 4                           # 264 bytes: not a multiple of 16
    assert _check(lib, d3, p) == 3
    d4 = _dims(lib)
    d4.o_stride[1] = 32                                   # heads of out overlap
    assert _check(lib, d4, p) == 4


def test_head_count_rules(lib):
    """FlashInfer docs, parameters q/k/v: num_k_heads equals num_q_heads or
    num_v_heads, and the query and value head counts are equal or one a
    multiple of the other; states, gates and output are per state head,
    max(H, HV)."""
    def dims(H, HV, HK=0):
        d = gdn2.Dims()
        st = lib.gdn2_dims_init(ctypes.byref(d), 256, 2, H, HV, 64, 64)
        d.HK = HK
        return st, d

    ok = [(4, 2, 0), (4, 2, 2), (4, 2, 4), (2, 4, 0), (2, 4, 4), (3, 6, 6), (6, 3, 3), (1, 8, 8), (8, 1, 1)]
    for H, HV, HK in ok:
        st, d = dims(H, HV, HK)
        assert st == 0
        p = _ptrs(d, 0)
        assert _check(lib, d, p, ws_bytes=1 << 30) == 0, (H, HV, HK)
    for H, HV, HK in ((4, 2, 3), (4, 2, 1), (2, 4, 1), (4, 6, 0), (2, 3, 2)):
        _, d = dims(H, HV, HK)
        assert _check(lib, d, _ptrs(d, 0), ws_bytes=1 << 30) == 2, (H, HV, HK)
    # per-state-head tensors are laid out with HS = max(H, HV) heads
    st, d = dims(4, 2)
    assert d.v_stride[0] == 2 * 64 and d.w_stride[0] == 4 * 64 and d.o_stride[0] == 4 * 64
    assert d.g_stride[0] == 4 * 64 and d.beta_stride[0] == 4 * 64 and d.q_stride[0] == 4 * 64
    # the workspace follows the state heads, not the value heads
    _, d44 = dims(4, 4)
    assert lib.gdn2_workspace_bytes(ctypes.byref(d)) == lib.gdn2_workspace_bytes(ctypes.byref(d44))


def test_launch_plan(lib):
    """The host-side description of the launch sequence (also printed with
    GDN2_LOG=1) names the kernels and grids each shape gets."""
    def plan(T, N, H, HV, K, impl=0, segments=0, sms=152):
        d = gdn2.Dims()
        assert lib.gdn2_dims_init(ctypes.byref(d), T, N, H, HV, K, K) == 0
        d.impl, d.state_segments = impl, segments
        return gdn2.launch_plan(d, sms)

    long5 = plan(4 * 32768, 4, 32, 32, 128)
    assert "intra first pass 304 x256" in long5 and "gdn2_tc_state_la128_kernel 128 CTAs of 128 columns" in long5
    few = plan(16384 * 2, 2, 16, 32, 128)
    assert "gdn2_tc_state_la_kernel 128 CTAs of 64 columns" in few
    seg = plan(4096, 1, 16, 16, 128)
    assert "chunk-parallel state pass, 5 segments" in seg
    assert "gdn2_tc_state_la128_kernel 112 CTAs of 128 columns" in seg   # segment 0, transitions of 1-3
    assert "combine 1x16x8, 3 steps" in seg
    assert "replay of segments 1-4 gdn2_tc_state_la_kernel 128 CTAs of 64 columns" in seg
    two = plan(4096, 1, 16, 16, 128, segments=2)
    assert "combine" not in two and "replay of segments 1-1" in two
    assert "simt_intra" in plan(256, 1, 2, 2, 64, impl=1)
    assert "state_kernel<64>" in plan(256, 1, 2, 2, 64)
    d = gdn2.Dims()
    assert lib.gdn2_dims_init(ctypes.byref(d), 256, 1, 2, 3, 64, 64) != 0
    assert lib.gdn2_launch_plan(ctypes.byref(d), 152, None, 0) == 0
    small = ctypes.create_string_buffer(8)
    assert lib.gdn2_launch_plan(ctypes.byref(gdn2.Dims()), 0, None, 0) == 0
    d = gdn2.Dims()
    lib.gdn2_dims_init(ctypes.byref(d), 256, 1, 2, 2, 64, 64)
    n = lib.gdn2_launch_plan(ctypes.byref(d), 0, small, 8)
    assert n > 8 and len(small.value) == 7  # truncated like snprintf


def test_chunk_fwd_rejects_before_launch(lib):
    """gdn2_chunk_fwd returns the argument error without any CUDA call."""
    d = _dims(lib)
    p = _ptrs(d, 0)
    ws = lib.gdn2_workspace_bytes(ctypes.byref(d))
    st = lib.gdn2_chunk_fwd(None, p["k"], p["v"], p["g"], p["beta"], p["w"], ctypes.c_float(0.0),
                            p["h0"], p["cu"], p["out"], p["hT"], ctypes.byref(d), p["ws"], ws, None)
    assert st == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error")
def test_chunk_fwd_without_device_fails_loudly(lib):
    """With valid arguments but no CUDA device the call fails with ERR_ARCH
    (there is no CPU path)."""
    d = _dims(lib)
    p = _ptrs(d, 0)
    ws = lib.gdn2_workspace_bytes(ctypes.byref(d))
    st = lib.gdn2_chunk_fwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["w"], ctypes.c_float(0.0),
                            p["h0"], p["cu"], p["out"], p["hT"], ctypes.byref(d), p["ws"], ws, None)
    assert st == 6


def test_binding_refuses_cpu_tensors(lib):
    q = torch.zeros(64, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 64], dtype=torch.int32)
    with pytest.raises(ValueError):
        gdn2.chunk_gdn2_fwd(q, q, q, cu_seqlens=cu)


def test_product_package_does_not_import_oracle():
    """The product package never reaches into oracle/ (no CPU fallback)."""
    pkg = os.path.join(ROOT, "gated_deltanet_prefill_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), f
                assert "gdn2_oracle" not in src, f


def _recurrent(lib, d, p, ws_bytes=64, **over):
    p = {**p, **over}
    return lib.gdn2_recurrent_fwd(p["q"], p["k"], p["v"], p["g"], p["beta"], p["w"], ctypes.c_float(0.0),
                                  p["h0"], p["cu"], p["out"], p["hT"], ctypes.byref(d), p["ws"], ws_bytes, None)


def test_recurrent_argument_checks(lib):
    """gdn2_recurrent_fwd: a 64-byte workspace, the state may be updated in
    place (same pointer), any other state overlap is refused; the checks run
    before any CUDA call (without a device a valid call reports ERR_ARCH)."""
    d = _dims(lib)
    assert lib.gdn2_recurrent_workspace_bytes(ctypes.byref(d)) == 64
    bad = _dims(lib)
    bad.K = 96
    assert lib.gdn2_recurrent_workspace_bytes(ctypes.byref(bad)) == 0
    p = _ptrs(d, 64)
    no_gpu = 6  # GDN2_ERR_ARCH: argument checks passed, no sm_103 device here
    if torch.cuda.is_available():
        pytest.skip("the valid-call cases would launch on this machine's GPU")
    assert _recurrent(lib, d, p) == no_gpu
    assert _recurrent(lib, d, p, hT=p["h0"]) == no_gpu          # in place
    assert _recurrent(lib, d, p, hT=p["h0"] + 1024) == 4       # partial overlap: ERR_ALIAS
    assert _recurrent(lib, d, p, ws_bytes=32) == 5              # ERR_WORKSPACE
    assert _recurrent(lib, d, p, ws=0) == 1                      # ERR_NULL
    assert _recurrent(lib, d, p, out=p["q"]) == 4                # out overlaps an input
    # the chunked call keeps refusing an in-place state
    assert _check(lib, d, p, hT=p["h0"]) == 4


def test_state_segments_host_logic(lib):
    """The chunk-parallel state pass: argument range, where it is allowed,
    the automatic choice (visible in the launch count) and its workspace."""
    p = _ptrs(None, 0)
    for val, impl, K, code in ((-1, 0, 128, 2), (65, 0, 128, 2), (64, 0, 128, 0), (4, 0, 64, 2),
                               (4, 1, 128, 2), (1, 1, 128, 0), (1, 0, 64, 0)):
        d = _dims(lib, K=K, V=K)
        d.impl, d.state_segments = impl, val
        assert _check(lib, d, p, ws_bytes=1 << 34) == code, (val, impl, K)
    # few (sequence, head) pairs on long sequences: P >= 3 chosen automatically
    few = _dims(lib, T=4096, N=1, H=16, HV=16, K=128, V=128)
    assert gdn2.launch_count(few) == 6            # map, intra (2 passes), transitions, combine, replay
    two = _dims(lib, T=4096, N=1, H=16, HV=16, K=128, V=128)
    two.state_segments = 2
    assert gdn2.launch_count(two) == 5            # two segments: nothing to combine
    seq = _dims(lib, T=4096, N=1, H=16, HV=16, K=128, V=128)
    seq.state_segments = 1
    assert gdn2.launch_count(seq) == 4            # map, intra (2 passes), state
    assert lib.gdn2_workspace_bytes(ctypes.byref(few)) > lib.gdn2_workspace_bytes(ctypes.byref(seq))
    many = _dims(lib, T=4096, N=2, H=16, HV=16, K=128, V=128)   # 32 pairs: sequential
    assert gdn2.launch_count(many) == 4
    short = _dims(lib, T=1024, N=1, H=2, HV=2, K=128, V=128)    # 16 chunks: too short to split
    assert gdn2.launch_count(short) == 4


def test_selftest_wait_timeout_argument_checks(lib):
    """The bounded-wait self-test validates its arguments before any launch;
    without a device a valid call reports ERR_ARCH."""
    ws = ctypes.c_void_p(BASE)
    assert lib.gdn2_selftest_wait_timeout(None, 64, 1_000_000, None) == 1      # ERR_NULL
    assert lib.gdn2_selftest_wait_timeout(ws, 32, 1_000_000, None) == 5        # ERR_WORKSPACE
    assert lib.gdn2_selftest_wait_timeout(ws, 64, 10, None) == 2               # limit below 1 us
    assert lib.gdn2_selftest_wait_timeout(ws, 64, 10**9, None) == 2            # limit above 100 ms
    if not torch.cuda.is_available():
        assert lib.gdn2_selftest_wait_timeout(ws, 64, 1_000_000, None) == 6    # ERR_ARCH


def test_sliced_host_runner_plan():
    """The piece bounds the pinned-host runner cuts sequences into (host
    logic, no device): whole 64-token chunks, increasing, covering every
    sequence, sized by the slice weights (by default the last two pieces are
    half and a quarter of the others), and bad weights refused."""
    g = gdn2

    def plan(lens, slices, weights):
        r = g._SlicedRunner.__new__(g._SlicedRunner)
        r.S, r.N = slices, len(lens)
        r.weights = weights
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        return r._plan(cu)

    lens = [32768, 32768 - 100, 1, 0, 640]
    for weights in ([1] * 8, [4, 4, 4, 4, 4, 4, 2, 1], [1, 3, 2, 5, 1, 1, 1, 1]):
        b, rows = plan(lens, 8, weights)
        for n, L in enumerate(lens):
            assert b[n][0] == 0 and b[n][-1] == L
            assert all(x % 64 == 0 for x in b[n][:-1])
            assert all(x <= y for x, y in zip(b[n], b[n][1:]))
        assert sum(rows) == sum(lens)
        w = sum(weights)
        for j in range(8):  # piece j of the long sequence: its share within one chunk
            assert abs((b[0][j + 1] - b[0][j]) - 32768 * weights[j] / w) <= 64
    dummy = {"v": torch.zeros(4, 1, 64), "q": torch.zeros(4, 1, 64), "cu_seqlens": torch.tensor([0, 4])}
    with pytest.raises(ValueError):
        g._SlicedRunner(dummy, "tc", False, True, 4, slice_weights=[1, 1, 1])
    with pytest.raises(ValueError):
        g._SlicedRunner(dummy, "tc", False, True, 2, slice_weights=[1, 0])
