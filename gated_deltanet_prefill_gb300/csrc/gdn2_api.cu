// C ABI of the GDN-2 chunked prefill forward: argument checks, workspace
// layout and the launch sequence.  See include/gdn2.h for the contract.
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gdn2_internal.cuh"

namespace gdn2 {

namespace {

// cuTensorMapEncodeTiled from the driver (looked up once; nullptr if absent)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Tensor map over a token-major [T, heads, D] tensor (element strides st_t,
// st_h; channel stride 1) whose box is 64 tokens x D channels of one head,
// written to shared memory as [64][D].  The two outer dimensions go in
// increasing stride order (*order = 0: (channel, head, token), 1: (channel,
// token, head)).  False if the driver rejects the layout.
bool encode_rows(CUtensorMap *map, int *order, const void *base, CUtensorMapDataType type, int64_t esize,
                 int64_t D, int64_t heads, int64_t T, int64_t st_t, int64_t st_h) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || !base || T < 1 || T > INT32_MAX || heads < 1) return false;
    const bool head_inner = st_h < st_t;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(head_inner ? heads : T),
                                static_cast<cuuint64_t>(head_inner ? T : heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>((head_inner ? st_h : st_t) * esize),
                                   static_cast<cuuint64_t>((head_inner ? st_t : st_h) * esize)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), head_inner ? 1u : 64u, head_inner ? 64u : 1u};
    const cuuint32_t estr[3] = {1, 1, 1};
    *order = head_inner ? 0 : 1;
    return enc(map, type, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int64_t nc_max(const gdn2_dims &d) { return d.T_tot / kChunk + d.N; }


// Byte range [lo, hi) covered by a strided token-major tensor.
struct Range {
    uintptr_t lo, hi;
};

Range tensor_range(const void *base, int64_t T, int heads, int ch, const int64_t *st, size_t esize) {
    if (!base || T <= 0) return {0, 0};
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    const int64_t last = (T - 1) * st[0] + static_cast<int64_t>(heads - 1) * st[1] + ch;
    return {b, b + static_cast<uintptr_t>(last) * esize};
}

Range flat_range(const void *base, size_t bytes) {
    if (!base || bytes == 0) return {0, 0};
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    return {b, b + bytes};
}

bool overlap(Range a, Range b) { return a.hi > a.lo && b.hi > b.lo && a.lo < b.hi && b.lo < a.hi; }

bool strides_ok(const void *base, const int64_t *st, size_t esize, int heads, int ch) {
    if (!base) return true;
    if (reinterpret_cast<uintptr_t>(base) % 16) return false;
    if (st[0] < 0 || st[1] < 0) return false;
    if ((st[0] * esize) % 16 || (st[1] * esize) % 16) return false;
    (void)heads; (void)ch;
    return true;
}

}  // namespace

bool shape_ok(const gdn2_dims &d) {
    if (d.T_tot < 0 || d.N < 0 || d.H <= 0 || d.HV <= 0 || d.HK < 0) return false;
    const int hk = dims_hk(d);
    if (hk != d.H && hk != d.HV) return false;            // num_k_heads = num_q_heads or num_v_heads
    if (d.HV % d.H != 0 && d.H % d.HV != 0) return false;  // one a multiple of the other
    if (d.K != d.V || (d.K != 64 && d.K != 128)) return false;
    if (nc_max(d) > (1ll << 30)) return false;
    return true;
}

// Segments of the chunk-parallel state pass.  The chain of a sequence's
// chunks is cut into P equal segments; the price is a first launch that
// replays segment 0 (128-column tiles) beside the transitions over K + V
// columns of segments 1 .. P - 2 (2 x 128-column tiles each), a combine of
// P - 2 steps and a replay of segments 1 .. P - 1.  P is the minimum of a
// time model per chunk of the longest pass, counted in waves of a GB300's 152
// SMs (one CTA per SM): 2.2 us for a 64-column tile, 3.1 us for a 128-column
// tile (the first launch's replay of segment 0 bounds that launch; its
// transition tiles take about 2.3 us) and 10 us per launch, fitted to the
// plain state kernel (the lookahead kernels are faster by similar factors in
// every pass), and 3.5 us per step of the tensor-core combine.  On the
// 4096-token, 16-head shape it picks P = 5, the best measured (state stage
// 0.080 ms, against 0.092 ms at P = 4 and 0.086 ms at P = 6).  Segments keep
// at least 8 chunks.
int scan_segments(const gdn2_dims &d) {
    if (d.impl != GDN2_IMPL_TC || d.K != 128 || d.V != 128 || d.N <= 0) return 1;
    if (d.state_segments > 0) return d.state_segments;
    constexpr int64_t kWave = 152;
    const int64_t units = static_cast<int64_t>(d.N) * dims_hs(d);
    const int64_t chunks = d.T_tot / (static_cast<int64_t>(kChunk) * d.N);  // mean per sequence
    auto waves = [](int64_t ctas) { return static_cast<double>((ctas + kWave - 1) / kWave); };
    auto pass = [&](int64_t S) {  // one state pass over S segments per (sequence, head)
        return 2 * units * S <= kWave ? 2.2 * waves(2 * units * S) : 3.1 * waves(units * S);
    };
    double best = 10.0 + chunks * pass(1);
    int best_P = 1;
    for (int64_t P = 2; P <= 16 && chunks >= 8 * P; ++P) {
        // segment 0 beside the transitions of segments 1 .. P - 2 (128
        // columns), P - 2 combine steps, the replay of segments 1 .. P - 1
        const double L = static_cast<double>((chunks + P - 1) / P);
        const double t = (P > 2 ? 3 : 2) * 10.0 + 3.5 * (P - 2) + L * (3.1 * waves(units * (2 * P - 3)) + pass(P - 1));
        if (t < best) {
            best = t;
            best_P = static_cast<int>(P);
        }
    }
    return best_P;
}

WsLayout workspace_layout(const gdn2_dims &d) {
    WsLayout L;
    memset(&L, 0, sizeof(L));
    const size_t T = static_cast<size_t>(d.T_tot), NC = static_cast<size_t>(nc_max(d));
    const size_t HS = static_cast<size_t>(dims_hs(d)), HK = static_cast<size_t>(dims_hk(d));
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t o = off; off += align_up(bytes); return o; };
    L.status = take(64);
    L.chunk_seq = take(NC * 4);
    L.chunk_len = take(NC * 4);
    L.chunk_start = take(NC * 8);
    L.seq_first = take((static_cast<size_t>(d.N) + 1) * 4);
    L.seq_order = take(static_cast<size_t>(d.N) * 4);
    if (d.impl == GDN2_IMPL_SIMT) {
        L.G = take(T * HS * d.K * 4);
        L.qn = take(d.use_qk_l2norm ? T * d.H * d.K * 2 : 0);
        L.kn = take(d.use_qk_l2norm ? T * HK * d.K * 2 : 0);
        L.Wt = take(T * HS * d.K * 2);
        L.Ut = take(T * HS * d.V * 2);
        L.hbuf = take(NC * HS * d.K * d.V * 2);
        L.vnew = take(T * HS * d.V * 2);
    } else {
        off = (off + 1023) & ~static_cast<size_t>(1023);  // records are 1 KB aligned
        L.rec = take(NC * HS * tc_record_bytes(d.K));
        L.exact_list = take(NC * HS * 4);
        const size_t P = static_cast<size_t>(scan_segments(d));
        if (P > 1) {
            const size_t units = static_cast<size_t>(d.N) * (P - 1) * HS;
            L.sc_tr = take(units * d.K * (d.K + d.V) * 4);
            L.sc_si = take(units * d.K * d.V * 4);
            L.sc_mimg = take(units * d.K * d.K * 4);  // hi and lo bf16 parts of M
        }
    }
    L.total = off;
    return L;
}

}  // namespace gdn2

using namespace gdn2;

extern "C" {

int32_t gdn2_version(void) { return (1 << 16) | 1; }

const char *gdn2_status_string(int status) {
    switch (status) {
        case GDN2_OK: return "ok";
        case GDN2_ERR_NULL: return "a required pointer is NULL";
        case GDN2_ERR_SHAPE: return "unsupported sizes (need K == V in {64,128}, key heads equal to query or value heads, query and value heads equal or one a multiple of the other, N >= 0, T_tot >= 0)";
        case GDN2_ERR_STRIDE: return "bad stride or alignment (innermost stride 1; strides and base pointers multiples of 16 bytes)";
        case GDN2_ERR_ALIAS: return "an output overlaps an input (or final_state overlaps initial_state)";
        case GDN2_ERR_WORKSPACE: return "workspace missing or smaller than gdn2_workspace_bytes()";
        case GDN2_ERR_ARCH: return "current CUDA device is not compute capability 10.3 (sm_103a)";
        case GDN2_ERR_LAUNCH: return "kernel launch failed";
        case GDN2_ERR_DTYPE: return "unsupported dtype or layout (q/k/v/beta/w/out bf16 or fp16; g fp32, bf16 or fp16; states fp32 or bf16; the SIMT path: defaults only)";
        case GDN2_ERR_CU_SEQLENS: return "cu_seqlens invalid on the device (cu[0] != 0, decreasing, or cu[N] != T_tot)";
        case GDN2_ERR_CUDA: return "CUDA runtime error";
        case GDN2_ERR_IMPL: return "unknown implementation selector";
        case GDN2_ERR_TIMEOUT: return "a tensor-core kernel timed out waiting on its own pipeline (outputs invalid)";
        case GDN2_ERR_NOALLOC_LIMIT: return "problem needs more scratch than the allocation-free entry point holds (GDN2_NOALLOC_SCRATCH_BYTES)";
        case GDN2_ERR_RANGE: return "a value passed the range of the fp16 intermediates and was clipped (outputs invalid)";
        case GDN2_ERR_BOUNDS: return "an index check of the checked build failed (outputs invalid; a library defect)";
        default: return "unknown status";
    }
}

gdn2_status gdn2_dims_init(gdn2_dims *d, int64_t T_tot, int32_t N, int32_t H, int32_t HV, int32_t K,
                           int32_t V) {
    if (!d) return GDN2_ERR_NULL;
    memset(d, 0, sizeof(*d));
    d->T_tot = T_tot; d->N = N; d->H = H; d->HV = HV; d->K = K; d->V = V;
    d->HK = 0;  // key heads = query heads
    const int64_t HS = H > HV ? H : HV;  // state heads: g, beta, w, out
    d->q_stride[0] = d->k_stride[0] = static_cast<int64_t>(H) * K;
    d->q_stride[1] = d->k_stride[1] = K;
    d->v_stride[0] = static_cast<int64_t>(HV) * V;
    d->w_stride[0] = d->o_stride[0] = HS * V;
    d->v_stride[1] = d->w_stride[1] = d->o_stride[1] = V;
    d->g_stride[0] = d->beta_stride[0] = HS * K;
    d->g_stride[1] = d->beta_stride[1] = K;
    d->dtype_qkv = GDN2_DTYPE_BF16;
    d->dtype_g = GDN2_DTYPE_F32;
    d->impl = GDN2_IMPL_TC;
    d->state_v_major = 0;
    d->dtype_state = GDN2_DTYPE_F32;
    return shape_ok(*d) ? GDN2_OK : GDN2_ERR_SHAPE;
}

size_t gdn2_workspace_bytes(const gdn2_dims *d) {
    if (!d || !shape_ok(*d)) return 0;
    return workspace_layout(*d).total;
}

}  // extern "C"

namespace gdn2 {

gdn2_status check_args(const void *q, const void *k, const void *v, const void *g, const void *beta,
                       const void *w, const void *initial_state, const void *cu_seqlens, const void *out,
                       const void *final_state, const gdn2_dims *d, const void *workspace,
                       size_t workspace_bytes, bool recurrent) {
    if (!d) return GDN2_ERR_NULL;
    if (d->dtype_qkv != GDN2_DTYPE_BF16 && d->dtype_qkv != GDN2_DTYPE_F16) return GDN2_ERR_DTYPE;
    if (d->dtype_g != GDN2_DTYPE_F32 && d->dtype_g != GDN2_DTYPE_BF16 && d->dtype_g != GDN2_DTYPE_F16)
        return GDN2_ERR_DTYPE;
    if (d->dtype_state != GDN2_DTYPE_F32 && d->dtype_state != GDN2_DTYPE_BF16) return GDN2_ERR_DTYPE;
    if (d->state_v_major != 0 && d->state_v_major != 1) return GDN2_ERR_DTYPE;
    if (d->state_segments < 0 || d->state_segments > 64) return GDN2_ERR_SHAPE;
    if (!recurrent && d->state_segments > 1 && (d->impl != GDN2_IMPL_TC || d->K != 128 || d->V != 128))
        return GDN2_ERR_SHAPE;  // the chunk-parallel state pass: tensor-core path, K = V = 128
    if (!recurrent && d->impl != GDN2_IMPL_TC && d->impl != GDN2_IMPL_SIMT) return GDN2_ERR_IMPL;
    if (!recurrent && d->impl == GDN2_IMPL_SIMT &&
        (d->dtype_qkv != GDN2_DTYPE_BF16 || d->dtype_g != GDN2_DTYPE_F32 || d->dtype_state != GDN2_DTYPE_F32 ||
         d->state_v_major != 0))
        return GDN2_ERR_DTYPE;  // the SIMT path supports the default dtypes and layout only
    const size_t g_es = d->dtype_g == GDN2_DTYPE_F32 ? 4 : 2;
    const size_t s_es = d->dtype_state == GDN2_DTYPE_F32 ? 4 : 2;
    if (!shape_ok(*d)) return GDN2_ERR_SHAPE;
    if (!cu_seqlens || !workspace) return GDN2_ERR_NULL;
    if (d->T_tot > 0 && (!q || !k || !v || !out)) return GDN2_ERR_NULL;
    const int64_t T = d->T_tot;
    const int HS = dims_hs(*d), HK = dims_hk(*d);
    if (!strides_ok(q, d->q_stride, 2, d->H, d->K) || !strides_ok(k, d->k_stride, 2, HK, d->K) ||
        !strides_ok(v, d->v_stride, 2, d->HV, d->V) || !strides_ok(w, d->w_stride, 2, HS, d->V) ||
        !strides_ok(beta, d->beta_stride, 2, HS, d->K) || !strides_ok(g, d->g_stride, g_es, HS, d->K) ||
        !strides_ok(out, d->o_stride, 2, HS, d->V))
        return GDN2_ERR_STRIDE;
    if ((initial_state && reinterpret_cast<uintptr_t>(initial_state) % 16) ||
        (final_state && reinterpret_cast<uintptr_t>(final_state) % 16))
        return GDN2_ERR_STRIDE;
    // out rows must not overlap each other
    if (T > 0 && (d->o_stride[1] < d->V || d->o_stride[0] < static_cast<int64_t>(HS - 1) * d->o_stride[1] + d->V))
        return GDN2_ERR_ALIAS;
    const size_t state_bytes = static_cast<size_t>(d->N) * HS * d->K * d->V * s_es;
    const Range r_out = tensor_range(out, T, HS, d->V, d->o_stride, 2);
    const Range r_fs = flat_range(final_state, state_bytes);
    // the recurrent call may update the state in place (the same pointer)
    const bool in_place = recurrent && initial_state && initial_state == final_state;
    const Range ins[] = {
        tensor_range(q, T, d->H, d->K, d->q_stride, 2),     tensor_range(k, T, HK, d->K, d->k_stride, 2),
        tensor_range(v, T, d->HV, d->V, d->v_stride, 2),    tensor_range(w, T, HS, d->V, d->w_stride, 2),
        tensor_range(beta, T, HS, d->K, d->beta_stride, 2), tensor_range(g, T, HS, d->K, d->g_stride, g_es),
        flat_range(cu_seqlens, (static_cast<size_t>(d->N) + 1) * (d->cu_seqlens_i64 ? 8 : 4)),
        flat_range(workspace, workspace_bytes)};
    for (const Range &r : ins)
        if (overlap(r_out, r) || overlap(r_fs, r)) return GDN2_ERR_ALIAS;
    const Range r_is = flat_range(initial_state, state_bytes);
    if (overlap(r_out, r_is) || (!in_place && overlap(r_fs, r_is))) return GDN2_ERR_ALIAS;
    if (overlap(r_out, r_fs)) return GDN2_ERR_ALIAS;
    const size_t need = recurrent ? kRecurrentWorkspaceBytes : workspace_layout(*d).total;
    if (workspace_bytes < need) return GDN2_ERR_WORKSPACE;
    return GDN2_OK;
}

bool pdl_on() {
    const char *e = getenv("GDN2_PDL");
    return !(e && e[0] == '0');
}

bool device_is_sm103(int *dev_out) {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (dev_out) *dev_out = dev;
    return major == 10 && minor == 3;
}

}  // namespace gdn2

namespace gdn2 {
namespace {

// The state-pass V tile the call uses: two 64-column tiles per (sequence,
// head) when the untiled grid would leave more than half of the SMs idle.
// Columns per CTA of the sequential pass or the replay (segs segments per
// sequence): 64 while two such tiles per (sequence, head, segment) fit one
// wave on the SMs.
int state_vtile(const gdn2_dims &d, int segs, int sms) {
    return d.K == 128 && 2ll * d.N * dims_hs(d) * segs <= sms ? 64 : d.K;
}

// The launch sequence of one call as text (what each launch runs and its grid).
int describe_plan(const gdn2_dims &d, int sms, char *buf, size_t len) {
    char tmp[1024];
    const int HS = dims_hs(d);
    const long long NCmax = nc_max(d), items = NCmax * HS;
    int n = snprintf(tmp, sizeof(tmp), "N=%d T_tot=%lld H=%d HK=%d HV=%d (state heads %d) K=V=%d; workspace %zu B; ",
                     d.N, static_cast<long long>(d.T_tot), d.H, dims_hk(d), d.HV, HS, d.K, workspace_layout(d).total);
    auto add = [&](const char *fmt, auto... a) {
        if (n >= 0 && static_cast<size_t>(n) < sizeof(tmp)) n += snprintf(tmp + n, sizeof(tmp) - n, fmt, a...);
    };
    add("%s", "chunk_map 1x1024");
    if (d.N > 0 && d.impl == GDN2_IMPL_SIMT) {
        if (d.use_qk_l2norm && d.T_tot > 0) add("; l2norm %lld warps", static_cast<long long>(d.T_tot) * (d.H + dims_hk(d)));
        add("; cumsum %lldx%d; simt_intra %lldx%d x256; simt_state %dx%dx%d x%d; simt_output %lldx%d x256",
            NCmax, HS, NCmax, HS, d.N, HS, d.K / 32, d.K, NCmax, HS);
    } else if (d.N > 0) {
        const long long grid = items < 2ll * sms ? items : 2ll * sms;
        add("; intra first pass %lld x256 (persistent, 2 CTAs/SM)", grid);
        add("; intra exact pass %lld x256 (programmatic dependent; only with g; runs the listed items)", grid);
        const int P = scan_segments(d);
        const int vt = state_vtile(d, P > 1 ? P - 1 : 1, sms);
        if (d.K == 64) {
            add("; state_output gdn2_tc_state_kernel<64> %dx%d", d.N, HS);
        } else if (P > 1) {
            add("; chunk-parallel state pass, %d segments: segment 0 and the transitions of segments 1-%d "
                "gdn2_tc_state_la128_kernel %lld CTAs of 128 columns",
                P, P - 2, 1ll * d.N * HS * (1 + 2 * (P - 2)));
            if (P > 2) add("; combine %dx%dx8, %d steps", d.N, HS, P - 2);
            add("; replay of segments 1-%d %s %lld CTAs of %d columns", P - 1,
                vt == 64 ? "gdn2_tc_state_la_kernel" : "gdn2_tc_state_la128_kernel", 1ll * d.N * (P - 1) * HS * (128 / vt),
                vt);
        } else {
            add("; state_output %s %lld CTAs of %d columns", vt == 64 ? "gdn2_tc_state_la_kernel" : "gdn2_tc_state_la128_kernel",
                1ll * d.N * HS * (128 / vt), vt);
        }
    }
    if (buf && len > 0) {
        const size_t m = static_cast<size_t>(n) < len - 1 ? static_cast<size_t>(n) : len - 1;
        memcpy(buf, tmp, m);
        buf[m] = 0;
    }
    return n;
}

}  // namespace
}  // namespace gdn2

extern "C" {

int32_t gdn2_launch_plan(const gdn2_dims *d, int32_t sm_count, char *buf, size_t len) {
    if (!d || !shape_ok(*d)) return 0;
    return describe_plan(*d, sm_count > 0 ? sm_count : 152, buf, len);
}

gdn2_status gdn2_check_args(const void *q, const void *k, const void *v, const void *g, const void *beta,
                            const void *w, const void *initial_state, const void *cu_seqlens,
                            const void *out, const void *final_state, const gdn2_dims *d,
                            const void *workspace, size_t workspace_bytes) {
    return check_args(q, k, v, g, beta, w, initial_state, cu_seqlens, out, final_state, d, workspace,
                      workspace_bytes, false);
}

namespace {

const char *const kSimtStages[] = {"prep", "intra", "state", "output"};
constexpr int kNumSimtStages = 4;
const char *const kTcStages[] = {"chunk_map", "intra", "state_output"};
constexpr int kNumTcStages = 3;

gdn2_status run(const void *q, const void *k, const void *v, const void *g, const void *beta, const void *w,
                float scale, const void *initial_state, const void *cu_seqlens, void *out, void *final_state,
                const gdn2_dims *d, void *workspace, size_t workspace_bytes, void *stream,
                void *const *events, int32_t n_events) {
    const gdn2_status st = gdn2_check_args(q, k, v, g, beta, w, initial_state, cu_seqlens, out, final_state,
                                           d, workspace, workspace_bytes);
    if (st != GDN2_OK) return st;
    if (events && n_events < gdn2_num_stages(d) + 1) return GDN2_ERR_NULL;
    int dev = 0;
    if (!device_is_sm103(&dev)) return GDN2_ERR_ARCH;

    const WsLayout L = workspace_layout(*d);
    char *ws = static_cast<char *>(workspace);
    Params p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const bf16 *>(q); p.k = static_cast<const bf16 *>(k); p.v = static_cast<const bf16 *>(v);
    p.beta = static_cast<const bf16 *>(beta); p.w = static_cast<const bf16 *>(w);
    p.g = static_cast<const float *>(g);
    p.sq_t = d->q_stride[0]; p.sq_h = d->q_stride[1];
    p.sk_t = d->k_stride[0]; p.sk_h = d->k_stride[1];
    p.sv_t = d->v_stride[0]; p.sv_h = d->v_stride[1];
    p.sg_t = d->g_stride[0]; p.sg_h = d->g_stride[1];
    p.sb_t = d->beta_stride[0]; p.sb_h = d->beta_stride[1];
    p.sw_t = d->w_stride[0]; p.sw_h = d->w_stride[1];
    p.so_t = d->o_stride[0]; p.so_h = d->o_stride[1];
    p.o = static_cast<bf16 *>(out);
    p.h0 = initial_state; p.hT = final_state;
    p.cu = cu_seqlens; p.cu64 = d->cu_seqlens_i64 ? 1 : 0;
    const int HS = dims_hs(*d), HK = dims_hk(*d);
    p.T_tot = d->T_tot; p.N = d->N; p.H = d->H; p.HK = HK; p.HV = HS; p.K = d->K; p.V = d->V;
    p.gq = HS / d->H; p.gk = HS / HK; p.gv = HS / d->HV;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d->K));
    p.has_g = g != nullptr; p.has_beta = beta != nullptr; p.has_w = w != nullptr;
    p.l2norm = d->use_qk_l2norm ? 1 : 0;
    p.in_f16 = d->dtype_qkv == GDN2_DTYPE_F16;
    p.g_dtype = d->dtype_g;
    p.state_vmajor = d->state_v_major;
    p.state_bf16 = d->dtype_state == GDN2_DTYPE_BF16;
    p.NCmax = static_cast<int>(d->T_tot / kChunk + d->N);
    p.status = reinterpret_cast<int *>(ws + L.status);
    p.chunk_seq = reinterpret_cast<int *>(ws + L.chunk_seq);
    p.chunk_len = reinterpret_cast<int *>(ws + L.chunk_len);
    p.chunk_start = reinterpret_cast<int64_t *>(ws + L.chunk_start);
    p.seq_first = reinterpret_cast<int *>(ws + L.seq_first);
    p.seq_order = reinterpret_cast<int *>(ws + L.seq_order);
    p.G = reinterpret_cast<float *>(ws + L.G);
    p.qn = reinterpret_cast<bf16 *>(ws + L.qn);
    p.kn = reinterpret_cast<bf16 *>(ws + L.kn);
    p.Wt = reinterpret_cast<bf16 *>(ws + L.Wt);
    p.Ut = reinterpret_cast<bf16 *>(ws + L.Ut);
    p.hbuf = reinterpret_cast<bf16 *>(ws + L.hbuf);
    p.vnew = reinterpret_cast<bf16 *>(ws + L.vnew);
    p.rec = reinterpret_cast<uint8_t *>(ws + L.rec);
    p.exact_list = reinterpret_cast<int *>(ws + L.exact_list);
    // State-kernel V tile: V columns of S evolve independently, so splitting V
    // is exact.  Two 64-column tiles per (sequence, head) when the untiled
    // grid would leave more than half of the SMs idle.
    p.sc_P = d->impl == GDN2_IMPL_TC ? scan_segments(*d) : 1;
    p.sc_mode = 0;
    p.sc_tr = p.sc_P > 1 ? reinterpret_cast<float *>(ws + L.sc_tr) : nullptr;
    p.sc_si = p.sc_P > 1 ? reinterpret_cast<float *>(ws + L.sc_si) : nullptr;
    p.sc_mimg = p.sc_P > 1 ? reinterpret_cast<uint8_t *>(ws + L.sc_mimg) : nullptr;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        sms = 0;
    }
    p.vtile = sms > 0 ? state_vtile(*d, p.sc_P > 1 ? p.sc_P - 1 : 1, sms) : d->K;
    const char *log = getenv("GDN2_LOG");
    if (log && log[0] == '1') {  // the launch plan on stderr (diagnostics)
        char plan[1024];
        describe_plan(*d, sms > 0 ? sms : 152, plan, sizeof(plan));
        fprintf(stderr, "gdn2: %s\n", plan);
    }
    // tensor maps for the intra kernel's g / v / w tiles (GDN2_ROW_COPIES=1
    // forces the row-by-row copies)
    if (d->impl == GDN2_IMPL_TC) {
        const char *rows = getenv("GDN2_ROW_COPIES");
        const bool force_rows = rows && rows[0] == '1';
        // 16-bit inputs: the maps only move bytes, so fp16 and bf16 share them
        const CUtensorMapDataType t16 =
            p.in_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapDataType tg = d->dtype_g == GDN2_DTYPE_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : d->dtype_g == GDN2_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const int64_t g_es = d->dtype_g == GDN2_DTYPE_F32 ? 4 : 2;
        p.tmap = !force_rows &&
                 (!p.has_g || encode_rows(&p.tm_g, &p.tm_order_g, g, tg, g_es, d->K, HS, d->T_tot, p.sg_t,
                                          p.sg_h)) &&
                 encode_rows(&p.tm_v, &p.tm_order_v, v, t16, 2, d->V, d->HV, d->T_tot, p.sv_t, p.sv_h) &&
                 (!p.has_w || encode_rows(&p.tm_w, &p.tm_order_w, w, t16, 2, d->V, HS, d->T_tot, p.sw_t, p.sw_h));
        p.tpre = p.tmap &&
                 encode_rows(&p.tm_k, &p.tm_order_k, k, t16, 2, d->K, HK, d->T_tot, p.sk_t, p.sk_h) &&
                 encode_rows(&p.tm_q, &p.tm_order_q, q, t16, 2, d->K, d->H, d->T_tot, p.sq_t, p.sq_h) &&
                 (!p.has_beta ||
                  encode_rows(&p.tm_b, &p.tm_order_b, beta, t16, 2, d->K, HS, d->T_tot, p.sb_t, p.sb_h));
    }
    p.q_in = p.q; p.k_in = p.k;
    p.sq_in_t = p.sq_t; p.sq_in_h = p.sq_h; p.sk_in_t = p.sk_t; p.sk_in_h = p.sk_h;
    if (p.l2norm && d->impl == GDN2_IMPL_SIMT) {  // SIMT kernels read the normalised packed copies
        p.q = p.qn; p.k = p.kn;
        p.sq_t = static_cast<int64_t>(p.H) * p.K;
        p.sk_t = static_cast<int64_t>(p.HK) * p.K;
        p.sq_h = p.sk_h = p.K;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();  // clear a stale error so the checks below see only ours
    int stage = 0;
    auto mark = [&]() {
        if (events) cudaEventRecord(static_cast<cudaEvent_t>(events[stage]), s);
        ++stage;
    };
    mark();
    if (launch_chunk_map(p, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
    if (d->impl == GDN2_IMPL_TC) {
        mark();
        if (p.N > 0 && launch_tc_intra(p, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
        mark();
        if (p.N > 0 && p.sc_P > 1) {  // chunk-parallel: transitions, combine, replay
            Params pt = p;
            pt.sc_mode = 1;
            pt.vtile = 128;
            if (launch_tc_state(pt, s) != cudaSuccess || launch_tc_scan_combine(p, s) != cudaSuccess)
                return GDN2_ERR_LAUNCH;
            Params pr = p;
            pr.sc_mode = 2;
            if (launch_tc_state(pr, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
        } else if (p.N > 0 && launch_tc_state(p, s) != cudaSuccess) {
            return GDN2_ERR_LAUNCH;
        }
        mark();
    } else {
        if (p.N > 0 && launch_prep(p, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
        mark();
        if (p.N > 0 && launch_simt_intra(p, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
        mark();
        if (p.N > 0 && launch_simt_state(p, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
        mark();
        if (p.N > 0 && launch_simt_output(p, s) != cudaSuccess) return GDN2_ERR_LAUNCH;
        mark();
    }
    if (events && cudaGetLastError() != cudaSuccess) return GDN2_ERR_CUDA;
    return GDN2_OK;
}

}  // namespace

int32_t gdn2_num_stages(const gdn2_dims *d) {
    if (!d || !shape_ok(*d)) return 0;
    return d->impl == GDN2_IMPL_SIMT ? kNumSimtStages : kNumTcStages;
}

const char *gdn2_stage_name(const gdn2_dims *d, int32_t i) {
    if (i < 0 || i >= gdn2_num_stages(d)) return nullptr;
    return d->impl == GDN2_IMPL_SIMT ? kSimtStages[i] : kTcStages[i];
}

int32_t gdn2_launch_count(const gdn2_dims *d) {
    if (!d || !shape_ok(*d)) return 0;
    if (d->N == 0) return 1;
    const int64_t ncmax = nc_max(*d);
    if (d->impl != GDN2_IMPL_SIMT) {  // map, intra (two passes), state; segmented: transitions, combine, replay
        const int P = scan_segments(*d);
        return 1 + (ncmax > 0 ? 2 : 0) + 1 + (P > 1 ? 1 : 0) + (P > 2 ? 1 : 0);
    }
    int n = 1;                                          // chunk map
    n += (d->use_qk_l2norm && d->T_tot > 0) ? 1 : 0;    // q/k L2 norm
    n += ncmax > 0 ? 1 : 0;                             // cumsum
    n += ncmax > 0 ? 1 : 0;                             // intra
    n += 1;                                             // state
    n += ncmax > 0 ? 1 : 0;                             // output
    return n;
}

gdn2_status gdn2_chunk_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                           const void *w, float scale, const void *initial_state, const void *cu_seqlens,
                           void *out, void *final_state, const gdn2_dims *d, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return run(q, k, v, g, beta, w, scale, initial_state, cu_seqlens, out, final_state, d, workspace,
               workspace_bytes, stream, nullptr, 0);
}

gdn2_status gdn2_chunk_fwd_staged(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                  const void *w, float scale, const void *initial_state, const void *cu_seqlens,
                                  void *out, void *final_state, const gdn2_dims *d, void *workspace,
                                  size_t workspace_bytes, void *stream, void *const *events, int32_t n_events) {
    if (!events) return GDN2_ERR_NULL;
    return run(q, k, v, g, beta, w, scale, initial_state, cu_seqlens, out, final_state, d, workspace,
               workspace_bytes, stream, events, n_events);
}

gdn2_status gdn2_device_status(const void *workspace, void *stream, int32_t *status) {
    if (!workspace || !status) return GDN2_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status words sit at offset 0 of the workspace: [0] cu_seqlens,
    // [1] chunk count, [2] wait timeout, [3] 16-bit range, [4] exact-list
    // length, [5] failed index check (checked builds)
    int32_t host[6] = {0, 0, 0, 0, 0, 0};
    if (cudaMemcpyAsync(host, workspace, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return GDN2_ERR_CUDA;
    }
    *status = host[0] != GDN2_OK   ? host[0]
              : host[2] != GDN2_OK ? host[2]
              : host[3] != GDN2_OK ? host[3]
              : host[5] != 0       ? static_cast<int32_t>(GDN2_ERR_BOUNDS)
                                   : static_cast<int32_t>(GDN2_OK);
    return GDN2_OK;
}

}  // extern "C"
