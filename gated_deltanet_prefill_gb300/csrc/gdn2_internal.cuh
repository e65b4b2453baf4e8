// Internal declarations shared by the library's translation units.
// Not part of the public ABI (that is include/gdn2.h).
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn2.h"

namespace gdn2 {

constexpr int kChunk = 64;     // WY chunk length (FlashRT "64-token WY blocks")
constexpr int kSub = 16;       // sub-chunk length for decay re-referencing (burn-gdn2)
constexpr int kNumSub = kChunk / kSub;

using bf16 = __nv_bfloat16;

// Everything a kernel needs, passed by value.  Token-major tensors carry
// element strides (token, head); the channel stride is 1.
struct Params {
    // q, k: what the chunk kernels read.  With the fused L2 norm these point
    // at the normalised copies in the workspace (packed [T_tot, H, K]) and
    // q_in / k_in hold the caller's tensors for the norm kernel.
    const bf16 *q, *k, *v, *beta, *w;
    const bf16 *q_in, *k_in;
    int64_t sq_in_t, sq_in_h, sk_in_t, sk_in_h;
    const float *g;
    int64_t sq_t, sq_h, sk_t, sk_h, sv_t, sv_h, sg_t, sg_h, sb_t, sb_h, sw_t, sw_h, so_t, so_h;
    bf16 *o;                    // dtype of the inputs (in_f16: the bits are fp16)
    const void *h0;             // states: fp32 or bf16 (state_bf16), [K][V] per
    void *hT;                   // (sequence, value head) or [V][K] (state_vmajor)
    const void *cu;
    int cu64;
    int64_t T_tot;
    // Heads: H query heads, HK key heads, and HV here counts the STATE heads
    // HS = max(H, value heads) (g, beta, w, the states and the output are per
    // state head).  State head hv reads q head hv / gq, k head hv / gk and v
    // head hv / gv (gq = HS / H, gk = HS / HK, gv = HS / value heads).
    int N, H, HK, HV, K, V;
    int gq, gk, gv;
    float scale;
    int has_g, has_beta, has_w, l2norm;
    int in_f16;                 // q, k, v, beta, w, out are fp16 (else bf16)
    int g_dtype;                // gdn2_dtype of g
    int state_vmajor, state_bf16;
    int NCmax;                  // upper bound on the chunk count: T_tot/64 + N
    // ---- workspace ----
    int *status;                // [0] cu_seqlens status, [1] chunk count NC, [2] wait timeout,
                                // [3] 16-bit range, [4] length of exact_list,
                                // [5] first failed index check (checked builds)
    int *chunk_seq;             // [NCmax]  sequence of chunk c, -1 past NC
    int *chunk_len;             // [NCmax]  tokens in chunk c (1..64)
    int64_t *chunk_start;       // [NCmax]  first token of chunk c
    int *seq_first;             // [N + 1]  first chunk of sequence n; [N] = NC
    int *seq_order;             // [N]      sequences by chunk count, longest first
    float *G;                   // [T_tot, HV, K]  chunk-local inclusive cumsum of g
    bf16 *qn, *kn;              // [T_tot, H, K], [T_tot, HK, K]  L2-normalised q, k (l2norm only)
    bf16 *Wt, *Ut;              // [T_tot, HV, K], [T_tot, HV, V]  WY pseudo-keys / values
    bf16 *hbuf;                 // [NCmax, HV, K, V] state entering each chunk (bf16)
    bf16 *vnew;                 // [T_tot, HV, V]  u_t (v_new) per token
    uint8_t *rec;               // [NCmax, HV] records of the tensor-core path
    int *exact_list;            // [NCmax * HV] items (c * HV + hv) for the intra kernel's exact pass
    int vtile;                  // V columns per state CTA (tensor-core path)
    // chunk-parallel state pass (tensor-core path, K = V = 128): each sequence's
    // chunks in sc_P segments.  sc_mode 0: one sequential pass (sc_P = 1);
    // 1: segment 0 replayed from the initial state, its final state into
    // sc_si [N, P-1, HV, K, V] unit 0, and the transitions [M | B] of
    // S_out = M S_in + B for segments 1 .. P-2 into sc_tr [N, P-1, HV, K, K+V]
    // (unit 0 unused); the combine fills sc_si units 1 .. P-2 (sc_si unit s is
    // the incoming state of segment s + 1); 2: segments 1 .. P-1 from their
    // incoming states.
    // sc_mimg [N, P-1, HV]: each transition's M split into bf16 hi and lo parts,
    // as K-major 128B-swizzled operand images (64 KB each; written by the
    // lookahead transitions, read by the tensor-core combine)
    int sc_P, sc_mode;
    float *sc_tr, *sc_si;
    uint8_t *sc_mimg;
    // TMA tensor maps over the rows of g, v, w (tensor-core intra kernel): a
    // box is 64 tokens x D channels of one head.  tm_order = 0: coordinates
    // (channel, head, token); 1: (channel, token, head).  tmap = 0: the maps
    // are not set and the kernel copies the rows one by one.
    CUtensorMap tm_g, tm_v, tm_w;
    int tmap;
    int tm_order_g, tm_order_v, tm_order_w;
    // maps over k, q (key heads) and beta (value heads) with the same box,
    // used only to prefetch the next item's tiles into L2 (tpre = 0: none)
    CUtensorMap tm_k, tm_q, tm_b;
    int tpre;
    int tm_order_k, tm_order_q, tm_order_b;
};

// The CTAs of one state launch, grouped by (sequence rank in the
// longest-first order, state head), `per` CTAs per group, the group's CTAs
// adjacent.  rt = V / VT column tiles cover one segment's state; a transition
// covers the K + V columns of [M | B] in 2 rt tiles.  sc_mode 0 (the
// sequential pass): rt tiles of the one segment.  sc_mode 1 (transitions):
// segment 0 runs as a replay from the initial state (rt tiles; its final state
// is the incoming state of segment 1), then 2 rt transition tiles for each of
// segments 1 .. P - 2.  sc_mode 2 (replay): rt tiles for each of segments
// 1 .. P - 1.
__host__ __device__ inline int scan_ctas_per_group(int mode, int P, int rt) {
    return mode == 1 ? rt + 2 * rt * (P - 2) : mode == 2 ? rt * (P - 1) : rt;
}
struct ScanCta {
    int rank, hv, seg, tile;
    bool trans;  // a transition tile (its tile indexes the 2 rt tiles of [M | B])
};
__host__ __device__ __forceinline__ ScanCta scan_cta(int b, int mode, int P, int HV, int rt) {
    const int per = scan_ctas_per_group(mode, P, rt);
    const int x = b % per, grp = b / per;
    ScanCta c;
    c.hv = grp % HV;
    c.rank = grp / HV;
    c.trans = mode == 1 && x >= rt;
    if (c.trans) {
        c.seg = 1 + (x - rt) / (2 * rt);
        c.tile = (x - rt) % (2 * rt);
    } else if (mode == 2) {
        c.seg = 1 + x / rt;
        c.tile = x % rt;
    } else {
        c.seg = 0;
        c.tile = x;
    }
    return c;
}

// Workspace layout (byte offsets), a function of the problem only.
struct WsLayout {
    size_t status, chunk_seq, chunk_len, chunk_start, seq_first, seq_order, G, qn, kn, Wt, Ut, hbuf, vnew, rec,
        exact_list, sc_tr, sc_si, sc_mimg;
    size_t total;
};

WsLayout workspace_layout(const gdn2_dims &d);

// Workspace of the recurrent (decode) call: the status words only.
constexpr size_t kRecurrentWorkspaceBytes = 64;

// Host-side argument checks shared by the chunked and the recurrent calls
// (the recurrent one allows initial_state == final_state and needs only
// kRecurrentWorkspaceBytes of workspace).
gdn2_status check_args(const void *q, const void *k, const void *v, const void *g, const void *beta,
                       const void *w, const void *initial_state, const void *cu_seqlens, const void *out,
                       const void *final_state, const gdn2_dims *d, const void *workspace,
                       size_t workspace_bytes, bool recurrent);
// Head counts of a problem: key heads (dims.HK, 0 = H) and state heads
// HS = max(H, HV), one state per state head.
inline int dims_hk(const gdn2_dims &d) { return d.HK > 0 ? d.HK : d.H; }
inline int dims_hs(const gdn2_dims &d) { return d.H > d.HV ? d.H : d.HV; }
// True if the current device is compute capability 10.3 (its index in *dev).
bool device_is_sm103(int *dev);
// Shapes the library supports (K = V in {64, 128}, HK equal to H or HV, H and
// HV equal or one a multiple of the other, ...).
bool shape_ok(const gdn2_dims &d);

// One element of a 16-bit input (bf16, or fp16 when f16) as fp32.
__device__ __forceinline__ float in_ld(const bf16 *base, int64_t i, bool f16) {
    const unsigned short b = reinterpret_cast<const unsigned short *>(base)[i];
    return f16 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}
// One element of g (fp32, bf16 or fp16) as fp32.
__device__ __forceinline__ float g_ld(const float *base, int64_t i, int dtype) {
    if (dtype == GDN2_DTYPE_F32) return base[i];
    const unsigned short b = reinterpret_cast<const unsigned short *>(base)[i];
    return dtype == GDN2_DTYPE_F16 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}
// Offset of element (key channel c, value channel j) in one (sequence, head)
// state block: [K][V] (K-major) or [V][K] (V-major).
__device__ __forceinline__ size_t state_off(int c, int j, int K, int V, bool vmajor) {
    return vmajor ? static_cast<size_t>(j) * K + c : static_cast<size_t>(c) * V + j;
}
__device__ __forceinline__ float state_ld(const void *base, size_t i, bool is_bf16) {
    return is_bf16 ? __bfloat162float(static_cast<const bf16 *>(base)[i]) : static_cast<const float *>(base)[i];
}
__device__ __forceinline__ void state_st(void *base, size_t i, float x, bool is_bf16) {
    if (is_bf16)
        static_cast<bf16 *>(base)[i] = __float2bfloat16_rn(x);
    else
        static_cast<float *>(base)[i] = x;
}

// Checked builds (compiled with -DGDN2_CHECK_BOUNDS, build.py's checked
// library): device-side index checks.  An index outside [lo, hi) is recorded
// in status word 5 (the site of the first failure) and clamped into range, so
// the access it guards stays inside its buffer and the control flow is that
// of the normal build; gdn2_device_status then reports GDN2_ERR_BOUNDS.
// Normal builds compile the checks away.
template <typename T>
__device__ __forceinline__ T chk(T x, T lo, T hi, int site, int *status) {
#ifdef GDN2_CHECK_BOUNDS
    if (x < lo || x >= hi) {
        atomicCAS(status + 5, 0, site);
        return x < lo ? lo : hi - 1;
    }
#else
    (void)lo; (void)hi; (void)site; (void)status;
#endif
    return x;
}

// Status word 3 of the workspace: a kernel converted a value past the range of
// its 16-bit intermediates (the conversion clipped it); gdn2_device_status
// reports GDN2_ERR_RANGE.
__device__ __forceinline__ void report_range(int *status, bool clipped) {
    if (clipped) atomicExch(status + 3, static_cast<int>(GDN2_ERR_RANGE));
}

__device__ __forceinline__ int64_t cu_at(const Params &p, int i) {
    return p.cu64 ? static_cast<const int64_t *>(p.cu)[i]
                  : static_cast<int64_t>(static_cast<const int32_t *>(p.cu)[i]);
}

// Programmatic dependent launches.  A forward call is a chain of kernels in
// one stream; each kernel after the first is launched with the programmatic
// serialization attribute, so it may be scheduled while its predecessor
// drains and the launch gap between them disappears.  Every kernel of a chain
// executes pdl_wait() in every thread before its first global access: the
// wait returns once the predecessor grid has completed and its writes are
// visible, and since the predecessor waited the same way, so have all earlier
// kernels of the chain.  pdl_trigger() allows the successor to be launched
// before this grid ends.  Both are no-ops for a kernel launched without the
// attribute.  GDN2_PDL=0 launches every kernel plainly (for comparison).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
bool pdl_on();
// Launch kern(p) as the next kernel of a chain (see above).
template <typename P>
cudaError_t launch_chained(void (*kern)(P), dim3 grid, dim3 block, size_t smem, cudaStream_t s, const P &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_on() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Launchers (each returns cudaGetLastError() of its launches).
cudaError_t launch_chunk_map(const Params &p, cudaStream_t s);
cudaError_t launch_prep(const Params &p, cudaStream_t s);
cudaError_t launch_simt_intra(const Params &p, cudaStream_t s);
cudaError_t launch_simt_state(const Params &p, cudaStream_t s);
cudaError_t launch_simt_output(const Params &p, cudaStream_t s);
cudaError_t launch_tc_intra(const Params &p, cudaStream_t s);
cudaError_t launch_tc_state(const Params &p, cudaStream_t s);
cudaError_t launch_tc_state_la(const Params &p, cudaStream_t s);
cudaError_t launch_tc_state_la128(const Params &p, cudaStream_t s);
cudaError_t launch_tc_scan_combine(const Params &p, cudaStream_t s);
// Segments per sequence of the chunk-parallel state pass for `d` (1 = none).
int scan_segments(const gdn2_dims &d);
size_t tc_record_bytes(int D);

}  // namespace gdn2
