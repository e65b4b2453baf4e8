// Token-by-token GDN-2 recurrence from a carried state: decode steps and short
// continuations of a prefill (FlashGDN-2 README quick start: prefill, then
// decode from the returned state; FlashInfer docs, chunk_gated_delta_rule2:
// the per-token recurrence).  Per token t of sequence n and value head hv
// (key head h = hv / (HV / H)):
//   S <- diag(e^{g_t}) S;  u = w_t v_t - S^T (beta_t k_t);  S <- S + k_t u^T;
//   o_t = scale S^T q_t
// The work is a matrix-vector product per token on a state read and written
// once per call, so it runs on CUDA cores and is bound by the state traffic.
//
// One CTA per (sequence, value head, 32-column V tile), K threads: warp w
// holds rows 32w .. 32w + 31 of the tile's columns, lane l column 32 z + l, in
// registers for the whole sequence.  Per token the CTA stages k, beta k, q
// and e^{g} in shared memory, each thread folds the decay, the erase read
// (beta k)^T S and q^T S over its 32 rows, the partial sums meet in shared
// memory, and o uses q^T S_new = q^T S' + (q . k) u.  (Prefetching the next
// token, double-buffered vectors with two barriers per token, and 16-byte
// vector reads were each measured slower for multi-token sequences.)
#include <string.h>

#include "gdn2_internal.cuh"

namespace gdn2 {

namespace {

struct RecParams {
    const bf16 *q, *k, *v, *beta, *w;
    const float *g;
    int64_t sq_t, sq_h, sk_t, sk_h, sv_t, sv_h, sg_t, sg_h, sb_t, sb_h, sw_t, sw_h, so_t, so_h;
    bf16 *o;          // at the inputs' dtype
    const void *h0;   // fp32 or bf16, [K][V] or [V][K] per (sequence, head)
    void *hT;
    const void *cu;
    int cu64;
    int64_t T_tot;
    int N, HV, gq, gk, gv;  // HV: state heads HS; q / k / v head of state head hv: hv / gq, gk, gv
    float scale;
    int has_g, has_beta, has_w, l2norm;
    int in_f16, g_dtype, state_vmajor, state_bf16;
    int *status;  // [0] cu_seqlens status, [1] 0, [2] 0, [3] 0
};

__device__ __forceinline__ int64_t rec_cu(const RecParams &p, int i) {
    return p.cu64 ? static_cast<const int64_t *>(p.cu)[i]
                  : static_cast<int64_t>(static_cast<const int32_t *>(p.cu)[i]);
}

// cu_seqlens checks (cu[0] = 0, non-decreasing, cu[N] = T_tot) into status[0];
// a bad cu_seqlens turns the recurrence kernel into a no-op.
__global__ void __launch_bounds__(256) gdn2_recurrent_check_kernel(RecParams p) {
    __shared__ int bad;
    pdl_trigger();  // the step kernel may launch now; it waits for this one
    if (threadIdx.x == 0) {
        bad = rec_cu(p, 0) != 0 || rec_cu(p, p.N) != p.T_tot;
        p.status[1] = 0;
        p.status[2] = 0;
        p.status[3] = 0;
        p.status[5] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < p.N; i += blockDim.x)
        if (rec_cu(p, i) > rec_cu(p, i + 1)) bad = 1;
    __syncthreads();
    if (threadIdx.x == 0) p.status[0] = bad ? static_cast<int>(GDN2_ERR_CU_SEQLENS) : static_cast<int>(GDN2_OK);
}

// GEN = false: bf16 inputs, fp32 g, fp32 K-major states through plain typed
// loads and stores.  (The dtype-generic helpers cost this instance 4
// registers, one CTA per SM less at K = 128, and 10 % of its time.)
template <int K, bool GEN>
__global__ void __launch_bounds__(K) gdn2_recurrent_kernel(RecParams p) {
    constexpr int W = K / 32;
    const bool f16 = GEN && p.in_f16, vmajor = GEN && p.state_vmajor, sbf16 = GEN && p.state_bf16;
    const int gdt = GEN ? p.g_dtype : static_cast<int>(GDN2_DTYPE_F32);
    auto ld16 = [&](const bf16 *b, int64_t i) { return GEN ? in_ld(b, i, f16) : __bfloat162float(b[i]); };
    __shared__ float s_k[K], s_bk[K], s_q[K], s_eg[K];
    __shared__ float s_part[2][W][32];
    __shared__ float s_red[3][W];
    pdl_wait();  // the check kernel's status is complete
    if (p.status[0] != GDN2_OK) return;
    const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
    const int n = blockIdx.x, hv = blockIdx.y, j = 32 * blockIdx.z + lane;
    const int hk = hv / p.gk, hq = hv / p.gq, hvv = hv / p.gv;  // key, query and value heads
    const int64_t t0 = rec_cu(p, n), t1 = rec_cu(p, n + 1);
    const size_t sbase = (static_cast<size_t>(n) * p.HV + hv) * K * K;  // [N, HV, K, V], K == V

    float S[32];
#pragma unroll
    for (int r = 0; r < 32; ++r)
        S[r] = !p.h0 ? 0.f
               : GEN ? state_ld(p.h0, sbase + state_off(32 * wp + r, j, K, K, vmajor), sbf16)
                     : static_cast<const float *>(p.h0)[sbase + static_cast<size_t>(32 * wp + r) * K + j];
    for (int64_t t = t0; t < t1; ++t) {
        float kc = ld16(p.k, t * p.sk_t + static_cast<int64_t>(hk) * p.sk_h + tid);
        float qc = ld16(p.q, t * p.sq_t + static_cast<int64_t>(hq) * p.sq_h + tid);
        const float bc = p.has_beta ? ld16(p.beta, t * p.sb_t + static_cast<int64_t>(hv) * p.sb_h + tid) : 1.f;
        const float gc = p.has_g ? (GEN ? g_ld(p.g, t * p.sg_t + static_cast<int64_t>(hv) * p.sg_h + tid, gdt)
                                 : p.g[t * p.sg_t + static_cast<int64_t>(hv) * p.sg_h + tid]) : 0.f;
        float a0 = kc * kc, a1 = qc * qc, a2 = qc * kc;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            a0 += __shfl_xor_sync(0xffffffffu, a0, off);
            a1 += __shfl_xor_sync(0xffffffffu, a1, off);
            a2 += __shfl_xor_sync(0xffffffffu, a2, off);
        }
        if (lane == 0) { s_red[0][wp] = a0; s_red[1][wp] = a1; s_red[2][wp] = a2; }
        __syncthreads();
        float kk = 0.f, qq = 0.f, qk = 0.f;
#pragma unroll
        for (int x = 0; x < W; ++x) { kk += s_red[0][x]; qq += s_red[1][x]; qk += s_red[2][x]; }
        if (p.l2norm) {
            const float ik = 1.f / fmaxf(sqrtf(kk), 1e-12f), iq = 1.f / fmaxf(sqrtf(qq), 1e-12f);
            kc *= ik; qc *= iq; qk *= ik * iq;
        }
        s_k[tid] = kc; s_bk[tid] = bc * kc; s_q[tid] = qc; s_eg[tid] = expf(gc);
        const float vj = ld16(p.v, t * p.sv_t + static_cast<int64_t>(hvv) * p.sv_h + j);
        const float wj = p.has_w ? ld16(p.w, t * p.sw_t + static_cast<int64_t>(hv) * p.sw_h + j) : 1.f;
        __syncthreads();
        float pr = 0.f, po = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int c = 32 * wp + r;
            S[r] *= s_eg[c]; pr += s_bk[c] * S[r]; po += s_q[c] * S[r];
        }
        s_part[0][wp][lane] = pr; s_part[1][wp][lane] = po;
        __syncthreads();
        float rj = 0.f, oj = 0.f;
#pragma unroll
        for (int x = 0; x < W; ++x) { rj += s_part[0][x][lane]; oj += s_part[1][x][lane]; }
        const float u = wj * vj - rj;
#pragma unroll
        for (int r = 0; r < 32; ++r) S[r] += s_k[32 * wp + r] * u;
        if (wp == 0) {  // o at the inputs' dtype
            const float ov = p.scale * (oj + qk * u);
            const int64_t oi = t * p.so_t + static_cast<int64_t>(hv) * p.so_h + j;
            if (f16)
                reinterpret_cast<__half *>(p.o)[oi] = __float2half_rn(ov);
            else
                p.o[oi] = __float2bfloat16_rn(ov);
        }
        __syncthreads();
    }
    if (p.hT) {
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if (GEN)
                state_st(p.hT, sbase + state_off(32 * wp + r, j, K, K, vmajor), S[r], sbf16);
            else
                static_cast<float *>(p.hT)[sbase + static_cast<size_t>(32 * wp + r) * K + j] = S[r];
    }
}

}  // namespace

}  // namespace gdn2

using namespace gdn2;

extern "C" {

size_t gdn2_recurrent_workspace_bytes(const gdn2_dims *d) {
    if (!d || !shape_ok(*d)) return 0;
    return kRecurrentWorkspaceBytes;
}

gdn2_status gdn2_recurrent_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                               const void *w, float scale, const void *initial_state, const void *cu_seqlens,
                               void *out, void *final_state, const gdn2_dims *d, void *workspace,
                               size_t workspace_bytes, void *stream) {
    const gdn2_status st = check_args(q, k, v, g, beta, w, initial_state, cu_seqlens, out, final_state, d,
                                      workspace, workspace_bytes, true);
    if (st != GDN2_OK) return st;
    if (!device_is_sm103(nullptr)) return GDN2_ERR_ARCH;
    RecParams p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const bf16 *>(q);
    p.k = static_cast<const bf16 *>(k);
    p.v = static_cast<const bf16 *>(v);
    p.beta = static_cast<const bf16 *>(beta);
    p.w = static_cast<const bf16 *>(w);
    p.g = static_cast<const float *>(g);
    p.sq_t = d->q_stride[0]; p.sq_h = d->q_stride[1];
    p.sk_t = d->k_stride[0]; p.sk_h = d->k_stride[1];
    p.sv_t = d->v_stride[0]; p.sv_h = d->v_stride[1];
    p.sg_t = d->g_stride[0]; p.sg_h = d->g_stride[1];
    p.sb_t = d->beta_stride[0]; p.sb_h = d->beta_stride[1];
    p.sw_t = d->w_stride[0]; p.sw_h = d->w_stride[1];
    p.so_t = d->o_stride[0]; p.so_h = d->o_stride[1];
    p.o = static_cast<bf16 *>(out);
    p.h0 = initial_state;
    p.hT = final_state;
    p.cu = cu_seqlens;
    p.cu64 = d->cu_seqlens_i64 ? 1 : 0;
    p.T_tot = d->T_tot;
    p.N = d->N;
    p.HV = dims_hs(*d);
    p.gq = p.HV / d->H;
    p.gk = p.HV / dims_hk(*d);
    p.gv = p.HV / d->HV;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d->K));
    p.has_g = g != nullptr;
    p.has_beta = beta != nullptr;
    p.has_w = w != nullptr;
    p.l2norm = d->use_qk_l2norm ? 1 : 0;
    p.in_f16 = d->dtype_qkv == GDN2_DTYPE_F16;
    p.g_dtype = d->dtype_g;
    p.state_vmajor = d->state_v_major;
    p.state_bf16 = d->dtype_state == GDN2_DTYPE_BF16;
    p.status = static_cast<int *>(workspace);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    gdn2_recurrent_check_kernel<<<1, 256, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return GDN2_ERR_LAUNCH;
    if (d->N > 0) {
        const dim3 grid(d->N, p.HV, d->V / 32);
        const bool gen = p.in_f16 || p.g_dtype != GDN2_DTYPE_F32 || p.state_vmajor || p.state_bf16;
        const cudaError_t e =
            d->K == 64
                ? launch_chained(gen ? gdn2_recurrent_kernel<64, true> : gdn2_recurrent_kernel<64, false>, grid,
                                 dim3(64), 0, s, p)
                : launch_chained(gen ? gdn2_recurrent_kernel<128, true> : gdn2_recurrent_kernel<128, false>, grid,
                                 dim3(128), 0, s, p);
        if (e != cudaSuccess) return GDN2_ERR_LAUNCH;
    }
    return GDN2_OK;
}

}  // extern "C"
