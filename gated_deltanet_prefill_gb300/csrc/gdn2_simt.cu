// CUDA-core (fp32 FMA) kernels of the chunked GDN-2 forward.
//
// This is the same chunked WY algorithm as the tensor-core path, with every
// contraction done in fp32 on CUDA cores: a second GPU implementation used to
// cross-check the tensor-core kernels.  It is selected explicitly
// (GDN2_IMPL_SIMT) and is never a fallback.
//
// Chunk algebra (unrolling the FlashInfer docs' recurrence over one 64-token
// chunk with incoming state S0, G_t = chunk-local inclusive cumsum of g):
//   A_ts = sum_c beta_t[c] k_t[c] e^{G_t[c]-G_s[c]} k_s[c]   (s < t)
//   T    = (I + A)^{-1}
//   Wt   = T (beta * k * e^G),   Ut = T (w * v)             (WY pseudo-keys/values)
//   U    = Ut - Wt S0                                       (u_t of every token)
//   O    = scale [ (q * e^G) S0 + P U ],  P_ts = sum_c q_t e^{G_t-G_s} k_s  (s <= t)
//   S_C  = diag(e^{G_L}) S0 + (k * e^{G_L - G})^T U         (L = last row)
// Decay factors e^{G_t - G_s} are split through 16-token sub-chunk references
// (burn-gdn2 README, "Numerical stability"): for column sub-chunk J with last
// row E_J and rows t below sub-chunk J, e^{G_t-G_s} = e^{G_t-G_{E_J}} *
// e^{G_{E_J}-G_s}, both factors <= 1.  Pairs inside one sub-chunk take
// e^{G_t-G_s} <= 1 directly, so no factor exceeds 1 for any g <= 0.
#include "gdn2_internal.cuh"

namespace gdn2 {

namespace {

constexpr int kIntraThreads = 256;
constexpr int kOutThreads = 256;

__device__ __forceinline__ int sub_end(int r, int len) {  // last row of r's sub-chunk
    return min((r / kSub) * kSub + kSub - 1, len - 1);
}

// ---------------------------------------------------------------------------
// Intra-chunk: A, T = (I + A)^{-1}, Wt, Ut.  One CTA per (chunk, value head).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kIntraThreads) gdn2_simt_intra_kernel(Params p) {
    constexpr int LD = D + 1;
    extern __shared__ float sm[];
    float *Gs = sm;               // [64][LD] G
    float *Ks = Gs + 64 * LD;     // [64][LD] k, later w * v
    float *Bs = Ks + 64 * LD;     // [64][LD] beta
    float *Rs = Bs + 64 * LD;     // [64][LD] right factor k e^{G_E - G}
    float *Ls = Rs + 64 * LD;     // [64][LD] left factor, later beta k e^G
    float *As = Ls + 64 * LD;     // [64][65]
    float *Ts = As + 64 * 65;     // [64][65]

    const int c = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
    const int seq = p.chunk_seq[c];
    if (seq < 0) return;
    const int64_t start = p.chunk_start[c];
    const int len = p.chunk_len[c];
    const int h = hv / p.gk;  // key head

    for (int i = tid; i < 64 * D; i += kIntraThreads) {
        const int r = i / D, ch = i % D;
        const int rr = min(r, len - 1);
        const int64_t t = start + rr;
        Gs[r * LD + ch] = p.G[(t * p.HV + hv) * D + ch];
        float kv = 0.f, bv = 0.f;
        if (r < len) {
            kv = __bfloat162float(p.k[t * p.sk_t + h * p.sk_h + ch]);
            bv = p.has_beta ? __bfloat162float(p.beta[t * p.sb_t + hv * p.sb_h + ch]) : 1.f;
        }
        Ks[r * LD + ch] = kv;
        Bs[r * LD + ch] = bv;
    }
    for (int i = tid; i < 64 * 65; i += kIntraThreads) As[i] = 0.f;
    __syncthreads();
    for (int i = tid; i < 64 * D; i += kIntraThreads) {
        const int r = i / D, ch = i % D;
        const int e = sub_end(r, len);
        Rs[r * LD + ch] = Ks[r * LD + ch] * __expf(Gs[e * LD + ch] - Gs[r * LD + ch]);
    }
    __syncthreads();
    for (int J = 0; J < kNumSub && J * kSub < len; ++J) {
        const int e = min(J * kSub + kSub - 1, len - 1);
        for (int i = tid; i < 64 * D; i += kIntraThreads) {
            const int r = i / D, ch = i % D;
            float x = 0.f;
            if (r > e && r < len)
                x = Bs[r * LD + ch] * Ks[r * LD + ch] * __expf(Gs[r * LD + ch] - Gs[e * LD + ch]);
            Ls[r * LD + ch] = x;
        }
        __syncthreads();
        for (int i = tid; i < 64 * kSub; i += kIntraThreads) {
            const int t = i / kSub, s = J * kSub + i % kSub;
            if (s < t && t < len) {
                float acc = 0.f;
                if (t > e) {
#pragma unroll 8
                    for (int ch = 0; ch < D; ++ch) acc += Ls[t * LD + ch] * Rs[s * LD + ch];
                } else {  // same sub-chunk: the decay of each pair directly
#pragma unroll 8
                    for (int ch = 0; ch < D; ++ch)
                        acc += Bs[t * LD + ch] * Ks[t * LD + ch] * Ks[s * LD + ch] *
                               __expf(Gs[t * LD + ch] - Gs[s * LD + ch]);
                }
                As[t * 65 + s] = acc;
            }
        }
        __syncthreads();
    }
    // forward substitution, one thread per column of T: T = (I + A)^{-1}
    if (tid < 64) {
        const int col = tid;
        for (int i = 0; i < 64; ++i) {
            float x = (i == col) ? 1.f : 0.f;
            for (int j = col; j < i; ++j) x -= As[i * 65 + j] * Ts[j * 65 + col];
            Ts[i * 65 + col] = x;
        }
    }
    // X1 = beta k e^G (into Ls), X2 = w v (into Ks)
    for (int i = tid; i < 64 * D; i += kIntraThreads) {
        const int r = i / D, ch = i % D;
        float x1 = 0.f, x2 = 0.f;
        if (r < len) {
            const int64_t t = start + r;
            x1 = Bs[r * LD + ch] * Ks[r * LD + ch] * __expf(Gs[r * LD + ch]);
            const float vv = __bfloat162float(p.v[t * p.sv_t + static_cast<int64_t>(hv / p.gv) * p.sv_h + ch]);
            const float ww = p.has_w ? __bfloat162float(p.w[t * p.sw_t + hv * p.sw_h + ch]) : 1.f;
            x2 = ww * vv;
        }
        Ls[r * LD + ch] = x1;
        Ks[r * LD + ch] = x2;
    }
    __syncthreads();
    {
        constexpr int RSTEP = kIntraThreads / D;
        const int ch = tid % D;
        for (int t = tid / D; t < len; t += RSTEP) {
            float a1 = 0.f, a2 = 0.f;
            for (int s = 0; s <= t; ++s) {
                const float tv = Ts[t * 65 + s];
                a1 += tv * Ls[s * LD + ch];
                a2 += tv * Ks[s * LD + ch];
            }
            const int64_t row = (start + t) * p.HV + hv;
            p.Wt[row * D + ch] = __float2bfloat16(a1);
            p.Ut[row * D + ch] = __float2bfloat16(a2);
        }
    }
}

// ---------------------------------------------------------------------------
// State passing: sequential over the chunks of one sequence.  One CTA per
// (sequence, value head, 32-column V tile); thread c owns row c of S.
// Writes the state entering each chunk (bf16), u_t (bf16), final state (fp32).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) gdn2_simt_state_kernel(Params p) {
    constexpr int VT = 32;
    constexpr int LD = D + 1;
    extern __shared__ float sm[];
    float *Ss = sm;                // [D][VT + 1]
    float *Ws = Ss + D * (VT + 1); // [64][LD]
    float *Us = Ws + 64 * LD;      // [64][VT + 1]

    if (p.status[0] != GDN2_OK) return;
    const int n = blockIdx.x, hv = blockIdx.y, v0 = blockIdx.z * VT, c = threadIdx.x;
    const int h = hv / p.gk;  // key head
    float S[VT];
    const size_t sbase = ((static_cast<size_t>(n) * p.HV + hv) * D + c) * D + v0;
#pragma unroll
    for (int j = 0; j < VT; ++j) S[j] = p.h0 ? static_cast<const float *>(p.h0)[sbase + j] : 0.f;  // fp32, K-major

    const int first = p.seq_first[n], last = p.seq_first[n + 1];
    for (int ck = first; ck < last; ++ck) {
        const int64_t start = p.chunk_start[ck];
        const int len = p.chunk_len[ck];
        bf16 *hp = p.hbuf + ((static_cast<size_t>(ck) * p.HV + hv) * D + c) * D + v0;
#pragma unroll
        for (int j = 0; j < VT; ++j) {
            hp[j] = __float2bfloat16(S[j]);
            Ss[c * (VT + 1) + j] = S[j];
        }
        for (int i = c; i < 64 * D; i += D) {
            const int r = i / D, cc = i % D;
            Ws[r * LD + cc] = r < len ? __bfloat162float(p.Wt[((start + r) * p.HV + hv) * D + cc]) : 0.f;
        }
        __syncthreads();
        for (int e = c; e < 64 * VT; e += D) {
            const int t = e / VT, j = e % VT;
            if (t < len) {
                const int64_t row = (start + t) * p.HV + hv;
                float acc = __bfloat162float(p.Ut[row * D + v0 + j]);
#pragma unroll 8
                for (int cc = 0; cc < D; ++cc) acc -= Ws[t * LD + cc] * Ss[cc * (VT + 1) + j];
                Us[t * (VT + 1) + j] = acc;
                p.vnew[row * D + v0 + j] = __float2bfloat16(acc);
            }
        }
        __syncthreads();
        const float GL = p.G[((start + len - 1) * p.HV + hv) * D + c];
        const float a = __expf(GL);
#pragma unroll
        for (int j = 0; j < VT; ++j) S[j] *= a;
        for (int t = 0; t < len; ++t) {
            const int64_t tok = start + t;
            const float kd = __bfloat162float(p.k[tok * p.sk_t + h * p.sk_h + c]) *
                             __expf(GL - p.G[(tok * p.HV + hv) * D + c]);
#pragma unroll
            for (int j = 0; j < VT; ++j) S[j] += kd * Us[t * (VT + 1) + j];
        }
        __syncthreads();
    }
    if (p.hT) {
#pragma unroll
        for (int j = 0; j < VT; ++j) static_cast<float *>(p.hT)[sbase + j] = S[j];
    }
}

// ---------------------------------------------------------------------------
// Output: O = scale [ (q e^G) S_chunk + P U ].  One CTA per (chunk, value head).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kOutThreads) gdn2_simt_output_kernel(Params p) {
    constexpr int LD = D + 1;
    extern __shared__ float sm[];
    float *Gs = sm;               // [64][LD]   } reused together as Hs [D][LD]
    float *Rs = Gs + 64 * LD;     // [64][LD]   }
    float *Qs = Rs + 64 * LD;     // [64][LD] q
    float *Ls = Qs + 64 * LD;     // [64][LD] left factor, later q e^G
    float *Us = Ls + 64 * LD;     // [64][LD] u
    float *Ps = Us + 64 * LD;     // [64][65]
    float *Hs = sm;               // [D][LD]
    static_assert(2 * 64 >= D, "Hs must fit in the G and R buffers");

    const int c = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
    const int seq = p.chunk_seq[c];
    if (seq < 0) return;
    const int64_t start = p.chunk_start[c];
    const int len = p.chunk_len[c];
    const int h = hv / p.gk, hq = hv / p.gq;  // key and query heads

    for (int i = tid; i < 64 * D; i += kOutThreads) {
        const int r = i / D, ch = i % D;
        const int64_t t = start + min(r, len - 1);
        Gs[r * LD + ch] = p.G[(t * p.HV + hv) * D + ch];
        Rs[r * LD + ch] = r < len ? __bfloat162float(p.k[t * p.sk_t + h * p.sk_h + ch]) : 0.f;
        Qs[r * LD + ch] = r < len ? __bfloat162float(p.q[t * p.sq_t + hq * p.sq_h + ch]) : 0.f;
    }
    for (int i = tid; i < 64 * 65; i += kOutThreads) Ps[i] = 0.f;
    __syncthreads();
    // pairs inside one sub-chunk (s <= t): the decay of each pair directly,
    // from the raw k rows
    for (int i = tid; i < 64 * kSub; i += kOutThreads) {
        const int t = i / kSub, s = (t / kSub) * kSub + i % kSub;
        if (s <= t && t < len) {
            float acc = 0.f;
#pragma unroll 8
            for (int ch = 0; ch < D; ++ch)
                acc += Qs[t * LD + ch] * Rs[s * LD + ch] * __expf(Gs[t * LD + ch] - Gs[s * LD + ch]);
            Ps[t * 65 + s] = acc;
        }
    }
    __syncthreads();
    for (int i = tid; i < 64 * D; i += kOutThreads) {
        const int r = i / D, ch = i % D;
        const int e = sub_end(r, len);
        Rs[r * LD + ch] *= __expf(Gs[e * LD + ch] - Gs[r * LD + ch]);
    }
    __syncthreads();
    for (int J = 0; J < kNumSub && J * kSub < len; ++J) {
        const int e = min(J * kSub + kSub - 1, len - 1);
        for (int i = tid; i < 64 * D; i += kOutThreads) {
            const int r = i / D, ch = i % D;
            float x = 0.f;
            if (r > e && r < len) x = Qs[r * LD + ch] * __expf(Gs[r * LD + ch] - Gs[e * LD + ch]);
            Ls[r * LD + ch] = x;
        }
        __syncthreads();
        for (int i = tid; i < 64 * kSub; i += kOutThreads) {
            const int t = i / kSub, s = J * kSub + i % kSub;
            if (t > e && t < len) {  // rows below sub-chunk J
                float acc = 0.f;
#pragma unroll 8
                for (int ch = 0; ch < D; ++ch) acc += Ls[t * LD + ch] * Rs[s * LD + ch];
                Ps[t * 65 + s] = acc;
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < 64 * D; i += kOutThreads) {
        const int r = i / D, ch = i % D;
        Ls[r * LD + ch] = Qs[r * LD + ch] * __expf(Gs[r * LD + ch]);
    }
    __syncthreads();  // G and R are dead: load the chunk state over them
    const bf16 *hp = p.hbuf + (static_cast<size_t>(c) * p.HV + hv) * D * D;
    for (int i = tid; i < D * D; i += kOutThreads) Hs[(i / D) * LD + i % D] = __bfloat162float(hp[i]);
    for (int i = tid; i < 64 * D; i += kOutThreads) {
        const int r = i / D, j = i % D;
        Us[r * LD + j] = r < len ? __bfloat162float(p.vnew[((start + r) * p.HV + hv) * D + j]) : 0.f;
    }
    __syncthreads();
    constexpr int RSTEP = kOutThreads / D;
    const int j = tid % D;
    for (int t = tid / D; t < len; t += RSTEP) {
        float acc = 0.f;
#pragma unroll 8
        for (int ch = 0; ch < D; ++ch) acc += Ls[t * LD + ch] * Hs[ch * LD + j];
        for (int s = 0; s <= t; ++s) acc += Ps[t * 65 + s] * Us[s * LD + j];
        const int64_t tok = start + t;
        p.o[tok * p.so_t + hv * p.so_h + j] = __float2bfloat16(acc * p.scale);
    }
}

template <int D>
cudaError_t launch_intra_d(const Params &p, cudaStream_t s) {
    const size_t smem = (5 * 64 * (D + 1) + 2 * 64 * 65) * sizeof(float);
    cudaFuncSetAttribute(gdn2_simt_intra_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (p.NCmax > 0) gdn2_simt_intra_kernel<D><<<dim3(p.NCmax, p.HV), kIntraThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_state_d(const Params &p, cudaStream_t s) {
    const size_t smem = (D * 33 + 64 * (D + 1) + 64 * 33) * sizeof(float);
    cudaFuncSetAttribute(gdn2_simt_state_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (p.N > 0) gdn2_simt_state_kernel<D><<<dim3(p.N, p.HV, D / 32), D, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_output_d(const Params &p, cudaStream_t s) {
    const size_t smem = (5 * 64 * (D + 1) + 64 * 65) * sizeof(float);
    cudaFuncSetAttribute(gdn2_simt_output_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (p.NCmax > 0) gdn2_simt_output_kernel<D><<<dim3(p.NCmax, p.HV), kOutThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_intra(const Params &p, cudaStream_t s) {
    return p.K == 64 ? launch_intra_d<64>(p, s) : launch_intra_d<128>(p, s);
}
cudaError_t launch_simt_state(const Params &p, cudaStream_t s) {
    return p.K == 64 ? launch_state_d<64>(p, s) : launch_state_d<128>(p, s);
}
cudaError_t launch_simt_output(const Params &p, cudaStream_t s) {
    return p.K == 64 ? launch_output_d<64>(p, s) : launch_output_d<128>(p, s);
}

}  // namespace gdn2
