// Tensor-core intra-chunk kernel: everything of a 64-token chunk that does
// not depend on the incoming state, written as the record the state kernel
// consumes (gdn2_record.cuh).  One CTA per (chunk, value head), 256 threads,
// two CTAs per SM.
//
// Steps (FlashRT gated-delta-attention page: norm/cumsum, kkt, solve_tril,
// recompute_wu; here fused into one kernel, GDN-2 channel-wise gates):
//  1. load k, q (key head), v, w, beta, g (value head); optional q/k L2 norm;
//     G = chunk-local inclusive cumsum of g.
//  2. decay factors through 16-token sub-chunk references (burn-gdn2 README,
//     "Numerical stability"): with B_I the row before sub-chunk I and E_J the
//     last row of sub-chunk J,
//        e^{G_t - G_s} = F_t * m_{I,J} * eR_s,   F_t = e^{G_t - G_{B_I}} <= 1,
//        eR_s = e^{G_{E_J} - G_s} <= 1, m_{I,J} = e^{G_{B_I} - G_{E_J}}
//     (m <= 1 for J < I; m = e^{+decay of sub-chunk I} for J = I).  Every m is
//     a product of the per-sub-chunk decays ge_J = e^{G_{E_J} - G_{E_{J-1}}}.
//  3. tcgen05: for each row block I, [beta k F ; q F] (M=128) x R_I^T where
//     R_I = k eR m_{I,.} (N = 16(I+1)): rows of block I give A (strict lower)
//     and P (lower incl. diagonal).
//  4. T = (I + A)^{-1} by blocked forward substitution in fp32 (16x16
//     diagonal blocks, then off-diagonal blocks level by level).
//  5. tcgen05: [Wt | Ut] = T x [beta k e^G | w v]  (M=128, N=2D, K=64).
//  6. write Qe, Kd^T, P, Wt, Ut, eGL as shared-memory images.
#include "gdn2_internal.cuh"
#include "gdn2_record.cuh"
#include "gdn2_tc.cuh"

namespace gdn2 {

namespace {

using namespace tc;

constexpr int kIntraThreads = 256;

template <int D>
struct IntraCfg {
    // region X: A_left image (M=128, K=D) then the four R_I images
    static constexpr uint32_t oAL = 0;
    static constexpr uint32_t kAL = (D / 64) * 16384;
    __host__ __device__ static constexpr uint32_t rows_R(int I) { return 16u * (I + 1); }
    __host__ __device__ static constexpr uint32_t oR(int I) {  // cumulative (D/64) * rows * 128 bytes
        return kAL + (D / 64) * 128u * 16u * (I * (I + 1) / 2);
    }
    static constexpr uint32_t kOperands = kAL + (D / 64) * 128u * 160u;
    static constexpr uint32_t kX = kOperands > 45056u ? kOperands : 45056u;
    // reused after the A/P MMA: solver buffers and the T image (last 8 KB of X)
    static constexpr uint32_t oAf = 0;                      // [64][65] fp32
    static constexpr uint32_t oTf = 16640;                  // [64][65] fp32
    static constexpr uint32_t oY = 33280;                   // 3 x [16][16] fp32
    static constexpr uint32_t oTimg = kX - 8192;            // [64 t][64 s] K-major bf16
    // B operand [beta k e^G | w v], MN-major, N = 2D, K = 64; holds G before
    static constexpr uint32_t oBWU = kX;
    static constexpr uint32_t kBWU = (2 * D / 64) * 8192;
    // per-channel tables: gE[4][D], ge[4][D], inv_ge[4][D]
    static constexpr uint32_t oTab = oBWU + kBWU;
    static constexpr uint32_t kSmem = oTab + 3 * 4 * D * 4 + 1024;
    static constexpr uint32_t kTmemCols = 256;
    static_assert(oTimg >= oY + 3 * 1024, "solver buffers overlap the T image");
    static_assert(kBWU >= 64 * D * 4, "G scratch must fit in the B operand area");
    static_assert(kSmem <= 113 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        f[2 * e] = x.x;
        f[2 * e + 1] = x.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}
__device__ __forceinline__ uint4 ldg16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

template <int D>
__global__ void __launch_bounds__(kIntraThreads, 2) gdn2_tc_intra_kernel(Params p) {
    using C = IntraCfg<D>;
    constexpr int SEG = D / 4;       // channels per thread (row t, segment seg)
    constexpr int NH = SEG / 16;     // halves of 16 channels
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_slot;

    const int c = blockIdx.x, hv = blockIdx.y;
    const int seq = p.chunk_seq[c];
    if (seq < 0) return;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int64_t start = p.chunk_start[c];
    const int len = p.chunk_len[c];
    const int h = hv / p.group;
    const int t = tid / 4, seg = tid % 4;   // row and channel segment owned in steps 1-2
    const int cb = seg * SEG;               // first channel of the segment
    const bool live = t < len;
    const int64_t tok = start + (live ? t : 0);
    uint8_t *rec = p.rec + (static_cast<size_t>(c) * p.HV + hv) * Rec<D>::bytes;

    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }

    // ---- 1. g -> shared scratch, cumsum over the chunk's tokens -------------
    float *Gs = reinterpret_cast<float *>(sm + C::oBWU);  // [64][D] fp32
    {
        const float *gp = p.g + tok * p.sg_t + static_cast<int64_t>(hv) * p.sg_h + cb;
#pragma unroll
        for (int e = 0; e < SEG; e += 4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live && p.has_g) x = __ldg(reinterpret_cast<const float4 *>(gp + e));
            *reinterpret_cast<float4 *>(Gs + t * D + cb + e) = x;
        }
    }
    // q/k L2 norm factors (fp32, per row) when requested
    float kscale = 1.f, qscale = 1.f;
    if (p.l2norm) {
        float sk = 0.f, sq = 0.f;
        if (live) {
            const bf16 *kp = p.k + tok * p.sk_t + static_cast<int64_t>(h) * p.sk_h + cb;
            const bf16 *qp = p.q + tok * p.sq_t + static_cast<int64_t>(h) * p.sq_h + cb;
#pragma unroll
            for (int e = 0; e < SEG; e += 8) {
                float a[8], b[8];
                unpack8(ldg16(kp + e), a);
                unpack8(ldg16(qp + e), b);
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    sk += a[x] * a[x];
                    sq += b[x] * b[x];
                }
            }
        }
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        kscale = 1.f / fmaxf(sqrtf(sk), 1e-12f);
        qscale = 1.f / fmaxf(sqrtf(sq), 1e-12f);
    }
    __syncthreads();
    if (tid < D) {
        float acc = 0.f;
#pragma unroll 8
        for (int r = 0; r < 64; ++r) {
            acc += Gs[r * D + tid];
            Gs[r * D + tid] = acc;
        }
    }
    __syncthreads();
    float *gE = reinterpret_cast<float *>(sm + C::oTab);      // [4][D]  G at E_J
    float *ge = gE + 4 * D;                                   // [4][D]  e^{G_{E_J} - G_{E_{J-1}}}
    float *ige = ge + 4 * D;                                  // [4][D]  1 / ge
    if (tid < D) {
        float prev = 0.f, egl = 1.f;
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            const int e = min(16 * J + 15, len - 1);
            const float gv = Gs[e * D + tid];
            gE[J * D + tid] = gv;
            ge[J * D + tid] = __expf(gv - prev);
            ige[J * D + tid] = __expf(prev - gv);
            egl *= __expf(gv - prev);
            prev = gv;
        }
        reinterpret_cast<float *>(rec + Rec<D>::eGL)[tid] = __expf(prev);
        (void)egl;
    }
    float Gr[SEG];
#pragma unroll
    for (int e = 0; e < SEG; e += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(Gs + t * D + cb + e);
        Gr[e] = x.x; Gr[e + 1] = x.y; Gr[e + 2] = x.z; Gr[e + 3] = x.w;
    }
    __syncthreads();  // G scratch is dead from here on; tables are visible

    // ---- 2. operand images --------------------------------------------------
    {
        const int I = t / 16;
        const bf16 *kp = p.k + tok * p.sk_t + static_cast<int64_t>(h) * p.sk_h;
        const bf16 *qp = p.q + tok * p.sq_t + static_cast<int64_t>(h) * p.sq_h;
        const bf16 *bp = p.beta + tok * p.sb_t + static_cast<int64_t>(hv) * p.sb_h;
        const bf16 *vp = p.v + tok * p.sv_t + static_cast<int64_t>(hv) * p.sv_h;
        const bf16 *wp = p.w + tok * p.sw_t + static_cast<int64_t>(hv) * p.sw_h;
#pragma unroll
        for (int hf = 0; hf < NH; ++hf) {
            const int c0 = cb + 16 * hf;   // 16 channels: two 8-element chunks
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const int cc = c0 + 8 * ch;
                float kk[8], qq[8], bb[8], vv[8], ww[8];
                if (live) {
                    unpack8(ldg16(kp + cc), kk);
                    unpack8(ldg16(qp + cc), qq);
                    unpack8(ldg16(vp + cc), vv);
                    if (p.has_beta) unpack8(ldg16(bp + cc), bb);
                    else {
#pragma unroll
                        for (int x = 0; x < 8; ++x) bb[x] = 1.f;
                    }
                    if (p.has_w) unpack8(ldg16(wp + cc), ww);
                    else {
#pragma unroll
                        for (int x = 0; x < 8; ++x) ww[x] = 1.f;
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 8; ++x) kk[x] = qq[x] = vv[x] = bb[x] = ww[x] = 0.f;
                }
                float Lk[8], Lq[8], kr[8], X1[8], X2[8], Qe[8], Kd[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int ci = cc + x;
                    const float gt = Gr[16 * hf + 8 * ch + x];
                    const float gB = I > 0 ? gE[(I - 1) * D + ci] : 0.f;
                    const float F = __expf(gt - gB);
                    const float eR = __expf(gE[I * D + ci] - gt);
                    const float kx = kk[x] * kscale;
                    float eGB = 1.f, eLE = 1.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        if (m < I) eGB *= ge[m * D + ci];
                        if (m > I) eLE *= ge[m * D + ci];
                    }
                    Lk[x] = bb[x] * kx * F;
                    Lq[x] = qq[x] * qscale * F;
                    kr[x] = kx * eR;
                    X1[x] = Lk[x] * eGB;
                    Qe[x] = Lq[x] * eGB;
                    Kd[x] = kr[x] * eLE;
                    X2[x] = ww[x] * vv[x];
                }
                const int kb = cc / 64, chunk = (cc % 64) / 8;
                // A_left rows t (beta k F) and 64 + t (q F)
                *reinterpret_cast<uint4 *>(sm + C::oAL + kb * 16384 + swz(t, chunk)) = pack8(Lk);
                *reinterpret_cast<uint4 *>(sm + C::oAL + kb * 16384 + swz(64 + t, chunk)) = pack8(Lq);
                // R_{I'} for I' >= I: k eR m_{I',I}
#pragma unroll
                for (int Ip = 0; Ip < 4; ++Ip) {
                    if (Ip < I) continue;
                    float r8[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const int ci = cc + x;
                        float m = 1.f;
                        if (Ip == I) m = ige[I * D + ci];
                        else
                            for (int mm = I + 1; mm < Ip; ++mm) m *= ge[mm * D + ci];
                        r8[x] = kr[x] * m;
                    }
                    *reinterpret_cast<uint4 *>(sm + C::oR(Ip) + kb * (C::rows_R(Ip) * 128u) + swz(t, chunk)) =
                        pack8(r8);
                }
                // B operand [X1 | X2], MN-major: n = cc (X1), n = D + cc (X2)
                *reinterpret_cast<uint4 *>(sm + C::oBWU + (cc / 64) * 8192 + swz(t, chunk)) = pack8(X1);
                *reinterpret_cast<uint4 *>(sm + C::oBWU + ((D + cc) / 64) * 8192 + swz(t, chunk)) = pack8(X2);
                // record: Qe (A1 rows 0-63) and Kd^T (MN-major A)
                *reinterpret_cast<uint4 *>(rec + Rec<D>::A1 + kb * 16384 + swz(t, chunk)) = pack8(Qe);
                *reinterpret_cast<uint4 *>(rec + Rec<D>::KdT + kb * 8192 + swz(t, chunk)) = pack8(Kd);
            }
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_slot;

    // ---- 3. A and P on the tensor cores ---------------------------------------
    if (tid == 0) {
        const uint32_t al = smem_u32(sm + C::oAL);
        uint32_t col = 0;
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            const uint32_t N = C::rows_R(I);
            const uint32_t id = idesc_bf16(128, N, false, false);
            const uint32_t rb = smem_u32(sm + C::oR(I));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16(tm + col, desc_kmajor(al, 128, kk), desc_kmajor(rb, N, kk), id, kk > 0);
            col += N;
        }
        mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 0)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    tc_fence_after();

    float *Af = reinterpret_cast<float *>(sm + C::oAf);
    if (warp < 4) {
        // TMEM row r: r < 64 -> A row t = r, r >= 64 -> P row t = r - 64.  The
        // 32 rows of a warp span row blocks Ilo and Ilo + 1; the warp loads the
        // union of their column groups at warp-uniform addresses (tcgen05.ld is
        // warp-collective) and each lane keeps the groups of its own block.
        const int r = 32 * warp + lane;
        const int tt = r & 63;
        const int I = tt / 16;
        const int Ilo = 2 * (warp & 1);
        const uint32_t cbeg = 16u * (Ilo * (Ilo + 1) / 2);
        const uint32_t cend = 16u * ((Ilo + 2) * (Ilo + 3) / 2);
        const uint32_t mycol0 = 16u * (I * (I + 1) / 2);
        const uint32_t mycols = 16u * (I + 1);
        __syncwarp();
#pragma unroll 1
        for (uint32_t cg = cbeg; cg < cend; cg += 16) {
            uint32_t v[16];
            tmem_ld16(tm + (static_cast<uint32_t>(32 * warp) << 16) + cg, v);
            tmem_ld_wait();
            if (cg >= mycol0 && cg < mycol0 + mycols) {
                const int s0 = static_cast<int>(cg - mycol0);
                if (r < 64) {
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int s = s0 + x;
                        Af[tt * 65 + s] = s < tt ? __uint_as_float(v[x]) : 0.f;
                    }
                } else {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float f[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            const int s = s0 + 8 * half + x;
                            f[x] = s <= tt ? __uint_as_float(v[8 * half + x]) : 0.f;
                        }
                        *reinterpret_cast<uint4 *>(rec + Rec<D>::P + swz(tt, s0 / 8 + half)) = pack8(f);
                    }
                }
            }
        }
        if (r >= 64) {  // P columns past this row's block are zero
            for (int chunk = 2 * (I + 1); chunk < 8; ++chunk)
                *reinterpret_cast<uint4 *>(rec + Rec<D>::P + swz(tt, chunk)) = make_uint4(0, 0, 0, 0);
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- 4. T = (I + A)^{-1}, blocked forward substitution -----------------
    float *Tf = reinterpret_cast<float *>(sm + C::oTf);
    float *Yb = reinterpret_cast<float *>(sm + C::oY);
    if (tid < 64) {  // diagonal 16x16 blocks, one thread per (block, column)
        const int I = tid / 16, j = tid % 16, o = 16 * I;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) acc -= Af[(o + i) * 65 + o + m] * x[m];
            x[i] = (i < j) ? 0.f : acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tf[(o + i) * 65 + o + j] = x[i];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;  // blocks (I, J) = (J + d, J), J = 0..nb-1
        for (int e = tid; e < nb * 256; e += kIntraThreads) {
            const int J = e / 256, i = (e % 256) / 16, j = e % 16;
            const int I = J + d;
            float acc = 0.f;  // Y = sum_{m=J}^{I-1} A_{I m} T_{m J}, row i, col j
            for (int m = 16 * J; m < 16 * I; ++m) acc += Af[(16 * I + i) * 65 + m] * Tf[m * 65 + 16 * J + j];
            Yb[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nb * 256; e += kIntraThreads) {
            const int J = e / 256, i = (e % 256) / 16, j = e % 16;
            const int I = J + d;
            float acc = 0.f;  // T_{IJ} = -T_{II} Y
#pragma unroll
            for (int m = 0; m < 16; ++m) acc -= Tf[(16 * I + i) * 65 + 16 * I + m] * Yb[J * 256 + m * 16 + j];
            Tf[(16 * I + i) * 65 + 16 * J + j] = acc;
        }
        __syncthreads();
    }
    // T -> bf16 K-major image [64 t][64 s]; zeros above the diagonal
    for (int e = tid; e < 64 * 8; e += kIntraThreads) {
        const int tt = e / 8, chunk = e % 8;
        float f[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const int s = 8 * chunk + x;
            f[x] = s <= tt ? Tf[tt * 65 + s] : 0.f;
        }
        *reinterpret_cast<uint4 *>(sm + C::oTimg + swz(tt, chunk)) = pack8(f);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 5. [Wt | Ut] = T x [X1 | X2] ------------------------------------------
    if (tid == 0) {
        constexpr uint32_t id = idesc_bf16(128, 2 * D, false, true);
        const uint32_t ti = smem_u32(sm + C::oTimg), bw = smem_u32(sm + C::oBWU);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(tm, desc_kmajor(ti, 128, kk), desc_mnmajor(bw, 64, kk), id, kk > 0);
        mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 1)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    tc_fence_after();

    // ---- 6. Wt -> A1 rows 64-127, Ut -> Ut image ------------------------------
    if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {
        __syncwarp();
        const int q = warp & 3;
        const int tt = 32 * q + lane;
        const bool is_u = warp >= 4;
        const uint32_t cbase = is_u ? D : 0;
#pragma unroll 1
        for (int j = 0; j < D / 32; ++j) {
            uint32_t v[32];
            tmem_ld32(tm + (static_cast<uint32_t>(32 * q) << 16) + cbase + 32 * j, v);
            tmem_ld_wait();
            const int n0 = 32 * j, kb = n0 / 64, c0 = (n0 % 64) / 8;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint4 o = make_uint4(pack2(__uint_as_float(v[8 * cc]), __uint_as_float(v[8 * cc + 1])),
                                           pack2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3])),
                                           pack2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5])),
                                           pack2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7])));
                uint8_t *dst = is_u ? rec + Rec<D>::Ut + kb * 8192 + swz(tt, c0 + cc)
                                    : rec + Rec<D>::A1 + kb * 16384 + swz(64 + tt, c0 + cc);
                *reinterpret_cast<uint4 *>(dst) = o;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tm, C::kTmemCols);
    }
}

template <int D>
cudaError_t launch_intra(const Params &p, cudaStream_t s) {
    using C = IntraCfg<D>;
    auto kern = gdn2_tc_intra_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    if (p.NCmax > 0) kern<<<dim3(p.NCmax, p.HV), kIntraThreads, C::kSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t tc_record_bytes(int D) { return D == 64 ? Rec<64>::bytes : Rec<128>::bytes; }

cudaError_t launch_tc_intra(const Params &p, cudaStream_t s) {
    return p.K == 64 ? launch_intra<64>(p, s) : launch_intra<128>(p, s);
}

}  // namespace gdn2
