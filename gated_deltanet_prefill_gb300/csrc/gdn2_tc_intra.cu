// Tensor-core intra-chunk kernel: everything of a 64-token chunk that does
// not depend on the incoming state, written as the record the state kernel
// consumes (gdn2_record.cuh).  Persistent: two CTAs of 256 threads per SM walk
// the (chunk, state head) items.  While an item is being processed the next
// one is prepared: its g, v, w tiles arrive by TMA (tensor maps built on the
// host, row copies when a layout cannot be mapped), its k, q, beta tiles are
// prefetched into L2, and the four warps idle in the W/U epilogue compute its
// prefix sums and decay tables.
//
// Steps (FlashRT gated-delta-attention page: norm/cumsum, kkt, solve_tril,
// recompute_wu; fused into one kernel here, with GDN-2's channel-wise gates):
//  1. G = chunk-local inclusive cumsum of g (log2-scaled, in shared memory);
//     k, q (key and query heads), beta (state head) read per thread one channel chunk
//     ahead; optional q/k L2 norm; w v formed from the staged v, w tiles.
//  2. decay factors through 16-token sub-chunk references (burn-gdn2 README,
//     "Numerical stability"): with B_I the row before sub-chunk I and E_J the
//     last row of sub-chunk J,
//        e^{G_t - G_s} = F_t * m_{I,J} * eR_s,   F_t = e^{G_t - G_{B_I}} <= 1,
//        eR_s = e^{G_{E_J} - G_s} <= 1, m_{I,J} = e^{G_{B_I} - G_{E_J}}
//     (m <= 1 for J < I; m = e^{+decay of sub-chunk I} for J = I).  Every m is
//     a product of the per-sub-chunk decays ge_J = e^{G_{E_J} - G_{E_{J-1}}}.
//     m for J = I stays below 2^92 (63.8 nats of decay in the sub-chunk); a
//     key channel that decays faster gets m = 0 there, and its terms of the
//     diagonal 16 x 16 blocks come from the exact path (e^{G_t - G_s} <= 1 per
//     pair), which a second launch of this kernel runs over the items the
//     first one lists.  So no factor exceeds its range for any g <= 0.
//  3. tcgen05 (bf16): [beta k F ; q F] (M=128) x [R_0; R_1; R_2; R_3]^T, one
//     N = 160 product, where R_I = k eR m_{I,.} holds the 16(I+1) tokens of row
//     blocks <= I; the rows of block I against R_I give A (strictly lower) and
//     P (lower incl. diagonal).
//  4. T = (I + A)^{-1} in fp32: 16 x 16 diagonal inverses by forward
//     substitution, 16 -> 32 merges, one 32 -> 64 merge (block inverse of a
//     lower triangular matrix, [[Ta, 0], [Aba, Tb]]^{-1} -> -Tb Aba Ta).
//  5. tcgen05 (fp16): [Wt | Ut] = T x [beta k e^G | w v]  (M=128, N=2D, K=64).
//  6. write Qe, Kd^T, P, Wt, Ut (fp16) and eGL (fp32) as shared-memory images.
// Every fp16 conversion tracks the largest magnitude it wrote; one that
// clipped (past 65504) sets GDN2_ERR_RANGE in the device status.
//
// Thread (t, seg = tid % 4) owns token row t and the 8-channel chunks seg,
// seg + 4, seg + 8, ...: the four segments of a row fall in different
// shared-memory banks for every per-channel table read.  Warp w covers rows
// 8w .. 8w + 7, its quarter-warps rows k and k + 4, which land in the two
// halves of the 128-byte swizzle pattern (conflict-free 16-byte stores).
#include "gdn2_internal.cuh"
#include "gdn2_record.cuh"
#include "gdn2_tc.cuh"

namespace gdn2 {

namespace {

using namespace tc;

constexpr int kIntraThreads = 256;
constexpr int kLD = 68;  // row stride (floats) of the fp32 solver matrices
// Largest decay (log2 units, 92 = 63.8 nats) of one key channel inside one
// 16-token sub-chunk for which the factorised diagonal block stays exact: its
// factors F_t >= 2^-92 and m = 2^92 stay normal in bf16 / fp32.  A channel
// that decays faster is taken out of the diagonal block's product and added
// back by the exact path (e^{G_t - G_s} per pair, fp32).
constexpr float kWideLog2 = 92.f;

template <int D>
struct IntraCfg {
    // region X: A_left image (bf16, M=128, K=D), then the right operands R_0..R_3
    // stacked as one K-major tile of 160 rows (R_I at row 16 I (I + 1) / 2)
    static constexpr uint32_t oAL = 0;
    static constexpr uint32_t kAL = (D / 64) * 16384;
    static constexpr uint32_t oR = kAL;
    static constexpr uint32_t kRrows = 160;
    __host__ __device__ static constexpr uint32_t row_R(int I) { return 16u * (I * (I + 1) / 2); }
    static constexpr uint32_t kOperands = kAL + (D / 64) * 128u * kRrows;
    static constexpr uint32_t kX = kOperands > 47104u ? kOperands : 47104u;
    // before the operand images: the G scratch [64][D] fp32 (plain rows), which
    // receives the item's g (bulk copies) while the previous item is in its
    // W/U product
    static constexpr uint32_t oG = 0;
    // reused after the A/P MMA: fp32 solver matrices and the fp16 T image
    static constexpr uint32_t oAf = 0;                         // [64][kLD]
    static constexpr uint32_t oTf = 64 * kLD * 4;              // [64][kLD]
    static constexpr uint32_t oY = 2 * 64 * kLD * 4;           // merge scratch, [32][32]
    static constexpr uint32_t oTimg = kX - 8192;               // [64 t][64 s] K-major fp16
    // [beta k e^G | w v] fp16 MN-major B (N = 2D, K = 64).  Before the item's
    // operand images it holds the item's raw v and w rows (bf16, [64][D] each),
    // copied in while the previous item is in its W/U epilogue.
    static constexpr uint32_t oBWU = kX;
    static constexpr uint32_t kBWU = (2 * D / 64) * 8192;
    // per-channel tables (log2-scaled G): gE[4][D] = G'_{E_J}, tGB[4][D] =
    // e^{G_{B_I}}, tI[4][D] = e^{G_{B_I} - G_{E_I}}, t2[2][D] = e^{G_{E_{I+1}} -
    // G_{E_I}}, t3[D] = e^{G_{E_3} - G_{E_2}}; the scan totals use the same
    // area before the tables exist
    static constexpr uint32_t oTab = oBWU + kBWU;
    static constexpr uint32_t kTab = 15 * D * 4;
    // mbarriers (MMA, g copies, v/w copies) and the TMEM slot; then the
    // staged item's exact-diagonal flag and the rows' k scales (exact path)
    static constexpr uint32_t oBar = oTab + kTab;
    static constexpr uint32_t oFlag = oBar + 32;
    static constexpr uint32_t oKs = oBar + 64;                  // [64] fp32
    static constexpr uint32_t kSmem = oKs + 256 + 1024;         // + alignment slack
    static constexpr uint32_t kTmemCols = 256;
    static_assert(oTimg >= oY + 4096, "solver buffers overlap the T image");
    static_assert(oG + 64 * D * 4 <= oTimg, "G scratch must not overlap the T image");
    static_assert(kBWU >= 2 * 64 * D * 2, "raw v and w must fit in the B operand area");
    static_assert(kTab >= (kIntraThreads / D) * D * 4, "scan totals must fit in the table area");
    // two CTAs per SM: 2 x (dynamic + 1 KB reserved) <= 228 KB
    static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ uint4 ldg16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

// Exact diagonal blocks for the wide-decay channels of one item (thread
// (t, seg); called by the whole CTA at the start of the item).  For the rows
// s of t's sub-chunk I (s <= t), the sums over the channels that decay by more
// than kWideLog2 inside sub-chunk I of beta_t k_t k_s e^{G_t - G_s} (A, s < t)
// and q_t k_s e^{G_t - G_s} (P), with e^{G_t - G_s} <= 1 taken per pair in
// fp32.  They go to the record's Ut area as fp32 [64 t][16] (A, then P);
// exact_diag_apply adds them to the product's diagonal blocks, and Ut itself
// is written later.  Gs: the item's G' rows; gE: G' at the sub-chunks' last
// rows; ks: scratch for each row's k scale.  Separate functions, off the
// per-item path, so that path keeps its own register allocation.
template <int D, bool F16>
__device__ __noinline__ void exact_diag_sums(const Params &p, const float *Gs, const float *gE, float *ks,
                                             uint8_t *rec, const bf16 *kp, const bf16 *qp, const bf16 *bp,
                                             int64_t start, int h, int t, int seg, bool live) {
    constexpr int NJ = D / 32;
    const int I = t / 16;
    float kscale = 1.f, qscale = 1.f;
    if (p.l2norm) {  // the row's scales, as the operand images take them
        float sk = 0.f, sq = 0.f;
        if (live) {
#pragma unroll 1
            for (int j = 0; j < NJ; ++j) {
                float a[8], b[8];
                unpack8_in(ldg16(kp + 8 * (seg + 4 * j)), a, F16);
                unpack8_in(ldg16(qp + 8 * (seg + 4 * j)), b, F16);
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
    if (seg == 0) ks[t] = kscale;
    __syncthreads();
    float cA[16], cP[16];
#pragma unroll
    for (int si = 0; si < 16; ++si) cA[si] = cP[si] = 0.f;
    if (live) {
#pragma unroll 1
        for (int j = 0; j < NJ; ++j) {
            const int cb = 8 * (seg + 4 * j);
            uint32_t wm = 0;  // wide channels of this 8-channel chunk
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float b = I > 0 ? gE[(I - 1) * D + cb + x] : 0.f;
                if (b - gE[I * D + cb + x] > kWideLog2) wm |= 1u << x;
            }
            if (!wm) continue;
            float kt[8], qt[8], bt[8], gt[8];
            unpack8_in(ldg16(kp + cb), kt, F16);
            unpack8_in(ldg16(qp + cb), qt, F16);
            if (p.has_beta) unpack8_in(ldg16(bp + cb), bt, F16);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                kt[x] *= kscale;
                qt[x] *= qscale;
                bt[x] = (p.has_beta ? bt[x] : 1.f) * kt[x];
                gt[x] = Gs[t * D + cb + x];
            }
#pragma unroll 1
            for (int si = 0; si < 16; ++si) {
                const int s = 16 * I + si;
                if (s > t) break;
                float kv[8];
                unpack8_in(ldg16(p.k + (start + s) * p.sk_t + static_cast<int64_t>(h) * p.sk_h + cb), kv, F16);
                const float sc = ks[s];
                float a = 0.f, q = 0.f;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    if (!((wm >> x) & 1u)) continue;
                    const float kw = kv[x] * sc * ex2(gt[x] - Gs[s * D + cb + x]);
                    a += bt[x] * kw;
                    q += qt[x] * kw;
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {  // register arrays take constant indices
                    if (u == si) {
                        cA[u] += s < t ? a : 0.f;
                        cP[u] += q;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {  // the four segments of the row hold partial sums
        cA[u] += __shfl_xor_sync(0xffffffffu, cA[u], 1);
        cA[u] += __shfl_xor_sync(0xffffffffu, cA[u], 2);
        cP[u] += __shfl_xor_sync(0xffffffffu, cP[u], 1);
        cP[u] += __shfl_xor_sync(0xffffffffu, cP[u], 2);
    }
    float4 a4 = make_float4(cA[0], cA[1], cA[2], cA[3]), p4 = make_float4(cP[0], cP[1], cP[2], cP[3]);
    if (seg == 1) {
        a4 = make_float4(cA[4], cA[5], cA[6], cA[7]);
        p4 = make_float4(cP[4], cP[5], cP[6], cP[7]);
    } else if (seg == 2) {
        a4 = make_float4(cA[8], cA[9], cA[10], cA[11]);
        p4 = make_float4(cP[8], cP[9], cP[10], cP[11]);
    } else if (seg == 3) {
        a4 = make_float4(cA[12], cA[13], cA[14], cA[15]);
        p4 = make_float4(cP[12], cP[13], cP[14], cP[15]);
    }
    float *corr = reinterpret_cast<float *>(rec + Rec<D>::Ut);
    *reinterpret_cast<float4 *>(corr + t * 16 + 4 * seg) = a4;
    *reinterpret_cast<float4 *>(corr + 64 * 16 + t * 16 + 4 * seg) = p4;
}

// Adds the exact path's sums (exact_diag_sums) to the four diagonal 16 x 16
// blocks of A (fp32, shared memory, row stride kLD; s < t) and of P (the
// record's fp16 image; s <= t), once the A/P epilogue has written both.
// Thread (block, row, 4-column group); called by the whole CTA.
template <int D>
__device__ __noinline__ void exact_diag_apply(float *Af, uint8_t *rec, int tid) {
    const int I = tid / 64, r = (tid / 4) % 16, q4 = tid % 4;
    const int tt = 16 * I + r, s0 = 16 * I + 4 * q4;
    const float *corr = reinterpret_cast<const float *>(rec + Rec<D>::Ut) + tt * 16 + 4 * q4;
    const float4 ca = *reinterpret_cast<const float4 *>(corr);
    const float4 cp = *reinterpret_cast<const float4 *>(corr + 64 * 16);
    const float a4[4] = {ca.x, ca.y, ca.z, ca.w}, p4[4] = {cp.x, cp.y, cp.z, cp.w};
    float *arow = Af + tt * kLD + s0;
    uint2 *prow = reinterpret_cast<uint2 *>(rec + Rec<D>::P + swz(tt, s0 / 8) + (s0 % 8) * 2);
    const uint2 ph = *prow;
    float2 pa = unpack_h2(ph.x), pb = unpack_h2(ph.y);
    float pv[4] = {pa.x, pa.y, pb.x, pb.y};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        if (s0 + x < tt) arow[x] += a4[x];
        if (s0 + x <= tt) pv[x] += p4[x];
    }
    *prow = make_uint2(pack_h2(pv[0], pv[1]), pack_h2(pv[2], pv[3]));
}

// F16: q, k, v, beta, w are fp16 (else bf16); a template parameter so that the
// operand-image loop carries no dtype branch.  EXACT = false: the pass over
// every (chunk, state head) item; an item with a wide-decay channel gets its
// record without that channel's diagonal terms and is appended to the exact
// list.  EXACT = true: the second launch, over the listed items only, with the
// exact path; it rewrites their records.  Two instantiations keep the exact
// path's code out of the first pass.
template <int D, bool F16, bool EXACT>
__global__ void __launch_bounds__(kIntraThreads, 2) gdn2_tc_intra_kernel(const __grid_constant__ Params p) {
    using C = IntraCfg<D>;
    constexpr int NJ = D / 32;         // 8-channel chunks per thread
    // D = 128, first pass: the record's P and [Wt | Ut] images are staged in
    // shared memory that is dead at that point and written by bulk copies
    // (the tensor memory accelerator reads them out of shared memory, so the
    // stores leave the LSU/L1 path; 2.93 -> 2.78 ms on the long workload).
    // P (8 KB) goes past the solver matrices, below the T image, during the
    // solve; [Wt | Ut] (32 KB) over the dead R operand and T image during the
    // W/U epilogue.  D = 64 has no such room, and the exact pass rewrites P
    // in the record with its own diagonal sums: both store from registers.
    constexpr bool kBulk = D == 128 && !EXACT;
    constexpr uint32_t oStg = 38912;
    static_assert(!kBulk || (oStg >= IntraCfg<D>::oY + 4096 && oStg + 8192 <= IntraCfg<D>::oTimg &&
                             oStg + 32768 <= IntraCfg<D>::kX), "staging area");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t &bar_mma = *reinterpret_cast<uint64_t *>(sm + C::oBar);
    uint32_t &tmem_slot = *reinterpret_cast<uint32_t *>(sm + C::oBar + 8);
    uint64_t &bar_g = *reinterpret_cast<uint64_t *>(sm + C::oBar + 16);
    uint64_t &bar_vw = *reinterpret_cast<uint64_t *>(sm + C::oBar + 24);

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    // thread (t, seg): a warp covers 8 rows; lanes 8k .. 8k+7 take rows k and
    // k + 4 of them, so a quarter-warp's 16-byte stores into a 128-byte
    // swizzled row pair hit 8 different chunks
    const int seg = tid % 4;
    const int t = 8 * warp + (((lane >> 2) & 1) << 2) + (lane >> 3);
    const int I = t / 16;
    // Both passes are programmatic dependents of the kernel before them: the
    // first pass of the chunk map, the exact pass of the first pass (the exact
    // list).  Each waits here until its predecessor has completed.  The first
    // pass lets the exact pass launch at once (its CTAs wait for this grid);
    // the exact pass lets the state kernel launch once the first pass is done.
    if (EXACT) {
        pdl_wait();
        pdl_trigger();
    } else {
        pdl_trigger();
        pdl_wait();
    }
    // (chunk, state head) items: all of them, or the exact list
    const int total = p.status[0] != GDN2_OK ? 0 : EXACT ? p.status[4] : p.status[1] * p.HV;
    if (static_cast<int>(blockIdx.x) >= total) return;  // before any barrier or TMEM allocation

    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_vw, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }

    // Per-item inputs.  The CTA walks items it = blockIdx.x, + gridDim.x, ...
    // The next item's chunk metadata is loaded after the A/P epilogue.  Its g
    // rows are bulk-copied into the G scratch once the T image is written
    // (warp 7), its v and w rows into the B operand area once the W/U product
    // has read it (warp 2); both land during the W/U product and epilogue.
    // k, q and beta are read by every thread during the operand images.
    int c = 0, hv = 0, len = 1, h = 0, item = 0;
    int nc = 0, nhv = 0, nlen = 1;
    int64_t nstart = 0, start = 0;
    bool live = false;
    const bf16 *kp = nullptr, *qp = nullptr, *bp = nullptr;
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    uint4 nk = z4, nq = z4, nb = z4;
    int nitem = 0;  // item index c * HV + hv of the staged item
    auto meta = [&](int it) {
        nitem = chk(EXACT ? p.exact_list[it] : it, 0, p.status[1] * p.HV, 101, p.status);
        nc = nitem / p.HV;
        nhv = nitem - nc * p.HV;
        nlen = chk(p.chunk_len[nc], 1, kChunk + 1, 102, p.status);
        nstart = chk(p.chunk_start[nc], int64_t(0), p.T_tot - nlen + 1, 103, p.status);
    };
    float *Gs = reinterpret_cast<float *>(sm + C::oG);
    uint8_t *raw_v = sm + C::oBWU;
    uint8_t *raw_w = sm + C::oBWU + 64 * D * 2;
    // TMA tile coordinates of token row t0 of head hh (the tile covers 64 rows;
    // rows past the chunk hold other tokens or zeros and are never used)
    auto tile = [&](void *dst, const CUtensorMap *map, int order, int hh, uint64_t *bar) {
        const int t0 = static_cast<int>(nstart);
        tma_load_3d(dst, map, 0, order ? t0 : hh, order ? hh : t0, bar);
    };
    // g rows: fp32 straight into the G scratch; 16-bit g into its upper half
    // (converted by the prefix-sum warps)
    const uint32_t g_es = p.g_dtype == GDN2_DTYPE_F32 ? 4u : 2u;
    uint8_t *g_dst = reinterpret_cast<uint8_t *>(Gs) + (g_es == 4u ? 0u : 64u * D * 2u);
    auto stage_g = [&]() {  // warp 7
        if (p.tmap) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_g, p.has_g ? 64u * D * g_es : 0u);
                if (p.has_g) tile(g_dst, &p.tm_g, p.tm_order_g, nhv, &bar_g);
            }
            return;
        }
        const uint32_t rows = p.has_g ? static_cast<uint32_t>(nlen) : 0u;
        if (lane == 0) mbar_arrive_expect_tx(&bar_g, rows * D * g_es);
        __syncwarp();
        const uint8_t *gb = reinterpret_cast<const uint8_t *>(p.g);
        for (uint32_t r = lane; r < rows; r += 32)
            bulk_g2s(g_dst + r * D * g_es,
                     gb + ((nstart + r) * p.sg_t + static_cast<int64_t>(nhv) * p.sg_h) * g_es, D * g_es, &bar_g);
    };
    auto stage_vw = [&]() {  // warp 2
        if (p.tmap) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_vw, 64u * D * 2 * (p.has_w ? 2u : 1u));
                tile(raw_v, &p.tm_v, p.tm_order_v, nhv / p.gv, &bar_vw);
                if (p.has_w) tile(raw_w, &p.tm_w, p.tm_order_w, nhv, &bar_vw);
            }
            return;
        }
        const uint32_t rows = static_cast<uint32_t>(nlen);
        if (lane == 0) mbar_arrive_expect_tx(&bar_vw, rows * D * 2 * (p.has_w ? 2u : 1u));
        __syncwarp();
        for (uint32_t r = lane; r < rows; r += 32) {
            const int64_t tok = nstart + r;
            bulk_g2s(raw_v + r * D * 2, p.v + tok * p.sv_t + static_cast<int64_t>(nhv / p.gv) * p.sv_h, D * 2,
                     &bar_vw);
            if (p.has_w)
                bulk_g2s(raw_w + r * D * 2, p.w + tok * p.sw_t + static_cast<int64_t>(nhv) * p.sw_h, D * 2, &bar_vw);
        }
    };
    auto adopt = [&]() {  // the staged item becomes the current one
        c = nc;
        hv = nhv;
        item = nitem;
        len = nlen;
        start = nstart;
        h = hv / p.gk;  // key head; the query head is hv / gq
        live = t < len;
        const int64_t tok = nstart + (live ? t : 0);
        kp = p.k + tok * p.sk_t + static_cast<int64_t>(h) * p.sk_h;
        qp = p.q + tok * p.sq_t + static_cast<int64_t>(hv / p.gq) * p.sq_h;
        bp = p.beta + tok * p.sb_t + static_cast<int64_t>(hv) * p.sb_h;
    };
    // G' = G log2(e): every decay factor below is an exact power of two of a
    // difference of G' values.  The staged item's prefix sums (in place in the
    // G scratch) and per-channel decay tables are computed by the four warps
    // that are idle in the W/U epilogue: warps 2, 3, 6, 7 (named barrier 1).
    constexpr float kLog2e = 1.4426950408889634f;
    constexpr int P4 = 128 / D;     // scan parts (rows split in P4 ranges)
    constexpr int R4 = 64 / P4;     // rows per part
    float *gE = reinterpret_cast<float *>(sm + C::oTab);  // G' at E_J
    float *tGB = gE + 4 * D;                              // e^{G_{B_I}}
    float *tI = tGB + 4 * D;                              // e^{G_{B_I} - G_{E_I}}
    float *t2 = tI + 4 * D;                               // e^{G_{E_{I+1}} - G_{E_I}}, I = 0, 1
    float *t3 = t2 + 2 * D;                               // e^{G_{E_3} - G_{E_2}}
    volatile uint32_t *exact_flag = reinterpret_cast<volatile uint32_t *>(sm + C::oFlag);
    float *ks_row = reinterpret_cast<float *>(sm + C::oKs);  // k scale of each row (exact path)
    uint32_t gph = 0, vph = 0;  // parities of the g and v/w staging barriers
    uint32_t hmax = 0;           // largest magnitude converted to fp16 (range check)
    const bool aux = (warp & 2) != 0;
    auto scan_tables = [&](int ilen, uint8_t *irec) {
        const int lt = 32 * ((warp & 1) + 2 * (warp >> 2)) + lane;  // 0 .. 127
        if (!mbar_wait(&bar_g, gph)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
        const int glen = p.has_g ? ilen : 0;  // rows past it read as 0
        const int ch = lt % D, part = lt / D;
        float *base = Gs + part * R4 * D + ch;
        float acc = 0.f;
        if (g_es == 2u) {
            // 16-bit g in the upper half of the scratch: rows in blocks of 8 are
            // read, then (after a barrier) written back as fp32 prefix sums; the
            // fp32 rows of block b overwrite only 16-bit rows <= 8b + 7
            const unsigned short *g16 = reinterpret_cast<const unsigned short *>(g_dst);
            const bool gf16 = p.g_dtype == GDN2_DTYPE_F16;
#pragma unroll 1
            for (int b = 0; b < 8; ++b) {
                float x[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int row = 8 * b + k;
                    const unsigned short u = lt < D && row < glen ? g16[row * D + lt] : 0;
                    x[k] = gf16 ? __half2float(__ushort_as_half(u)) : __bfloat162float(__ushort_as_bfloat16(u));
                }
                named_sync(1, 128);
                if (lt < D) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        acc += __fmul_rn(x[k], kLog2e);
                        Gs[(8 * b + k) * D + lt] = acc;
                    }
                }
            }
        } else {
#pragma unroll 1
        for (int r8 = 0; r8 < R4; r8 += 8) {
            float *b8 = base + r8 * D;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int row = part * R4 + r8 + k;
                acc += row < glen ? __fmul_rn(b8[k * D], kLog2e) : 0.f;
                b8[k * D] = acc;
            }
        }
        }
        if (P4 > 1 && g_es == 4u) {
            float *tot = reinterpret_cast<float *>(sm + C::oTab);  // [P4][D], before the tables
            tot[part * D + ch] = acc;
            named_sync(1, 128);
            float off = 0.f;
            for (int pp = 0; pp < part; ++pp) off += tot[pp * D + ch];
            if (part > 0) {
#pragma unroll 1
                for (int r8 = 0; r8 < R4; r8 += 8) {
                    float *b8 = base + r8 * D;
#pragma unroll
                    for (int k = 0; k < 8; ++k) b8[k * D] += off;
                }
            }
        }
        if (lt == 0) *exact_flag = 0u;
        named_sync(1, 128);
        if (lt < D) {
            float e[4];
#pragma unroll
            for (int J = 0; J < 4; ++J) e[J] = Gs[min(16 * J + 15, ilen - 1) * D + lt];
            bool wide = false;
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                const float b = J > 0 ? e[J - 1] : 0.f;
                gE[J * D + lt] = e[J];
                tGB[J * D + lt] = ex2(b);
                // a channel that decays by more than kWideLog2 inside sub-chunk
                // J takes its diagonal block from the exact path (m = 0 here)
                const bool wj = b - e[J] > kWideLog2;
                tI[J * D + lt] = wj ? 0.f : ex2(b - e[J]);
                wide |= wj;
            }
            if (wide) *exact_flag = 1u;
            t2[lt] = ex2(e[1] - e[0]);
            t2[D + lt] = ex2(e[2] - e[1]);
            t3[lt] = ex2(e[3] - e[2]);
            reinterpret_cast<float *>(irec + Rec<D>::eGL)[lt] = ex2(e[3]);
        }
    };
    auto rec_of = [&](int ic, int ihv) { return p.rec + (static_cast<size_t>(ic) * p.HV + ihv) * Rec<D>::bytes; };

    if (static_cast<int>(blockIdx.x) < total) meta(blockIdx.x);
    __syncthreads();  // barriers initialised
    if (static_cast<int>(blockIdx.x) < total) {
        if (warp == 7) stage_g();
        if (warp == 2) stage_vw();
        if (aux) scan_tables(nlen, rec_of(nc, nhv));
    }
    gph ^= 1u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_slot;

#pragma unroll 1
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
    adopt();
    uint8_t *rec = rec_of(c, hv);
    // some key channel decays past the factorised range inside a sub-chunk of
    // this item: its diagonal blocks take the exact path (CTA-uniform)
    const bool exact = *exact_flag != 0u;
    const uint32_t hmax_in = hmax;
    if (!EXACT && exact && tid == 0)
        p.exact_list[chk(atomicAdd(p.status + 4, 1), 0, p.NCmax * p.HV, 104, p.status)] = item;
    if (EXACT && exact) exact_diag_sums<D, F16>(p, Gs, gE, ks_row, rec, kp, qp, bp, start, h, t, seg, live);

    // ---- 1. cumsum (g is in the G scratch) ----------------------------------------
    nk = nq = nb = z4;
    if (live) {  // first operand chunk; later chunks are fetched one ahead
        const int cb = 8 * seg;
        nk = ldg16(kp + cb);
        nq = ldg16(qp + cb);
        if (p.has_beta) nb = ldg16(bp + cb);
    }
    float kscale = 1.f, qscale = 1.f;
    if (p.l2norm) {
        float sk = 0.f, sq = 0.f;
        if (live) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                float a[8], b[8];
                unpack8_in(ldg16(kp + 8 * (seg + 4 * j)), a, F16);
                unpack8_in(ldg16(qp + 8 * (seg + 4 * j)), b, F16);
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
    // G' prefix sums and tables are ready (computed during the previous item's
    // W/U epilogue, or before the loop); raw v and w are in the B operand area
    if (!mbar_wait(&bar_vw, vph)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    vph ^= 1u;
    // w v for this thread's chunks, stored to its operand image after the
    // barrier below (it overwrites the raw rows)
    uint4 wX2[NJ];
    // raw rows are 256 bytes apart and an eight-lane group holds rows t and
    // t + 4: rows with bit 2 of t set read each pair of chunks in the other
    // order, so the two rows of a group hit different banks
    const bool rsw = (t >> 2) & 1;
#pragma unroll
    for (int j = 0; j < NJ; j += 2) {
        uint4 rv[2], rw[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int cb = 8 * (seg + 4 * (j + (h ^ static_cast<int>(rsw))));
            rv[h] = live ? *reinterpret_cast<const uint4 *>(raw_v + (t * D + cb) * 2) : z4;
            rw[h] = live && p.has_w ? *reinterpret_cast<const uint4 *>(raw_w + (t * D + cb) * 2) : z4;
        }
        auto sel = [](bool c, const uint4 &x, const uint4 &y) {
            return make_uint4(c ? x.x : y.x, c ? x.y : y.y, c ? x.z : y.z, c ? x.w : y.w);
        };
        const uint4 v0 = sel(rsw, rv[1], rv[0]), v1 = sel(rsw, rv[0], rv[1]);
        const uint4 w0 = sel(rsw, rw[1], rw[0]), w1 = sel(rsw, rw[0], rw[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float vv[8], ww[8];
            unpack8_in(h ? v1 : v0, vv, F16);
            unpack8_in(h ? w1 : w0, ww, F16);
#pragma unroll
            for (int x = 0; x < 8; ++x) ww[x] = (p.has_w || !live) ? ww[x] * vv[x] : vv[x];
            wX2[j + h] = pack8_hm(ww, hmax);
        }
    }
    float Gr[8 * NJ];
    // G rows are 512 bytes apart, so the same channels of different rows share
    // banks.  A 16-byte load is served eight lanes at a time, and those lanes
    // hold rows t and t + 4: rows with bit 2 of t set load each chunk's two
    // halves in the other order, so every eight-lane group covers all 32 banks
    const int gsw = ((t >> 2) & 1) ? 4 : 0;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int cb = 8 * (seg + 4 * j);
        const float4 x0 = *reinterpret_cast<const float4 *>(Gs + t * D + cb + gsw);
        const float4 x1 = *reinterpret_cast<const float4 *>(Gs + t * D + cb + (4 - gsw));
        const float4 a = gsw ? x1 : x0, b = gsw ? x0 : x1;
        Gr[8 * j + 0] = a.x; Gr[8 * j + 1] = a.y; Gr[8 * j + 2] = a.z; Gr[8 * j + 3] = a.w;
        Gr[8 * j + 4] = b.x; Gr[8 * j + 5] = b.y; Gr[8 * j + 6] = b.z; Gr[8 * j + 7] = b.w;
    }
    if (kBulk && tid == 0) bulk_wait_read0();  // the [Wt | Ut] staging (the R operand area) is free
    __syncthreads();  // G scratch and raw v, w are dead from here on
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int cb = 8 * (seg + 4 * j);
        *reinterpret_cast<uint4 *>(sm + C::oBWU + ((D + cb) / 64) * 8192 + swz(t, (cb % 64) / 8)) = wX2[j];
    }

    // ---- 2. operand images -------------------------------------------------------
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int cb = 8 * (seg + 4 * j);
        float kk[8], qq[8], bb[8];
        unpack8_in(nk, kk, F16);
        unpack8_in(nq, qq, F16);
        unpack8_in(nb, bb, F16);
        if (!p.has_beta && live) {
#pragma unroll
            for (int x = 0; x < 8; ++x) bb[x] = 1.f;
        }
        if (j + 1 < NJ && live) {  // fetch the next chunk
            const int cn = 8 * (seg + 4 * (j + 1));
            nk = ldg16(kp + cn);
            nq = ldg16(qp + cn);
            if (p.has_beta) nb = ldg16(bp + cn);
        }
        // outputs packed two channels per 32-bit word as they are produced
        uint32_t wLk[4], wLq[4], wkr[4], wX1[4], wQe[4], wKd[4], wr0[4], wr2[4], wr3[4];
        const float4 z4f = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            // per-channel tables for channels cb + 4 hh .. + 3: one 16-byte load
            // each, shared by the four channels
            const int c4 = cb + 4 * hh;
            const float4 vB4 = I > 0 ? *reinterpret_cast<const float4 *>(gE + (I - 1) * D + c4) : z4f;
            const float4 vE4 = *reinterpret_cast<const float4 *>(gE + I * D + c4);
            const float4 v44 = *reinterpret_cast<const float4 *>(t3 + c4);
            const float4 vG4 = *reinterpret_cast<const float4 *>(tGB + I * D + c4);
            const float4 vI4 = *reinterpret_cast<const float4 *>(tI + I * D + c4);
            const float4 v24 = *reinterpret_cast<const float4 *>(t2 + (I & 1) * D + c4);
            const float4 v34 = *reinterpret_cast<const float4 *>(t2 + D + c4);
            const float vB[4] = {vB4.x, vB4.y, vB4.z, vB4.w}, vE[4] = {vE4.x, vE4.y, vE4.z, vE4.w};
            const float v4[4] = {v44.x, v44.y, v44.z, v44.w}, vG[4] = {vG4.x, vG4.y, vG4.z, vG4.w};
            const float vI[4] = {vI4.x, vI4.y, vI4.z, vI4.w}, v2[4] = {v24.x, v24.y, v24.z, v24.w};
            const float v3[4] = {v34.x, v34.y, v34.z, v34.w};
            float lk[4], lq[4], kr[4], x1[4], qe[4], kd[4], r0[4], r2[4], r3[4];
#pragma unroll
            for (int ce = 0; ce < 4; ++ce) {
                const int x = 4 * hh + ce;
                const float gt = Gr[8 * j + x];
                const float F = ex2(gt - vB[ce]);                // e^{G_t - G_{B_I}}
                const float eR = ex2(vE[ce] - gt);               // e^{G_{E_I} - G_t}
                // e^{G_L - G_t} = eR e^{G_L - G_{E_I}}, the second factor a
                // product of the sub-chunk decays after sub-chunk I (L = E_3)
                float fL = I == 3 ? 1.f : v4[ce];
                if (I <= 1) fL *= v2[ce];
                if (I == 0) fL *= v3[ce];
                const float eL = eR * fL;
                const float kx = kk[x] * kscale;
                lk[ce] = bb[x] * kx * F;
                lq[ce] = qq[x] * qscale * F;
                kr[ce] = kx * eR;
                x1[ce] = lk[ce] * vG[ce];                        // * e^{G_{B_I}}
                qe[ce] = lq[ce] * vG[ce];
                kd[ce] = kx * eL;
                r0[ce] = kr[ce] * vI[ce];                        // row of R_I
                r2[ce] = kr[ce] * v2[ce];                        // row of R_{I+2}, I <= 1
                r3[ce] = r2[ce] * v3[ce];                        // row of R_3, I = 0
            }
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int x2 = 2 * hh + e2, a = 2 * e2;
                wLk[x2] = pack_bf2(lk[a], lk[a + 1]);
                wLq[x2] = pack_bf2(lq[a], lq[a + 1]);
                wkr[x2] = pack_bf2(kr[a], kr[a + 1]);
                wr0[x2] = pack_bf2(r0[a], r0[a + 1]);
                wr2[x2] = pack_bf2(r2[a], r2[a + 1]);
                wr3[x2] = pack_bf2(r3[a], r3[a + 1]);
                wX1[x2] = pack_h2mh(x1[a], x1[a + 1], hmax);
                wQe[x2] = pack_h2mh(qe[a], qe[a + 1], hmax);
                wKd[x2] = pack_h2mh(kd[a], kd[a + 1], hmax);
            }
        }
        auto u4 = [](const uint32_t (&w)[4]) { return make_uint4(w[0], w[1], w[2], w[3]); };
        const int kb = cb / 64, chunk = (cb % 64) / 8;
        *reinterpret_cast<uint4 *>(sm + C::oAL + kb * 16384 + swz(t, chunk)) = u4(wLk);
        *reinterpret_cast<uint4 *>(sm + C::oAL + kb * 16384 + swz(64 + t, chunk)) = u4(wLq);
        // rows of R_{I'} for I' >= I (R_{I+1} takes m = 1) in the stacked 160-row tile
        uint8_t *rt = sm + C::oR + kb * (C::kRrows * 128u);
        *reinterpret_cast<uint4 *>(rt + swz(C::row_R(I) + t, chunk)) = u4(wr0);
        if (I + 1 < 4) *reinterpret_cast<uint4 *>(rt + swz(C::row_R(I + 1) + t, chunk)) = u4(wkr);
        if (I + 2 < 4) *reinterpret_cast<uint4 *>(rt + swz(C::row_R(I + 2) + t, chunk)) = u4(wr2);
        if (I == 0) *reinterpret_cast<uint4 *>(rt + swz(C::row_R(3) + t, chunk)) = u4(wr3);
        *reinterpret_cast<uint4 *>(sm + C::oBWU + (cb / 64) * 8192 + swz(t, chunk)) = u4(wX1);
        *reinterpret_cast<uint4 *>(rec + Rec<D>::A1 + kb * 16384 + swz(t, chunk)) = u4(wQe);
        *reinterpret_cast<uint4 *>(rec + Rec<D>::KdT + kb * 8192 + swz(t, chunk)) = u4(wKd);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 3. A and P on the tensor cores (bf16) --------------------------------
    if (tid == 0) {  // one N = 160 chain: columns 16 I (I + 1) / 2 .. hold R_I
        const uint32_t al = smem_u32(sm + C::oAL), rb = smem_u32(sm + C::oR);
        constexpr uint32_t id = idesc_bf16(128, C::kRrows, false, false);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            mma_f16(tm, desc_kmajor(al, 128, kk), desc_kmajor(rb, C::kRrows, kk), id, kk > 0);
        mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 0)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    tc_fence_after();

    float *Af = reinterpret_cast<float *>(sm + C::oAf);
    {
        // TMEM row r: r < 64 -> A row r, r >= 64 -> P row r - 64.  A warp's 32
        // rows span row blocks Ilo and Ilo + 1; the warp loads the union of their
        // 16-column groups at warp-uniform addresses (tcgen05.ld is
        // warp-collective) and each lane keeps the groups of its own block.
        // Warps w and w + 4 share lane quarter w % 4 and take alternate groups.
        const int wq = warp & 3;
        const int r = 32 * wq + lane;
        const int tt = r & 63;
        const int Ir = tt / 16;
        const int Ilo = 2 * (wq & 1);
        const uint32_t cbeg = 16u * (Ilo * (Ilo + 1) / 2) + 16u * (warp >> 2);
        const uint32_t cend = 16u * ((Ilo + 2) * (Ilo + 3) / 2);
        const uint32_t mycol0 = 16u * (Ir * (Ir + 1) / 2);
        const uint32_t mycols = 16u * (Ir + 1);
        __syncwarp();
        auto keep = [&](uint32_t cg, const uint32_t (&v)[16]) {
            if (cg >= mycol0 && cg < mycol0 + mycols) {
                const int s0 = static_cast<int>(cg - mycol0);
                if (r < 64) {
#pragma unroll
                    for (int x4 = 0; x4 < 4; ++x4) {
                        float4 f;
                        f.x = s0 + 4 * x4 + 0 < tt ? __uint_as_float(v[4 * x4 + 0]) : 0.f;
                        f.y = s0 + 4 * x4 + 1 < tt ? __uint_as_float(v[4 * x4 + 1]) : 0.f;
                        f.z = s0 + 4 * x4 + 2 < tt ? __uint_as_float(v[4 * x4 + 2]) : 0.f;
                        f.w = s0 + 4 * x4 + 3 < tt ? __uint_as_float(v[4 * x4 + 3]) : 0.f;
                        *reinterpret_cast<float4 *>(Af + tt * kLD + s0 + 4 * x4) = f;
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
                        *reinterpret_cast<uint4 *>((kBulk ? sm + oStg : rec + Rec<D>::P) + swz(tt, s0 / 8 + half)) =
                            pack8_hm(f, hmax);
                    }
                }
            }
        };
#pragma unroll 1
        for (uint32_t cg = cbeg; cg < cend; cg += 32) {
            uint32_t v0[16];
            tmem_ld16(tm + (static_cast<uint32_t>(32 * wq) << 16) + cg, v0);
            tmem_ld_wait();
            keep(cg, v0);
        }
        if (r >= 64 && warp < 4) {  // P columns past this row's block are zero
            for (int chunk = 2 * (Ir + 1); chunk < 8; ++chunk)
                *reinterpret_cast<uint4 *>((kBulk ? sm + oStg : rec + Rec<D>::P) + swz(tt, chunk)) =
                    make_uint4(0, 0, 0, 0);
        }
        if (kBulk) fence_proxy_async();  // the staged P is read by a bulk copy after the next barrier
    }
    if (EXACT && exact) {  // the exact path's sums join the diagonal blocks of A and P
        __syncthreads();
        exact_diag_apply<D>(Af, rec, tid);
        __syncthreads();
    }
    const bool has_next = it + static_cast<int>(gridDim.x) < total;
    if (has_next) meta(it + static_cast<int>(gridDim.x));
    tc_fence_before();

    // ---- 4. T = (I + A)^{-1}, blocked forward substitution (fp32) ---------------
    // The diagonal inverses start once the A warps (0, 1, 4, 5) have written
    // A (named barrier 2); the P warps are still storing P meanwhile.
    float *Tf = reinterpret_cast<float *>(sm + C::oTf);
    float *Yb = reinterpret_cast<float *>(sm + C::oY);
    if (!aux) named_sync(2, 128);
    if (has_next && p.tpre && warp == 6 && lane == 0) {  // next item's k, q, beta into L2
        const int t0 = static_cast<int>(nstart), nk_h = nhv / p.gk, nq_h = nhv / p.gq;
        tma_prefetch_3d(&p.tm_k, 0, p.tm_order_k ? t0 : nk_h, p.tm_order_k ? nk_h : t0);
        tma_prefetch_3d(&p.tm_q, 0, p.tm_order_q ? t0 : nq_h, p.tm_order_q ? nq_h : t0);
        if (p.has_beta) tma_prefetch_3d(&p.tm_b, 0, p.tm_order_b ? t0 : nhv, p.tm_order_b ? nhv : t0);
    }
    // The fp16 T image (K-major [64 t][64 s]) is written as its blocks are
    // computed: zeros above the diagonal blocks here, each diagonal block by
    // its inverse, each off-diagonal block by its merge.
    uint8_t *timg = sm + C::oTimg;
    if (tid >= 64) {  // 16-byte zero chunks: rows of block I, chunks 2 (I + 1) .. 7
        for (int e = tid - 64; e < 192; e += kIntraThreads - 64) {
            const int Ib = e < 96 ? 0 : e < 160 ? 1 : 2;
            const int e0 = e - (Ib == 0 ? 0 : Ib == 1 ? 96 : 160), nz = 6 - 2 * Ib;
            const int row = 16 * Ib + e0 / nz, chunk = 2 * (Ib + 1) + e0 % nz;
            *reinterpret_cast<uint4 *>(timg + swz(row, chunk)) = make_uint4(0, 0, 0, 0);
        }
    }
    if (tid < 64) {  // diagonal 16x16 blocks, one thread per (block, column)
        const int Ib = tid / 16, j = tid % 16, o = 16 * Ib;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == j) ? 1.f : 0.f;
            const float *arow = Af + (o + i) * kLD + o;  // 16-byte aligned (kLD = 68)
#pragma unroll
            for (int m4 = 0; m4 < i; m4 += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(arow + m4);
                acc -= a.x * x[m4];
                if (m4 + 1 < i) acc -= a.y * x[m4 + 1];
                if (m4 + 2 < i) acc -= a.z * x[m4 + 2];
                if (m4 + 3 < i) acc -= a.w * x[m4 + 3];
            }
            x[i] = (i < j) ? 0.f : acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tf[(o + i) * kLD + o + j] = x[i];
    }
    __syncthreads();
    if (kBulk && tid == 0) {  // the staged P image into the record
        bulk_s2g(rec + Rec<D>::P, sm + oStg, 8192);
        bulk_commit();
    }
    // 16 -> 32 merges: T_{I+1,I} = -T_{I+1,I+1} (A_{I+1,I} T_{I,I}), I = 0 and 2,
    // a 1 x 2 tile per thread
    {
        const int b = tid / 128, e = tid % 128, Ib = 2 * b;
        const int i = e / 8, j0 = 2 * (e % 8);
        const int r0 = 16 * (Ib + 1), c0 = 16 * Ib;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 16; m4 += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(Af + (r0 + i) * kLD + c0 + m4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const float2 tv = *reinterpret_cast<const float2 *>(Tf + (c0 + m4 + mm) * kLD + c0 + j0);
                y0 += av[mm] * tv.x;
                y1 += av[mm] * tv.y;
            }
        }
        *reinterpret_cast<float2 *>(Yb + b * 256 + i * 16 + j0) = make_float2(y0, y1);
        // row i, columns j0, j0 + 1 of the diagonal blocks I and I + 1 into the image
#pragma unroll
        for (int d = 0; d < 2; ++d) {
            const int o = d ? r0 : c0;
            const float2 tv = *reinterpret_cast<const float2 *>(Tf + (o + i) * kLD + o + j0);
            *reinterpret_cast<uint32_t *>(timg + swz(o + i, (o + j0) / 8) + ((o + j0) % 8) * 2) =
                pack_h2mh(tv.x, tv.y, hmax);
        }
        __syncthreads();
        float z0 = 0.f, z1 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 16; m4 += 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(Tf + (r0 + i) * kLD + r0 + m4);
            const float tvv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const float2 yv = *reinterpret_cast<const float2 *>(Yb + b * 256 + (m4 + mm) * 16 + j0);
                z0 -= tvv[mm] * yv.x;
                z1 -= tvv[mm] * yv.y;
            }
        }
        *reinterpret_cast<float2 *>(Tf + (r0 + i) * kLD + c0 + j0) = make_float2(z0, z1);
        *reinterpret_cast<uint32_t *>(timg + swz(r0 + i, (c0 + j0) / 8) + ((c0 + j0) % 8) * 2) = pack_h2mh(z0, z1, hmax);
    }
    __syncthreads();
    // 32 -> 64 merge on the 32 x 32 halves a (rows/cols 0-31) and b (32-63):
    // X = A_ba T_a, then T_ba = -T_b X; a 2 x 2 tile per thread.  T_a and T_b
    // are block lower triangular, so the sums skip their zero upper blocks.
    {
        const int i0 = 2 * (tid / 16), j0 = 2 * (tid % 16);
        float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
#pragma unroll 2
        for (int m4 = j0 & ~15; m4 < 32; m4 += 4) {
            const float4 p0 = *reinterpret_cast<const float4 *>(Af + (32 + i0) * kLD + m4);
            const float4 p1 = *reinterpret_cast<const float4 *>(Af + (33 + i0) * kLD + m4);
            const float a0v[4] = {p0.x, p0.y, p0.z, p0.w}, a1v[4] = {p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const float2 tv = *reinterpret_cast<const float2 *>(Tf + (m4 + mm) * kLD + j0);
                x00 += a0v[mm] * tv.x; x01 += a0v[mm] * tv.y; x10 += a1v[mm] * tv.x; x11 += a1v[mm] * tv.y;
            }
        }
        *reinterpret_cast<float2 *>(Yb + i0 * 32 + j0) = make_float2(x00, x01);
        *reinterpret_cast<float2 *>(Yb + (i0 + 1) * 32 + j0) = make_float2(x10, x11);
        __syncthreads();
        float z00 = 0.f, z01 = 0.f, z10 = 0.f, z11 = 0.f;
        const int mend = (i0 & ~15) + 16;
#pragma unroll 2
        for (int m4 = 0; m4 < mend; m4 += 4) {
            const float4 p0 = *reinterpret_cast<const float4 *>(Tf + (32 + i0) * kLD + 32 + m4);
            const float4 p1 = *reinterpret_cast<const float4 *>(Tf + (33 + i0) * kLD + 32 + m4);
            const float t0v[4] = {p0.x, p0.y, p0.z, p0.w}, t1v[4] = {p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const float2 xv = *reinterpret_cast<const float2 *>(Yb + (m4 + mm) * 32 + j0);
                z00 -= t0v[mm] * xv.x; z01 -= t0v[mm] * xv.y; z10 -= t1v[mm] * xv.x; z11 -= t1v[mm] * xv.y;
            }
        }
        *reinterpret_cast<float2 *>(Tf + (32 + i0) * kLD + j0) = make_float2(z00, z01);
        *reinterpret_cast<float2 *>(Tf + (33 + i0) * kLD + j0) = make_float2(z10, z11);
        *reinterpret_cast<uint32_t *>(timg + swz(32 + i0, j0 / 8) + (j0 % 8) * 2) = pack_h2mh(z00, z01, hmax);
        *reinterpret_cast<uint32_t *>(timg + swz(33 + i0, j0 / 8) + (j0 % 8) * 2) = pack_h2mh(z10, z11, hmax);
    }
    if (kBulk && tid == 0) bulk_wait_read0();  // the P staging is free for [Wt | Ut]
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (has_next && warp == 7) stage_g();  // the solver matrices are dead: the G scratch is free

    // ---- 5. [Wt | Ut] = T x [X1 | X2] (fp16) -----------------------------------
    if (tid == 0) {
        constexpr uint32_t id = idesc_fp16(128, 2 * D, false, true);
        const uint32_t ti = smem_u32(sm + C::oTimg), bw = smem_u32(sm + C::oBWU);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f16(tm, desc_kmajor(ti, 128, kk), desc_mnmajor(bw, 64, kk), id, kk > 0);
        mma_commit(&bar_mma);
    }
    if (!mbar_wait(&bar_mma, 1)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    tc_fence_after();
    if (has_next && warp == 2) stage_vw();  // the W/U product has read the B operand area
    if (has_next && aux) scan_tables(nlen, rec_of(nc, nhv));  // the next item's G' and tables
    if (has_next) gph ^= 1u;

    // ---- 6. Wt -> A1 rows 64-127, Ut -> Ut image (fp16) -------------------------
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
                const uint32_t *w = v + 8 * cc;
                const uint4 o = make_uint4(pack_h2mh(__uint_as_float(w[0]), __uint_as_float(w[1]), hmax),
                                           pack_h2mh(__uint_as_float(w[2]), __uint_as_float(w[3]), hmax),
                                           pack_h2mh(__uint_as_float(w[4]), __uint_as_float(w[5]), hmax),
                                           pack_h2mh(__uint_as_float(w[6]), __uint_as_float(w[7]), hmax));
                uint8_t *dst = kBulk ? sm + oStg + (is_u ? 16384 : 0) + kb * 8192 + swz(tt, c0 + cc)
                               : is_u ? rec + Rec<D>::Ut + kb * 8192 + swz(tt, c0 + cc)
                                      : rec + Rec<D>::A1 + kb * 16384 + swz(64 + tt, c0 + cc);
                *reinterpret_cast<uint4 *>(dst) = o;
            }
        }
        if (kBulk) {  // Wt (rows 64-127 of each A1 block) and Ut into the record
            fence_proxy_async();
            named_sync(2, 128);
            if (tid == 0) {
                bulk_s2g(rec + Rec<D>::A1 + 8192, sm + oStg, 8192);
                bulk_s2g(rec + Rec<D>::A1 + 16384 + 8192, sm + oStg + 8192, 8192);
                bulk_s2g(rec + Rec<D>::Ut, sm + oStg + 16384, 16384);
                bulk_commit();
            }
        }
    }
    // the first pass's record of a listed item is rewritten by the exact pass:
    // its values do not count for the range check
    if (!EXACT && exact) hmax = hmax_in;
    tc_fence_before();
    __syncthreads();  // the item's shared memory and TMEM are free for the next one
    tc_fence_after();
    }  // items
    if (kBulk && tid == 0) bulk_wait0();  // the last record's bulk copies are complete
    report_range(p.status, half_clipped(hmax));
    // every MMA has completed before Tensor Memory is released (after a timed
    // out wait one may still run); each item completed two phases of bar_mma
    if (tid == 0) {
        mma_commit(&bar_mma);
        if (!mbar_wait(&bar_mma, 0)) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tm, C::kTmemCols);
    }
}

template <int D, bool F16, bool EXACT>
cudaError_t launch_intra_pass(const Params &p, cudaStream_t s) {
    using C = IntraCfg<D>;
    auto kern = gdn2_tc_intra_kernel<D, F16, EXACT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaGetLastError();
    const long long items = static_cast<long long>(p.NCmax) * p.HV;  // upper bound; the kernel reads the count
    const int grid = static_cast<int>(items < 2ll * sms ? items : 2ll * sms);
    if (grid <= 0) return cudaGetLastError();
    return launch_chained(kern, dim3(grid), dim3(kIntraThreads), C::kSmem, s, p);
}

// Both passes: every item, then the exact pass over the items the first one
// listed (its CTAs return at once when the list is empty).  Without g there
// is no decay, so no item can be listed and the exact pass is not launched.
template <int D, bool F16>
cudaError_t launch_intra(const Params &p, cudaStream_t s) {
    const cudaError_t e = launch_intra_pass<D, F16, false>(p, s);
    if (e != cudaSuccess || !p.has_g) return e;
    return launch_intra_pass<D, F16, true>(p, s);
}

}  // namespace

size_t tc_record_bytes(int D) { return D == 64 ? Rec<64>::bytes : Rec<128>::bytes; }

cudaError_t launch_tc_intra(const Params &p, cudaStream_t s) {
    if (p.K == 64) return p.in_f16 ? launch_intra<64, true>(p, s) : launch_intra<64, false>(p, s);
    return p.in_f16 ? launch_intra<128, true>(p, s) : launch_intra<128, false>(p, s);
}

}  // namespace gdn2
