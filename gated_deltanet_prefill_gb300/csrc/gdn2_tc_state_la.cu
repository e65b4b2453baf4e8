// Tensor-core state-passing kernels with a one-chunk lookahead (K = V = 128):
// gdn2_tc_state_la_kernel for 64-column V tiles and gdn2_tc_state_la128_kernel
// for 128-column tiles (its layout at the second kernel).  They run the
// sequential pass and, instantiated with SCAN, the transition and replay
// launches of the chunk-parallel pass.
//
// The plain state kernel runs one dependent chain per chunk: S image ->
// [Qe ; Wt] S -> U = Ut - Wt S -> S += Kd^T U -> next S image.  Here the next
// chunk's product with the state is split along the state update.  With
// A1 = [Qe ; Wt] (the record's 128-row A operand) and E_c = diag(eGL_c) S_c
// (the state with its rows rescaled by e^{G_L}),
//   A1_{c+1} S_{c+1} = A1_{c+1} E_c + (A1_{c+1} Kd_c^T) U_c,
// so the first product and XY_{c+1} = A1_{c+1} Kd_c^T need no U and run ahead;
// only XY_{c+1} U_c (K = 64) stands between U_c and U_{c+1}.  The rows Qe give
// the output's inter-chunk term the same way.  Per chunk c (chunk 0 takes
// D_0 = A1_0 S_0 directly):
//   Ma  D_c  = A1_c img(E_{c-1})           fp16 image of E, MN-major B
//   Mb  XY_c = A1_c Kd_{c-1}^T             fp32 in TMEM -> fp16 A operand in TMEM
//   Mc  D_c += XY_c img(U_{c-1})           A from Tensor Memory
//   epi U_c  = Ut_c - D_c[64:128]          fp16 image (two buffers)
//   Me  S    = E_c + Kd_c^T U_c            S_{c+1}, fp32 in TMEM
//   Md  D_c[0:64] += P_c U_c               output -> scale -> global
// Tensor pipe order per chunk c: Ma_{c+1} once E_c is ready; once U_c and
// XY_{c+1} are, Mc_{c+1} (the chain), Me_c, Md_c in one burst; the stage of
// chunk c is released; then Mb_{c+2}.  Accumulators D are triple-buffered so
// that an output epilogue never delays the next chunk's first product.
//
// Warps (24): 0 bulk-copy producer, 1 MMA issuer (and TMEM owner), 2-3 and
// 6-7 U epilogue (D rows 64-127 live in TMEM lane quarters 2 and 3), 4-5
// output epilogue, 8-15 state epilogue (E = eGL S -> fp16 image and back to
// TMEM), 16-23 XY epilogue (fp32 -> fp16 A operand).  Every wait is
// time-bounded; a timeout sets the device status word and the CTA unwinds.
#include "gdn2_internal.cuh"
#include "gdn2_record.cuh"
#include "gdn2_tc.cuh"



namespace gdn2 {

namespace {

using namespace tc;

constexpr int kLaThreads = 768;

struct LaCfg {
    static constexpr int D = 128, VT = 64, NSTAGE = 3;
    // a stage holds the record's P, A1, Kd^T (one contiguous copy) and the
    // tile's 64 columns of Ut; the stages' eGL vectors live after the images
    static constexpr uint32_t sP = 0;
    static constexpr uint32_t sA1 = 8192;
    static constexpr uint32_t sKdT = sA1 + 2 * 16384;
    static constexpr uint32_t sUt = sKdT + 2 * 8192;
    static constexpr uint32_t kStage = sUt + 8192;
    static constexpr uint32_t oE = NSTAGE * kStage;         // E image: [128 K rows][64 columns] fp16
    static constexpr uint32_t oU = oE + D * 128;            // two U images: [64 t][64 columns] fp16
    static constexpr uint32_t oEGL = oU + 2 * 8192;         // eGL per stage, D fp32
    static constexpr uint32_t kSmem = oEGL + NSTAGE * D * 4 + 1024;  // + alignment slack
    static constexpr uint32_t kLoadBytes = Rec<D>::mma_prefix + 8192 + D * 4;
    // TMEM columns: S (64), D x 3 (64 each), XY fp32 (64), XY fp16 A operand (32)
    static constexpr uint32_t cS = 0, cD = 64, cXY = 256, cXa = 320, kTmemCols = 512;
    static_assert(Rec<D>::mma_prefix == sUt, "P, A1 and Kd^T are one contiguous copy");
    static_assert(kStage % 1024 == 0 && oE % 1024 == 0 && oU % 1024 == 0, "128B-swizzle operands");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void set_timeout_la(const Params &p) {
    atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
}

// SCAN: the replay of the chunk-parallel pass (sc_mode 2), as in the
// 128-column kernel below; the transitions always take 128-column tiles.
template <bool SCAN>
__global__ void __launch_bounds__(kLaThreads, 1) gdn2_tc_state_la_kernel(Params p) {
    using C = LaCfg;
    constexpr int D = C::D, VT = C::VT, NSTAGE = C::NSTAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t full_bar[NSTAGE], empty_bar[NSTAGE];
    __shared__ uint64_t s_ready, s_full, u_ready, xy_full, xy_ready, drain;
    __shared__ uint64_t d_full[3], o_full[3], d_free[3];
    __shared__ uint32_t tmem_slot;

    pdl_wait();  // the records (intra kernel) or incoming states (combine) are complete
    if (p.status[0] != GDN2_OK) return;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // one CTA per (sequence in longest-first order, value head, segment,
    // 64-column tile), the tile fastest (scan_cta); the sequential pass has
    // one segment, the replay segments 1 .. P - 1
    int P = 1, tile, seg = 0, hv, n, first, nck, c_lo = 0;
    if constexpr (SCAN) {
        P = p.sc_P;
        const ScanCta sc = scan_cta(blockIdx.x, 2, P, p.HV, 2);
        tile = sc.tile;
        hv = sc.hv;
        seg = sc.seg;
        n = chk(p.seq_order[sc.rank], 0, p.N, 301, p.status);
        const int seq0 = p.seq_first[n], nck_all = p.seq_first[n + 1] - seq0;
        const int L = (nck_all + P - 1) / P;
        c_lo = min(seg * L, nck_all);
        first = seq0 + c_lo;
        nck = min(c_lo + L, nck_all) - c_lo;
    } else {
        tile = blockIdx.x % 2;
        hv = (blockIdx.x / 2) % p.HV;
        n = chk(p.seq_order[blockIdx.x / (2 * p.HV)], 0, p.N, 301, p.status);
        first = p.seq_first[n];
        nck = p.seq_first[n + 1] - first;
    }
    const int v0 = tile * VT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&s_ready, 256);
        mbar_init(&s_full, 1);
        mbar_init(&u_ready, 128);
        mbar_init(&xy_full, 1);
        mbar_init(&xy_ready, 256);
        mbar_init(&drain, 1);
        for (int b = 0; b < 3; ++b) {
            mbar_init(&d_full[b], 1);
            mbar_init(&o_full[b], 1);
            mbar_init(&d_free[b], 64);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_slot + C::cS, tXY = tmem_slot + C::cXY, tXa = tmem_slot + C::cXa;
    auto tD = [&](int c) { return tmem_slot + C::cD + 64u * static_cast<uint32_t>(c % 3); };
    auto stage = [&](int c) { return sm + (c % NSTAGE) * C::kStage; };
    const uint32_t sE = smem_u32(sm + C::oE);
    auto sU = [&](int c) { return smem_u32(sm + C::oU + (c & 1) * 8192); };

    if (warp == 0) {
        // ------------------------------------------------ bulk-copy producer
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nck && ok; ++i) {
                const int s = i % NSTAGE;
                if (i >= NSTAGE && !mbar_wait(&empty_bar[s], ((i / NSTAGE) - 1) & 1)) {
                    set_timeout_la(p);
                    ok = false;
                    break;
                }
                const uint8_t *rec =
                    p.rec + (static_cast<size_t>(chk(first + i, 0, p.status[1], 302, p.status)) * p.HV + hv) *
                                Rec<D>::bytes;
                mbar_arrive_expect_tx(&full_bar[s], C::kLoadBytes);
                bulk_g2s(stage(i) + C::sP, rec + Rec<D>::P, Rec<D>::mma_prefix, &full_bar[s]);
                bulk_g2s(stage(i) + C::sUt, rec + Rec<D>::Ut + tile * 8192, 8192, &full_bar[s]);
                bulk_g2s(sm + C::oEGL + s * D * 4, rec + Rec<D>::eGL, D * 4, &full_bar[s]);
                ++issued;
            }
            if (!ok) {  // let every copy in flight land before the CTA exits
                for (int i = issued - NSTAGE > 0 ? issued - NSTAGE : 0; i < issued; ++i)
                    mbar_wait(&full_bar[i % NSTAGE], (i / NSTAGE) & 1);
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        // Its waits park the thread (the other roles poll), and the chunk's
        // dependent instructions go out in as few bursts as the inputs allow:
        // MMAs issued in short bursts pay the tensor pipe's fill latency per
        // burst.  On two sequences of 16384 tokens with 32 value heads: 0.465
        // -> 0.438 ms (parked waits) -> 0.424 ms (the stage released before
        // the XY product, Mc/Me/Md in one burst) -> 0.421 ms (Ma issued as
        // soon as E_c is ready).
        if (lane == 0 && nck > 0) {
            constexpr uint32_t idB = idesc_fp16(128, VT, false, true);   // B = state / U image (MN-major)
            constexpr uint32_t idS = idesc_fp16(128, VT, true, true);    // A = Kd^T (MN-major)
            constexpr uint32_t idXY = idesc_fp16(128, 64, false, false); // B = Kd^T read K-major (N = tokens)
            bool ok = true;
            // descriptors are linear in the address (below 256 KB): a k-step
            // adds a constant to the base descriptor
            auto kmaj = [](uint32_t rows, int kk) -> uint64_t {
                return ((kk >> 2) * rows * 128u + (kk & 3) * 32u) >> 4;
            };
            auto mnmaj = [](int kk) -> uint64_t { return static_cast<uint64_t>(kk) * (2048u >> 4); };
            const uint64_t dE = desc_mnmajor(sE, D, 0);
            auto product_a1 = [&](int j) {  // D_j = A1_j img(E)  (img(S_0) for j = 0)
                const uint64_t dA = desc_kmajor(smem_u32(stage(j) + C::sA1), 128, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_f16(tD(j), dA + kmaj(128, kk), dE + mnmaj(kk), idB, kk > 0);
            };
            auto product_xy = [&](int j) {  // XY_j = A1_j Kd_{j-1}^T
                const uint64_t dA = desc_kmajor(smem_u32(stage(j) + C::sA1), 128, 0);
                const uint64_t dK = desc_kmajor(smem_u32(stage(j - 1) + C::sKdT), 64, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_f16(tXY, dA + kmaj(128, kk), dK + kmaj(64, kk), idXY, kk > 0);
                mma_commit(&xy_full);
            };
            if (!mbar_wait_parked(&full_bar[0], 0) || !mbar_wait_parked(&s_ready, 0)) ok = false;
            if (ok) {
                tc_fence_after();
                product_a1(0);
                mma_commit(&d_full[0]);
                if (nck > 1) {
                    if (!mbar_wait_parked(&full_bar[1 % NSTAGE], 0)) {
                        ok = false;
                    } else {
                        tc_fence_after();
                        product_xy(1);
                    }
                }
            }
            for (int c = 0; c < nck && ok; ++c) {
                const bool next = c + 1 < nck;
                // E_c is ready: its image (for D_{c+1}) and Tensor Memory (for
                // the state update)
                if ((next && c + 1 >= 3 && !mbar_wait_parked(&d_free[(c + 1) % 3], ((c - 2) / 3) & 1)) ||
                    !mbar_wait_parked(&s_ready, (c + 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (next) product_a1(c + 1);
                if ((next && !mbar_wait_parked(&xy_ready, c & 1)) || !mbar_wait_parked(&u_ready, c & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dU = desc_mnmajor(sU(c), 64, 0);
                if (next) {  // the chain: D_{c+1} += XY_{c+1} U_c
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_f16_ta(tD(c + 1), tXa + 8 * kk, dU + mnmaj(kk), idB, 1);
                    mma_commit(&d_full[(c + 1) % 3]);
                }
                const uint64_t dK = desc_mnmajor(smem_u32(stage(c) + C::sKdT), 64, 0);
                const uint64_t dP = desc_kmajor(smem_u32(stage(c) + C::sP), 128, 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(tS, dK + mnmaj(kk), dU + mnmaj(kk), idS, 1);
                mma_commit(&s_full);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(tD(c), dP + kmaj(128, kk), dU + mnmaj(kk), idB, 1);
                mma_commit(&o_full[c % 3]);
                mma_commit(&empty_bar[c % NSTAGE]);
                if (c + 2 < nck) {
                    if (!mbar_wait_parked(&full_bar[(c + 2) % NSTAGE], ((c + 2) / NSTAGE) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    product_xy(c + 2);
                }
            }
            if (!ok) set_timeout_la(p);
            mma_commit(&drain);
            if (!mbar_wait_parked(&drain, 0)) set_timeout_la(p);
        }
    } else if (warp >= 8 && warp < 16) {
        // ------------------------- state epilogue: E_c = eGL_c S_c (rows = key channels)
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3, g = (warp - 8) >> 2;  // lane quarter, 32-column group
        const int row = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const size_t sblk = (static_cast<size_t>(n) * p.HV + hv) * D * D;  // this (sequence, head) block
        const bool plain = !p.state_vmajor && !p.state_bf16;           // fp32 [K][V]
        const int col0 = v0 + 32 * g;
        uint8_t *img = sm + C::oE;
        auto write_img = [&](const uint32_t (&r)[32]) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint4 v;
                v.x = pack_h2m(__uint_as_float(r[8 * cc + 0]), __uint_as_float(r[8 * cc + 1]), hmax);
                v.y = pack_h2m(__uint_as_float(r[8 * cc + 2]), __uint_as_float(r[8 * cc + 3]), hmax);
                v.z = pack_h2m(__uint_as_float(r[8 * cc + 4]), __uint_as_float(r[8 * cc + 5]), hmax);
                v.w = pack_h2m(__uint_as_float(r[8 * cc + 6]), __uint_as_float(r[8 * cc + 7]), hmax);
                *reinterpret_cast<uint4 *>(img + swz(row, 4 * g + cc)) = v;
            }
        };
        uint32_t r[32];
        // the segment's incoming state: the combined state (a later replay
        // segment) or the initial state
        const float *si = SCAN && seg > 0
                              ? p.sc_si + ((static_cast<size_t>(n) * (P - 1) + seg - 1) * p.HV + hv) * D * D
                              : nullptr;
        if (SCAN && si) {
            const float *src = si + static_cast<size_t>(row) * D + col0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(src + e);
                r[e] = __float_as_uint(x.x); r[e + 1] = __float_as_uint(x.y);
                r[e + 2] = __float_as_uint(x.z); r[e + 3] = __float_as_uint(x.w);
            }
        } else if (p.h0 && plain) {
            const float *h0 = static_cast<const float *>(p.h0) + sblk + static_cast<size_t>(row) * D + col0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(h0 + e);
                r[e] = __float_as_uint(x.x); r[e + 1] = __float_as_uint(x.y);
                r[e + 2] = __float_as_uint(x.z); r[e + 3] = __float_as_uint(x.w);
            }
        } else {  // zero, bf16 or V-major: element by element (lanes = consecutive rows)
#pragma unroll
            for (int e = 0; e < 32; ++e)
                r[e] = __float_as_uint(
                    p.h0 ? state_ld(p.h0, sblk + state_off(row, col0 + e, D, D, p.state_vmajor), p.state_bf16) : 0.f);
        }
        write_img(r);  // img(S_0) for D_0
        fence_proxy_async();
        mbar_arrive(&s_ready);
        bool ok = true;
        for (int c = 0; c < nck; ++c) {
            // S_c is in Tensor Memory (chunk 0: in registers) and the image is
            // free: after D_0's product, later after the state update (which
            // the tensor pipe runs after D_c's first product)
            if ((c == 0 ? !warp_wait(&d_full[0], 0) : !warp_wait(&s_full, (c - 1) & 1)) ||
                !warp_wait(&full_bar[c % NSTAGE], (c / NSTAGE) & 1)) {
                set_timeout_la(p);
                ok = false;
                break;
            }
            tc_fence_after();
            if (c > 0) {
                tmem_ld32(tS + lane_base + 32 * g, r);
                tmem_ld_wait();
            }
            const float egl = reinterpret_cast<const float *>(sm + C::oEGL + (c % NSTAGE) * D * 4)[row];
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * egl);
            write_img(r);
            tmem_st32(tS + lane_base + 32 * g, r);
            tmem_st_wait();
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&s_ready);
        }
        if (ok && nck > 0 && !warp_wait(&s_full, (nck - 1) & 1)) {
            set_timeout_la(p);
            ok = false;
        }
        tc_fence_after();
        // the replay writes the final state from the last segment only
        if (ok && p.hT && (!SCAN || seg == P - 1)) {
            if (nck > 0) {  // S_nck (with no chunk, S_0 is still in registers)
                tmem_ld32(tS + lane_base + 32 * g, r);
                tmem_ld_wait();
            }
            if (plain) {
                float *hT = static_cast<float *>(p.hT) + sblk + static_cast<size_t>(row) * D + col0;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(hT + e) = make_float4(
                        __uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                        __uint_as_float(r[e + 3]));
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    state_st(p.hT, sblk + state_off(row, col0 + e, D, D, p.state_vmajor), __uint_as_float(r[e]),
                             p.state_bf16);
            }
        }
        report_range(p.status, half_clipped(hmax));
    } else if (warp >= 16) {
        // ------------------- XY epilogue: fp32 accumulator -> fp16 A operand in TMEM
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3, g = (warp - 16) >> 2;  // lane quarter, 32 of the 64 token columns
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        for (int k = 0; k + 1 < nck; ++k) {  // XY of chunk k + 1
            if (!warp_wait(&xy_full, k & 1)) {
                set_timeout_la(p);
                break;
            }
            tc_fence_after();
            uint32_t r[32], h[16];
            tmem_ld32(tXY + lane_base + 32 * g, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = pack_h2m(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), hmax);
            tmem_st16(tXa + lane_base + 16 * g, h);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&xy_ready);
        }
        report_range(p.status, half_clipped(hmax));
    } else if (warp == 4 || warp == 5) {
        // ----------------------------------------- output epilogue (tokens 0-63)
        const int q = warp & 3;  // 0 or 1
        const int t = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int64_t seq_start = cu_at(p, n), seq_end = cu_at(p, n + 1);
        for (int c = 0; c < nck; ++c) {
            if (!warp_wait(&o_full[c % 3], (c / 3) & 1)) {
                set_timeout_la(p);
                break;
            }
            tc_fence_after();
            const int64_t tok = seq_start + static_cast<int64_t>(c_lo + c) * kChunk + t;
            const bool valid = tok < seq_end;
            bf16 *orow = p.o + tok * p.so_t + static_cast<int64_t>(hv) * p.so_h + v0;
#pragma unroll 1
            for (int j = 0; j < VT / 32; ++j) {
                uint32_t r[32];
                tmem_ld32(tD(c) + lane_base + 32 * j, r);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        // output at the inputs' dtype (plain round-to-nearest)
                        auto pk = [&](int e) {
                            const float a = __uint_as_float(r[8 * cc + e]) * p.scale;
                            const float b = __uint_as_float(r[8 * cc + e + 1]) * p.scale;
                            return p.in_f16 ? pack_f16_rn(a, b) : pack_bf2(a, b);
                        };
                        reinterpret_cast<uint4 *>(orow + 32 * j)[cc] = make_uint4(pk(0), pk(2), pk(4), pk(6));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&d_free[c % 3]);
        }
    } else {
        // ----------------------------------- U epilogue (D rows 64-127 = Wt S)
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3;  // 2 or 3
        const int t = 32 * (q - 2) + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int g = warp < 4 ? 0 : 1;  // 32-column group
        for (int c = 0; c < nck; ++c) {
            if (!warp_wait(&d_full[c % 3], (c / 3) & 1) || !warp_wait(&full_bar[c % NSTAGE], (c / NSTAGE) & 1)) {
                set_timeout_la(p);
                break;
            }
            tc_fence_after();
            const uint8_t *ut = stage(c) + C::sUt;
            uint8_t *dst = sm + C::oU + (c & 1) * 8192;
            uint32_t r[32];
            tmem_ld32(tD(c) + lane_base + 32 * g, r);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint4 u = *reinterpret_cast<const uint4 *>(ut + swz(t, 4 * g + cc));
                const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
                uint32_t ow[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 a = unpack_h2(uw[e]);
                    ow[e] = pack_h2m(a.x - __uint_as_float(r[8 * cc + 2 * e]), a.y - __uint_as_float(r[8 * cc + 2 * e + 1]), hmax);
                }
                *reinterpret_cast<uint4 *>(dst + swz(t, 4 * g + cc)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&u_ready);
        }
        report_range(p.status, half_clipped(hmax));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_slot, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// The same lookahead pass for 128-column tiles (one CTA per (sequence, value
// head)).  The layout differs so that it fits 227 KB of shared memory and 512
// Tensor Memory columns:
//  * a stage holds P, A1 and Kd^T (one copy, 56 KB).  A1_c's slot is dead once
//    its two products (XY_c, D_c) are done, which the state update of chunk
//    c - 1 implies; the state epilogue then writes img(E_c) there, and the
//    stage is released after D_{c+1}'s product has read it;
//  * Ut_c is copied into the U image buffer of chunk c (two buffers), and the
//    U epilogue turns it into U_c in place.  Before the first chunk the two
//    buffers hold img(S_0);
//  * two accumulators D (128 columns each) instead of three.
// Tensor Memory columns: S (128), D x 2 (128 each), XY fp32 (64), XY fp16 (32).
struct La128Cfg {
    static constexpr int D = 128, NSTAGE = 3;
    static constexpr uint32_t sP = 0;
    static constexpr uint32_t sA1 = 8192;                      // A1_c, later img(E_c)
    static constexpr uint32_t sKdT = sA1 + 2 * 16384;
    static constexpr uint32_t kStage = sKdT + 2 * 8192;         // 56 KB
    static constexpr uint32_t oU = NSTAGE * kStage;             // two [64 t][128 columns] fp16 buffers
    static constexpr uint32_t kUBytes = 2 * 8192;
    static constexpr uint32_t oEGL = oU + 2 * kUBytes;          // eGL per stage, D fp32
    // the output epilogue's token rows (256 bytes each), staged for bulk
    // copies; the 272-byte stride puts the lanes' 16-byte stores in different
    // banks
    static constexpr uint32_t oO = oEGL + NSTAGE * D * 4;
    static constexpr uint32_t kOStride = 272;
    static constexpr uint32_t kSmem = oO + 64 * kOStride + 1024;
    static constexpr uint32_t kStageBytes = Rec<D>::mma_prefix + D * 4;
    static constexpr uint32_t cS = 0, cD = 128, cXY = 384, cXa = 448, kTmemCols = 512;
    static_assert(Rec<D>::mma_prefix == kStage, "P, A1 and Kd^T are one contiguous copy");
    static_assert(Rec<D>::eGL - Rec<D>::Ut == kUBytes, "Ut of all 128 columns is one copy");
    static_assert(kStage % 1024 == 0 && oU % 1024 == 0, "128B-swizzle operands");
    static_assert(2 * kUBytes == D * 128 * 2, "img(S_0) fills both U buffers");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// SCAN = false: the sequential pass.  SCAN = true: the chunk-parallel modes of
// the plain state kernel (sc_mode 1: segment 0 replayed from the initial
// state beside the transitions [M | B] of segments 1 .. P - 2 on two
// 128-column tiles, M from the identity with no Ut and no output; sc_mode 2:
// segments 1 .. P - 1 from their incoming states).
template <bool SCAN>
__global__ void __launch_bounds__(kLaThreads, 1) gdn2_tc_state_la128_kernel(Params p) {
    using C = La128Cfg;
    constexpr int D = C::D, NSTAGE = C::NSTAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t full_bar[NSTAGE], empty_bar[NSTAGE], ut_full[2];
    __shared__ uint64_t s_ready, s_full, u_ready, xy_full, xy_ready, drain;
    __shared__ uint64_t d_full[2], o_full[2], d_free[2];
    __shared__ uint32_t tmem_slot;

    pdl_wait();  // the records (intra kernel) or incoming states (combine) are complete
    if (SCAN && p.sc_mode == 1) pdl_trigger();  // the combine may launch and wait for the transitions
    if (p.status[0] != GDN2_OK) return;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // one CTA per (sequence in longest-first order, value head, segment,
    // tile), the tile fastest (scan_cta); the sequential pass has one segment
    // and one tile.  A segment's chunks are [seg L, seg L + L) of the
    // sequence's, L = ceil(chunks / P).
    int mode = 0, P = 1, tile = 0, seg = 0, hv, n, first, nck, c_lo = 0;
    bool trans_cta = false;
    if constexpr (SCAN) {
        mode = p.sc_mode;
        P = p.sc_P;
        const ScanCta sc = scan_cta(blockIdx.x, mode, P, p.HV, 1);
        tile = sc.tile;
        hv = sc.hv;
        seg = sc.seg;
        trans_cta = sc.trans;
        n = chk(p.seq_order[sc.rank], 0, p.N, 401, p.status);
        const int seq0 = p.seq_first[n], nck_all = p.seq_first[n + 1] - seq0;
        const int L = (nck_all + P - 1) / P;
        c_lo = min(seg * L, nck_all);
        first = seq0 + c_lo;
        nck = min(c_lo + L, nck_all) - c_lo;
    } else {
        hv = blockIdx.x % p.HV;
        n = chk(p.seq_order[blockIdx.x / p.HV], 0, p.N, 401, p.status);
        first = p.seq_first[n];
        nck = p.seq_first[n + 1] - first;
    }
    const bool trans = SCAN && trans_cta, is_m = trans && tile == 0;  // is_m: columns of M (no Ut)
    // segment 0 of the transitions launch: a replay whose final state is the
    // incoming state of segment 1
    const bool to_si = SCAN && mode == 1 && !trans;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ut_full[b], 1);
            mbar_init(&d_full[b], 1);
            mbar_init(&o_full[b], 1);
            mbar_init(&d_free[b], 64);
        }
        mbar_init(&s_ready, 256);
        mbar_init(&s_full, 1);
        mbar_init(&u_ready, 128);
        mbar_init(&xy_full, 1);
        mbar_init(&xy_ready, 256);
        mbar_init(&drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_slot + C::cS, tXY = tmem_slot + C::cXY, tXa = tmem_slot + C::cXa;
    auto tD = [&](int c) { return tmem_slot + C::cD + 128u * static_cast<uint32_t>(c & 1); };
    auto stage = [&](int c) { return sm + (c % NSTAGE) * C::kStage; };
    auto ubuf = [&](int c) { return sm + C::oU + (c & 1) * C::kUBytes; };
    auto rec_of = [&](int c) {
        return p.rec + (static_cast<size_t>(chk(first + c, 0, p.status[1], 402, p.status)) * p.HV + hv) *
                           Rec<D>::bytes;
    };

    if (warp == 0) {
        // ------------------------------------------------ bulk-copy producer
        if (lane == 0 && nck > 0) {
            auto load_stage = [&](int i) {
                const int s = i % NSTAGE;
                mbar_arrive_expect_tx(&full_bar[s], C::kStageBytes);
                bulk_g2s(stage(i) + C::sP, rec_of(i) + Rec<D>::P, Rec<D>::mma_prefix, &full_bar[s]);
                bulk_g2s(sm + C::oEGL + s * D * 4, rec_of(i) + Rec<D>::eGL, D * 4, &full_bar[s]);
            };
            auto load_ut = [&](int c) {
                if (SCAN && is_m) {  // Ut = 0: the U epilogue writes -Wt S without reading the buffer
                    mbar_arrive(&ut_full[c & 1]);
                    return;
                }
                mbar_arrive_expect_tx(&ut_full[c & 1], C::kUBytes);
                bulk_g2s(ubuf(c), rec_of(c) + Rec<D>::Ut, C::kUBytes, &ut_full[c & 1]);
            };
            int st_issued = 0, ut_issued = 0;
            bool ok = true;
            for (int i = 0; i < NSTAGE && i < nck; ++i) {
                load_stage(i);
                st_issued = i + 1;
            }
            // the U buffers hold img(S_0) until D_0's product is done
            if (!mbar_wait(&d_full[0], 0)) {
                ok = false;
            } else {
                for (int c = 0; c < 2 && c < nck; ++c) {
                    load_ut(c);
                    ut_issued = c + 1;
                }
            }
            // after chunk i - 3 is done: the stage of chunk i and the U buffer
            // of chunk i - 1
            for (int i = NSTAGE; ok && i <= nck; ++i) {
                if (!mbar_wait(&empty_bar[(i - NSTAGE) % NSTAGE], ((i - NSTAGE) / NSTAGE) & 1)) {
                    ok = false;
                    break;
                }
                if (i < nck) {
                    load_stage(i);
                    st_issued = i + 1;
                }
                load_ut(i - 1);
                ut_issued = i;
            }
            if (!ok) {  // let every copy in flight land before the CTA exits
                set_timeout_la(p);
                for (int i = st_issued - NSTAGE > 0 ? st_issued - NSTAGE : 0; i < st_issued; ++i)
                    mbar_wait(&full_bar[i % NSTAGE], (i / NSTAGE) & 1);
                for (int c = ut_issued - 2 > 0 ? ut_issued - 2 : 0; c < ut_issued; ++c)
                    mbar_wait(&ut_full[c & 1], (c >> 1) & 1);
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        // Parked waits, as in the 64-column kernel.  Here D_{c+1}'s first
        // product goes out as soon as E_c is ready, ahead of the wait for U_c:
        // at 128 columns the U epilogue is the longer chain (long workload,
        // 4 x 32768 tokens: state stage 1.158 -> 1.113 ms, against 1.184 ms
        // for the plain kernel).  Each pair of waits takes first the barrier
        // that usually completes first (1.115 -> 1.102 ms).
        if (lane == 0 && nck > 0) {
            constexpr uint32_t idB = idesc_fp16(128, 128, false, true);   // B = state / U image (MN-major)
            constexpr uint32_t idS = idesc_fp16(128, 128, true, true);    // A = Kd^T (MN-major)
            constexpr uint32_t idXY = idesc_fp16(128, 64, false, false);  // B = Kd^T read K-major (N = tokens)
            bool ok = true;
            auto kmaj = [](uint32_t rows, int kk) -> uint64_t {
                return ((kk >> 2) * rows * 128u + (kk & 3) * 32u) >> 4;
            };
            auto mnmaj = [](int kk) -> uint64_t { return static_cast<uint64_t>(kk) * (2048u >> 4); };
            // D_j = A1_j img  (img(S_0) in the U buffers for j = 0, img(E_{j-1}) after)
            auto product_a1 = [&](int j, uint32_t img) {
                const uint64_t dA = desc_kmajor(smem_u32(stage(j) + C::sA1), 128, 0);
                const uint64_t dE = desc_mnmajor(img, D, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_f16(tD(j), dA + kmaj(128, kk), dE + mnmaj(kk), idB, kk > 0);
            };
            auto product_xy = [&](int j) {  // XY_j = A1_j Kd_{j-1}^T
                const uint64_t dA = desc_kmajor(smem_u32(stage(j) + C::sA1), 128, 0);
                const uint64_t dK = desc_kmajor(smem_u32(stage(j - 1) + C::sKdT), 64, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_f16(tXY, dA + kmaj(128, kk), dK + kmaj(64, kk), idXY, kk > 0);
                mma_commit(&xy_full);
            };
            if (!mbar_wait_parked(&full_bar[0], 0) || !mbar_wait_parked(&s_ready, 0)) ok = false;
            if (ok) {
                tc_fence_after();
                product_a1(0, smem_u32(sm + C::oU));
                mma_commit(&d_full[0]);
                if (nck > 1) {
                    if (!mbar_wait_parked(&full_bar[1 % NSTAGE], 0)) {
                        ok = false;
                    } else {
                        tc_fence_after();
                        product_xy(1);
                    }
                }
            }
            for (int c = 0; c < nck && ok; ++c) {
                const bool next = c + 1 < nck;
                // E_c (image in stage c, and Tensor Memory), U_c and XY_{c+1}
                // are ready, and D_{c+1}'s buffer is free
                if ((next && c + 1 >= 2 && !mbar_wait_parked(&d_free[(c + 1) & 1], ((c - 1) >> 1) & 1)) ||
                    !mbar_wait_parked(&s_ready, (c + 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (next) product_a1(c + 1, smem_u32(stage(c) + C::sA1));
                if ((next && !mbar_wait_parked(&xy_ready, c & 1)) || !mbar_wait_parked(&u_ready, c & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dU = desc_mnmajor(smem_u32(ubuf(c)), 64, 0);
                if (next) {
                    // the chain: D_{c+1} += XY_{c+1} U_c
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_f16_ta(tD(c + 1), tXa + 8 * kk, dU + mnmaj(kk), idB, 1);
                    mma_commit(&d_full[(c + 1) & 1]);
                }
                const uint64_t dK = desc_mnmajor(smem_u32(stage(c) + C::sKdT), 64, 0);
                const uint64_t dP = desc_kmajor(smem_u32(stage(c) + C::sP), 128, 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(tS, dK + mnmaj(kk), dU + mnmaj(kk), idS, 1);
                mma_commit(&s_full);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(tD(c), dP + kmaj(128, kk), dU + mnmaj(kk), idB, 1);
                mma_commit(&o_full[c & 1]);
                mma_commit(&empty_bar[c % NSTAGE]);  // stage c and U buffer c are read
                if (c + 2 < nck) {
                    if (!mbar_wait_parked(&full_bar[(c + 2) % NSTAGE], ((c + 2) / NSTAGE) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    product_xy(c + 2);
                }
            }
            if (!ok) set_timeout_la(p);
            mma_commit(&drain);
            if (!mbar_wait_parked(&drain, 0)) set_timeout_la(p);
        }
    } else if (warp >= 8 && warp < 16) {
        // ------------------------- state epilogue: E_c = eGL_c S_c (rows = key channels)
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3, g2 = (warp - 8) >> 2;  // lane quarter, 64-column half
        const int row = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const size_t sblk = (static_cast<size_t>(n) * p.HV + hv) * D * D;  // this (sequence, head) block
        const bool plain = !p.state_vmajor && !p.state_bf16;           // fp32 [K][V]
        // one 32-column group of img (MN-major, two 64-column blocks of [128 rows][128 B])
        auto write_img = [&](uint8_t *img, int gcol, const uint32_t (&r)[32]) {
            uint8_t *blk = img + (gcol >> 1) * (D * 128);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint4 v;
                v.x = pack_h2m(__uint_as_float(r[8 * cc + 0]), __uint_as_float(r[8 * cc + 1]), hmax);
                v.y = pack_h2m(__uint_as_float(r[8 * cc + 2]), __uint_as_float(r[8 * cc + 3]), hmax);
                v.z = pack_h2m(__uint_as_float(r[8 * cc + 4]), __uint_as_float(r[8 * cc + 5]), hmax);
                v.w = pack_h2m(__uint_as_float(r[8 * cc + 6]), __uint_as_float(r[8 * cc + 7]), hmax);
                *reinterpret_cast<uint4 *>(blk + swz(row, 4 * (gcol & 1) + cc)) = v;
            }
        };
        // the segment's incoming state: [I | 0] (transitions), the combined
        // state (a later replay segment) or the initial state
        const float *si = SCAN && mode == 2 && seg > 0
                              ? p.sc_si + ((static_cast<size_t>(n) * (P - 1) + seg - 1) * p.HV + hv) * D * D
                              : nullptr;
        auto load_h0 = [&](int gcol, uint32_t (&r)[32]) {
            const int col0 = 32 * gcol;
            if (SCAN && trans) {
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(is_m && row == col0 + e ? 1.f : 0.f);
            } else if (SCAN && si) {
                const float *src = si + static_cast<size_t>(row) * D + col0;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(src + e);
                    r[e] = __float_as_uint(x.x); r[e + 1] = __float_as_uint(x.y);
                    r[e + 2] = __float_as_uint(x.z); r[e + 3] = __float_as_uint(x.w);
                }
            } else if (p.h0 && plain) {
                const float *h0 = static_cast<const float *>(p.h0) + sblk + static_cast<size_t>(row) * D + col0;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(h0 + e);
                    r[e] = __float_as_uint(x.x); r[e + 1] = __float_as_uint(x.y);
                    r[e + 2] = __float_as_uint(x.z); r[e + 3] = __float_as_uint(x.w);
                }
            } else {  // zero, bf16 or V-major: element by element (lanes = consecutive rows)
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    r[e] = __float_as_uint(
                        p.h0 ? state_ld(p.h0, sblk + state_off(row, col0 + e, D, D, p.state_vmajor), p.state_bf16) : 0.f);
            }
        };
        uint32_t r[32];
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {  // img(S_0) for D_0, in the U buffers
            load_h0(2 * g2 + h, r);
            write_img(sm + C::oU, 2 * g2 + h, r);
        }
        fence_proxy_async();
        mbar_arrive(&s_ready);
        bool ok = true;
        for (int c = 0; c < nck; ++c) {
            // S_c is in Tensor Memory (chunk 0: h0), and A1_c's slot is free:
            // after D_0's product, later after the state update (which the
            // tensor pipe runs after D_c's product)
            if ((c == 0 ? !warp_wait(&d_full[0], 0) : !warp_wait(&s_full, (c - 1) & 1)) ||
                !warp_wait(&full_bar[c % NSTAGE], (c / NSTAGE) & 1)) {
                set_timeout_la(p);
                ok = false;
                break;
            }
            tc_fence_after();
            const float egl = reinterpret_cast<const float *>(sm + C::oEGL + (c % NSTAGE) * D * 4)[row];
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int gcol = 2 * g2 + h;
                if (c > 0) {
                    tmem_ld32(tS + lane_base + 32 * gcol, r);
                    tmem_ld_wait();
                } else {
                    load_h0(gcol, r);
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * egl);
                write_img(stage(c) + C::sA1, gcol, r);
                tmem_st32(tS + lane_base + 32 * gcol, r);
                tmem_st_wait();
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&s_ready);
        }
        if (ok && nck > 0 && !warp_wait(&s_full, (nck - 1) & 1)) {
            set_timeout_la(p);
            ok = false;
        }
        tc_fence_after();
        // a transition writes [M | B], segment 0 of the transitions launch
        // sc_si unit (n, 0); the replay writes the final state from the last
        // segment only
        const bool write_final = (SCAN && trans) || to_si || (p.hT && (mode == 0 || seg == P - 1));
        if (ok && write_final) {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int col0 = 32 * (2 * g2 + h);
                if (nck > 0) {  // S_nck (with no chunk, S_0)
                    tmem_ld32(tS + lane_base + col0, r);
                    tmem_ld_wait();
                } else {
                    load_h0(2 * g2 + h, r);
                }
                if (SCAN && trans) {
                    const size_t u = (static_cast<size_t>(n) * (P - 1) + seg) * p.HV + hv;
                    float *tr = p.sc_tr + u * D * (2 * D) + static_cast<size_t>(row) * (2 * D) + tile * D + col0;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(tr + e) = make_float4(
                            __uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                            __uint_as_float(r[e + 3]));
                    if (is_m) {  // M's bf16 hi and lo parts as the combine's A operand images (row = M row)
                        uint8_t *img = p.sc_mimg + u * (2 * 32768);
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float a = __uint_as_float(r[8 * cc + 2 * e]), b = __uint_as_float(r[8 * cc + 2 * e + 1]);
                                hi[e] = pack_bf2(a, b);
                                const float2 hb = unpack_bf2(hi[e]);
                                lo[e] = pack_bf2(a - hb.x, b - hb.y);
                            }
                            const int chunk = col0 / 8 + cc;  // 8-column chunk of the K index
                            const uint32_t off = (chunk / 8) * 16384u + swz(row, chunk % 8);
                            *reinterpret_cast<uint4 *>(img + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            *reinterpret_cast<uint4 *>(img + 32768 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        }
                    }
                } else if (to_si) {  // fp32 [K][V]
                    float *dst = p.sc_si + static_cast<size_t>(n) * (P - 1) * p.HV * D * D +
                                 static_cast<size_t>(hv) * D * D + static_cast<size_t>(row) * D + col0;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + e) = make_float4(
                            __uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                            __uint_as_float(r[e + 3]));
                } else if (plain) {
                    float *hT = static_cast<float *>(p.hT) + sblk + static_cast<size_t>(row) * D + col0;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(hT + e) = make_float4(
                            __uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                            __uint_as_float(r[e + 3]));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        state_st(p.hT, sblk + state_off(row, col0 + e, D, D, p.state_vmajor), __uint_as_float(r[e]),
                                 p.state_bf16);
                }
            }
        }
        report_range(p.status, half_clipped(hmax));
    } else if (warp >= 16) {
        // ------------------- XY epilogue: fp32 accumulator -> fp16 A operand in TMEM
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3, g = (warp - 16) >> 2;  // lane quarter, 32 of the 64 token columns
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        for (int k = 0; k + 1 < nck; ++k) {  // XY of chunk k + 1
            if (!warp_wait(&xy_full, k & 1)) {
                set_timeout_la(p);
                break;
            }
            tc_fence_after();
            uint32_t r[32], h[16];
            tmem_ld32(tXY + lane_base + 32 * g, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = pack_h2m(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), hmax);
            tmem_st16(tXa + lane_base + 16 * g, h);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&xy_ready);
        }
        report_range(p.status, half_clipped(hmax));
    } else if (warp == 4 || warp == 5) {
        // ----------------------------------------- output epilogue (tokens 0-63)
        const int q = warp & 3;  // 0 or 1
        const int t = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int64_t seq_start = cu_at(p, n), seq_end = cu_at(p, n + 1);
        uint8_t *srow = sm + C::oO + t * C::kOStride;  // this lane's token row, staged
        for (int c = 0; c < nck; ++c) {
            if (!warp_wait(&o_full[c & 1], (c >> 1) & 1)) {
                set_timeout_la(p);
                break;
            }
            tc_fence_after();
            const int64_t tok = seq_start + static_cast<int64_t>(c_lo + c) * kChunk + t;
            const bool valid = !trans && tok < seq_end;
            bf16 *orow = p.o + tok * p.so_t + static_cast<int64_t>(hv) * p.so_h;
            bulk_wait_read0();  // the previous chunk's row copy has read the staging row
#pragma unroll 1
            for (int j = 0; j < D / 32; ++j) {
                uint32_t r[32];
                tmem_ld32(tD(c) + lane_base + 32 * j, r);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        // output at the inputs' dtype (plain round-to-nearest)
                        auto pk = [&](int e) {
                            const float a = __uint_as_float(r[8 * cc + e]) * p.scale;
                            const float b = __uint_as_float(r[8 * cc + e + 1]) * p.scale;
                            return p.in_f16 ? pack_f16_rn(a, b) : pack_bf2(a, b);
                        };
                        *reinterpret_cast<uint4 *>(srow + 64 * j + 16 * cc) = make_uint4(pk(0), pk(2), pk(4), pk(6));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&d_free[c & 1]);
            if (valid) {  // the row (256 bytes) by one bulk copy of this lane, after the D buffer is released
                fence_proxy_async();
                bulk_s2g(orow, srow, D * 2);
                bulk_commit();
            }
        }
        bulk_wait0();
    } else {
        // ------------------- U epilogue (D rows 64-127 = Wt S): U = Ut - Wt S in place
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3;  // 2 or 3
        const int t = 32 * (q - 2) + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int g = warp < 4 ? 0 : 1;  // 64-column block
        for (int c = 0; c < nck; ++c) {
            if (!warp_wait(&d_full[c & 1], (c >> 1) & 1) || !warp_wait(&ut_full[c & 1], (c >> 1) & 1)) {
                set_timeout_la(p);
                break;
            }
            tc_fence_after();
            uint8_t *blk = ubuf(c) + g * 8192;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
                tmem_ld32(tD(c) + lane_base + 64 * g + 32 * h, r);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint4 *at = reinterpret_cast<uint4 *>(blk + swz(t, 4 * h + cc));
                    const uint4 u = SCAN && is_m ? make_uint4(0, 0, 0, 0) : *at;
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
                    uint32_t ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 a = unpack_h2(uw[e]);
                        ow[e] = pack_h2m(a.x - __uint_as_float(r[8 * cc + 2 * e]),
                                        a.y - __uint_as_float(r[8 * cc + 2 * e + 1]), hmax);
                    }
                    *at = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&u_ready);
        }
        report_range(p.status, half_clipped(hmax));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_slot, C::kTmemCols);
    }
}

}  // namespace

cudaError_t launch_tc_state_la(const Params &p, cudaStream_t s) {
    if (p.sc_mode == 1) return cudaErrorInvalidValue;  // transitions: 128-column tiles only
    auto kern = p.sc_mode == 0 ? gdn2_tc_state_la_kernel<false> : gdn2_tc_state_la_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LaCfg::kSmem);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.N) * p.HV * scan_ctas_per_group(p.sc_mode, p.sc_P, 2);
    if (ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    if (ctas > 0) return launch_chained(kern, dim3(static_cast<unsigned>(ctas)), dim3(kLaThreads), LaCfg::kSmem, s, p);
    return cudaGetLastError();
}

cudaError_t launch_tc_state_la128(const Params &p, cudaStream_t s) {
    auto kern = p.sc_mode == 0 ? gdn2_tc_state_la128_kernel<false> : gdn2_tc_state_la128_kernel<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, La128Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.N) * p.HV * scan_ctas_per_group(p.sc_mode, p.sc_P, 1);
    if (ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    if (ctas > 0) return launch_chained(kern, dim3(static_cast<unsigned>(ctas)), dim3(kLaThreads), La128Cfg::kSmem, s, p);
    return cudaGetLastError();
}

}  // namespace gdn2
