// Tensor-core state-passing kernel with the output fused in.
//
// One CTA per (sequence, value head, V tile of VT columns) walks the
// sequence's chunks in order (the inter-chunk recurrence is sequential; V
// columns of S evolve independently, so V tiles are exact).  The state S
// (D x VT fp32) stays in Tensor Memory for the whole sequence.  Per chunk,
// with the intra kernel's record (gdn2_record.cuh):
//   MMA1  D1 = [Qe ; Wt] x S_fp16          (M=128, N=VT, K=D)
//   epi   U  = Ut - (Wt S)  -> fp16 smem   (rows 64-127 of D1)
//   MMA3  S  += Kd^T x U                   (M=128, K=64), S pre-scaled by eGL
//   MMA2  D1[0:64] += P x U                (M=128, K=64; rows 64-127 dead)
//   epi   o = scale * D1[0:64] -> bf16 global
// (the state update is issued first: it is on the chunk chain, the output
// product is not).  For 64-column tiles of the sequential pass the
// lookahead kernel (gdn2_tc_state_la.cu) is used instead.
// which is the FlashRT page's WY chain (chunk_h then output_o) fused into one
// pass, with burn-gdn2's "in-loop output phase".
//
// Warp roles (24 warps): 0 bulk-copy producer, 1 MMA issuer (and TMEM owner),
// 8-23 state epilogue (S -> fp16 operand, S *= eGL; four warps per TMEM lane
// quarter, one 32-column group each), 2-3 and 6-7 U epilogue (the Wt S rows
// live in lane quarters 2 and 3; two warps per quarter, half the columns
// each), 4-5 output epilogue.  Every wait is time-bounded; a timeout sets the device
// status word and the CTA unwinds.  Operands are fp16 (10-bit mantissa,
// saturating at +-65504); accumulation and the carried state are fp32.
#include <stdlib.h>

#include "gdn2_internal.cuh"
#include "gdn2_record.cuh"
#include "gdn2_tc.cuh"

namespace gdn2 {

namespace {

using namespace tc;

constexpr int kStateThreads = 768;

template <int D, int VT, int NSTAGE>
struct StateCfg {
    static constexpr uint32_t sP = 0;
    static constexpr uint32_t sA1 = 8192;
    static constexpr uint32_t sKdT = sA1 + (D / 64) * 16384;
    static constexpr uint32_t sZero = sKdT + (D / 64) * 8192;        // 8 KB zeros when D == 64
    static constexpr uint32_t sUt = sZero + (D == 64 ? 8192 : 0);
    static constexpr uint32_t sEGL = sUt + (VT / 64) * 8192;
    static constexpr uint32_t kStage = (sEGL + D * 4 + 1023) / 1024 * 1024;
    static constexpr uint32_t oS = NSTAGE * kStage;                   // S fp16, MN-major B
    static constexpr uint32_t oU = oS + (VT / 64) * D * 128;          // U fp16, MN-major B
    static constexpr uint32_t kSmem = oU + (VT / 64) * 8192 + 1024;   // + alignment slack
    static constexpr uint32_t kLoadBytes = Rec<D>::mma_prefix + (VT / 64) * 8192 + D * 4;
    static constexpr uint32_t kTmemCols = 3 * VT <= 256 ? 256 : 512;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void set_timeout(const Params &p) {
    atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
}

// SCAN = false: the sequential pass (sc_mode 0), compiled without the
// chunk-parallel modes' branches.
template <int D, int VT, int NSTAGE, bool SCAN>
__global__ void __launch_bounds__(kStateThreads, 1) gdn2_tc_state_kernel(Params p) {
    using C = StateCfg<D, VT, NSTAGE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t full_bar[NSTAGE], empty_bar[NSTAGE];
    __shared__ uint64_t s_ready, u_ready, s_full, drain;
    __shared__ uint64_t d1_full[2], o_full[2], d1_free[2];
    __shared__ uint32_t tmem_slot;

    pdl_wait();  // the records (intra kernel) or incoming states (combine) are complete
    if (SCAN && p.sc_mode == 1) pdl_trigger();  // the combine may launch and wait for the transitions
    if (p.status[0] != GDN2_OK) return;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // A CTA takes one (sequence, segment, value head, tile) (scan_cta); the
    // segment's chunks are [seg L, seg L + L) of the sequence's, L =
    // ceil(chunks / segments).  A transition's tiles cover the K + V columns
    // of [M | B]: M columns start from the identity and take no Ut
    // (S_out = M S_in + B).
    const int mode = SCAN ? p.sc_mode : 0;
    const int P = mode == 0 ? 1 : p.sc_P;
    const ScanCta sc = scan_cta(blockIdx.x, mode, P, p.HV, D / VT);
    const int tile = sc.tile, hv = sc.hv, seg = sc.seg;
    const int n = chk(p.seq_order[sc.rank], 0, p.N, 201, p.status);
    const bool trans = sc.trans;
    const int col0 = tile * VT;                     // first column of this tile
    const bool is_m = trans && col0 < D;            // a tile of M
    const int v0 = trans ? (is_m ? 0 : col0 - D) : col0;
    const int seq0 = p.seq_first[n], nck_all = p.seq_first[n + 1] - seq0;
    const int L = (nck_all + P - 1) / P;
    const int c_lo = min(seg * L, nck_all), c_hi = min(c_lo + L, nck_all);
    const int first = seq0 + c_lo, nck = c_hi - c_lo;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&s_ready, 512);
        mbar_init(&u_ready, 128);
        mbar_init(&s_full, 1);
        mbar_init(&drain, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&d1_full[b], 1);
            mbar_init(&o_full[b], 1);
            mbar_init(&d1_free[b], 64);
        }
        fence_mbar_init();
    }
    if (D == 64) {  // zero rows that pad the 64-channel Kd^T operand to M = 128
        for (int s = 0; s < NSTAGE; ++s)
            for (int i = threadIdx.x; i < 8192 / 16; i += kStateThreads)
                reinterpret_cast<uint4 *>(sm + s * C::kStage + C::sZero)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_slot;
    const uint32_t tD1[2] = {tmem_slot + VT, tmem_slot + 2 * VT};
    const uint32_t sS = smem_u32(sm + C::oS), sU = smem_u32(sm + C::oU);

    if (warp == 0) {
        // ------------------------------------------------ bulk-copy producer
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nck && ok; ++i) {
                const int s = i % NSTAGE;
                if (i >= NSTAGE && !mbar_wait(&empty_bar[s], ((i / NSTAGE) - 1) & 1)) {
                    set_timeout(p);
                    ok = false;
                    break;
                }
                const uint8_t *rec =
                    p.rec + (static_cast<size_t>(chk(first + i, 0, p.status[1], 202, p.status)) * p.HV + hv) *
                                Rec<D>::bytes;
                uint8_t *st = sm + s * C::kStage;
                mbar_arrive_expect_tx(&full_bar[s], C::kLoadBytes);
                bulk_g2s(st + C::sP, rec + Rec<D>::P, Rec<D>::mma_prefix, &full_bar[s]);
                bulk_g2s(st + C::sUt, rec + Rec<D>::Ut + (v0 / 64) * 8192, (VT / 64) * 8192, &full_bar[s]);
                bulk_g2s(st + C::sEGL, rec + Rec<D>::eGL, D * 4, &full_bar[s]);
                ++issued;
            }
            if (!ok) {  // let every copy in flight land before the CTA exits
                for (int i = issued - NSTAGE > 0 ? issued - NSTAGE : 0; i < issued; ++i)
                    mbar_wait(&full_bar[i % NSTAGE], (i / NSTAGE) & 1);
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id1 = idesc_fp16(128, VT, false, true);
            constexpr uint32_t id3 = idesc_fp16(128, VT, true, true);
            // descriptors are linear in the address (below 256 KB): a k-step
            // adds a constant to the base descriptor
            auto kmaj = [](uint32_t rows, int kk) -> uint64_t {
                return ((kk >> 2) * rows * 128u + (kk & 3) * 32u) >> 4;
            };
            auto mnmaj = [](int kk) -> uint64_t { return static_cast<uint64_t>(kk) * (2048u >> 4); };
            const uint64_t dS = desc_mnmajor(sS, D, 0), dU = desc_mnmajor(sU, 64, 0);
            for (int i = 0; i < nck; ++i) {
                const int s = i % NSTAGE, b = i & 1;
                if (!mbar_wait(&full_bar[s], (i / NSTAGE) & 1) || !mbar_wait(&s_ready, i & 1) ||
                    (i >= 2 && !mbar_wait(&d1_free[b], ((i >> 1) - 1) & 1))) {
                    set_timeout(p);
                    break;
                }
                tc_fence_after();
                const uint32_t st = smem_u32(sm + s * C::kStage);
                const uint64_t dA1 = desc_kmajor(st + C::sA1, 128, 0), dKd = desc_mnmajor(st + C::sKdT, 64, 0),
                               dP = desc_kmajor(st + C::sP, 128, 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_f16(tD1[b], dA1 + kmaj(128, kk), dS + mnmaj(kk), id1, kk > 0);
                mma_commit(&d1_full[b]);
                if (!mbar_wait(&u_ready, i & 1)) {
                    set_timeout(p);
                    break;
                }
                tc_fence_after();
                // the state update first: the S epilogue (the chain) starts
                // while the output product P U still runs
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(tS, dKd + mnmaj(kk), dU + mnmaj(kk), id3, 1);
                mma_commit(&s_full);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_f16(tD1[b], dP + kmaj(128, kk), dU + mnmaj(kk), id1, 1);
                mma_commit(&o_full[b]);
                mma_commit(&empty_bar[s]);
            }
            mma_commit(&drain);
            if (!mbar_wait(&drain, 0)) set_timeout(p);
        }
    } else if (warp >= 8) {
        // ------------------------------------- state epilogue (S rows = key channels)
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int grp = (warp - 8) >> 2;  // 32-column group of this warp
        const bool active = row < D && grp < VT / 32;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int j0 = grp, j1 = grp + 1;
        const size_t sblk = (static_cast<size_t>(n) * p.HV + hv) * D * D;  // this (sequence, head) block
        const bool plain = !p.state_vmajor && !p.state_bf16;           // fp32 [K][V]
        // a later segment of the replay pass starts from the combined state
        const float *si = mode == 2 && seg > 0
                              ? p.sc_si + ((static_cast<size_t>(n) * (P - 1) + seg - 1) * p.HV + hv) * D * D
                              : nullptr;
        if (active) {
#pragma unroll 1
            for (int j = j0; j < j1; ++j) {
                uint32_t r[32];
                if (trans) {  // [I | 0]
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(is_m && row == col0 + 32 * j + e ? 1.f : 0.f);
                } else if (si) {
                    const float *src = si + static_cast<size_t>(row) * D + v0 + 32 * j;
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(src + e);
                        r[e] = __float_as_uint(x.x); r[e + 1] = __float_as_uint(x.y);
                        r[e + 2] = __float_as_uint(x.z); r[e + 3] = __float_as_uint(x.w);
                    }
                } else if (p.h0 && plain) {
                    const float *h0 = static_cast<const float *>(p.h0) + sblk + static_cast<size_t>(row) * D + v0;
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(h0 + 32 * j + e);
                        r[e] = __float_as_uint(x.x); r[e + 1] = __float_as_uint(x.y);
                        r[e + 2] = __float_as_uint(x.z); r[e + 3] = __float_as_uint(x.w);
                    }
                } else {  // zero, bf16 or V-major: element by element (lanes = consecutive rows)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r[e] = __float_as_uint(
                            p.h0 ? state_ld(p.h0, sblk + state_off(row, v0 + 32 * j + e, D, D, p.state_vmajor),
                                            p.state_bf16)
                                 : 0.f);
                }
                tmem_st32(tS + lane_base + 32 * j, r);
            }
            tmem_st_wait();
        }
        bool ok = true;
        for (int i = 0; i < nck; ++i) {
            const int s = i % NSTAGE;
            if ((i > 0 && !warp_wait(&s_full, (i - 1) & 1)) || !warp_wait(&full_bar[s], (i / NSTAGE) & 1)) {
                set_timeout(p);
                ok = false;
                break;
            }
            tc_fence_after();
            if (active) {
                const float egl = reinterpret_cast<const float *>(sm + s * C::kStage + C::sEGL)[row];
#pragma unroll 1
                for (int j = j0; j < j1; ++j) {
                    uint32_t r[32];
                    tmem_ld32(tS + lane_base + 32 * j, r);
                    tmem_ld_wait();
                    uint8_t *dst = sm + C::oS + ((32 * j) / 64) * D * 128;
                    const int c0 = ((32 * j) % 64) / 8;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint4 v;
                        v.x = pack_h2m(__uint_as_float(r[8 * cc + 0]), __uint_as_float(r[8 * cc + 1]), hmax);
                        v.y = pack_h2m(__uint_as_float(r[8 * cc + 2]), __uint_as_float(r[8 * cc + 3]), hmax);
                        v.z = pack_h2m(__uint_as_float(r[8 * cc + 4]), __uint_as_float(r[8 * cc + 5]), hmax);
                        v.w = pack_h2m(__uint_as_float(r[8 * cc + 6]), __uint_as_float(r[8 * cc + 7]), hmax);
                        *reinterpret_cast<uint4 *>(dst + swz(row, c0 + cc)) = v;
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * egl);
                    tmem_st32(tS + lane_base + 32 * j, r);
                }
                tmem_st_wait();
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&s_ready);
        }
        if (ok && nck > 0 && !warp_wait(&s_full, (nck - 1) & 1)) {
            set_timeout(p);
            ok = false;
        }
        tc_fence_after();
        // final state: a transition writes [M | B]; segment 0 of the
        // transitions launch the incoming state of segment 1; the replay only
        // from the last segment
        const bool to_si = mode == 1 && !trans;
        const bool write_final = trans || to_si || (p.hT && (mode == 0 || seg == P - 1));
        if (ok && active && write_final) {
#pragma unroll 1
            for (int j = j0; j < j1; ++j) {
                uint32_t r[32];
                tmem_ld32(tS + lane_base + 32 * j, r);
                tmem_ld_wait();
                if (trans) {
                    float *tr = p.sc_tr +
                                ((static_cast<size_t>(n) * (P - 1) + seg) * p.HV + hv) * D * (2 * D) +
                                static_cast<size_t>(row) * (2 * D) + col0 + 32 * j;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(tr + e) =
                            make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                        __uint_as_float(r[e + 3]));
                } else if (to_si) {  // sc_si unit (n, 0): fp32 [K][V]
                    float *dst = p.sc_si + static_cast<size_t>(n) * (P - 1) * p.HV * D * D +
                                 static_cast<size_t>(hv) * D * D + static_cast<size_t>(row) * D + v0 + 32 * j;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + e) =
                            make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                        __uint_as_float(r[e + 3]));
                } else if (plain) {
                    float *hT = static_cast<float *>(p.hT) + sblk + static_cast<size_t>(row) * D + v0;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(hT + 32 * j + e) =
                            make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                        __uint_as_float(r[e + 3]));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        state_st(p.hT, sblk + state_off(row, v0 + 32 * j + e, D, D, p.state_vmajor),
                                 __uint_as_float(r[e]), p.state_bf16);
                }
            }
        }
        report_range(p.status, half_clipped(hmax));
    } else if (warp == 4 || warp == 5) {
        // ----------------------------------------- output epilogue (tokens 0-63)
        const int q = warp & 3;  // 0 or 1
        const int t = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        // chunk i of sequence n covers tokens [cu[n] + 64 i, min(cu[n] + 64 i + 64, cu[n + 1]))
        const int64_t seq_start = cu_at(p, n), seq_end = cu_at(p, n + 1);
        for (int i = 0; i < nck; ++i) {
            const int b = i & 1;
            if (!warp_wait(&o_full[b], (i >> 1) & 1)) {
                set_timeout(p);
                break;
            }
            tc_fence_after();
            const int64_t tok = seq_start + static_cast<int64_t>(c_lo + i) * kChunk + t;
            const bool valid = !trans && tok < seq_end;  // a transition writes no output
            bf16 *orow = p.o + tok * p.so_t + static_cast<int64_t>(hv) * p.so_h + v0;
#pragma unroll 1
            for (int j = 0; j < VT / 32; ++j) {
                uint32_t r[32];
                tmem_ld32(tD1[b] + lane_base + 32 * j, r);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint4 v;
                        // output at the inputs' dtype (plain round-to-nearest)
                        auto pk = [&](int e) {
                            const float a = __uint_as_float(r[8 * cc + e]) * p.scale;
                            const float b = __uint_as_float(r[8 * cc + e + 1]) * p.scale;
                            return p.in_f16 ? pack_f16_rn(a, b) : pack_bf2(a, b);
                        };
                        v.x = pk(0);
                        v.y = pk(2);
                        v.z = pk(4);
                        v.w = pk(6);
                        reinterpret_cast<uint4 *>(orow + 32 * j)[cc] = v;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&d1_free[b]);
        }
    } else if (warp == 2 || warp == 3 || warp == 6 || warp == 7) {
        // ----------------------------------- U epilogue (D1 rows 64-127 = Wt S)
        uint32_t hmax = 0;  // largest magnitude converted to fp16 (range check)
        const int q = warp & 3;  // 2 or 3
        const int t = 32 * (q - 2) + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const int j0 = warp < 4 ? 0 : VT / 64, j1 = warp < 4 ? VT / 64 : VT / 32;  // 32-column groups
        for (int i = 0; i < nck; ++i) {
            const int s = i % NSTAGE, b = i & 1;
            if (!warp_wait(&d1_full[b], (i >> 1) & 1) || !warp_wait(&full_bar[s], (i / NSTAGE) & 1)) {
                set_timeout(p);
                break;
            }
            tc_fence_after();
            const uint8_t *ut = sm + s * C::kStage + C::sUt;
#pragma unroll 1
            for (int j = j0; j < j1; ++j) {
                uint32_t r[32];
                tmem_ld32(tD1[b] + lane_base + 32 * j, r);
                tmem_ld_wait();
                const int blk = (32 * j) / 64, c0 = ((32 * j) % 64) / 8;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const uint4 u = is_m ? make_uint4(0, 0, 0, 0)  // M columns: U = -Wt S
                                         : *reinterpret_cast<const uint4 *>(ut + blk * 8192 + swz(t, c0 + cc));
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
                    uint32_t ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 a = unpack_h2(uw[e]);
                        ow[e] = pack_h2m(a.x - __uint_as_float(r[8 * cc + 2 * e]),
                                        a.y - __uint_as_float(r[8 * cc + 2 * e + 1]), hmax);
                    }
                    *reinterpret_cast<uint4 *>(sm + C::oU + blk * 8192 + swz(t, c0 + cc)) =
                        make_uint4(ow[0], ow[1], ow[2], ow[3]);
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
        tmem_dealloc(tS, C::kTmemCols);
    }
}

template <int D, int VT, int NSTAGE, bool SCAN>
cudaError_t launch_state(const Params &p, cudaStream_t s) {
    using C = StateCfg<D, VT, NSTAGE>;
    auto kern = gdn2_tc_state_kernel<D, VT, NSTAGE, SCAN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.N) * p.HV * scan_ctas_per_group(p.sc_mode, p.sc_P, D / VT);
    if (ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    if (ctas > 0) return launch_chained(kern, dim3(static_cast<unsigned>(ctas)), dim3(kStateThreads), C::kSmem, s, p);
    return cudaGetLastError();
}

// Chunk-parallel state pass, between the transition and the replay passes:
// S_in(s + 1) = M_s S_in(s) + B_s for s = 1 .. P - 2, into sc_si unit s,
// starting from S_in(1), which the transitions launch wrote into unit 0 (it
// replays segment 0 from the initial state).  One CTA per (sequence, value
// head, CW value columns); fp32 on CUDA cores, the running 128 x CW tile in
// shared memory.  The chain of P - 2 dependent steps is latency-bound: each step's M_s
// (128 x 128 fp32, shared by the head's column tiles) is copied into shared
// memory one step ahead by per-thread 16-byte asynchronous copies (rows
// padded to 132 floats, so that rows read together start 4 banks apart), so
// a step waits on shared memory only.  (Bulk copies of the 128 rows, 512 bytes
// each, were slower.)
constexpr int kCombineLd = 132;
template <int CW>
constexpr size_t combine_smem() {
    return (2 * 128 * kCombineLd + 128 * CW) * sizeof(float);
}
template <int CW>
__global__ void __launch_bounds__(256, 1) gdn2_scan_combine_kernel(Params p) {
    // thread: rows r0, r0 + 1 and 4 columns c0 .. c0 + 3 of the CTA's 128 x CW
    // tile (CW = 16): per 4 steps of k, 2 + 4 16-byte shared loads feed 32
    // multiply-adds into 8 independent accumulators
    constexpr int D = 128, NC = 4;
    static_assert(CW == 16, "256 threads cover 128 rows x 16 columns");
    extern __shared__ float4 combine_smem_raw[];
    float *Ms = reinterpret_cast<float *>(combine_smem_raw);  // [2][D][kCombineLd]
    float *Ss = Ms + 2 * D * kCombineLd;                      // [D][CW]
    pdl_wait();     // the transitions are complete
    pdl_trigger();  // the replay may launch and wait for this grid
    if (p.status[0] != GDN2_OK) return;
    const int n = blockIdx.x, hv = blockIdx.y, cbase = CW * blockIdx.z;
    const int tid = threadIdx.x, r0 = 2 * (tid / 4), c0 = NC * (tid % 4);
    const int P = p.sc_P;
    auto unit = [&](int sg) { return (static_cast<size_t>(n) * (P - 1) + sg) * p.HV + hv; };
    auto load_m = [&](int sg) {  // M_sg: the first D columns of [M | B]
        const float *tr = p.sc_tr + unit(sg) * D * (2 * D);
        float *dst = Ms + (sg & 1) * D * kCombineLd;
#pragma unroll 4
        for (int i = tid; i < D * D / 4; i += 256) {
            const int row = i / (D / 4), c4 = i % (D / 4);
            cp_async16(dst + row * kCombineLd + 4 * c4, tr + static_cast<size_t>(row) * (2 * D) + 4 * c4, 16);
        }
        cp_async_commit();
    };
    if (P > 2) load_m(1);
    {  // S_in(1): sc_si unit 0, fp32 [K][V]
        const float *s1 = p.sc_si + unit(0) * D * D;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
            *reinterpret_cast<float4 *>(Ss + (r0 + rr) * CW + c0) =
                *reinterpret_cast<const float4 *>(s1 + static_cast<size_t>(r0 + rr) * D + cbase + c0);
    }
    for (int sg = 1; sg < P - 1; ++sg) {
        const bool ahead = sg + 1 < P - 1;
        if (ahead) load_m(sg + 1);  // its buffer was last read in step sg - 1
        const float *tr = p.sc_tr + unit(sg) * D * (2 * D);
        float acc[2][NC];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float4 b = *reinterpret_cast<const float4 *>(tr + static_cast<size_t>(r0 + rr) * (2 * D) + D + cbase + c0);
            acc[rr][0] = b.x; acc[rr][1] = b.y; acc[rr][2] = b.z; acc[rr][3] = b.w;
        }
        if (ahead)
            cp_async_wait_group<1>();
        else
            cp_async_wait_group<0>();
        __syncthreads();  // M_sg and S_in(sg) are in shared memory
        const float *m0 = Ms + (sg & 1) * D * kCombineLd + r0 * kCombineLd;
        const float *m1 = m0 + kCombineLd;
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
            const float4 a0 = *reinterpret_cast<const float4 *>(m0 + k);
            const float4 a1 = *reinterpret_cast<const float4 *>(m1 + k);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 sv = *reinterpret_cast<const float4 *>(Ss + (k + kk) * CW + c0);
                acc[0][0] += av0[kk] * sv.x; acc[0][1] += av0[kk] * sv.y;
                acc[0][2] += av0[kk] * sv.z; acc[0][3] += av0[kk] * sv.w;
                acc[1][0] += av1[kk] * sv.x; acc[1][1] += av1[kk] * sv.y;
                acc[1][2] += av1[kk] * sv.z; acc[1][3] += av1[kk] * sv.w;
            }
        }
        __syncthreads();  // every read of S_in(sg) and of M_sg is done
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float4 o = make_float4(acc[rr][0], acc[rr][1], acc[rr][2], acc[rr][3]);
            *reinterpret_cast<float4 *>(Ss + (r0 + rr) * CW + c0) = o;
            *reinterpret_cast<float4 *>(p.sc_si + unit(sg) * D * D + static_cast<size_t>(r0 + rr) * D + cbase + c0) = o;
        }
    }
}

// The same combine on the tensor cores, one CTA per (sequence, value head,
// 16 value columns) as above, from S_in(1) over segments 1 .. P - 2.  The
// CTA's product M_s S (128 x 128 x 16) is three bf16 products with fp32
// accumulation, M_hi S_hi + M_hi S_lo +
// M_lo S_hi, where x_hi = bf16(x) and x_lo = bf16(x - x_hi): about 16
// mantissa bits per operand, far finer than the fp16 operand rounding the
// state pass applies at every chunk (the dropped M_lo S_lo term is below
// 2^-16 of the product).  Both operands are K-major:
// M as A (128 rows; the transitions write its hi and lo images, sc_mimg),
// the 16 state columns as B (16 rows, K = the 128 state rows).  Per step:
// one thread issues the 24 MMAs; warps 0-3 (one TMEM lane quarter each) add
// B_s to the product, write S_in(s + 1) and split it into the next B
// operand; warps 4-7 copy the M images two steps ahead (per-thread 16-byte
// asynchronous copies into two buffers).
struct CombineTcCfg {
    static constexpr uint32_t kMimg = 65536;           // hi (32 KB) then lo: [2 blocks of 64 K][128 rows][128 B]
    static constexpr uint32_t oSh = 2 * kMimg;         // B: [2 blocks of 64 K][16 rows][128 B]
    static constexpr uint32_t oSl = oSh + 4096;
    static constexpr uint32_t kSmem = oSl + 4096 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 32;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t split_bf(float x, float &lo) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    lo = x - __bfloat162float(h);
    return static_cast<uint32_t>(__bfloat16_as_ushort(h));
}

__global__ void __launch_bounds__(256, 1) gdn2_scan_combine_tc_kernel(Params p) {
    using C = CombineTcCfg;
    constexpr int D = 128, CW = 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t mma_done, drain;
    __shared__ uint32_t tmem_slot;
    pdl_wait();     // the transitions are complete
    pdl_trigger();  // the replay may launch and wait for this grid
    if (p.status[0] != GDN2_OK) return;
    const int n = blockIdx.x, hv = blockIdx.y, cbase = CW * blockIdx.z;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int P = p.sc_P, steps = P - 2;  // step s: segment s + 1
    auto unit = [&](int sg) { return (static_cast<size_t>(n) * (P - 1) + sg) * p.HV + hv; };
    if (tid == 0) {
        mbar_init(&mma_done, 1);
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
    const uint32_t tD = tmem_slot;
    bool ok = true;
    auto load_m = [&](int st) {  // step st's M images (segment st + 1) into buffer st & 1 (warps 4-7)
        const uint8_t *src = p.sc_mimg + unit(st + 1) * C::kMimg;
        uint8_t *dst = sm + (st & 1) * C::kMimg;
#pragma unroll 4
        for (int i = tid - 128; i < static_cast<int>(C::kMimg / 16); i += 128) cp_async16(dst + 16 * i, src + 16 * i, 16);
        cp_async_commit();
    };
    // state row r (the K index), column j (0..15) of the B operands: row j of a
    // K-major [16][128] tile, element r
    auto put_s = [&](int r, int j, float x) {
        float lo;
        const uint32_t hi = split_bf(x, lo);
        const uint32_t off = (r / 64) * 2048u + swz(j, (r % 64) / 8) + (r % 8) * 2;
        *reinterpret_cast<unsigned short *>(sm + C::oSh + off) = static_cast<unsigned short>(hi);
        *reinterpret_cast<unsigned short *>(sm + C::oSl + off) = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    };
    {  // S_in(1): sc_si unit 0 (fp32 [K][V]), two threads per row, 8 columns each
        const int r = tid / 2, j0 = 8 * (tid % 2);
        const float *s1 = p.sc_si + unit(0) * D * D + static_cast<size_t>(r) * D + cbase + j0;
#pragma unroll
        for (int x = 0; x < 8; ++x) put_s(r, j0 + x, s1[x]);
    }
    if (warp >= 4 && steps > 0) {
        load_m(0);
        if (steps > 1) load_m(1);
        if (steps > 1) cp_async_wait_group<1>(); else cp_async_wait_group<0>();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();  // step 0's M images (each thread's own copies waited for) and S_in(1) are in place
    tc_fence_after();
    for (int s = 0; s < steps; ++s) {
        const bool next = s + 1 < steps;
        if (tid == 0) {
            constexpr uint32_t id = idesc_bf16(128, CW, false, false);
            const uint32_t mh = smem_u32(sm + (s & 1) * C::kMimg), ml = mh + 32768;
            const uint32_t sh = smem_u32(sm + C::oSh), sl = smem_u32(sm + C::oSl);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_f16(tD, desc_kmajor(mh, 128, kk), desc_kmajor(sh, CW, kk), id, kk > 0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) mma_f16(tD, desc_kmajor(mh, 128, kk), desc_kmajor(sl, CW, kk), id, 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) mma_f16(tD, desc_kmajor(ml, 128, kk), desc_kmajor(sh, CW, kk), id, 1);
            mma_commit(&mma_done);
        }
        if (warp < 4) {
            // S_in(s + 2) = M_{s+1} S_in(s + 1) + B_{s+1}: row r of the product is TMEM lane r
            const int r = 32 * warp + lane;
            const float *brow = p.sc_tr + unit(s + 1) * D * (2 * D) + static_cast<size_t>(r) * (2 * D) + D + cbase;
            float bv[CW];
#pragma unroll
            for (int x = 0; x < CW; x += 4) {
                const float4 b = *reinterpret_cast<const float4 *>(brow + x);
                bv[x] = b.x; bv[x + 1] = b.y; bv[x + 2] = b.z; bv[x + 3] = b.w;
            }
            if (!warp_wait(&mma_done, s & 1)) ok = false;
            tc_fence_after();
            uint32_t acc[16];
            tmem_ld16(tD + (static_cast<uint32_t>(32 * warp) << 16), acc);
            tmem_ld_wait();
            float v[CW];
#pragma unroll
            for (int x = 0; x < CW; ++x) v[x] = __uint_as_float(acc[x]) + bv[x];
            float *si = p.sc_si + unit(s + 1) * D * D + static_cast<size_t>(r) * D + cbase;
#pragma unroll
            for (int x = 0; x < CW; x += 4) *reinterpret_cast<float4 *>(si + x) = make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
            if (next) {
#pragma unroll
                for (int x = 0; x < CW; ++x) put_s(r, x, v[x]);
            }
        } else if (next) {
            // M_{s+2} into the buffer M_s leaves once its products are done;
            // then this thread's copies of M_{s+1} must have landed
            if (s + 2 < steps) {
                if (!mbar_wait(&mma_done, s & 1)) ok = false;
                load_m(s + 2);
                cp_async_wait_group<1>();
            } else {
                cp_async_wait_group<0>();
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // every MMA has completed before Tensor Memory is released (after a timed
    // out wait one may still run)
    if (tid == 0) {
        mma_commit(&drain);
        if (!mbar_wait(&drain, 0)) ok = false;
    }
    if (!ok) atomicExch(p.status + 2, static_cast<int>(GDN2_ERR_TIMEOUT));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tD, C::kTmemCols);
    }
}

}  // namespace

// The 128-column lookahead kernel runs unless GDN2_STATE_LOOKAHEAD is 0 or 64
// (the plain kernel, for comparison).
bool lookahead128_on() {
    const char *la = getenv("GDN2_STATE_LOOKAHEAD");
    return !(la && (la[0] == '0' || (la[0] == '6' && la[1] == '4')));
}

cudaError_t launch_tc_scan_combine(const Params &p, cudaStream_t s) {
    constexpr int CW = 16;
    if (p.N <= 0 || p.sc_P <= 2) return cudaSuccess;  // two segments: nothing to combine
    // the tensor-core combine reads the M images the lookahead transitions
    // write; GDN2_SCAN_COMBINE=cuda (or the plain state kernel) keeps the
    // CUDA-core one
    const char *cmb = getenv("GDN2_SCAN_COMBINE");
    if (!(cmb && cmb[0] == 'c') && lookahead128_on()) {
        const cudaError_t e = cudaFuncSetAttribute(gdn2_scan_combine_tc_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(CombineTcCfg::kSmem));
        if (e != cudaSuccess) return e;
        return launch_chained(gdn2_scan_combine_tc_kernel, dim3(p.N, p.HV, 128 / CW), dim3(256), CombineTcCfg::kSmem,
                              s, p);
    }
    const cudaError_t e = cudaFuncSetAttribute(gdn2_scan_combine_kernel<CW>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(combine_smem<CW>()));
    if (e != cudaSuccess) return e;
    return launch_chained(gdn2_scan_combine_kernel<CW>, dim3(p.N, p.HV, 128 / CW), dim3(256), combine_smem<CW>(), s,
                          p);
}

cudaError_t launch_tc_state(const Params &p, cudaStream_t s) {
    if (p.K == 64) return launch_state<64, 64, 3, false>(p, s);
    // the sequential pass and the chunk-parallel modes run the one-chunk
    // lookahead kernels (GDN2_STATE_LOOKAHEAD=0 selects the plain kernel for
    // both tile widths, =64 for 128-column tiles only; for comparison)
    const char *la = getenv("GDN2_STATE_LOOKAHEAD");
    const bool la_off = la && la[0] == '0', la128_off = !lookahead128_on();
    if (p.vtile == 64 && p.sc_mode != 1 && !la_off) return launch_tc_state_la(p, s);
    if (p.vtile == 128 && !la128_off) return launch_tc_state_la128(p, s);
    if (p.sc_mode != 0)
        return p.vtile == 64 ? launch_state<128, 64, 3, true>(p, s) : launch_state<128, 128, 2, true>(p, s);
    if (p.vtile == 64) return launch_state<128, 64, 3, false>(p, s);
    return launch_state<128, 128, 2, false>(p, s);
}

}  // namespace gdn2
