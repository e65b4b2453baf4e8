// Blackwell (sm_103a) building blocks written as inline PTX: mbarriers with
// time-bounded waits, bulk global->shared copies, Tensor Memory (TMEM)
// allocation / loads / stores, tcgen05.mma (bf16 x bf16 -> fp32) and its
// shared-memory matrix descriptors.
//
// Shared-memory operand images use the 128-byte swizzle: a tile is a stack
// of 1024-byte atoms of 8 rows x 128 bytes, and inside an atom the 16-byte
// chunk j of row r is stored at chunk j ^ (r % 8).  Two orientations are used:
//  * K-major  (rows = M or N, 64 K-elements per 128-byte row): blocks of 64 K
//    columns, each [rows][128 B]; an MMA step of 16 K advances 32 bytes.
//  * MN-major (rows = K, 64 M/N-elements per 128-byte row): blocks of 64 M/N
//    columns, each [K rows][128 B]; an MMA step of 16 K advances 2048 bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdn2 {
namespace tc {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete; gives up after
// limit_ns of wall time and returns false (the caller records the timeout
// and unwinds instead of hanging).
__device__ __forceinline__ bool mbar_wait_ns(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_ns(bar, parity, kWaitLimitNs);
}
// The same bounded wait with a suspend-time hint: a thread whose phase is not
// complete is parked by the hardware (for at most hint_ns per try) until the
// phase completes, instead of polling.  Which waits gain from it is measured
// per kernel and per role.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_parked(uint64_t *bar, uint32_t parity) {
    constexpr uint32_t kHintNs = 20000;
    if (mbar_try_wait_hint(bar, parity, kHintNs)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity, kHintNs)) return true;
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

// The same wait taken by a whole warp, with a warp-uniform result, so that the
// warp-collective tcgen05 loads and stores that follow never diverge.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// ---------------------------------------------------------- bulk copies
// Contiguous global -> shared copy completing on an mbarrier (transaction
// bytes).  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Contiguous shared -> global copy in a bulk async-group of the issuing
// thread (addresses 16-byte aligned, size a multiple of 16).  The writers of
// the shared source issue fence_proxy_async() before the barrier that
// precedes the copy.  bulk_commit closes the group; bulk_wait_read0 returns
// once every committed group has read its shared source (which may then be
// overwritten), bulk_wait0 once every group's writes are complete.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tile of a 3-D tensor map (box given by the map) -> shared memory, completing
// on an mbarrier.  tmap: generic address of a CUtensorMap in kernel-parameter,
// constant or global memory; c0 (innermost) .. c2: element coordinates, with
// c0 * element size a multiple of 16 bytes.  dst 128-byte aligned.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Prefetch a tile of a 3-D tensor map into L2 (no completion to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const void *tmap, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tmap), "r"(c0),
                 "r"(c1), "r"(c2)
                 : "memory");
}

// Per-thread 16-byte global -> shared copy (L2 only); src_bytes = 0 writes
// zeros without reading src.  Completion: cp_async_wait_all by the issuing
// thread, then a block barrier before other threads read the data.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Close the thread's pending cp.async copies into a group; wait until at
// most N of its groups are still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Named barrier `id` (1..15) over `nthreads` threads of the block (a
// multiple of 32, whole warps); id 0 is __syncthreads.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (tcgen05.mma operand reads, bulk copies).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------- TMEM
// Allocation is warp-wide; the TMEM address is written to *slot (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// TMEM address of (lane, column)
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane
// (lane_base + i), registers r[j] = column (col + j).
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(addr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(addr));
}
__device__ __forceinline__ void tmem_st32(uint32_t addr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(addr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// -------------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2),
// descriptor version 1.  lbo / sbo in bytes.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}
// K-major SW128 operand at k-step kk (16 elements) for a tile of `rows`
// rows: blocks of 64 K-columns, [rows][128 B] each.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, uint32_t rows, uint32_t kk) {
    return sdesc(base + (kk >> 2) * rows * 128u + (kk & 3u) * 32u, 16u, 1024u);
}
// MN-major SW128 operand at k-step kk for a tile with `krows` K rows: blocks
// of 64 M/N-columns, [krows][128 B] each.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, uint32_t krows, uint32_t kk) {
    return sdesc(base + kk * 2048u, krows * 128u, 1024u);
}

// Instruction descriptor, kind::f16, fp32 D; A and B both bf16 or both fp16.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool a_mn, bool b_mn, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return idesc_f16kind(M, N, a_mn, b_mn, true);
}
__host__ __device__ constexpr uint32_t idesc_fp16(int M, int N, bool a_mn, bool b_mn) {
    return idesc_f16kind(M, N, a_mn, b_mn, false);
}

// D[tmem] (+)= A[smem] x B[smem], kind::f16 (bf16 or fp16 operands per the
// instruction descriptor); issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same with A in Tensor Memory (row m of A in lane m, K packed two fp16
// per 32-bit column; a K = 16 step spans 8 columns); B from shared memory.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128B-swizzled block whose rows are 128 bytes.
__host__ __device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero): used on
// log2(e)-prescaled decay exponents, which are <= 0 except for the diagonal
// sub-chunk factors, which the intra kernel keeps below 2^92.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ----------------------------------------------------------- conversions
// fp16 intermediates saturate at +-65504 instead of overflowing to inf.
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    uint32_t r;  // a -> low half; out-of-range finite values saturate to +-65504
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
// The same conversion, tracking in m the largest fp16 magnitude written, so
// that a clipped value can be reported: a lane whose magnitude bits are 0x7bff
// (65504, where the conversion saturates) or above (inf, NaN) means a value was
// clipped, and the kernel then reports GDN2_ERR_RANGE in the device status
// instead of returning it silently.  Two forms, each where it measured faster:
//  - pack_h2m: the sign bits cleared, then a 16-bit unsigned max (two integer
//    instructions; the state kernels, whose epilogues keep the fp16 units busy);
//  - pack_h2mh: one packed fp16 maximum of the magnitudes (max.xorsign.abs,
//    whose sign is the xor of the operands' signs and is ignored; NaN
//    propagated; the intra kernel, which is bound by its instruction count).
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t pack_h2m(float a, float b, uint32_t &m) {
    const uint32_t r = pack_h2(a, b);
    m = umax16x2(m, r & 0x7fff7fffu);
    return r;
}
__device__ __forceinline__ uint32_t pack_h2mh(float a, float b, uint32_t &m) {
    const uint32_t r = pack_h2(a, b);
    asm("max.NaN.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(r));
    return r;
}
// either form's m: magnitude bits of each lane at or past the clipping point
__device__ __forceinline__ bool half_clipped(uint32_t m) {
    return (m & 0x7fffu) >= 0x7bffu || ((m >> 16) & 0x7fffu) >= 0x7bffu;
}
// a -> low half, IEEE round-to-nearest (overflow gives inf, as a cast would)
__device__ __forceinline__ uint32_t pack_f16_rn(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_h2(uint32_t x) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&x));
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack_bf2(uint32_t x) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x));
}
__device__ __forceinline__ uint4 pack8_h(const float (&f)[8]) {
    return make_uint4(pack_h2(f[0], f[1]), pack_h2(f[2], f[3]), pack_h2(f[4], f[5]), pack_h2(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack8_hm(const float (&f)[8], uint32_t &m) {  // pack_h2mh's tracking
    return make_uint4(pack_h2mh(f[0], f[1], m), pack_h2mh(f[2], f[3], m), pack_h2mh(f[4], f[5], m),
                      pack_h2mh(f[6], f[7], m));
}
__device__ __forceinline__ uint4 pack8_bf(const float (&f)[8]) {
    return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]), pack_bf2(f[6], f[7]));
}
// eight fp16 values of a 16-byte chunk
__device__ __forceinline__ void unpack8_f16(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = unpack_h2(w[i]);
        f[2 * i] = a.x;
        f[2 * i + 1] = a.y;
    }
}
// eight 16-bit inputs (fp16 when f16, else bf16)
__device__ __forceinline__ void unpack8_bf(const uint4 &u, float (&f)[8]);
__device__ __forceinline__ void unpack8_in(const uint4 &u, float (&f)[8], bool f16) {
    if (f16)
        unpack8_f16(u, f);
    else
        unpack8_bf(u, f);
}
__device__ __forceinline__ void unpack8_bf(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = unpack_bf2(w[e]);
        f[2 * e] = x.x;
        f[2 * e + 1] = x.y;
    }
}

}  // namespace tc
}  // namespace gdn2
