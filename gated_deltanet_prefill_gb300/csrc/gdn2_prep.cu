// Chunk map and per-chunk prep (cumsum of the log-decay, optional q/k L2 norm).
//
// Chunk map: packed variable-length sequences (FlashInfer docs,
// chunk_gated_delta_rule2: cu_seqlens) are cut into 64-token chunks that never
// span two sequences; the last chunk of a sequence may be partial.  The map is
// built on the device so the host never waits on cu_seqlens.
//
// Prep: G_t = sum_{s <= t, s in chunk} g_s per key channel (the chunk-local
// cumulative log-decay of the FlashRT WY chain's norm/cumsum stage), and, when
// requested, q, k <- x / max(||x||_2, 1e-12) (FlashInfer docs:
// use_qk_l2norm_in_kernel).
#include "gdn2_internal.cuh"

namespace gdn2 {

namespace {

constexpr int kMapThreads = 1024;
constexpr int kSeqCache = 4096;  // seq_first entries kept in shared memory

// Inclusive prefix sum of x over the CTA's 1024 threads: a shuffle scan in
// each warp, then one over the 32 warp totals.  sums: 32 ints of shared
// memory, free again after the call's second barrier.
__device__ __forceinline__ int block_scan(int x, int *sums) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) sums[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        sums[lane] = t;
    }
    __syncthreads();
    return w > 0 ? x + sums[w - 1] : x;
}

// One CTA: validate cu_seqlens, scan the per-sequence chunk counts, fill the
// per-chunk table.  Invalid cu_seqlens -> status word set, zero chunks.
__global__ void __launch_bounds__(kMapThreads) gdn2_chunk_map_kernel(Params p) {
    __shared__ int s_bad;
    __shared__ int s_sums[32];
    __shared__ int s_pos[kMapThreads];  // chunk-count buckets of the sequence order
    __shared__ int s_first[kSeqCache];  // seq_first[0 .. N] when N < kSeqCache
    const int tid = threadIdx.x;
    pdl_trigger();  // the chain's first kernel: the intra kernel may launch now and waits for this one
    if (tid == 0) {
        s_bad = 0;
        p.status[2] = GDN2_OK;
        p.status[3] = GDN2_OK;
        p.status[4] = 0;
        p.status[5] = 0;
    }
    __syncthreads();
    for (int n = tid; n < p.N; n += kMapThreads)
        if (cu_at(p, n + 1) < cu_at(p, n)) s_bad = 1;
    if (tid == 0 && (cu_at(p, 0) != 0 || cu_at(p, p.N) != p.T_tot)) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            p.status[0] = GDN2_ERR_CU_SEQLENS;
            p.status[1] = 0;
        }
        for (int c = tid; c < p.NCmax; c += kMapThreads) p.chunk_seq[c] = -1;
        for (int n = tid; n <= p.N; n += kMapThreads) p.seq_first[n] = 0;
        return;
    }
    const bool cached = p.N < kSeqCache;
    int running = 0;
    for (int base = 0; base < p.N; base += kMapThreads) {
        const int n = base + tid;
        int cnt = 0;
        if (n < p.N) cnt = static_cast<int>((cu_at(p, n + 1) - cu_at(p, n) + kChunk - 1) / kChunk);
        const int incl = block_scan(cnt, s_sums);
        if (n < p.N) {
            p.seq_first[n] = running + incl - cnt;
            if (cached) s_first[n] = running + incl - cnt;
        }
        running += s_sums[31];  // the batch total
        __syncthreads();        // read by every thread before the next batch's scan writes s_sums
    }
    const int NC = running;
    if (tid == 0) {
        p.seq_first[p.N] = NC;
        if (cached) s_first[p.N] = NC;
        p.status[0] = GDN2_OK;
        p.status[1] = NC;
    }
    s_pos[tid] = 0;
    __syncthreads();  // seq_first (global, and its shared copy) is now visible to the CTA
    auto first = [&](int n) { return cached ? s_first[n] : p.seq_first[n]; };
    // Sequence order for the state pass: longest first, so that the longest
    // chunk chains start in the first wave of CTAs.  A counting sort over
    // chunk counts (kMapThreads buckets, the last one open-ended); the order
    // inside a bucket follows the shared-memory atomics and only decides
    // which CTA starts first, never a result.
    auto bucket = [&](int n) { return min(first(n + 1) - first(n), kMapThreads - 1); };
    for (int n = tid; n < p.N; n += kMapThreads) atomicAdd(&s_pos[bucket(n)], 1);
    __syncthreads();
    {  // s_pos[b] = number of sequences in buckets above b (descending exclusive scan)
        const int b = kMapThreads - 1 - tid;
        const int cnt = s_pos[b];
        const int incl = block_scan(cnt, s_sums);
        s_pos[b] = incl - cnt;
    }
    __syncthreads();
    for (int n = tid; n < p.N; n += kMapThreads) p.seq_order[atomicAdd(&s_pos[bucket(n)], 1)] = n;
    for (int c = tid; c < p.NCmax; c += kMapThreads) {
        if (c >= NC) {
            p.chunk_seq[c] = -1;
            continue;
        }
        // owner of chunk c = the last n with seq_first[n] <= c (empty sequences
        // before it share its seq_first; those after it start past c)
        int lo = 0, hi = p.N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (first(mid) <= c) lo = mid; else hi = mid - 1;
        }
        const int64_t start = cu_at(p, lo) + static_cast<int64_t>(c - first(lo)) * kChunk;
        const int64_t end = cu_at(p, lo + 1);
        p.chunk_seq[c] = lo;
        p.chunk_start[c] = start;
        p.chunk_len[c] = static_cast<int>(end - start < kChunk ? end - start : kChunk);
    }
}

// Chunk-local inclusive cumsum of g, one CTA per (chunk, value head), one
// thread per key channel.  Absent g -> G = 0.
__global__ void gdn2_cumsum_kernel(Params p) {
    const int c = blockIdx.x, hv = blockIdx.y, ch = threadIdx.x;
    const int seq = p.chunk_seq[c];
    if (seq < 0) return;
    const int64_t start = p.chunk_start[c];
    const int len = p.chunk_len[c];
    float acc = 0.f;
    for (int i = 0; i < len; ++i) {
        const int64_t t = start + i;
        if (p.has_g) acc += p.g[t * p.sg_t + hv * p.sg_h + ch];
        p.G[(t * p.HV + hv) * p.K + ch] = acc;
    }
}

// Row L2 norm of q (H heads) and k (HK heads), one warp per (token, head)
// row (the q rows first, then the k rows), fp32 math, bf16 out.
__global__ void gdn2_l2norm_kernel(Params p) {
    int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int64_t qrows = p.T_tot * p.H;
    if (row >= qrows + p.T_tot * p.HK) return;
    const int which = row >= qrows;  // 0: q, 1: k
    if (which) row -= qrows;
    const int heads = which ? p.HK : p.H;
    const int64_t t = row / heads;
    const int h = static_cast<int>(row % heads);
    {
        const bf16 *src = which ? p.k_in + t * p.sk_in_t + h * p.sk_in_h : p.q_in + t * p.sq_in_t + h * p.sq_in_h;
        bf16 *dst = (which ? p.kn : p.qn) + row * p.K;
        float x[4];
        float ss = 0.f;
        const int per = p.K / 32;
        for (int i = 0; i < per; ++i) {
            x[i] = __bfloat162float(src[lane + 32 * i]);
            ss += x[i] * x[i];
        }
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float d = fmaxf(sqrtf(ss), 1e-12f);
        for (int i = 0; i < per; ++i) dst[lane + 32 * i] = __float2bfloat16(x[i] / d);
    }
}

}  // namespace

cudaError_t launch_chunk_map(const Params &p, cudaStream_t s) {
    gdn2_chunk_map_kernel<<<1, kMapThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prep(const Params &p, cudaStream_t s) {
    if (p.l2norm && p.T_tot > 0) {
        const int64_t rows = p.T_tot * (p.H + p.HK);
        const int per_block = 8;
        gdn2_l2norm_kernel<<<static_cast<unsigned>((rows + per_block - 1) / per_block), 32 * per_block, 0, s>>>(p);
    }
    if (p.NCmax > 0) gdn2_cumsum_kernel<<<dim3(p.NCmax, p.HV), p.K, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn2
