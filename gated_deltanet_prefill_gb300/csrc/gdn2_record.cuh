// The per-(chunk, value head) record that the tensor-core intra kernel writes
// and the tensor-core state kernel reads.  Every operand the state kernel
// feeds to tcgen05.mma is stored as its shared-memory image (128B swizzle,
// see gdn2_tc.cuh), so a bulk copy places it ready for the MMA.
//
// Chunk algebra (64 tokens, incoming state S0, chunk-local cumsum G, last
// valid row L; FlashInfer docs' recurrence unrolled over the chunk):
//   U   = Ut - Wt S0                           Wt = T (beta k e^G),  Ut = T (w v)
//   O   = scale [ Qe S0 + P U ]                Qe = q e^G,  P_ts = sum_c q_t e^{G_t-G_s} k_s (s <= t)
//   S_C = diag(eGL) S0 + Kd^T U                Kd = k e^{G_L - G},  eGL = e^{G_L}
// with T = (I + A)^{-1}, A_ts = sum_c beta_t k_t e^{G_t-G_s} k_s (s < t).
//
// Layout for head dim D (= K = V, 64 or 128), byte offsets:
//   P    [64 t][64 s]          K-major A image, one 8 KB block
//   A1   [Qe ; Wt]             K-major A image, M = 128 rows (Qe rows 0-63,
//                              Wt rows 64-127), D/64 blocks of 16 KB
//   KdT  Kd as an MN-major A   D/64 blocks of [64 s][128 B] = 8 KB
//   Ut   [64 t][D]             D/64 blocks of [64 t][128 B], swizzled
//   eGL  D fp32
// Qe, Wt, P, KdT and Ut are fp16 (10-bit mantissa; conversions saturate at
// +-65504).  Rows of tokens past the chunk's length are zero (eGL is always
// defined).
#pragma once

#include <stdint.h>

namespace gdn2 {

template <int D>
struct Rec {
    static constexpr uint32_t P = 0;
    static constexpr uint32_t A1 = 8192;
    static constexpr uint32_t KdT = A1 + (D / 64) * 16384;
    static constexpr uint32_t Ut = KdT + (D / 64) * 8192;
    static constexpr uint32_t eGL = Ut + (D / 64) * 8192;
    static constexpr uint32_t bytes = ((eGL + D * 4) + 1023) / 1024 * 1024;
    static constexpr uint32_t mma_prefix = Ut;  // P, A1 and KdT are contiguous
};

}  // namespace gdn2
