// kvp_vec.cuh -- per-warp vector machinery of the pool decoder (the
// register / warp-shuffle Walsh-Hadamard transform), the packed f32x2
// helpers, and the 3-bit Lloyd-Max codebook shared by the encoder, the
// decoder and the attention kernels.
//
// Decoder lane mapping.  A value vector of d = 64 or 128 coordinates is held by
// LPV = d/32 lanes, 32 coordinates per lane, as 4 chunks of 8 consecutive
// coordinates: lane l of the vector holds chunks c = j*LPV + l (j = 0..3),
// coordinate i = 8c + e (e = 0..7).  So coordinate bits 0-2 live in
// registers (e), the next log2(LPV) bits in the lane index (l) and the top 2
// bits in registers again (j); a warp holds 32/LPV vectors.  With this
// mapping every 16-byte access of a warp instruction is part of a fully used
// 32-byte sector (chunk j of the LPV lanes of a vector is contiguous).
#pragma once

#include "kvp_internal.cuh"

namespace kvp {

// Packed f32x2 add and subtract; a - b is fma(b, -1, a), rounded once like
// the subtraction.
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2sub(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }

// Unnormalised Sylvester-order Walsh-Hadamard transform ("PolyKV" 2.B.2
// rotation, y_i = sum_j (-1)^popcount(i & j) x_j, one butterfly stage per
// index bit) of the vector held by the LPV lanes of each vector, on packed
// pairs: x[j][p] holds coordinates (8c + 2p, 8c + 2p + 1) of chunk
// c = j*LPV + l, and the caller has already applied the butterfly of
// coordinate bit 0 (x[j][p] = (a + b, a - b)).  The remaining stages run as
// f32x2 operations.
template <int LPV>
__device__ __forceinline__ void fwht_pairs(float2 (&x)[4][4], int lane) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int h = 1; h < 4; h <<= 1) {       // coordinate bits 1, 2
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                if ((p & h) == 0) {
                    const float2 a = x[j][p], b = x[j][p + h];
                    x[j][p] = f2add(a, b);
                    x[j][p + h] = f2sub(a, b);
                }
            }
        }
    }
#pragma unroll
    for (int h = 1; h < 4; h <<= 1) {           // the two register-held top bits
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if ((j & h) == 0) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float2 a = x[j][p], b = x[j + h][p];
                    x[j][p] = f2add(a, b);
                    x[j + h][p] = f2sub(a, b);
                }
            }
        }
    }
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) {         // lane bits
        const float sg = (lane & m) ? -1.0f : 1.0f;
        const float2 sgn = make_float2(sg, sg);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                float2 o;
                o.x = __shfl_xor_sync(0xffffffffu, x[j][p].x, m);
                o.y = __shfl_xor_sync(0xffffffffu, x[j][p].y, m);
                x[j][p] = __ffma2_rn(sgn, x[j][p], o);
            }
        }
    }
}

// Lloyd-Max 8-level codebook for N(0,1) (+-0.2451, 0.7560, 1.3440, 2.1520)
// and its decision thresholds (midpoints of adjacent centroids), positive
// half.  Codes 0..7 index the centroids in ascending order.
constexpr float THR1 = 0.50055f;  // (0.2451 + 0.7560) / 2
constexpr float THR2 = 1.05f;     // (0.7560 + 1.3440) / 2
constexpr float THR3 = 1.748f;    // (1.3440 + 2.1520) / 2

// Centroid of a code scaled by 10^4 -- the codebook's values are integers at
// that scale (2451, 7560, 13440, 21520), so a Walsh-Hadamard transform of
// them is exact in fp32 (|sum| <= 128 * 21520 < 2^24); the 10^-4 is folded
// into the final rescale.
__device__ __forceinline__ float centroid_e4(uint32_t code) {
    const uint32_t up = code >> 2;                  // 1 for the positive half
    const uint32_t rank = (code ^ (up - 1u)) & 3u;  // 0..3 by magnitude
    const float m = (rank & 2u) ? ((rank & 1u) ? 21520.0f : 13440.0f)
                                : ((rank & 1u) ? 7560.0f : 2451.0f);
    return up ? m : -m;
}

}  // namespace kvp
