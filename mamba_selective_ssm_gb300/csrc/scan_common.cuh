// Geometry and warp reductions shared by the selective-scan forward and backward kernels.
//
// A CTA owns DT = 64 consecutive channels of one batch row at a time and walks
// the sequence in tiles of TT = 16 steps that TMA stages into shared memory
// ([TT x DT] boxes of delta, x, z, dy; [TT*N] boxes of B_t, C_t).
//
// Inside a warp, lane = cg * NG + ng: the NG = N/4 lanes of channel-pair group
// cg share two channels and split the N states four apiece, so every thread
// advances 2 channels x 4 states = 8 (d, n) recurrences with packed f32x2
// arithmetic.  Sums over n (y, and the delta / x gradients) are reduce-scatters
// across the NG lanes of a pair group (lane bits below log2 NG); sums over d
// (dB, dC) are reduce-scatters across the pair groups (the bits above), then
// across warps in shared memory.
#pragma once

#include "common.cuh"

namespace ssk {

constexpr int kTT = 16;  // time steps per TMA tile
constexpr int kDT = 64;  // channels per CTA
constexpr int kS = 8;    // backward register window: steps whose a_t, h_t stay in registers

template <int N>
struct Geo {
  static_assert(N == 4 || N == 8 || N == 16, "N must be 4, 8 or 16");
  static constexpr int NG = N / 4;    // lanes sharing a channel pair
  static constexpr int CG = 32 / NG;  // channel pairs per warp
  static constexpr int WC = 2 * CG;   // channels per warp
  static constexpr int W = kDT / WC;  // warps per CTA
  static constexpr int NT = 32 * W;   // threads per CTA
  // channel-group lane bits that remain after the 4 -> 1 reduce-scatter
  static constexpr int kDupMask = NG == 4 ? 4 : (NG == 2 ? 6 : 7);
};

// Sum over the channel-pair groups of a warp of four per-thread values
// (entries 0..3 = states n0..n0+3 of the thread).  Reduce-scatter on lane
// bits 4 and 3, then all-reduce on the remaining group bits.  Afterwards the
// lane holds the warp total of entry dsum_index(lane); among the duplicates,
// lanes with (lane & Geo<N>::kDupMask) == 0 store it.
template <int N>
__device__ __forceinline__ float dsum4(float v0, float v1, float v2, float v3, int lane) {
  const bool hi1 = lane & 16;
  float s0 = hi1 ? v2 : v0, s1 = hi1 ? v3 : v1;
  const float o0 = hi1 ? v0 : v2, o1 = hi1 ? v1 : v3;
  s0 += __shfl_xor_sync(0xffffffffu, o0, 16);
  s1 += __shfl_xor_sync(0xffffffffu, o1, 16);
  const bool hi2 = lane & 8;
  float k = hi2 ? s1 : s0;
  const float o = hi2 ? s0 : s1;
  k += __shfl_xor_sync(0xffffffffu, o, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  if constexpr (Geo<N>::NG <= 2) k += __shfl_xor_sync(0xffffffffu, k, 2);
  if constexpr (Geo<N>::NG <= 1) k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}
__device__ __forceinline__ int dsum_index(int lane) { return ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1); }

}  // namespace ssk
