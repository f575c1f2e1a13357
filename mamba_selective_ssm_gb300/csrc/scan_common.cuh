// Geometry and warp reductions shared by the selective-scan forward and backward kernels.
//
// A CTA owns DT consecutive channels of one batch row at a time and walks
// the sequence in tiles of TT = 16 steps that TMA stages into shared memory
// ([TT x DT] boxes of delta, x, z, dy; [TT*N] boxes of B_t, C_t).
//
// Inside a warp, lane = cg * NG + ng: the NG = N/4 lanes of channel-pair group
// cg share two channels and split the N states four apiece, so every thread
// advances 2 channels x 4 states = 8 (d, n) recurrences with packed f32x2
// arithmetic.  Sums over n (y, and the delta / x gradients) are reduce-scatters
// across the NG lanes of a pair group (lane bits below log2 NG); sums over d
// (dB, dC) run across the pair groups and the warps of the CTA.
#pragma once

#include "common.cuh"

namespace ssk {

constexpr int kTT = 16;  // time steps per TMA tile
constexpr int kDT = 64;  // default channels per CTA
constexpr int kS = 8;    // backward register window: steps whose a_t, h_t stay in registers

template <int N, int DT = kDT>
struct Geo {
  static_assert(N == 4 || N == 8 || N == 16, "N must be 4, 8 or 16");
  static constexpr int NG = N / 4;    // lanes sharing a channel pair
  static constexpr int CG = 32 / NG;  // channel pairs per warp
  static constexpr int WC = 2 * CG;   // channels per warp
  static constexpr int W = DT / WC;   // warps per CTA
  static constexpr int NT = 32 * W;   // threads per CTA
  static_assert(W >= 1 && DT % WC == 0, "a CTA holds whole warps");
};

}  // namespace ssk
