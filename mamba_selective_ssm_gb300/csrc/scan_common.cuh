// Geometry and warp reductions shared by the selective-scan forward and backward kernels.
//
// A CTA owns DT consecutive channels of one batch row at a time and walks
// the sequence in tiles of TT = 16 steps that TMA stages into shared memory
// ([TT x DT] boxes of delta, x, z, dy; [TT*N] boxes of B_t, C_t).
//
// Backward: inside a warp, lane = cg * NG + ng: the NG = N/4 lanes of
// channel-pair group cg share two channels and split the N states four apiece,
// so every thread advances 2 channels x 4 states = 8 (d, n) recurrences with
// packed f32x2 arithmetic.  Sums over n (y, and the delta / x gradients) add
// the NG lanes' shares in shared memory; sums over d (dB, dC) run across the
// pair groups and the warps of the CTA.
// Forward: 1 channel x 4 states per thread with lane = ng * CG + cg, so that
// the CG lanes reading the same four B_t / C_t values are consecutive: a
// 128-bit shared load whose lanes share addresses in runs of 8 costs two
// wavefronts, against four when the sharing lanes are interleaved.
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

// ---------------------------------------------------------------- sequence segments
// When a layer has too few (batch, channel-tile) pairs to fill the GPU, the
// sequence is cut into P segments of Ls steps (a multiple of `unit`).  A
// summary kernel computes each segment's contribution from a zero carry and
// its total step size sum(delta); a main-kernel CTA then composes its own
// carry from the summaries of the segments before (forward) or after
// (backward) it:  carry <- exp2(A log2e * sum(delta)) * carry + contribution.

// Upper bound on P used to size the summary workspace: aims at ~2400 CTAs.
inline int seg_pmax(long long ctas, int L, int unit) {
  long long pm = (2432 + ctas - 1) / ctas;
  const long long units = (L + unit - 1) / unit;
  if (pm > 64) pm = 64;
  if (pm > units) pm = units;
  return pm < 1 ? 1 : (int)pm;
}

struct SegPlan {
  int P, Ls;
};

// Segments of equal length (a multiple of unit) covering L with about p_want pieces.
inline SegPlan seg_plan(int p_want, int L, int unit) {
  if (p_want <= 1) return SegPlan{1, L};
  const int per = (L + p_want - 1) / p_want;
  const int Ls = ((per + unit - 1) / unit) * unit;
  return SegPlan{(L + Ls - 1) / Ls, Ls};
}

// ---------------------------------------------------------------- fused discretisation
// log(1 + u) for u in [0, 1]: the Taylor series u - u^2/2 + u^3/3 below 1/32
// (truncation below u^4/4, i.e. 7e-6 relative), the fast logarithm of 1 + u
// above (where 1 + u keeps u to 2e-6 relative).
__device__ __forceinline__ float log1p_unit(float u) {
  return u < 0.03125f ? u * fmaf(u, fmaf(u, 1.0f / 3.0f, -0.5f), 1.0f) : __logf(1.0f + u);
}

// softplus(v) = log(1 + e^v) = max(v, 0) + log(1 + e^-|v|).
__device__ __forceinline__ float softplus_f(float v) { return fmaxf(v, 0.f) + log1p_unit(__expf(-fabsf(v))); }

// softplus'(v) = sigmoid(v) = 1 - e^-softplus(v), from delta = softplus(v):
// the series delta - delta^2/2 + delta^3/6 below 1/32 (no cancellation), else 1 - e^-delta.
__device__ __forceinline__ float softplus_grad_from_delta(float dl) {
  return dl < 0.03125f ? dl * fmaf(dl, fmaf(dl, 1.0f / 6.0f, -0.5f), 1.0f) : 1.0f - __expf(-dl);
}

// The delta the recurrence uses, from the caller's raw values: raw + bias, and
// softplus of that when asked.  Steps past L and channels past D are forced to
// 0 so that they leave the state unchanged, as the zero-filled raw delta does
// without the transform.
__device__ __forceinline__ void delta_transform4(float* dv, const float* bias_s, int c4, bool row_ok, int d_left,
                                                 int softplus) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float v = dv[e] + bias_s[c4 + e];
    if (softplus) v = softplus_f(v);
    dv[e] = (row_ok && e < d_left) ? v : 0.f;
  }
}

}  // namespace ssk
