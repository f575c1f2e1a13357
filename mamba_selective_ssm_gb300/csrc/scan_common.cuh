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
// its total step size sum(delta); seg_combine_kernel below composes the maps
// carry <- exp2(A log2e * sum(delta)) * carry + contribution of the segments
// before (forward) or after (backward) each one, and the main kernel runs
// every segment from its carry.

// Upper bound on P used to size the summary workspace: aims at about `target`
// CTAs in all (16 per SM of 152 by default).
inline int seg_pmax(long long ctas, int L, int unit, long long target = 2432) {
  long long pm = (target + ctas - 1) / ctas;
  const long long units = (L + unit - 1) / unit;
  if (pm > 64) pm = 64;
  if (pm > units) pm = units;
  return pm < 1 ? 1 : (int)pm;
}

struct SegPlan {
  int P, Ls;
};

// CTA rows of a grid whose CTAs walk batch rows y, y + gy, ...: all B rows at
// once when the B x tiles CTAs fit the `resident` slots, else the fewest rows
// of CTAs that fit and give every CTA the same number of batch rows up to one
// (one wave of equal CTAs instead of a full wave and a partial one).
inline int balanced_rows(int B, int tiles, long long resident) {
  const long long fit = tiles > 0 ? resident / tiles : 0;
  if (fit < 1 || fit >= B) return fit < 1 ? 1 : B;
  const long long per = (B + fit - 1) / fit;  // batch rows per CTA
  return (int)((B + per - 1) / per);
}

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

// Segment carries by a warp-shuffle associative scan.  Segment v maps the
// carry entering it to the carry leaving it by c -> alpha_v c + beta_v, with
// alpha_v = exp2(A log2e * sum of delta over v) and beta_v the segment's
// summary (its contribution from a zero carry).  The maps are composed by an
// inclusive scan of the affine pairs, (a1, b1) then (a2, b2) = (a1 a2,
// a2 b1 + b2), and applied to `init` (NULL: zero).  Forward (REV = false):
// segments run v = 0 .. P-1, summaries of 0 .. P-2 exist, out[v] is the state
// entering v.  Backward (REV = true): the adjoint runs from the last segment
// to the first, so v counts segments from the end (segment P-1-v), summaries of
// segments 1 .. P-1 exist, and out[segment] is the carry arriving at its end.
// CTA (32 x 8) = 32 consecutive (d, n) columns of one batch row (blockIdx.y):
// the pairs pass through shared memory so that global accesses stay coalesced;
// warp w scans columns w, w + 8, w + 16, w + 24 with lane l holding segments
// 2l and 2l + 1 of the scan order (P <= kSegMax).
constexpr int kSegMax = 64;

struct SegCombine {
  const float* A;     // [D, N]
  const float* dsum;  // [B][P][D]    sum of delta over each segment
  const float* summ;  // [B][P][D][N] each segment's contribution from a zero carry
  const float* init;  // [B][D][N]    carry entering the scan (h0 or dh_last), or NULL
  float* out;         // [B][P][D][N]
  int P, D, N;
  int sb, sv;         // row of (batch b, segment v) in dsum / summ / out: b * sb + v * sv
                      // (sb = P, sv = 1 for the layout above; sb = 1, sv = B for segment-major [P][B])
};

template <bool REV>
__global__ void __launch_bounds__(256) seg_combine_kernel(const SegCombine c) {
  __shared__ float al[kSegMax][33], be[kSegMax][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int b = blockIdx.y, P = c.P;
  const long long DN = (long long)c.D * c.N;
  const long long col = (long long)blockIdx.x * 32 + tx;
  const bool ok = col < DN;
  for (int v = ty; v < kSegMax; v += 8) {
    float a = 1.f, bv = 0.f;  // identity map where the scan has no segment
    if (ok && v < P - 1) {
      const size_t row = (size_t)b * c.sb + (size_t)(REV ? P - 1 - v : v) * c.sv;
      a = ex2(c.A[col] * kLog2e * c.dsum[row * c.D + col / c.N]);
      bv = c.summ[row * DN + col];
    }
    al[v][tx] = a;
    be[v][tx] = bv;
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const long long cc = (long long)blockIdx.x * 32 + k;
    const float a0 = al[2 * tx][k], b0 = be[2 * tx][k], a1 = al[2 * tx + 1][k], b1 = be[2 * tx + 1][k];
    float Ac = a0 * a1, Bc = fmaf(a1, b0, b1);  // segment 2l, then 2l + 1
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ap = __shfl_up_sync(0xffffffffu, Ac, off), bp = __shfl_up_sync(0xffffffffu, Bc, off);
      if (tx >= off) {
        Bc = fmaf(Ac, bp, Bc);
        Ac *= ap;
      }
    }
    float Ae = __shfl_up_sync(0xffffffffu, Ac, 1), Be = __shfl_up_sync(0xffffffffu, Bc, 1);
    if (tx == 0) {
      Ae = 1.f;
      Be = 0.f;
    }
    const float c0 = (c.init != nullptr && cc < DN) ? c.init[(size_t)b * DN + cc] : 0.f;
    const float in0 = fmaf(Ae, c0, Be);  // entering segment 2l of the scan order
    __syncwarp();
    al[2 * tx][k] = in0;
    al[2 * tx + 1][k] = fmaf(a0, in0, b0);  // entering segment 2l + 1
  }
  __syncthreads();
  for (int v = ty; v < P; v += 8)
    if (ok) c.out[((size_t)b * c.sb + (size_t)(REV ? P - 1 - v : v) * c.sv) * DN + col] = al[v][tx];
}

template <bool REV>
inline cudaError_t seg_combine(const SegCombine& c, int B, cudaStream_t s) {
  const long long DN = (long long)c.D * c.N;
  seg_combine_kernel<REV><<<dim3((unsigned)((DN + 31) / 32), B), 256, 0, s>>>(c);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- lane reductions
// Reduce-scatter step between lane and lane ^ mask, which each hold v0 and v1:
// afterwards the lane with `hi` set holds the pair's sum of v1, the other lane
// the pair's sum of v0.  Each lane adds in a fixed order (its own value first),
// so the result does not depend on timing.
__device__ __forceinline__ float rs_pair(float v0, float v1, bool hi, int mask) {
  const float send = hi ? v0 : v1;
  return (hi ? v1 : v0) + __shfl_xor_sync(0xffffffffu, send, mask);
}

}  // namespace ssk
