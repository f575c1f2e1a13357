// Depthwise causal conv1d backward (conv1d_causal_bwd) for sm_103a.
//
//   out[t,d] = bias[d] + sum_k w[d,k] x[t-(K-1)+k, d]     (newest input at tap K-1)
//   dx[s,d]  = sum_j dout[s+j, d] w[d, K-1-j]             (terms past the end dropped)
//   dw[d,k] += sum_{b,t} dout[t,d] x[t-(K-1)+k, d],   db[d] += sum_{b,t} dout[t,d]
//
// A thread owns 4 adjacent channels (one 16-byte fp32 vector of dout per
// step) over a 16-step tile of one batch row and slides two K-wide register
// windows along time: dout ahead of the output step (for dx) and x behind it
// (for dw).  One wave of CTAs (four per SM, at most 128 registers a thread)
// loops over the (batch, tile) items, keeping dw / db in registers, and writes
// one partial per CTA row; colsum_kernel adds the partials in fixed order into
// dw / db.  HBM traffic is one read of dout and x plus one write of dx (the
// K-1 halo steps per tile come from L2).
//
// conv1d_causal_silu_bwd takes the gradient after a SiLU on the conv output
// instead: a thread walks the input steps t of its tile and K-1 beyond, turns
// each incoming dout[t] into g[t] = dout[t] * silu'(pre[t]) with
// pre[t] = bias + sum_k w[k] x[t-(K-1)+k] recomputed from the x window behind
// t, and completes dx[t-(K-1)] from the last K values of g; the loads of eight
// steps are issued together, at three CTAs per SM (with fp32 x, 2 channels per
// thread at six CTAs per SM).  The four-channel arithmetic runs as packed
// f32x2 operations (two per step where scalar code takes four).
#include "common.cuh"

namespace {

using namespace ssk;

constexpr int kCTile = 16;     // time steps per tile (short tiles: the (batch row, tile) items spread evenly over the CTAs)
constexpr int kCTileSilu = 24;  // the SiLU-fused form recomputes K-1 steps of g per tile (16: 84 us, 24: 81, 32: 82)
constexpr int kCtasSilu = 3;    // SiLU-fused form: CTAs per SM (~170 registers for its eight loads in flight)
constexpr int kCThreads = 128;  // threads per CTA: 512 channels

template <typename T>
__device__ __forceinline__ float4 ld_x4(const T* p);
template <>
__device__ __forceinline__ float4 ld_x4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 ld_x4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}

// raw x vector of 4 channels as loaded (8 bytes for bf16, 16 for fp32) and its widening
template <typename T>
struct RawX4;
template <>
struct RawX4<float> {
  using V = float4;
  static __device__ __forceinline__ V ld(const float* p) { return *reinterpret_cast<const float4*>(p); }
  static __device__ __forceinline__ float4 wide(V v) { return v; }
  static __device__ __forceinline__ V zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct RawX4<__nv_bfloat16> {
  using V = uint2;
  static __device__ __forceinline__ V ld(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ float4 wide(V v) { return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)); }
  static __device__ __forceinline__ V zero() { return make_uint2(0u, 0u); }
};

// four-channel arithmetic as two packed f32x2 operations (the same roundings as four scalar ones)
__device__ __forceinline__ float4 f4fma(float4 a, float4 b, float4 c) {
  const float2 lo = fma2(f2(a.x, a.y), f2(b.x, b.y), f2(c.x, c.y));
  const float2 hi = fma2(f2(a.z, a.w), f2(b.z, b.w), f2(c.z, c.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
  const float2 lo = add2(f2(a.x, a.y), f2(b.x, b.y)), hi = add2(f2(a.z, a.w), f2(b.z, b.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
// g * silu'(v) for two channels: sigmoid s = 1 / (1 + 2^(-v log2 e)), silu'(v) = s (1 + v (1 - s))
__device__ __forceinline__ float2 gdsilu2(float2 g, float2 v) {
  const float2 e = ex2_2(mul2(v, bc2(-kLog2e)));
  const float2 den = add2(e, bc2(1.0f));
  const float2 sg = f2(rcp(den.x), rcp(den.y));
  const float2 t = fma2(v, fma2(sg, bc2(-1.0f), bc2(1.0f)), bc2(1.0f));
  return mul2(g, mul2(sg, t));
}
__device__ __forceinline__ float4 f4z() { return make_float4(0.f, 0.f, 0.f, 0.f); }


template <int K, typename T, bool SILU>
__global__ void __launch_bounds__(kCThreads, SILU ? kCtasSilu : 4) conv_bwd_kernel(const float* __restrict__ dout, const T* __restrict__ x,
                                                             const float* __restrict__ w, const float* __restrict__ bias,
                                                             float* __restrict__ dx, float* __restrict__ ws, int B, int L,
                                                             int D) {
  pdl_trigger();  // the column sum of the partials may launch now; it waits for this grid's end
  // Rows narrower than a CTA (D/4 < kCThreads channel quads) pack ipc items per
  // CTA step: thread slot `sub` takes every ipc-th item of its CTA row.
  const int cpr = D / 4;
  const int ipc = cpr >= kCThreads ? 1 : kCThreads / cpr;
  const int sub = cpr >= kCThreads ? 0 : (int)threadIdx.x / cpr;
  const int d = (cpr >= kCThreads ? (int)(blockIdx.x * kCThreads + threadIdx.x) : (int)threadIdx.x % cpr) * 4;
  const bool valid = d < D && sub < ipc;  // D % 8 == 0, so all four channels are in range
  constexpr int TILE = SILU ? kCTileSilu : kCTile;
  const int ntt = (L + TILE - 1) / TILE;
  float4 wk[K];  // wk[k] = w[d..d+3, k]
#pragma unroll
  for (int k = 0; k < K; ++k)
    wk[k] = valid ? make_float4(w[(size_t)d * K + k], w[(size_t)(d + 1) * K + k], w[(size_t)(d + 2) * K + k],
                                w[(size_t)(d + 3) * K + k])
                  : f4z();
  float4 dw[K], db = f4z();
#pragma unroll
  for (int k = 0; k < K; ++k) dw[k] = f4z();
  const float4 b4 = (SILU && valid && bias != nullptr) ? *reinterpret_cast<const float4*>(bias + d) : f4z();
  // g[t] = dout[t] * silu'(pre[t]); xs points at x[t-(K-1)] .. x[t]
  auto gact = [&](float4 g, const float4* xs) {
    float4 pre = b4;
#pragma unroll
    for (int k = 0; k < K; ++k) pre = f4fma(wk[k], xs[k], pre);
    const float2 lo = gdsilu2(f2(g.x, g.y), f2(pre.x, pre.y)), hi = gdsilu2(f2(g.z, g.w), f2(pre.z, pre.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  };

  if (valid && SILU) {
    // walk the input steps t = t0 .. t1+K-2: g[t] is formed once from the x window behind t, enters dw / db
    // when t < t1, and completes dx[t-(K-1)] when that is in the tile; loads issued U steps at a time
    constexpr int U = 8;  // loads issued together, at three CTAs per SM (four CTAs with 4 loads: 80.4 us, 78.5 here)
    using R = RawX4<T>;
    for (int bt = blockIdx.y * ipc + sub; bt < B * ntt; bt += gridDim.y * ipc) {
      const int b = bt / ntt, t0 = (bt % ntt) * TILE;
      const int t1 = min(L, t0 + TILE);
      const int tend = t1 + K - 1, tl = min(L, tend);
      const float* g = dout + (size_t)b * L * D + d;
      const T* xb = x + (size_t)b * L * D + d;
      float4 xw[K], gw[K];  // xw[k] = x[t-(K-1)+k], gw[j] = g[t-(K-1)+j]
#pragma unroll
      for (int j = 0; j < K - 1; ++j) {
        const int tx = t0 - (K - 1) + j;
        xw[j + 1] = tx >= 0 ? ld_x4(xb + (size_t)tx * D) : f4z();
        gw[j + 1] = f4z();  // only ever combined into outputs before t0
      }
      for (int tb = t0; tb < tend; tb += U) {
        float4 gr[U];
        typename R::V xr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool in = tb + u < tl;
          gr[u] = in ? *reinterpret_cast<const float4*>(g + (size_t)(tb + u) * D) : f4z();
          xr[u] = in ? R::ld(xb + (size_t)(tb + u) * D) : R::zero();
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int t = tb + u;
          if (t < tend) {
#pragma unroll
            for (int j = 0; j < K - 1; ++j) {
              xw[j] = xw[j + 1];
              gw[j] = gw[j + 1];
            }
            xw[K - 1] = R::wide(xr[u]);
            gw[K - 1] = gact(gr[u], xw);
            if (t < t1) {
#pragma unroll
              for (int k = 0; k < K; ++k) dw[k] = f4fma(gw[K - 1], xw[k], dw[k]);
              db = f4add(db, gw[K - 1]);
            }
            const int s = t - (K - 1);
            if (s >= t0) {
              float4 acc = f4z();
#pragma unroll
              for (int j = 0; j < K; ++j) acc = f4fma(gw[j], wk[K - 1 - j], acc);
              *reinterpret_cast<float4*>(dx + ((size_t)b * L + s) * D + d) = acc;
            }
          }
        }
      }
    }
  } else if (valid) {
    for (int bt = blockIdx.y * ipc + sub; bt < B * ntt; bt += gridDim.y * ipc) {
      const int b = bt / ntt, t0 = (bt % ntt) * TILE;
      const int t1 = min(L, t0 + TILE);
      const float* g = dout + (size_t)b * L * D + d;
      const T* xb = x + (size_t)b * L * D + d;
      float4 gw[K], xw[K];  // gw[j] = dout[s+j], xw[k] = x[s-(K-1)+k]
#pragma unroll
      for (int j = 0; j < K - 1; ++j) {
        const int t = t0 + j;
        gw[j + 1] = t < L ? *reinterpret_cast<const float4*>(g + (size_t)t * D) : f4z();
        const int tx = t0 - (K - 1) + j;
        xw[j + 1] = tx >= 0 ? ld_x4(xb + (size_t)tx * D) : f4z();
      }
#pragma unroll 8
      for (int s = t0; s < t1; ++s) {
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
          gw[j] = gw[j + 1];
          xw[j] = xw[j + 1];
        }
        const int tg = s + K - 1;
        gw[K - 1] = tg < L ? *reinterpret_cast<const float4*>(g + (size_t)tg * D) : f4z();
        xw[K - 1] = ld_x4(xb + (size_t)s * D);
        float4 acc = f4z();
#pragma unroll
        for (int j = 0; j < K; ++j) acc = f4fma(gw[j], wk[K - 1 - j], acc);
        *reinterpret_cast<float4*>(dx + ((size_t)b * L + s) * D + d) = acc;
#pragma unroll
        for (int k = 0; k < K; ++k) dw[k] = f4fma(gw[0], xw[k], dw[k]);
        db = f4add(db, gw[0]);
      }
    }
  }
  if (valid) {
    float* o = ws + ((size_t)blockIdx.y * ipc + sub) * (K + 1) * D + d;  // partial row: [K+1][D]
#pragma unroll
    for (int k = 0; k < K; ++k) *reinterpret_cast<float4*>(o + (size_t)k * D) = dw[k];
    *reinterpret_cast<float4*>(o + (size_t)K * D) = db;
  }
}

// The SiLU-fused backward with 2 channels per thread (twice the threads of the
// 4-channel form, half the registers each), for fp32 x and rows of at least 256
// channels: the same input-step walk, loads of U steps issued together.
constexpr int kCtasSilu2 = 6;

template <int K>
__global__ void __launch_bounds__(kCThreads, kCtasSilu2) conv_silu_bwd2_kernel(const float* __restrict__ dout,
                                                                              const float* __restrict__ x,
                                                                              const float* __restrict__ w,
                                                                              const float* __restrict__ bias,
                                                                              float* __restrict__ dx,
                                                                              float* __restrict__ ws, int B, int L,
                                                                              int D) {
  pdl_trigger();  // the column sum of the partials may launch now; it waits for this grid's end
  constexpr int TILE = kCTileSilu;
  constexpr int U = 8;
  const int d = (int)(blockIdx.x * kCThreads + threadIdx.x) * 2;
  const bool valid = d < D;  // D % 8 == 0: both channels of a thread are in range
  const int ntt = (L + TILE - 1) / TILE;
  float2 wk[K], dw[K], db = f2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    wk[k] = valid ? f2(w[(size_t)d * K + k], w[(size_t)(d + 1) * K + k]) : f2(0.f, 0.f);
    dw[k] = f2(0.f, 0.f);
  }
  const float2 b2 = (valid && bias != nullptr) ? *reinterpret_cast<const float2*>(bias + d) : f2(0.f, 0.f);
  if (valid) {
    for (int bt = blockIdx.y; bt < B * ntt; bt += gridDim.y) {
      const int b = bt / ntt, t0 = (bt % ntt) * TILE;
      const int t1 = min(L, t0 + TILE);
      const int tend = t1 + K - 1, tl = min(L, tend);
      const float* g = dout + (size_t)b * L * D + d;
      const float* xb = x + (size_t)b * L * D + d;
      float2 xw[K], gw[K];  // xw[k] = x[t-(K-1)+k], gw[j] = g[t-(K-1)+j]
#pragma unroll
      for (int j = 0; j < K - 1; ++j) {
        const int tx = t0 - (K - 1) + j;
        xw[j + 1] = tx >= 0 ? *reinterpret_cast<const float2*>(xb + (size_t)tx * D) : f2(0.f, 0.f);
        gw[j + 1] = f2(0.f, 0.f);  // only ever combined into outputs before t0
      }
      for (int tb = t0; tb < tend; tb += U) {
        float2 gr[U], xr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool in = tb + u < tl;
          gr[u] = in ? *reinterpret_cast<const float2*>(g + (size_t)(tb + u) * D) : f2(0.f, 0.f);
          xr[u] = in ? *reinterpret_cast<const float2*>(xb + (size_t)(tb + u) * D) : f2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int t = tb + u;
          if (t < tend) {
#pragma unroll
            for (int j = 0; j < K - 1; ++j) {
              xw[j] = xw[j + 1];
              gw[j] = gw[j + 1];
            }
            xw[K - 1] = xr[u];
            float2 pre = b2;
#pragma unroll
            for (int k = 0; k < K; ++k) pre = fma2(wk[k], xw[k], pre);
            gw[K - 1] = gdsilu2(gr[u], pre);
            if (t < t1) {
#pragma unroll
              for (int k = 0; k < K; ++k) dw[k] = fma2(gw[K - 1], xw[k], dw[k]);
              db = add2(db, gw[K - 1]);
            }
            const int sdx = t - (K - 1);
            if (sdx >= t0) {
              float2 acc = f2(0.f, 0.f);
#pragma unroll
              for (int j = 0; j < K; ++j) acc = fma2(gw[j], wk[K - 1 - j], acc);
              *reinterpret_cast<float2*>(dx + ((size_t)b * L + sdx) * D + d) = acc;
            }
          }
        }
      }
    }
    float* o = ws + (size_t)blockIdx.y * (K + 1) * D + d;  // partial row: [K+1][D]
#pragma unroll
    for (int k = 0; k < K; ++k) *reinterpret_cast<float2*>(o + (size_t)k * D) = dw[k];
    *reinterpret_cast<float2*>(o + (size_t)K * D) = db;
  }
}

// column i = k * D + d of the partials: dw[d, k] (k < K) or db[d] (k = K)
struct ConvStore {
  float* dw;
  float* db;
  int D, K;
  __device__ void put(long long i, float v) const {
    const int k = (int)(i / D), d = (int)(i % D);
    if (k < K) dw[(size_t)d * K + k] += v;
    else db[d] += v;
  }
};

struct ConvPlan {
  int gx, gy, rows;
  size_t bytes;
};

inline ConvPlan conv_plan(int B, int L, int D, int K) {
  ConvPlan p;
  p.gx = (D / 4 + kCThreads - 1) / kCThreads;
  const long long pairs = (long long)B * ((L + kCTile - 1) / kCTile);
  long long cap = 608 / p.gx;  // one wave: 4 resident CTAs on each of 152 SMs, each looping over its items
  if (cap < 1) cap = 1;
  const int ipc = D / 4 >= kCThreads ? 1 : kCThreads / (D / 4);  // items per CTA step (narrow rows)
  const long long rows_needed = (pairs + ipc - 1) / ipc;
  p.gy = (int)(rows_needed < cap ? rows_needed : cap);
  p.rows = p.gy * ipc;  // partial rows: one per (CTA row, item slot)
  p.bytes = (size_t)p.rows * D * (K + 1) * sizeof(float);
  return p;
}

int conv_validate(int B, int L, int D, int K, int x_dtype) {
  if (B <= 0 || L <= 0 || D <= 0 || K <= 0) return SS_ERR_DIM;
  if (K > 4) return SS_ERR_UNSUPPORTED;
  if (x_dtype != SS_F32 && x_dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (D % 8 != 0) return SS_ERR_ALIGN;
  if ((long long)B * ((L + kCTile - 1) / kCTile) >= (1ll << 31)) return SS_ERR_DIM;
  return SS_OK;
}

template <int K, typename T, bool SILU>
int conv_launch(const float* dout, const void* x, const float* w, const float* bias, float* dx, float* dw, float* db,
                int B, int L, int D, float* ws, const ConvPlan& pl, cudaStream_t s) {
  // fp32 x: two channels per thread, one wave of kCtasSilu2 CTAs per SM (mamba130m 70 -> 64 us); bf16 x keeps four
  // (its two-channel loads of x would be 4 bytes: 81 -> 99 us on the 1.4B layer)
  if constexpr (SILU && sizeof(T) == 4) {
    if (D >= 2 * kCThreads) {
      const int gx2 = (D / 2 + kCThreads - 1) / kCThreads;
      int gy2 = (kCtasSilu2 * device_sm_count()) / gx2;
      if (gy2 < 1) gy2 = 1;
      if (gy2 > pl.rows) gy2 = pl.rows;  // the workspace holds pl.rows partial rows
      const long long items = (long long)B * ((L + kCTileSilu - 1) / kCTileSilu);
      if (gy2 > items) gy2 = (int)items;
      conv_silu_bwd2_kernel<K><<<dim3(gx2, gy2), kCThreads, 0, s>>>(dout, static_cast<const float*>(x), w, bias, dx, ws,
                                                                     B, L, D);
      if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
      return colsum(ws, (long long)D * (K + 1), gy2, ConvStore{dw, db, D, K}, s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
    }
  }
  // one wave: the SiLU-fused form holds three CTAs per SM, so it runs fewer CTA rows (and partial rows)
  int gy = pl.gy, rows = pl.rows;
  if (SILU) {
    const int cap = (kCtasSilu * device_sm_count()) / pl.gx > 0 ? (kCtasSilu * device_sm_count()) / pl.gx : 1;
    if (gy > cap) {
      rows = rows / gy * cap;
      gy = cap;
    }
  }
  conv_bwd_kernel<K, T, SILU>
      <<<dim3(pl.gx, gy), kCThreads, 0, s>>>(dout, static_cast<const T*>(x), w, bias, dx, ws, B, L, D);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  return colsum(ws, (long long)D * (K + 1), rows, ConvStore{dw, db, D, K}, s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

extern "C" size_t conv1d_causal_bwd_workspace_size(int B, int L, int D, int d_conv) {
  if (conv_validate(B, L, D, d_conv, SS_F32) != SS_OK) return 0;
  return conv_plan(B, L, D, d_conv).bytes;
}

namespace {

template <typename T, bool SILU>
int conv_dispatch(const float* dout, const void* x, const float* w, const float* bias, float* dx, float* dw, float* db,
                  int B, int L, int D, int K, float* ws, const ConvPlan& pl, cudaStream_t s) {
  switch (K) {
    case 1: return conv_launch<1, T, SILU>(dout, x, w, bias, dx, dw, db, B, L, D, ws, pl, s);
    case 2: return conv_launch<2, T, SILU>(dout, x, w, bias, dx, dw, db, B, L, D, ws, pl, s);
    case 3: return conv_launch<3, T, SILU>(dout, x, w, bias, dx, dw, db, B, L, D, ws, pl, s);
    default: return conv_launch<4, T, SILU>(dout, x, w, bias, dx, dw, db, B, L, D, ws, pl, s);
  }
}

template <bool SILU>
int conv_bwd_entry(const float* dout, const void* x, const float* w, const float* bias, float* dx, float* dw, float* db,
                   int B, int L, int D, int d_conv, int x_dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (!dout || !x || !w || !dx || !dw || !db) return SS_ERR_NULL;
  const int v = conv_validate(B, L, D, d_conv, x_dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {dout, x, w, dx, dw, db};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  if (bias && !ssh::aligned16(bias)) return SS_ERR_ALIGN;
  const ConvPlan pl = conv_plan(B, L, D, d_conv);
  if (workspace == nullptr || ws_bytes < pl.bytes) return SS_ERR_WORKSPACE;
  if (!ssh::aligned16(workspace)) return SS_ERR_ALIGN;
  float* ws = static_cast<float*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (x_dtype == SS_F32) return conv_dispatch<float, SILU>(dout, x, w, bias, dx, dw, db, B, L, D, d_conv, ws, pl, s);
  return conv_dispatch<__nv_bfloat16, SILU>(dout, x, w, bias, dx, dw, db, B, L, D, d_conv, ws, pl, s);
}

}  // namespace

extern "C" int conv1d_causal_bwd(const float* dout, const void* x, const float* w, float* dx, float* dw, float* db, int B,
                                 int L, int D, int d_conv, int x_dtype, void* workspace, size_t ws_bytes, void* stream) {
  return conv_bwd_entry<false>(dout, x, w, nullptr, dx, dw, db, B, L, D, d_conv, x_dtype, workspace, ws_bytes, stream);
}

extern "C" int conv1d_causal_silu_bwd(const float* dact, const void* x, const float* w, const float* bias, float* dx,
                                      float* dw, float* db, int B, int L, int D, int d_conv, int x_dtype, void* workspace,
                                      size_t ws_bytes, void* stream) {
  return conv_bwd_entry<true>(dact, x, w, bias, dx, dw, db, B, L, D, d_conv, x_dtype, workspace, ws_bytes, stream);
}
