// Depthwise causal conv1d forward (conv1d_causal_fwd) for sm_103a, with an
// optional SiLU on the output:
//
//   pre[t,d] = bias[d] + sum_k w[d,k] x[t-(K-1)+k, d]     (x at t < 0 is 0; newest input at tap K-1)
//   out[t,d] = silu ? pre * sigmoid(pre) : pre
//
// One CTA per (512-channel block, batch row, 16-step tile): a thread owns 4
// adjacent channels over the tile, issues the tile's 16 + K - 1 loads of its
// x column together and then forms the 16 outputs on channel pairs (packed
// f32x2 arithmetic).  HBM traffic is one read of x and one write of out (the
// K - 1 halo steps of a tile come from L2).  A persistent form (CTAs looping
// over tiles with a sliding register window) measured 35 us on the 1.4B layer
// against 29 us for this one.
#include "common.cuh"

namespace {

using namespace ssk;

constexpr int kFThreads = 128;  // threads per CTA: 512 channels

template <typename T>
__device__ __forceinline__ void st4g(T* p, float4 v);
template <>
__device__ __forceinline__ void st4g<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <>
__device__ __forceinline__ void st4g<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(ActT<__nv_bfloat16>::pack2(v.x, v.y), ActT<__nv_bfloat16>::pack2(v.z, v.w));
}

// raw activation vector of 4 channels as loaded (8 bytes for bf16, 16 for fp32) and its widening
template <typename T>
struct Raw4;
template <>
struct Raw4<float> {
  using V = float4;
  static __device__ __forceinline__ V ld(const float* p) { return *reinterpret_cast<const float4*>(p); }
  static __device__ __forceinline__ float4 wide(V v) { return v; }
  static __device__ __forceinline__ V zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct Raw4<__nv_bfloat16> {
  using V = uint2;
  static __device__ __forceinline__ V ld(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ float4 wide(V v) { return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)); }
  static __device__ __forceinline__ V zero() { return make_uint2(0u, 0u); }
};

constexpr int kFTile = 16;  // time steps per CTA (measured: 8 and 32 slower on the 1.4B layer)

// One (channel block, batch row, TS-step tile) per CTA, no loop: a thread owns
// 4 channels over TS steps, issues all TS + K - 1 loads of its x column at once
// (the K - 1 halo rows are the previous tile's last rows, read again from L2),
// then forms and stores the TS outputs.  blockIdx.x = item * gx + channel block.
// The arithmetic runs on channel pairs (packed f32x2: the same roundings as
// scalar code), the taps of a channel come as one 16-byte row of w when K = 4,
// and tiles away from the sequence ends skip every bounds test.
template <int K>
__device__ __forceinline__ void load_taps(const float* __restrict__ w, int d, float2 (&wlo)[K], float2 (&whi)[K]) {
  if constexpr (K == 4) {
    const float4 r0 = __ldg(reinterpret_cast<const float4*>(w + (size_t)d * 4));
    const float4 r1 = __ldg(reinterpret_cast<const float4*>(w + (size_t)(d + 1) * 4));
    const float4 r2 = __ldg(reinterpret_cast<const float4*>(w + (size_t)(d + 2) * 4));
    const float4 r3 = __ldg(reinterpret_cast<const float4*>(w + (size_t)(d + 3) * 4));
    wlo[0] = f2(r0.x, r1.x); wlo[1] = f2(r0.y, r1.y); wlo[2] = f2(r0.z, r1.z); wlo[3] = f2(r0.w, r1.w);
    whi[0] = f2(r2.x, r3.x); whi[1] = f2(r2.y, r3.y); whi[2] = f2(r2.z, r3.z); whi[3] = f2(r2.w, r3.w);
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      wlo[k] = f2(__ldg(w + (size_t)d * K + k), __ldg(w + (size_t)(d + 1) * K + k));
      whi[k] = f2(__ldg(w + (size_t)(d + 2) * K + k), __ldg(w + (size_t)(d + 3) * K + k));
    }
  }
}

// silu(v) = v / (1 + 2^(-v log2 e)) on a channel pair
__device__ __forceinline__ float2 silu2(float2 v) {
  const float2 e = ex2_2(mul2(v, bc2(-kLog2e)));
  const float2 den = add2(e, bc2(1.0f));
  return mul2(v, f2(rcp(den.x), rcp(den.y)));
}

template <int K, typename T, bool SILU, int TS>
__global__ void __launch_bounds__(kFThreads) conv_fwd_tile_kernel(const T* __restrict__ x, const float* __restrict__ w,
                                                                  const float* __restrict__ bias, T* __restrict__ out,
                                                                  int L, int D, int gx, int ntt) {
  using R = Raw4<T>;
  const int cx = (int)(blockIdx.x % (unsigned)gx);
  const long long item = blockIdx.x / (unsigned)gx;
  const int b = (int)(item / ntt), t0 = (int)(item % ntt) * TS;
  const int d = (cx * kFThreads + (int)threadIdx.x) * 4;
  if (d >= D) return;  // D % 8 == 0: all four channels of a thread are in range
  const bool inner = t0 >= K - 1 && t0 + TS <= L;
  const T* xb = x + ((size_t)b * L + t0) * D + d;  // row t0 of this thread's column
  typename R::V xr[TS + K - 1];  // xr[j] = x[t0 - (K-1) + j]
  if (inner) {
#pragma unroll
    for (int j = 0; j < TS + K - 1; ++j) xr[j] = R::ld(xb + (j - (K - 1)) * D);
  } else {
#pragma unroll
    for (int j = 0; j < TS + K - 1; ++j) {
      const int t = t0 - (K - 1) + j;
      xr[j] = (t >= 0 && t < L) ? R::ld(xb + (j - (K - 1)) * D) : R::zero();
    }
  }
  float2 wlo[K], whi[K];
  load_taps<K>(w, d, wlo, whi);
  float2 blo = f2(0.f, 0.f), bhi = f2(0.f, 0.f);
  if (bias != nullptr) {
    const float4 b4 = __ldg(reinterpret_cast<const float4*>(bias + d));
    blo = f2(b4.x, b4.y);
    bhi = f2(b4.z, b4.w);
  }
  T* ob = out + ((size_t)b * L + t0) * D + d;
#pragma unroll
  for (int s = 0; s < TS; ++s) {
    if (inner || t0 + s < L) {
      float2 lo = blo, hi = bhi;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const float4 xv = R::wide(xr[s + k]);
        lo = fma2(wlo[k], f2(xv.x, xv.y), lo);
        hi = fma2(whi[k], f2(xv.z, xv.w), hi);
      }
      if (SILU) {
        lo = silu2(lo);
        hi = silu2(hi);
      }
      st4g(ob + s * D, make_float4(lo.x, lo.y, hi.x, hi.y));
    }
  }
}

int conv_fwd_validate(int B, int L, int D, int K, int x_dtype) {
  if (B <= 0 || L <= 0 || D <= 0 || K <= 0) return SS_ERR_DIM;
  if (K > 4) return SS_ERR_UNSUPPORTED;
  if (x_dtype != SS_F32 && x_dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (D % 8 != 0) return SS_ERR_ALIGN;
  if ((long long)B * ((L + kFTile - 1) / kFTile) >= (1ll << 31)) return SS_ERR_DIM;
  return SS_OK;
}

template <int K, typename T>
int conv_fwd_launch(const void* x, const float* w, const float* bias, void* out, int B, int L, int D, int silu,
                    cudaStream_t s) {
  const int gx = (D / 4 + kFThreads - 1) / kFThreads;
  const int ntt = (L + kFTile - 1) / kFTile;
  const long long blocks = (long long)gx * B * ntt;
  if (blocks >= (1ll << 31) || (long long)(kFTile + 4) * D >= (1ll << 31)) return SS_ERR_DIM;
  const T* xx = static_cast<const T*>(x);
  T* o = static_cast<T*>(out);
  if (silu) conv_fwd_tile_kernel<K, T, true, kFTile><<<(unsigned)blocks, kFThreads, 0, s>>>(xx, w, bias, o, L, D, gx, ntt);
  else conv_fwd_tile_kernel<K, T, false, kFTile><<<(unsigned)blocks, kFThreads, 0, s>>>(xx, w, bias, o, L, D, gx, ntt);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename T>
int conv_fwd_dispatch(const void* x, const float* w, const float* bias, void* out, int B, int L, int D, int K, int silu,
                      cudaStream_t s) {
  switch (K) {
    case 1: return conv_fwd_launch<1, T>(x, w, bias, out, B, L, D, silu, s);
    case 2: return conv_fwd_launch<2, T>(x, w, bias, out, B, L, D, silu, s);
    case 3: return conv_fwd_launch<3, T>(x, w, bias, out, B, L, D, silu, s);
    default: return conv_fwd_launch<4, T>(x, w, bias, out, B, L, D, silu, s);
  }
}

}  // namespace

extern "C" int conv1d_causal_fwd(const void* x, const float* w, const float* bias, void* out, int B, int L, int D,
                                 int d_conv, int silu, int x_dtype, void* stream) {
  if (!x || !w || !out) return SS_ERR_NULL;
  const int v = conv_fwd_validate(B, L, D, d_conv, x_dtype);
  if (v != SS_OK) return v;
  if (!ssh::aligned16(x) || !ssh::aligned16(out) || (bias && !ssh::aligned16(bias))) return SS_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (x_dtype == SS_F32) return conv_fwd_dispatch<float>(x, w, bias, out, B, L, D, d_conv, silu, s);
  return conv_fwd_dispatch<__nv_bfloat16>(x, w, bias, out, B, L, D, d_conv, silu, s);
}
