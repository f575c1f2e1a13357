// Depthwise causal conv1d forward (conv1d_causal_fwd) for sm_103a, with an
// optional SiLU on the output:
//
//   pre[t,d] = bias[d] + sum_k w[d,k] x[t-(K-1)+k, d]     (x at t < 0 is 0; newest input at tap K-1)
//   out[t,d] = silu ? pre * sigmoid(pre) : pre
//
// A thread owns 4 adjacent channels over a 64-step tile of one batch row and
// slides a K-wide register window of x along time; CTAs loop over (batch row,
// tile) pairs.  HBM traffic is one read of x and one write of out (the K-1
// halo steps of a tile come from L2).
#include "common.cuh"

namespace {

using namespace ssk;

constexpr int kFTile = 64;      // time steps per tile
constexpr int kFThreads = 128;  // threads per CTA: 512 channels

template <typename T>
__device__ __forceinline__ float4 ld4g(const T* p);
template <>
__device__ __forceinline__ float4 ld4g<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 ld4g<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
}

template <typename T>
__device__ __forceinline__ void st4g(T* p, float4 v);
template <>
__device__ __forceinline__ void st4g<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <>
__device__ __forceinline__ void st4g<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(ActT<__nv_bfloat16>::pack2(v.x, v.y), ActT<__nv_bfloat16>::pack2(v.z, v.w));
}

__device__ __forceinline__ float silu(float v) { return v * sigmoid(v); }

template <int K, typename T, bool SILU>
__global__ void __launch_bounds__(kFThreads) conv_fwd_kernel(const T* __restrict__ x, const float* __restrict__ w,
                                                             const float* __restrict__ bias, T* __restrict__ out, int B,
                                                             int L, int D) {
  // rows narrower than a CTA pack ipc (batch row, tile) items per CTA step
  const int cpr = D / 4;
  const int ipc = cpr >= kFThreads ? 1 : kFThreads / cpr;
  const int sub = cpr >= kFThreads ? 0 : (int)threadIdx.x / cpr;
  const int d = (cpr >= kFThreads ? (int)(blockIdx.x * kFThreads + threadIdx.x) : (int)threadIdx.x % cpr) * 4;
  if (d >= D || sub >= ipc) return;  // D % 8 == 0: all four channels of a thread are in range
  const int ntt = (L + kFTile - 1) / kFTile;
  float4 wk[K];
#pragma unroll
  for (int k = 0; k < K; ++k)
    wk[k] = make_float4(w[(size_t)d * K + k], w[(size_t)(d + 1) * K + k], w[(size_t)(d + 2) * K + k],
                        w[(size_t)(d + 3) * K + k]);
  const float4 b4 = bias != nullptr ? *reinterpret_cast<const float4*>(bias + d) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int bt = blockIdx.y * ipc + sub; bt < B * ntt; bt += gridDim.y * ipc) {
    const int b = bt / ntt, t0 = (bt % ntt) * kFTile;
    const int t1 = min(L, t0 + kFTile);
    const T* xb = x + (size_t)b * L * D + d;
    T* ob = out + (size_t)b * L * D + d;
    float4 xw[K];  // xw[k] = x[s-(K-1)+k]
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      const int tx = t0 - (K - 1) + j;
      xw[j + 1] = tx >= 0 ? ld4g(xb + (size_t)tx * D) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 4
    for (int s = t0; s < t1; ++s) {
#pragma unroll
      for (int j = 0; j < K - 1; ++j) xw[j] = xw[j + 1];
      xw[K - 1] = ld4g(xb + (size_t)s * D);
      float4 acc = b4;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        acc.x = fmaf(wk[k].x, xw[k].x, acc.x);
        acc.y = fmaf(wk[k].y, xw[k].y, acc.y);
        acc.z = fmaf(wk[k].z, xw[k].z, acc.z);
        acc.w = fmaf(wk[k].w, xw[k].w, acc.w);
      }
      if (SILU) acc = make_float4(silu(acc.x), silu(acc.y), silu(acc.z), silu(acc.w));
      st4g(ob + (size_t)s * D, acc);
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
  const long long pairs = (long long)B * ((L + kFTile - 1) / kFTile);
  long long cap = 4096 / gx;
  if (cap < 1) cap = 1;
  const int gy = (int)(pairs < cap ? pairs : cap);
  const T* xx = static_cast<const T*>(x);
  T* o = static_cast<T*>(out);
  if (silu) conv_fwd_kernel<K, T, true><<<dim3(gx, gy), kFThreads, 0, s>>>(xx, w, bias, o, B, L, D);
  else conv_fwd_kernel<K, T, false><<<dim3(gx, gy), kFThreads, 0, s>>>(xx, w, bias, o, B, L, D);
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
