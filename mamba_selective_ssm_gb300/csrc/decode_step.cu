// Single-token recurrent updates (decode) for sm_103a: ss_scan_step and
// conv1d_causal_step.  One call advances B independent sequences by one step.
//
// ss_scan_step, per (b, d):
//   h[d,n] <- exp(delta[d] A[d,n]) h[d,n] + delta[d] B[n] x[d]
//   y[d]    = (sum_n C[n] h[d,n] + D[d] x[d]) * silu(z[d])
// The N/4 lanes of a channel are consecutive; each loads and stores its four
// states as one 16-byte vector (so a warp moves contiguous 512-byte runs of
// h), and the state sum over n is a shuffle reduction over those lanes.
//
// conv1d_causal_step, per (b, d): the shift register state[0..K-1] (newest at
// K-1) moves one tap towards 0, takes x at tap K-1, and
//   out[d] = act(bias[d] + sum_k w[d,k] state[k]).
#include "common.cuh"

namespace {

using namespace ssk;

constexpr int kStepThreads = 256;

template <int N, typename T>
__global__ void __launch_bounds__(kStepThreads) ss_step_kernel(const T* __restrict__ x, const T* __restrict__ delta,
                                                               const float* __restrict__ A, const T* __restrict__ Bm,
                                                               const T* __restrict__ Cm, const float* __restrict__ Dv,
                                                               const T* __restrict__ z, float* __restrict__ h,
                                                               T* __restrict__ y, int B, int D) {
  using AT = ActT<T>;
  constexpr int NG = N / 4;  // lanes per channel
  const long long gid = (long long)blockIdx.x * kStepThreads + threadIdx.x;
  const long long q = gid / NG;  // channel index over B*D
  const int ng = (int)(gid % NG);
  const bool ok = q < (long long)B * D;
  const int b = ok ? (int)(q / D) : 0, d = ok ? (int)(q % D) : 0;
  float part = 0.f, xd = 0.f;
  if (ok) {
    const float dt = AT::ld(delta + q);
    xd = AT::ld(x + q);
    const float4 a4 = *reinterpret_cast<const float4*>(A + (size_t)d * N + ng * 4);
    float4 hv = *reinterpret_cast<const float4*>(h + q * N + ng * 4);
    const T* bb = Bm + (size_t)b * N + ng * 4;
    const T* cc = Cm + (size_t)b * N + ng * 4;
    const float dx = dt * xd;
    hv.x = fmaf(ex2(dt * (a4.x * kLog2e)), hv.x, dx * AT::ld(bb + 0));
    hv.y = fmaf(ex2(dt * (a4.y * kLog2e)), hv.y, dx * AT::ld(bb + 1));
    hv.z = fmaf(ex2(dt * (a4.z * kLog2e)), hv.z, dx * AT::ld(bb + 2));
    hv.w = fmaf(ex2(dt * (a4.w * kLog2e)), hv.w, dx * AT::ld(bb + 3));
    *reinterpret_cast<float4*>(h + q * N + ng * 4) = hv;
    part = fmaf(AT::ld(cc + 0), hv.x, fmaf(AT::ld(cc + 1), hv.y, fmaf(AT::ld(cc + 2), hv.z, AT::ld(cc + 3) * hv.w)));
  }
#pragma unroll
  for (int o = 1; o < NG; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (ok && ng == 0) {
    const float zz = AT::ld(z + q);
    const float s = fmaf(Dv[d], xd, part);
    const float o = s * zz * sigmoid(zz);
    if constexpr (sizeof(T) == 4) y[q] = o;
    else y[q] = __float2bfloat16_rn(o);
  }
}

template <int K, typename T, bool SILU>
__global__ void __launch_bounds__(kStepThreads) conv_step_kernel(const T* __restrict__ x, float* __restrict__ state,
                                                                 const float* __restrict__ w,
                                                                 const float* __restrict__ bias, T* __restrict__ out,
                                                                 int B, int D) {
  const long long q = (long long)blockIdx.x * kStepThreads + threadIdx.x;
  if (q >= (long long)B * D) return;
  const int d = (int)(q % D);
  float st[K];
#pragma unroll
  for (int k = 0; k < K; ++k) st[k] = state[q * K + k];
#pragma unroll
  for (int k = 0; k < K - 1; ++k) st[k] = st[k + 1];
  st[K - 1] = ActT<T>::ld(x + q);
  float acc = bias != nullptr ? bias[d] : 0.f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    acc = fmaf(w[(size_t)d * K + k], st[k], acc);
    state[q * K + k] = st[k];
  }
  if (SILU) acc = acc * sigmoid(acc);
  if constexpr (sizeof(T) == 4) out[q] = acc;
  else out[q] = __float2bfloat16_rn(acc);
}

template <int N, typename T>
int step_launch(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm, const float* Dv,
                const void* z, float* h, void* y, int B, int D, cudaStream_t s) {
  const long long threads = (long long)B * D * (N / 4);
  const long long blocks = (threads + kStepThreads - 1) / kStepThreads;
  ss_step_kernel<N, T><<<(unsigned)blocks, kStepThreads, 0, s>>>(
      static_cast<const T*>(x), static_cast<const T*>(delta), A, static_cast<const T*>(Bm), static_cast<const T*>(Cm), Dv,
      static_cast<const T*>(z), h, static_cast<T*>(y), B, D);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <int K, typename T>
int conv_step_launch(const void* x, float* state, const float* w, const float* bias, void* out, int B, int D, int silu,
                     cudaStream_t s) {
  const long long blocks = ((long long)B * D + kStepThreads - 1) / kStepThreads;
  const T* xx = static_cast<const T*>(x);
  T* o = static_cast<T*>(out);
  if (silu) conv_step_kernel<K, T, true><<<(unsigned)blocks, kStepThreads, 0, s>>>(xx, state, w, bias, o, B, D);
  else conv_step_kernel<K, T, false><<<(unsigned)blocks, kStepThreads, 0, s>>>(xx, state, w, bias, o, B, D);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename T>
int conv_step_dispatch(const void* x, float* state, const float* w, const float* bias, void* out, int B, int D, int K,
                       int silu, cudaStream_t s) {
  switch (K) {
    case 1: return conv_step_launch<1, T>(x, state, w, bias, out, B, D, silu, s);
    case 2: return conv_step_launch<2, T>(x, state, w, bias, out, B, D, silu, s);
    case 3: return conv_step_launch<3, T>(x, state, w, bias, out, B, D, silu, s);
    default: return conv_step_launch<4, T>(x, state, w, bias, out, B, D, silu, s);
  }
}

}  // namespace

extern "C" int ss_scan_step(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                            const float* Dv, const void* z, float* h, void* y, int B, int D, int N, int dtype,
                            void* stream) {
  if (!x || !delta || !A || !Bm || !Cm || !Dv || !z || !h || !y) return SS_ERR_NULL;
  if (B <= 0 || D <= 0 || N <= 0) return SS_ERR_DIM;
  if (N != 4 && N != 8 && N != 16) return SS_ERR_UNSUPPORTED;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if ((long long)B * D * (N / 4) >= (1ll << 38)) return SS_ERR_DIM;  // grid.x < 2^31 blocks
  if (!ssh::aligned16(A) || !ssh::aligned16(h)) return SS_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) {
    if (N == 4) return step_launch<4, float>(x, delta, A, Bm, Cm, Dv, z, h, y, B, D, s);
    if (N == 8) return step_launch<8, float>(x, delta, A, Bm, Cm, Dv, z, h, y, B, D, s);
    return step_launch<16, float>(x, delta, A, Bm, Cm, Dv, z, h, y, B, D, s);
  }
  if (N == 4) return step_launch<4, __nv_bfloat16>(x, delta, A, Bm, Cm, Dv, z, h, y, B, D, s);
  if (N == 8) return step_launch<8, __nv_bfloat16>(x, delta, A, Bm, Cm, Dv, z, h, y, B, D, s);
  return step_launch<16, __nv_bfloat16>(x, delta, A, Bm, Cm, Dv, z, h, y, B, D, s);
}

extern "C" int conv1d_causal_step(const void* x, float* conv_state, const float* w, const float* bias, void* out, int B,
                                  int D, int d_conv, int silu, int dtype, void* stream) {
  if (!x || !conv_state || !w || !out) return SS_ERR_NULL;
  if (B <= 0 || D <= 0 || d_conv <= 0) return SS_ERR_DIM;
  if (d_conv > 4) return SS_ERR_UNSUPPORTED;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if ((long long)B * D >= (1ll << 38)) return SS_ERR_DIM;  // grid.x < 2^31 blocks
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) return conv_step_dispatch<float>(x, conv_state, w, bias, out, B, D, d_conv, silu, s);
  return conv_step_dispatch<__nv_bfloat16>(x, conv_state, w, bias, out, B, D, d_conv, silu, s);
}
