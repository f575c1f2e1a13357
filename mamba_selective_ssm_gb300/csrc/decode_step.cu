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

// CTA (blockIdx.x = sequence b, blockIdx.y = a run of U * kStepThreads
// (channel, state quad) slots of that sequence): each thread advances U state
// vectors, with all their loads issued before the arithmetic.  U = 2 when the
// grid still has a few CTAs per SM (1024 sequences: 120.8 -> 115.6 us with the
// vector B_t / C_t loads), 1 for a handful of sequences, whose latency is the
// number of CTAs in flight.
template <int N, typename T, bool VBC, int U>
__global__ void __launch_bounds__(kStepThreads) ss_step_kernel(const T* __restrict__ x, const T* __restrict__ delta,
                                                               const float* __restrict__ A, const T* __restrict__ Bm,
                                                               const T* __restrict__ Cm, const float* __restrict__ Dv,
                                                               const T* __restrict__ z, float* __restrict__ h,
                                                               T* __restrict__ y, int B, int D) {
  using AT = ActT<T>;
  constexpr int NG = N / 4;  // lanes per channel
  const int b = (int)blockIdx.x;
  const T* bb = Bm + (size_t)b * N;
  const T* cc = Cm + (size_t)b * N;
  float4 hv[U], a4[U];
  float dt[U], xd[U];
  bool ok[U];
  int d[U], ng[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int slot = ((int)blockIdx.y * U + u) * kStepThreads + (int)threadIdx.x;  // d * NG + ng
    d[u] = slot / NG;
    ng[u] = slot % NG;
    ok[u] = d[u] < D;
    const size_t q = (size_t)b * D + (ok[u] ? d[u] : 0);
    dt[u] = ok[u] ? AT::ld(delta + q) : 0.f;
    xd[u] = ok[u] ? AT::ld(x + q) : 0.f;
    a4[u] = ok[u] ? *reinterpret_cast<const float4*>(A + (size_t)d[u] * N + ng[u] * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    hv[u] = ok[u] ? *reinterpret_cast<const float4*>(h + q * N + ng[u] * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const size_t q = (size_t)b * D + (ok[u] ? d[u] : 0);
    const T* bq = bb + ng[u] * 4;
    const T* cq = cc + ng[u] * 4;
    float bv[4], cv[4];  // one 8- or 16-byte load each when B_t / C_t rows are aligned for it
    if constexpr (VBC) {
      AT::ld4(bq, bv);
      AT::ld4(cq, cv);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bv[k] = AT::ld(bq + k);
        cv[k] = AT::ld(cq + k);
      }
    }
    const float dx = dt[u] * xd[u];
    float4 v = hv[u];
    v.x = fmaf(ex2(dt[u] * (a4[u].x * kLog2e)), v.x, dx * bv[0]);
    v.y = fmaf(ex2(dt[u] * (a4[u].y * kLog2e)), v.y, dx * bv[1]);
    v.z = fmaf(ex2(dt[u] * (a4[u].z * kLog2e)), v.z, dx * bv[2]);
    v.w = fmaf(ex2(dt[u] * (a4[u].w * kLog2e)), v.w, dx * bv[3]);
    if (ok[u]) *reinterpret_cast<float4*>(h + q * N + ng[u] * 4) = v;
    float part = fmaf(cv[0], v.x, fmaf(cv[1], v.y, fmaf(cv[2], v.z, cv[3] * v.w)));
#pragma unroll
    for (int o = 1; o < NG; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (ok[u] && ng[u] == 0) {
      const float zz = AT::ld(z + q);
      const float s = fmaf(Dv[d[u]], xd[u], part);
      const float o = s * zz * sigmoid(zz);
      if constexpr (sizeof(T) == 4) y[q] = o;
      else y[q] = __float2bfloat16_rn(o);
    }
  }
}

// CTA (blockIdx.x = sequence b, blockIdx.y = a run of U * kStepThreads
// channels): each thread shifts U channels' registers, loads first.  With VEC
// (K = 4, 16-byte aligned state) a channel's register is one 16-byte load and
// store.
template <int K, typename T, bool SILU, bool VEC, int U>
__global__ void __launch_bounds__(kStepThreads) conv_step_kernel(const T* __restrict__ x, float* __restrict__ state,
                                                                 const float* __restrict__ w,
                                                                 const float* __restrict__ bias, T* __restrict__ out,
                                                                 int B, int D) {
  const int b = (int)blockIdx.x;
  float st[U][K], xv[U];
  int d[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    d[u] = ((int)blockIdx.y * U + u) * kStepThreads + (int)threadIdx.x;
    const size_t q = (size_t)b * D + d[u];
    if (d[u] < D) {
      if constexpr (VEC) {
        const float4 v = *reinterpret_cast<const float4*>(state + q * K);
        st[u][0] = v.x; st[u][1] = v.y; st[u][2] = v.z; st[u][3] = v.w;
      } else {
#pragma unroll
        for (int k = 0; k < K; ++k) st[u][k] = state[q * K + k];
      }
      xv[u] = ActT<T>::ld(x + q);
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (d[u] >= D) continue;
    const size_t q = (size_t)b * D + d[u];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) st[u][k] = st[u][k + 1];
    st[u][K - 1] = xv[u];
    float acc = bias != nullptr ? bias[d[u]] : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) acc = fmaf(w[(size_t)d[u] * K + k], st[u][k], acc);
    if constexpr (VEC) {
      *reinterpret_cast<float4*>(state + q * K) = make_float4(st[u][0], st[u][1], st[u][2], st[u][3]);
    } else {
#pragma unroll
      for (int k = 0; k < K; ++k) state[q * K + k] = st[u][k];
    }
    if (SILU) acc = acc * sigmoid(acc);
    if constexpr (sizeof(T) == 4) out[q] = acc;
    else out[q] = __float2bfloat16_rn(acc);
  }
}

template <int N, typename T>
int step_launch(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm, const float* Dv,
                const void* z, float* h, void* y, int B, int D, cudaStream_t s) {
  const long long slots = (long long)D * (N / 4);  // per sequence
  const long long runs2 = (slots + 2 * kStepThreads - 1) / (2 * kStepThreads);
  const bool two = (long long)B * runs2 >= 2ll * device_sm_count();
  const long long runs = two ? runs2 : (slots + kStepThreads - 1) / kStepThreads;
  const uintptr_t quad = 4 * sizeof(T) - 1;  // a state quad of B_t / C_t: 8 bytes (bf16) or 16 (fp32)
  const bool vbc = ((reinterpret_cast<uintptr_t>(Bm) | reinterpret_cast<uintptr_t>(Cm)) & quad) == 0;
  auto kern = two ? (vbc ? ss_step_kernel<N, T, true, 2> : ss_step_kernel<N, T, false, 2>)
                  : (vbc ? ss_step_kernel<N, T, true, 1> : ss_step_kernel<N, T, false, 1>);
  kern<<<dim3((unsigned)B, (unsigned)runs), kStepThreads, 0, s>>>(
      static_cast<const T*>(x), static_cast<const T*>(delta), A, static_cast<const T*>(Bm), static_cast<const T*>(Cm), Dv,
      static_cast<const T*>(z), h, static_cast<T*>(y), B, D);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <int K, typename T>
int conv_step_launch(const void* x, float* state, const float* w, const float* bias, void* out, int B, int D, int silu,
                     cudaStream_t s) {
  const long long runs2 = (D + 2 * kStepThreads - 1) / (2 * kStepThreads);
  const bool two = (long long)B * runs2 >= 2ll * device_sm_count();
  const dim3 grid((unsigned)B, (unsigned)(two ? runs2 : (D + kStepThreads - 1) / kStepThreads));
  const T* xx = static_cast<const T*>(x);
  T* o = static_cast<T*>(out);
  constexpr bool kVec = K == 4;
  const bool vec = kVec && ssh::aligned16(state);
  using Kern = void (*)(const T*, float*, const float*, const float*, T*, int, int);
  Kern kern;
  if (vec) kern = silu ? (two ? conv_step_kernel<K, T, true, kVec, 2> : conv_step_kernel<K, T, true, kVec, 1>)
                       : (two ? conv_step_kernel<K, T, false, kVec, 2> : conv_step_kernel<K, T, false, kVec, 1>);
  else kern = silu ? (two ? conv_step_kernel<K, T, true, false, 2> : conv_step_kernel<K, T, true, false, 1>)
                   : (two ? conv_step_kernel<K, T, false, false, 2> : conv_step_kernel<K, T, false, false, 1>);
  kern<<<grid, kStepThreads, 0, s>>>(xx, state, w, bias, o, B, D);
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
  if ((long long)D * (N / 4) > 65535ll * kStepThreads) return SS_ERR_DIM;  // grid.y <= 65535
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
  if ((long long)D > 65535ll * kStepThreads) return SS_ERR_DIM;  // grid.y <= 65535
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) return conv_step_dispatch<float>(x, conv_state, w, bias, out, B, D, d_conv, silu, s);
  return conv_step_dispatch<__nv_bfloat16>(x, conv_state, w, bias, out, B, D, d_conv, silu, s);
}
