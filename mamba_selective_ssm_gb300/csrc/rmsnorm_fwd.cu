// RMSNorm forward (rmsnorm_fwd) for sm_103a.
//
//   rms_r = sqrt(mean_i x[r,i]^2 + eps),   y[r,i] = x[r,i] * scale_i / rms_r
//
// Same row walk as the backward: a CTA of T = ceil(dim / (8 VPT)) threads
// handles rows r = blockIdx.x, +gridDim.x, ...; each thread owns VPT groups of
// 8 consecutive columns, prefetches the next row while the current row's sum
// of squares is reduced (warp shuffles, then one shared-memory exchange whose
// buffer alternates with the row parity), and writes y in the input dtype
// (bf16 rounded to nearest even) and rms_r in fp32.
#include "common.cuh"

namespace {

using namespace ssk;

constexpr int kRmsFMaxThreads = 1024;
constexpr int kRmsFMaxDim = 32768;

template <typename T, int VPT>
__global__ void __launch_bounds__(kRmsFMaxThreads) rms_fwd_kernel(const T* __restrict__ x, const float* __restrict__ scale,
                                                                  float eps, T* __restrict__ y, float* __restrict__ rms,
                                                                  int rows, int dim) {
  __shared__ float red[2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
  float sc[VPT][8], xv[VPT][8], xvn[VPT][8];
  bool col_ok[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * blockDim.x + tid) * 8;
    col_ok[v] = c < dim;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sc[v][e] = col_ok[v] ? scale[c + e] : 0.f;
      xv[v][e] = 0.f;
    }
  }
  auto load_row = [&](int r, float (*xx)[8]) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * blockDim.x + tid) * 8;
      if (col_ok[v] && r < rows) {
        ActT<T>::ld8(x + (size_t)r * dim + c, xx[v]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) xx[v][e] = 0.f;
      }
    }
  };
  const float inv_dim = 1.0f / (float)dim;
  int parity = 0;
  int r = blockIdx.x;
  if (r < rows) load_row(r, xv);
  for (; r < rows; r += gridDim.x) {
    float part = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
      for (int e = 0; e < 8; ++e) part = fmaf(xv[v][e], xv[v][e], part);
    load_row(r + gridDim.x, xvn);  // next row in flight during the reduction
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[parity][warp] = part;
    __syncthreads();
    float ss = 0.f;
    for (int i = 0; i < nw; ++i) ss += red[parity][i];
    parity ^= 1;
    const float rr = sqrtf(fmaf(ss, inv_dim, eps));
    const float inv = 1.0f / rr;
    if (tid == 0 && rms != nullptr) rms[r] = rr;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * blockDim.x + tid) * 8;
      if (col_ok[v]) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (xv[v][e] * sc[v][e]) * inv;
        ActT<T>::st8(y + (size_t)r * dim + c, o);
      }
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[v][e] = xvn[v][e];
  }
}

int rms_fwd_validate(int rows, int dim, int dtype) {
  if (rows <= 0 || dim <= 0) return SS_ERR_DIM;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (dim % 8 != 0) return SS_ERR_ALIGN;
  if (dim > kRmsFMaxDim) return SS_ERR_DIM;
  return SS_OK;
}

template <typename T>
int rms_fwd_launch(const void* x, const float* scale, float eps, void* y, float* rms, int rows, int dim, cudaStream_t s) {
  const int groups = dim / 8;
  const int vpt = groups <= 1024 ? 1 : groups <= 2048 ? 2 : 4;
  const int threads = ((groups + vpt - 1) / vpt + 31) / 32 * 32;
  const int grid = rows < 1216 ? rows : 1216;  // 8 CTAs per SM; each walks rows / 1216 rows
  const T* xx = static_cast<const T*>(x);
  T* yy = static_cast<T*>(y);
  if (vpt == 1) rms_fwd_kernel<T, 1><<<grid, threads, 0, s>>>(xx, scale, eps, yy, rms, rows, dim);
  else if (vpt == 2) rms_fwd_kernel<T, 2><<<grid, threads, 0, s>>>(xx, scale, eps, yy, rms, rows, dim);
  else rms_fwd_kernel<T, 4><<<grid, threads, 0, s>>>(xx, scale, eps, yy, rms, rows, dim);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

extern "C" int rmsnorm_fwd(const void* x, const float* scale, float eps, void* y, float* rms, int rows, int dim, int dtype,
                           void* stream) {
  if (!x || !scale || !y) return SS_ERR_NULL;
  const int v = rms_fwd_validate(rows, dim, dtype);
  if (v != SS_OK) return v;
  if (!(eps >= 0.0f)) return SS_ERR_DIM;  // also rejects NaN
  if (!ssh::aligned16(x) || !ssh::aligned16(scale) || !ssh::aligned16(y) || (rms && !ssh::aligned16(rms)))
    return SS_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) return rms_fwd_launch<float>(x, scale, eps, y, rms, rows, dim, s);
  return rms_fwd_launch<__nv_bfloat16>(x, scale, eps, y, rms, rows, dim, s);
}
