// RMSNorm forward (rmsnorm_fwd) for sm_103a.
//
//   rms_r = sqrt(mean_i x[r,i]^2 + eps),   y[r,i] = x[r,i] * scale_i / rms_r
//
// Same row walk as the backward: a CTA of T = ceil(dim / (8 VPT)) threads
// handles rows r = blockIdx.x, +gridDim.x, ...; each thread owns VPT groups of
// 8 consecutive columns; the row's sum of squares is reduced with warp
// shuffles and one shared-memory exchange whose buffer alternates with the
// row parity; y is written in the input dtype (bf16 rounded to nearest even)
// and rms_r in fp32.  Rows of 257 .. 2048 columns (1024 for fp32) go one warp
// per row with the row in registers (rms_fwd_reg_kernel); fp32 rows of 1025 ..
// 2048 columns one warp per row through a per-warp ring of bulk-copied stages
// (rms_fwd_warp_kernel); rows of at most 8192 columns arrive through a per-CTA ring of
// shared-memory stages filled by untiled bulk copies (rms_fwd_tma_kernel);
// wider rows use the register-prefetch form (one row ahead).
#include "common.cuh"

namespace {

using namespace ssk;

__device__ unsigned g_rmsf_err;

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

template <typename T>
__global__ void __launch_bounds__(kRmsFMaxThreads) rms_fwd_tma_kernel(const T* __restrict__ x,
                                                                      const float* __restrict__ scale, float eps,
                                                                      T* __restrict__ y, float* __restrict__ rms, int rows,
                                                                      int dim, int nst) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ float red[2][32];
  const uint32_t row_bytes = (uint32_t)dim * sizeof(T);
  T* buf = reinterpret_cast<T*>(sm);  // [nst][dim]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)nst * row_bytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
  const int nk = (rows - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  auto issue = [&](int k) {
    fence_proxy_async_smem();  // the slot's earlier readers passed a barrier before this call
    const size_t r = (size_t)blockIdx.x + (size_t)k * gridDim.x;
    const int st = k % nst;
    mbar_arrive_expect_tx(&full[st], row_bytes);
    bulk_load(buf + (size_t)st * dim, x + r * dim, row_bytes, &full[st]);
  };
  if (tid == 0) {
    for (int st = 0; st < nst; ++st) mbar_init(&full[st], 1);
    fence_barrier_init();
    for (int k = 0; k < nst && k < nk; ++k) issue(k);
  }
  const int c = tid * 8;
  const bool col_ok = c < dim;
  float sc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sc[e] = col_ok ? scale[c + e] : 0.f;
  __syncthreads();
  const float inv_dim = 1.0f / (float)dim;
  int parity = 0;
  for (int k = 0; k < nk; ++k) {
    const int r = (int)blockIdx.x + k * (int)gridDim.x;
    const int st = k % nst;
    bool ok = true;
    if (tid == 0) ok = mbar_wait_bounded(&full[st], (k / nst) & 1, kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicOr(&g_rmsf_err, kErrTmaTimeout);
        for (int k2 = k; k2 < k + nst && k2 < nk; ++k2) mbar_wait_bounded(&full[k2 % nst], (k2 / nst) & 1, 100000000ull);
      }
      return;
    }
    float xv[8];
    if (col_ok) {
      ActT<T>::ld8(buf + (size_t)st * dim + c, xv);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[e] = 0.f;
    }
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) part = fmaf(xv[e], xv[e], part);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[parity][warp] = part;
    __syncthreads();  // every thread has its row values: the stage can be refilled
    if (tid == 0 && k + nst < nk) issue(k + nst);
    float ss = 0.f;
    for (int i = 0; i < nw; ++i) ss += red[parity][i];
    parity ^= 1;
    const float rr = sqrtf(fmaf(ss, inv_dim, eps));
    const float inv = 1.0f / rr;
    if (tid == 0 && rms != nullptr) rms[r] = rr;
    if (col_ok) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (xv[e] * sc[e]) * inv;
      ActT<T>::st8(y + (size_t)r * dim + c, o);
    }
  }
}

// Rows of 257 .. 2048 columns: one warp per row, no block barrier.  Lane l
// owns the 8-column groups l, l + 32, ... (VPW of them) and reads the row
// twice from its warp's ring of shared-memory stages (bulk copies, one
// mbarrier per stage): once for the sum of squares, reduced with shuffles, and
// once for y.
constexpr int kRmsFWarps = 4;

template <typename T, int VPW>
__global__ void __launch_bounds__(32 * kRmsFWarps) rms_fwd_warp_kernel(const T* __restrict__ x,
                                                                       const float* __restrict__ scale, float eps,
                                                                       T* __restrict__ y, float* __restrict__ rms, int rows,
                                                                       int dim, int nst) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t row_bytes = (uint32_t)dim * sizeof(T);
  T* buf = reinterpret_cast<T*>(sm) + (size_t)warp * nst * dim;  // this warp's [nst][dim]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)kRmsFWarps * nst * row_bytes) + warp * nst;
  const long long nwarps = (long long)gridDim.x * kRmsFWarps;
  const long long gw = (long long)blockIdx.x * kRmsFWarps + warp;
  const int nk = gw < rows ? (int)((rows - gw + nwarps - 1) / nwarps) : 0;
  auto issue = [&](int k) {  // lane 0; the stage's readers passed a warp sync
    fence_proxy_async_smem();
    const size_t r = (size_t)(gw + (long long)k * nwarps);
    const int st = k % nst;
    mbar_arrive_expect_tx(&full[st], row_bytes);
    bulk_load(buf + (size_t)st * dim, x + r * dim, row_bytes, &full[st]);
  };
  if (lane == 0) {
    for (int st = 0; st < nst; ++st) mbar_init(&full[st], 1);
    fence_barrier_init();
    for (int k = 0; k < nst && k < nk; ++k) issue(k);
  }
  float sc[VPW][8];
#pragma unroll
  for (int v = 0; v < VPW; ++v) {
    const int c = (v * 32 + lane) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) sc[v][e] = c < dim ? scale[c + e] : 0.f;
  }
  __syncwarp();
  const float inv_dim = 1.0f / (float)dim;
  for (int k = 0; k < nk; ++k) {
    const long long r = gw + (long long)k * nwarps;
    const int st = k % nst;
    const bool ok = mbar_wait_bounded(&full[st], (k / nst) & 1, kWaitLimitNs);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) {
        atomicOr(&g_rmsf_err, kErrTmaTimeout);
        for (int k2 = k; k2 < k + nst && k2 < nk; ++k2) mbar_wait_bounded(&full[k2 % nst], (k2 / nst) & 1, 100000000ull);
      }
      return;
    }
    const T* x_s = buf + (size_t)st * dim;
    float part = 0.f;
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      const int c = (v * 32 + lane) * 8;
      if (c < dim) {
        float xv[8];
        ActT<T>::ld8(x_s + c, xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(xv[e], xv[e], part);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    const float rr = sqrtf(fmaf(part, inv_dim, eps));
    const float inv = 1.0f / rr;
    if (lane == 0 && rms != nullptr) rms[r] = rr;
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      const int c = (v * 32 + lane) * 8;
      if (c < dim) {
        float xv[8], o[8];
        ActT<T>::ld8(x_s + c, xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (xv[e] * sc[v][e]) * inv;
        ActT<T>::st8(y + (size_t)r * dim + c, o);
      }
    }
    __syncwarp();
    if (lane == 0 && k + nst < nk) issue(k + nst);
  }
}

template <typename T>
int rms_fwd_warp_launch(const void* x, const float* scale, float eps, void* y, float* rms, int rows, int dim,
                        cudaStream_t s) {
  const size_t rb = (size_t)dim * sizeof(T);
  int nst = (int)((64u * 1024u) / (kRmsFWarps * rb));
  if (nst > 4) nst = 4;
  if (nst < 2) nst = 2;
  const size_t smem = (size_t)kRmsFWarps * nst * rb + (size_t)kRmsFWarps * nst * sizeof(uint64_t);
  auto run = [&](auto kern) -> int {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    const int per_sm = resident_ctas(kern, 32 * kRmsFWarps, smem);
    if (per_sm < 1) return SS_ERR_CUDA;
    long long grid = (long long)per_sm * device_sm_count();
    const long long need = ((long long)rows + kRmsFWarps - 1) / kRmsFWarps;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    kern<<<(int)grid, 32 * kRmsFWarps, smem, s>>>(static_cast<const T*>(x), scale, eps, static_cast<T*>(y), rms, rows, dim,
                                                   nst);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  };
  const int vpw = (dim + 255) / 256;
  if (vpw <= 2) return run(rms_fwd_warp_kernel<T, 2>);
  if (vpw <= 4) return run(rms_fwd_warp_kernel<T, 4>);
  return run(rms_fwd_warp_kernel<T, 8>);
}

// Rows of 257 .. 2048 columns (bf16; 1024 for fp32), held in registers: one
// warp per row, lane l owning the 8-column groups l, l + 32, ... (VPW of
// them), all of a row's loads issued together.  The warps of a CTA walk rows
// w, w + W, ... and the CTA stages scale in shared memory once (a lane reads
// its 8 values as two 16-byte words that neighbouring lanes' words follow, so
// the reads are conflict-free); reading scale from global memory per row
// measured 3 us slower on the 1.4B layer's [8192, 2048] rows, and a second row
// buffer per warp (loads of the next row in flight) no faster.
constexpr int kRmsRegWarps = 8;

template <typename T, int VPW>
__global__ void __launch_bounds__(32 * kRmsRegWarps, VPW >= 8 ? 3 : 4) rms_fwd_reg_kernel(const T* __restrict__ x,
                                                                        const float* __restrict__ scale, float eps,
                                                                        T* __restrict__ y, float* __restrict__ rms,
                                                                        int rows, int dim) {
  using R = Raw8<T>;
  extern __shared__ float4 ssc[];  // [2][dim / 8]: group g's first four values at g, last four at dim/8 + g
  const int ng = dim / 8;
  for (int i = threadIdx.x; i < ng; i += blockDim.x) {
    ssc[i] = __ldg(reinterpret_cast<const float4*>(scale) + 2 * i);
    ssc[ng + i] = __ldg(reinterpret_cast<const float4*>(scale) + 2 * i + 1);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * kRmsRegWarps;
  const float inv_dim = 1.0f / (float)dim;
  for (long long r = (long long)blockIdx.x * kRmsRegWarps + (threadIdx.x >> 5); r < rows; r += nw) {
    typename R::V b[VPW];
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      const int c = (v * 32 + lane) * 8;
      b[v] = c < dim ? R::ld(x + (size_t)r * dim + c) : R::zero();
    }
    float part = 0.f;
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      float xv[8];
      R::wide(b[v], xv);
#pragma unroll
      for (int e = 0; e < 8; ++e) part = fmaf(xv[e], xv[e], part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    const float rr = sqrtf(fmaf(part, inv_dim, eps));
    const float inv = 1.0f / rr;
    if (lane == 0 && rms != nullptr) rms[r] = rr;
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      const int c = (v * 32 + lane) * 8;
      if (c < dim) {
        float xv[8], o[8];
        R::wide(b[v], xv);
        const float4 s0 = ssc[v * 32 + lane], s1 = ssc[ng + v * 32 + lane];
        const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (xv[e] * sc[e]) * inv;
        ActT<T>::st8(y + (size_t)r * dim + c, o);
      }
    }
  }
}

template <typename T, int VPW>
int rms_fwd_reg_launch(const void* x, const float* scale, float eps, void* y, float* rms, int rows, int dim,
                       cudaStream_t s) {
  auto kern = rms_fwd_reg_kernel<T, VPW>;
  const size_t smem = (size_t)dim * sizeof(float);
  const int per_sm = resident_ctas(kern, 32 * kRmsRegWarps, smem);
  if (per_sm < 1) return SS_ERR_CUDA;
  long long grid = (long long)per_sm * device_sm_count();
  const long long need = ((long long)rows + kRmsRegWarps - 1) / kRmsRegWarps;
  if (grid > need) grid = need;
  kern<<<(int)grid, 32 * kRmsRegWarps, smem, s>>>(static_cast<const T*>(x), scale, eps, static_cast<T*>(y), rms, rows,
                                                  dim);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// Rows of at most 256 columns: G lanes per row (one 8-column group each), 32/G
// rows per warp, the sum of squares reduced by shuffles inside each G-lane
// segment, no block barrier per row.
template <typename T, int G>
__global__ void __launch_bounds__(256) rms_fwd_small_kernel(const T* __restrict__ x, const float* __restrict__ scale,
                                                            float eps, T* __restrict__ y, float* __restrict__ rms, int rows,
                                                            int dim) {
  constexpr int R = 32 / G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int slot = lane / G, c = (lane % G) * 8;
  const bool col_ok = c < dim;
  float sc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sc[e] = col_ok ? scale[c + e] : 0.f;
  const float inv_dim = 1.0f / (float)dim;
  const long long step = (long long)gridDim.x * nw * R;
  for (long long rb = ((long long)blockIdx.x * nw + warp) * R; rb < rows; rb += step) {
    const long long r = rb + slot;
    const bool row_ok = r < rows;
    float xv[8];
    if (row_ok && col_ok) {
      ActT<T>::ld8(x + r * dim + c, xv);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) xv[e] = 0.f;
    }
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) part = fmaf(xv[e], xv[e], part);
#pragma unroll
    for (int o = 1; o < G; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (row_ok) {
      const float rr = sqrtf(fmaf(part, inv_dim, eps));
      const float inv = 1.0f / rr;
      if (c == 0 && rms != nullptr) rms[r] = rr;
      if (col_ok) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (xv[e] * sc[e]) * inv;
        ActT<T>::st8(y + r * dim + c, o);
      }
    }
  }
}

template <typename T, int G>
int rms_fwd_small_launch(const void* x, const float* scale, float eps, void* y, float* rms, int rows, int dim,
                         cudaStream_t s) {
  constexpr int R = 32 / G;
  long long grid = ((long long)rows + 8 * R - 1) / (8 * R);
  const long long cap = 16ll * device_sm_count();
  if (cap > 0 && grid > cap) grid = cap;
  rms_fwd_small_kernel<T, G><<<(int)grid, 256, 0, s>>>(static_cast<const T*>(x), scale, eps, static_cast<T*>(y), rms, rows,
                                                       dim);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
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
  if (groups <= 32) {  // short rows: several rows per warp
    if (groups <= 1) return rms_fwd_small_launch<T, 1>(x, scale, eps, y, rms, rows, dim, s);
    if (groups <= 2) return rms_fwd_small_launch<T, 2>(x, scale, eps, y, rms, rows, dim, s);
    if (groups <= 4) return rms_fwd_small_launch<T, 4>(x, scale, eps, y, rms, rows, dim, s);
    if (groups <= 8) return rms_fwd_small_launch<T, 8>(x, scale, eps, y, rms, rows, dim, s);
    if (groups <= 16) return rms_fwd_small_launch<T, 16>(x, scale, eps, y, rms, rows, dim, s);
    return rms_fwd_small_launch<T, 32>(x, scale, eps, y, rms, rows, dim, s);
  }
  constexpr int kRegMaxGroups = sizeof(T) == 2 ? 256 : 128;  // rows held in registers: 64 columns a lane (bf16)
  if (groups <= kRegMaxGroups) {
    if (groups <= 64) return rms_fwd_reg_launch<T, 2>(x, scale, eps, y, rms, rows, dim, s);
    if (groups <= 128) return rms_fwd_reg_launch<T, 4>(x, scale, eps, y, rms, rows, dim, s);
    if constexpr (sizeof(T) == 2) return rms_fwd_reg_launch<T, 8>(x, scale, eps, y, rms, rows, dim, s);
  }
  if (groups <= 256) return rms_fwd_warp_launch<T>(x, scale, eps, y, rms, rows, dim, s);  // one warp per row
  if (groups <= 1024) {  // one 8-column group per thread: the bulk-copy ring, up to 16 rows or ~100 KB per CTA
    int nst = (int)((32u * 1024u) / ((size_t)dim * sizeof(T)));
    if (nst > 16) nst = 16;
    const int threads = (groups + 31) / 32 * 32;
    const size_t smem = (size_t)nst * dim * sizeof(T) + (size_t)nst * sizeof(uint64_t);
    auto kern = rms_fwd_tma_kernel<T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
  // prefer the largest shared-memory carveout, so that residency (and the occupancy
  // query the segment and grid choices rely on) is limited by the CTAs' own needs
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    int per_sm = 0;
    per_sm = resident_ctas(kern, threads, smem);
    if (per_sm < 1) return SS_ERR_CUDA;
    int grid = per_sm * device_sm_count();
    if (grid > rows) grid = rows;
    if (grid < 1) grid = 1;
    kern<<<grid, threads, smem, s>>>(static_cast<const T*>(x), scale, eps, static_cast<T*>(y), rms, rows, dim, nst);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  }
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

namespace ssh {
int read_clear_rmsf_err(cudaStream_t s, unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_rmsf_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SS_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_rmsf_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return SS_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
}  // namespace ssh

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
