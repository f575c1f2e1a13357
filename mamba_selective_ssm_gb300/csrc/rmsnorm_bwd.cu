// RMSNorm backward (rmsnorm_bwd) for sm_103a.
//
//   inv = 1/rms_r;  dot_r = inv^2 sum_i dy*scale*x
//   dx[r,i] = inv (scale_i dy[r,i] - x[r,i] dot_r / dim);   dscale_i += sum_r dy x inv
//
// A CTA of T = ceil(dim / (8 VPT)) threads walks rows r = blockIdx.x, +gridDim.x, ...
// Each thread owns VPT groups of 8 consecutive columns, keeps scale and its
// dscale partial in registers, and the row's dot product is reduced with warp
// shuffles and one shared-memory exchange whose buffer alternates with the
// row parity.  Rows reach the CTA through a ring of `nst` shared-memory stages
// filled by untiled bulk copies (cp.async.bulk, one mbarrier per stage), so
// up to nst rows of dy and x per CTA are in flight without holding registers
// (rms_bwd_tma_kernel, rows of 2049 .. 8192 columns); rows of 257 .. 2048
// columns are split over a CTA's threads, which walk the rows with the next
// row's loads in flight and one barrier per row (rms_bwd_cols_kernel);
// the register-prefetch form (rms_bwd_kernel, one row ahead) serves the
// fixed-grid no-alloc entry point and rows too wide for two stages.  Per-CTA
// dscale partials are added in fixed order by colsum_kernel.
#include <mutex>

#include "common.cuh"

// Scratch of rmsnorm_bwd_noalloc: one dscale partial row per CTA of its fixed
// 128-CTA grid, for dim up to 8192 (4 MiB).  Every GPU that loads the library
// keeps this array until the process exits.
constexpr int kNoAllocGrid = 128;
constexpr int kNoAllocMaxDim = 8192;
static __device__ __align__(256) float g_rms_noalloc_scratch[kNoAllocGrid * kNoAllocMaxDim];

namespace {

using namespace ssk;

__device__ unsigned g_rms_err;

constexpr int kRmsMaxThreads = 1024;
constexpr int kRmsMaxDim = 32768;

template <typename T, int VPT>
__global__ void __launch_bounds__(kRmsMaxThreads) rms_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ x,
                                                                 const float* __restrict__ scale,
                                                                 const float* __restrict__ rms, float* __restrict__ dx,
                                                                 float* __restrict__ ws, int rows, int dim) {
  pdl_trigger();  // the column sum of the partials may launch now; it waits for this grid's end
  __shared__ float red[2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
  float sc[VPT][8], acc[VPT][8], gy[VPT][8], xv[VPT][8], gyn[VPT][8], xvn[VPT][8];
  bool col_ok[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * blockDim.x + tid) * 8;
    col_ok[v] = c < dim;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sc[v][e] = col_ok[v] ? scale[c + e] : 0.f;
      acc[v][e] = 0.f;
      gy[v][e] = xv[v][e] = 0.f;
    }
  }
  auto load_row = [&](int r, float (*g)[8], float (*xx)[8]) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * blockDim.x + tid) * 8;
      if (col_ok[v] && r < rows) {
        ActT<T>::ld8(dy + (size_t)r * dim + c, g[v]);
        ActT<T>::ld8(x + (size_t)r * dim + c, xx[v]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) g[v][e] = xx[v][e] = 0.f;
      }
    }
  };
  const float inv_dim = 1.0f / (float)dim;
  int parity = 0;
  int r = blockIdx.x;
  if (r < rows) load_row(r, gy, xv);
  for (; r < rows; r += gridDim.x) {
    const float inv = 1.0f / rms[r];
    float part = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
      for (int e = 0; e < 8; ++e) part = fmaf(gy[v][e] * sc[v][e], xv[v][e], part);
    load_row(r + gridDim.x, gyn, xvn);  // next row in flight during the reduction
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[parity][warp] = part;
    __syncthreads();
    float dot = 0.f;
    for (int i = 0; i < nw; ++i) dot += red[parity][i];
    parity ^= 1;
    const float k = dot * inv * inv * inv_dim;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * blockDim.x + tid) * 8;
      if (col_ok[v]) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          o[e] = inv * (sc[v][e] * gy[v][e]) - inv * (xv[v][e] * k);
          acc[v][e] = fmaf(gy[v][e] * xv[v][e], inv, acc[v][e]);
        }
        ActT<float>::st8(dx + (size_t)r * dim + c, o);
      }
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        gy[v][e] = gyn[v][e];
        xv[v][e] = xvn[v][e];
      }
  }
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * blockDim.x + tid) * 8;
    if (col_ok[v]) ActT<float>::st8(ws + (size_t)blockIdx.x * dim + c, acc[v]);
  }
}

template <typename T, int VPT>
__global__ void __launch_bounds__(kRmsMaxThreads) rms_bwd_tma_kernel(const T* __restrict__ dy, const T* __restrict__ x,
                                                                     const float* __restrict__ scale,
                                                                     const float* __restrict__ rms, float* __restrict__ dx,
                                                                     float* __restrict__ ws, int rows, int dim, int nst) {
  pdl_trigger();  // the column sum of the partials may launch now; it waits for this grid's end
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ float red[2][32];
  const uint32_t row_bytes = (uint32_t)dim * sizeof(T);
  T* buf = reinterpret_cast<T*>(sm);  // [nst][dy | x][dim]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)nst * 2 * row_bytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (blockDim.x + 31) >> 5;
  const int nk = (rows - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;  // rows of this CTA
  auto issue = [&](int k) {
    fence_proxy_async_smem();  // the slot's earlier readers passed a barrier before this call
    const size_t r = (size_t)blockIdx.x + (size_t)k * gridDim.x;
    const int st = k % nst;
    mbar_arrive_expect_tx(&full[st], 2 * row_bytes);
    bulk_load(buf + (size_t)(2 * st) * dim, dy + r * dim, row_bytes, &full[st]);
    bulk_load(buf + (size_t)(2 * st + 1) * dim, x + r * dim, row_bytes, &full[st]);
  };
  if (tid == 0) {
    for (int st = 0; st < nst; ++st) mbar_init(&full[st], 1);
    fence_barrier_init();
    for (int k = 0; k < nst && k < nk; ++k) issue(k);
  }
  float sc[VPT][8], acc[VPT][8];
  bool col_ok[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * blockDim.x + tid) * 8;
    col_ok[v] = c < dim;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sc[v][e] = col_ok[v] ? scale[c + e] : 0.f;
      acc[v][e] = 0.f;
    }
  }
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
        atomicOr(&g_rms_err, kErrTmaTimeout);
        for (int k2 = k; k2 < k + nst && k2 < nk; ++k2) mbar_wait_bounded(&full[k2 % nst], (k2 / nst) & 1, 100000000ull);
      }
      // the column sum still adds this CTA's partial row: make it zero
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int c = (v * blockDim.x + tid) * 8;
        const float z8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (col_ok[v]) ActT<float>::st8(ws + (size_t)blockIdx.x * dim + c, z8);
      }
      return;
    }
    float gy[VPT][8], xv[VPT][8];
    float part = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * blockDim.x + tid) * 8;
      if (col_ok[v]) {
        ActT<T>::ld8(buf + (size_t)(2 * st) * dim + c, gy[v]);
        ActT<T>::ld8(buf + (size_t)(2 * st + 1) * dim + c, xv[v]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gy[v][e] = xv[v][e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) part = fmaf(gy[v][e] * sc[v][e], xv[v][e], part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[parity][warp] = part;
    __syncthreads();  // every thread has its row values: the stage can be refilled
    if (tid == 0 && k + nst < nk) issue(k + nst);
    float dot = 0.f;
    for (int i = 0; i < nw; ++i) dot += red[parity][i];
    parity ^= 1;
    const float inv = 1.0f / rms[r];
    const float kk = dot * inv * inv * inv_dim;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = (v * blockDim.x + tid) * 8;
      if (col_ok[v]) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          o[e] = inv * (sc[v][e] * gy[v][e]) - inv * (xv[v][e] * kk);
          acc[v][e] = fmaf(gy[v][e] * xv[v][e], inv, acc[v][e]);
        }
        ActT<float>::st8(dx + (size_t)r * dim + c, o);
      }
    }
  }
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = (v * blockDim.x + tid) * 8;
    if (col_ok[v]) ActT<float>::st8(ws + (size_t)blockIdx.x * dim + c, acc[v]);
  }
}

// Rows of at most 256 columns: G lanes per row (one 8-column group each), 32/G
// rows per warp, the dot product reduced by shuffles inside each G-lane
// segment, no block barrier per row.  The dscale partials of the CTA's
// (warp, row slot) pairs are added in fixed order at the end.
template <typename T, int G>
__global__ void __launch_bounds__(256) rms_bwd_small_kernel(const T* __restrict__ dy, const T* __restrict__ x,
                                                            const float* __restrict__ scale, const float* __restrict__ rms,
                                                            float* __restrict__ dx, float* __restrict__ ws, int rows,
                                                            int dim) {
  pdl_trigger();  // the column sum of the partials may launch now; it waits for this grid's end
  constexpr int R = 32 / G;
  __shared__ float red[8 * R][G * 8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int slot = lane / G, c = (lane % G) * 8;
  const bool col_ok = c < dim;
  float sc[8], acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sc[e] = col_ok ? scale[c + e] : 0.f;
    acc[e] = 0.f;
  }
  const float inv_dim = 1.0f / (float)dim;
  const long long step = (long long)gridDim.x * nw * R;
  for (long long rb = ((long long)blockIdx.x * nw + warp) * R; rb < rows; rb += step) {
    const long long r = rb + slot;
    const bool row_ok = r < rows;
    float gy[8], xv[8];
    if (row_ok && col_ok) {
      ActT<T>::ld8(dy + r * dim + c, gy);
      ActT<T>::ld8(x + r * dim + c, xv);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) gy[e] = xv[e] = 0.f;
    }
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) part = fmaf(gy[e] * sc[e], xv[e], part);
#pragma unroll
    for (int o = 1; o < G; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (row_ok && col_ok) {
      const float inv = 1.0f / rms[r];
      const float kk = part * inv * inv * inv_dim;
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        o[e] = inv * (sc[e] * gy[e]) - inv * (xv[e] * kk);
        acc[e] = fmaf(gy[e] * xv[e], inv, acc[e]);
      }
      ActT<float>::st8(dx + r * dim + c, o);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[warp * R + slot][(lane % G) * 8 + e] = acc[e];
  __syncthreads();
  for (int col = tid; col < dim; col += blockDim.x) {
    float a = 0.f;
    for (int i = 0; i < nw * R; ++i) a += red[i][col];
    ws[(size_t)blockIdx.x * dim + col] = a;
  }
}

struct AddTo {
  float* out;
  __device__ void put(long long i, float v) const { out[i] += v; }
};

struct RmsPlan {
  int vpt, threads, grid;
  int cgrid;  // partial rows the column-split kernel may use (rows of 257 .. 2048 columns)
  size_t bytes;
};

inline RmsPlan rms_plan(int rows, int dim) {
  RmsPlan p;
  const int groups = dim / 8;
  p.vpt = groups <= 1024 ? 1 : groups <= 2048 ? 2 : 4;
  p.threads = ((groups + p.vpt - 1) / p.vpt + 31) / 32 * 32;
  p.grid = rows < 608 ? rows : 608;  // 4 waves of 152 SMs; each CTA walks rows/608 rows
  // narrow rows make small column-split CTAs (dim/64 warps): allow enough of them for ~32 warps per SM
  const int cw = (dim / 8 + 31) / 32;
  const int cap = dim > 256 && dim <= 2048 ? 152 * (32 / cw > 4 ? 32 / cw : 4) : 608;
  p.cgrid = rows < cap ? rows : cap;
  p.bytes = (size_t)(p.cgrid > p.grid ? p.cgrid : p.grid) * dim * sizeof(float);
  return p;
}

int rms_validate(int rows, int dim, int dtype) {
  if (rows <= 0 || dim <= 0) return SS_ERR_DIM;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (dim % 8 != 0) return SS_ERR_ALIGN;
  if (dim > kRmsMaxDim) return SS_ERR_DIM;
  return SS_OK;
}

template <typename T, int G>
int rms_small_launch(const void* dy, const void* x, const float* scale, const float* rms, float* dx, float* dscale,
                     int rows, int dim, float* ws, const RmsPlan& pl, cudaStream_t s) {
  constexpr int R = 32 / G;
  long long grid = ((long long)rows + 8 * R - 1) / (8 * R);
  if (grid > pl.grid) grid = pl.grid;  // the workspace holds pl.grid partial rows
  rms_bwd_small_kernel<T, G><<<(int)grid, 256, 0, s>>>(static_cast<const T*>(dy), static_cast<const T*>(x), scale, rms, dx,
                                                       ws, rows, dim);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  return colsum(ws, dim, (int)grid, AddTo{dscale}, s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename T>
int rms_small_dispatch(const void* dy, const void* x, const float* scale, const float* rms, float* dx, float* dscale,
                       int rows, int dim, float* ws, const RmsPlan& pl, cudaStream_t s) {
  const int groups = dim / 8;
  if (groups <= 1) return rms_small_launch<T, 1>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  if (groups <= 2) return rms_small_launch<T, 2>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  if (groups <= 4) return rms_small_launch<T, 4>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  if (groups <= 8) return rms_small_launch<T, 8>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  if (groups <= 16) return rms_small_launch<T, 16>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  return rms_small_launch<T, 32>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
}

// Shared-memory stages of the bulk-copy form (rows of at most 8192 columns, one
// 8-column group per thread): ~32 KB per CTA, between 2 and 16 rows of dy and
// x; 0 when two stages do not fit.
inline int rms_tma_stages(int dim, int esize) {
  const size_t pair = (size_t)2 * dim * esize;
  int nst = (int)((32u * 1024u) / pair);
  if (nst > 16) nst = 16;
  return nst >= 2 ? nst : 0;
}

template <typename T>
int rms_tma_launch(const void* dy, const void* x, const float* scale, const float* rms, float* dx, float* dscale, int rows,
                   int dim, float* ws, const RmsPlan& pl, int nst, cudaStream_t s) {
  const size_t smem = (size_t)nst * 2 * dim * sizeof(T) + (size_t)nst * sizeof(uint64_t);
  const T* g = static_cast<const T*>(dy);
  const T* xx = static_cast<const T*>(x);
  auto run = [&](auto kern) -> int {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
  // prefer the largest shared-memory carveout, so that residency (and the occupancy
  // query the segment and grid choices rely on) is limited by the CTAs' own needs
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    int per_sm = 0;
    per_sm = resident_ctas(kern, pl.threads, smem);
    if (per_sm < 1) return SS_ERR_CUDA;
    int grid = per_sm * device_sm_count();
    if (grid > pl.grid) grid = pl.grid;  // the workspace holds pl.grid partial rows
    if (grid < 1) grid = 1;
    kern<<<grid, pl.threads, smem, s>>>(g, xx, scale, rms, dx, ws, rows, dim, nst);
    if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
    return colsum(ws, dim, grid, AddTo{dscale}, s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
  };
  return run(rms_bwd_tma_kernel<T, 1>);
}

// Rows of 257 .. 2048 columns, column-split: the CTA's threads share the
// columns (8 each, one 16- or 32-byte vector of a row) and walk groups of R
// rows.  A thread loads its columns of the R rows' dy and x at once; each row's
// dot product is summed over the thread's 8 columns, across the warp by
// shuffles and across the warps through shared memory in warp order (one
// barrier per R rows, parity-buffered); every thread keeps its columns' dscale
// partial in registers over all the rows it visits.
template <typename T, int R, bool PF>
__global__ void __launch_bounds__(256) rms_bwd_cols_kernel(const T* __restrict__ dy, const T* __restrict__ x,
                                                           const float* __restrict__ scale, const float* __restrict__ rms,
                                                           float* __restrict__ dx, float* __restrict__ ws, int rows,
                                                           int dim) {
  pdl_trigger();  // the column sum of the partials may launch now; it waits for this grid's end
  using Rw = Raw8<T>;
  using Buf = typename Rw::V[R];
  __shared__ float part[2][R][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = (int)blockDim.x >> 5;
  const int c = (int)threadIdx.x * 8;
  const bool cv = c < dim;
  float sc[8], acc[8];
  {
    const float4 s0 = cv ? __ldg(reinterpret_cast<const float4*>(scale + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 s1 = cv ? __ldg(reinterpret_cast<const float4*>(scale + c + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    sc[0] = s0.x; sc[1] = s0.y; sc[2] = s0.z; sc[3] = s0.w; sc[4] = s1.x; sc[5] = s1.y; sc[6] = s1.z; sc[7] = s1.w;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const float inv_dim = 1.0f / (float)dim;
  const long long step = (long long)gridDim.x * R;
  auto load = [&](Buf& gr, Buf& xr, long long r0) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long r = r0 + i;
      const bool ok = cv && r < rows;
      gr[i] = ok ? Rw::ld(dy + (size_t)r * dim + c) : Rw::zero();
      xr[i] = ok ? Rw::ld(x + (size_t)r * dim + c) : Rw::zero();
    }
  };
  int par = 0;
  auto finish = [&](const Buf& gr, const Buf& xr, long long r0) {
    float rinv[R];
#pragma unroll
    for (int i = 0; i < R; ++i) rinv[i] = r0 + i < rows ? 1.0f / __ldg(rms + r0 + i) : 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      float gv[8], xv[8];
      Rw::wide(gr[i], gv);
      Rw::wide(xr[i], xv);
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) a = fmaf(gv[e] * sc[e], xv[e], a);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (lane == 0) part[par][i][warp] = a;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long r = r0 + i;
      if (r < rows && cv) {
        float dot = part[par][i][0];
        for (int w = 1; w < nwarp; ++w) dot += part[par][i][w];
        const float inv = rinv[i];
        const float kk = dot * inv * inv * inv_dim;
        float gv[8], xv[8], o[8];
        Rw::wide(gr[i], gv);
        Rw::wide(xr[i], xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          o[e] = inv * (sc[e] * gv[e]) - inv * (xv[e] * kk);
          acc[e] = fmaf(gv[e] * xv[e], inv, acc[e]);
        }
        ActT<float>::st8(dx + (size_t)r * dim + c, o);
      }
    }
    par ^= 1;
  };
  Buf ga, xa, gb, xb;
  long long r0 = (long long)blockIdx.x * R;
  if constexpr (!PF) {
    for (; r0 < rows; r0 += step) {
      load(ga, xa, r0);
      finish(ga, xa, r0);
    }
  } else {
    if (r0 < rows) load(ga, xa, r0);
    for (; r0 < rows; r0 += 2 * step) {
      if (r0 + step < rows) load(gb, xb, r0 + step);
      finish(ga, xa, r0);
      if (r0 + step >= rows) break;
      if (r0 + 2 * step < rows) load(ga, xa, r0 + 2 * step);
      finish(gb, xb, r0 + step);
    }
  }
  if (cv) ActT<float>::st8(ws + (size_t)blockIdx.x * dim + c, acc);
}

template <typename T>
int rms_cols_launch(const void* dy, const void* x, const float* scale, const float* rms, float* dx, float* dscale,
                    int rows, int dim, float* ws, const RmsPlan& pl, cudaStream_t s) {
  constexpr int R = 1;  // one row per step, the next row's loads in flight (measured best of 1, 2, 4, 8 rows)
  auto kern = rms_bwd_cols_kernel<T, R, true>;
  const int threads = (dim / 8 + 31) / 32 * 32;
  const int per_sm = resident_ctas(kern, threads, 0);
  if (per_sm < 1) return SS_ERR_CUDA;
  long long grid = (long long)per_sm * device_sm_count();
  const long long need = ((long long)rows + R - 1) / R;
  if (grid > need) grid = need;
  if (grid > pl.cgrid) grid = pl.cgrid;  // the workspace holds pl.cgrid partial rows
  if (grid < 1) grid = 1;
  kern<<<(int)grid, threads, 0, s>>>(static_cast<const T*>(dy), static_cast<const T*>(x), scale, rms, dx, ws, rows, dim);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  return colsum(ws, dim, (int)grid, AddTo{dscale}, s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename T>
int rms_launch(const void* dy, const void* x, const float* scale, const float* rms, float* dx, float* dscale, int rows,
               int dim, float* ws, const RmsPlan& pl, cudaStream_t s) {
  const T* g = static_cast<const T*>(dy);
  const T* xx = static_cast<const T*>(x);
  if (pl.vpt == 1) rms_bwd_kernel<T, 1><<<pl.grid, pl.threads, 0, s>>>(g, xx, scale, rms, dx, ws, rows, dim);
  else if (pl.vpt == 2) rms_bwd_kernel<T, 2><<<pl.grid, pl.threads, 0, s>>>(g, xx, scale, rms, dx, ws, rows, dim);
  else rms_bwd_kernel<T, 4><<<pl.grid, pl.threads, 0, s>>>(g, xx, scale, rms, dx, ws, rows, dim);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  return colsum(ws, dim, pl.grid, AddTo{dscale}, s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

extern "C" size_t rmsnorm_bwd_workspace_size(int rows, int dim) {
  if (rms_validate(rows, dim, SS_F32) != SS_OK) return 0;
  return rms_plan(rows, dim).bytes;
}

extern "C" int rmsnorm_bwd(const void* dy, const void* x, const float* scale, const float* rms, float* dx, float* dscale,
                           int rows, int dim, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (!dy || !x || !scale || !rms || !dx || !dscale) return SS_ERR_NULL;
  const int v = rms_validate(rows, dim, dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {dy, x, scale, rms, dx, dscale};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  const RmsPlan pl = rms_plan(rows, dim);
  if (workspace == nullptr || ws_bytes < pl.bytes) return SS_ERR_WORKSPACE;
  if (!ssh::aligned16(workspace)) return SS_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  if (dim <= 256) {  // short rows: several rows per warp
    if (dtype == SS_F32) return rms_small_dispatch<float>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
    return rms_small_dispatch<__nv_bfloat16>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  }
  if (dim <= 2048) {  // columns split over a CTA
    if (dtype == SS_F32) return rms_cols_launch<float>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
    return rms_cols_launch<__nv_bfloat16>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  }
  const int nst = rms_tma_stages(dim, dtype == SS_F32 ? 4 : 2);
  if (nst > 0 && pl.vpt == 1) {  // dim <= 8192 and two stages fit
    if (dtype == SS_F32) return rms_tma_launch<float>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, nst, s);
    return rms_tma_launch<__nv_bfloat16>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, nst, s);
  }
  if (dtype == SS_F32) return rms_launch<float>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  return rms_launch<__nv_bfloat16>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
}

namespace {

// Device address of g_rms_noalloc_scratch on the current device, looked up
// once per device (in host code the array's name is only a stand-in).
std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 64;
float* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rms_noalloc_scratch) != cudaSuccess || p == nullptr) return SS_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return SS_OK;
}

}  // namespace

namespace ssh {
int read_clear_rms_err(cudaStream_t s, unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_rms_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SS_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_rms_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) return SS_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
}  // namespace ssh

extern "C" int rmsnorm_bwd_noalloc(const void* dy, const void* x, const float* scale, const float* rms, float* dx,
                                   float* dscale, int rows, int dim, int dtype, void* stream) {
  if (!dy || !x || !scale || !rms || !dx || !dscale) return SS_ERR_NULL;
  const int v = rms_validate(rows, dim, dtype);
  if (v != SS_OK) return v;
  if (dim > kNoAllocMaxDim) return SS_ERR_DIM;
  const void* ptrs[] = {dy, x, scale, rms, dx, dscale};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  float* ws = nullptr;
  const int rc = noalloc_scratch(&ws);
  if (rc != SS_OK) return rc;
  RmsPlan pl = rms_plan(rows, dim);
  pl.grid = rows < kNoAllocGrid ? rows : kNoAllocGrid;  // every CTA overwrites its own partial row
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) return rms_launch<float>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
  return rms_launch<__nv_bfloat16>(dy, x, scale, rms, dx, dscale, rows, dim, ws, pl, s);
}
