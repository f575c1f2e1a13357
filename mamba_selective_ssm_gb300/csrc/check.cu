// Non-finite check (ss_count_nonfinite) for sm_103a: the number of NaN and
// +-Inf values in a dense fp32 or bf16 device buffer, for the caller's
// failure detection (a step whose gradients hold any is to be dropped).
//
// A value is non-finite when its exponent field is all ones (fp32 bits
// 0x7f800000, bf16 bits 0x7f80).  Pass 1: every block counts its grid-stride
// share (16-byte vector loads, the tail one element at a time) and writes one
// partial; pass 2: one block adds the partials in a fixed order into a 64-bit
// total.  Integer sums, no atomics.
#include "common.cuh"

namespace {

using namespace ssk;

constexpr int kChkThreads = 256;
constexpr int kChkMaxBlocks = 1024;

__device__ __forceinline__ unsigned nf32(uint32_t u) { return (u & 0x7f800000u) == 0x7f800000u ? 1u : 0u; }
__device__ __forceinline__ unsigned nf16(uint32_t h) { return (h & 0x7f80u) == 0x7f80u ? 1u : 0u; }
// both bf16 halves of a 32-bit word
__device__ __forceinline__ unsigned nfbf2(uint32_t u) { return nf16(u & 0xffffu) + nf16(u >> 16); }

__device__ __forceinline__ unsigned block_sum(unsigned v) {
  __shared__ unsigned part[kChkThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned t = 0;
  if (threadIdx.x == 0)
    for (int w = 0; w < kChkThreads / 32; ++w) t += part[w];
  return t;  // valid in thread 0
}

// n elements; vectors of 4 (fp32) or 8 (bf16) elements, the tail past the last whole vector element by element
template <bool BF16>
__global__ void __launch_bounds__(kChkThreads) count_nonfinite_kernel(const void* __restrict__ p, size_t n,
                                                                      unsigned* __restrict__ partial) {
  constexpr size_t per_vec = BF16 ? 8 : 4;
  const size_t nvec = n / per_vec;
  const uint4* v = static_cast<const uint4*>(p);
  unsigned c = 0;
  for (size_t i = (size_t)blockIdx.x * kChkThreads + threadIdx.x; i < nvec; i += (size_t)gridDim.x * kChkThreads) {
    const uint4 q = v[i];
    if constexpr (BF16) c += nfbf2(q.x) + nfbf2(q.y) + nfbf2(q.z) + nfbf2(q.w);
    else c += nf32(q.x) + nf32(q.y) + nf32(q.z) + nf32(q.w);
  }
  if (blockIdx.x == 0) {
    for (size_t i = nvec * per_vec + threadIdx.x; i < n; i += kChkThreads) {
      if constexpr (BF16) c += nf16(static_cast<const uint16_t*>(p)[i]);
      else c += nf32(static_cast<const uint32_t*>(p)[i]);
    }
  }
  const unsigned t = block_sum(c);
  if (threadIdx.x == 0) partial[blockIdx.x] = t;
}

__global__ void __launch_bounds__(kChkThreads) sum_partials_kernel(const unsigned* __restrict__ partial, int nblocks,
                                                                   unsigned long long* __restrict__ count) {
  // thread t adds partials t, t + 256, ... in order; the 256 sums are added in thread order
  __shared__ unsigned long long s[kChkThreads];
  unsigned long long a = 0;
  for (int i = threadIdx.x; i < nblocks; i += kChkThreads) a += partial[i];
  s[threadIdx.x] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int i = 0; i < kChkThreads; ++i) t += s[i];
    *count = t;
  }
}

}  // namespace

extern "C" size_t ss_count_nonfinite_workspace_size(void) { return kChkMaxBlocks * sizeof(unsigned); }

extern "C" int ss_count_nonfinite(const void* p, size_t n, int dtype, unsigned long long* count, void* workspace,
                                  size_t ws_bytes, void* stream) {
  if (!count || (n > 0 && !p)) return SS_ERR_NULL;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (workspace == nullptr || ws_bytes < ss_count_nonfinite_workspace_size()) return SS_ERR_WORKSPACE;
  if ((n > 0 && !ssh::aligned16(p)) || !ssh::aligned16(workspace) || (reinterpret_cast<uintptr_t>(count) & 7u))
    return SS_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* partial = static_cast<unsigned*>(workspace);
  const size_t per_vec = dtype == SS_BF16 ? 8 : 4;
  const size_t nvec = n / per_vec;
  size_t blocks = (nvec + kChkThreads - 1) / kChkThreads;
  const size_t cap = (size_t)device_sm_count() * 4;
  if (blocks > cap) blocks = cap;
  if (blocks > (size_t)kChkMaxBlocks) blocks = kChkMaxBlocks;
  if (blocks < 1) blocks = 1;
  if (dtype == SS_BF16) count_nonfinite_kernel<true><<<(unsigned)blocks, kChkThreads, 0, s>>>(p, n, partial);
  else count_nonfinite_kernel<false><<<(unsigned)blocks, kChkThreads, 0, s>>>(p, n, partial);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  sum_partials_kernel<<<1, kChkThreads, 0, s>>>(partial, (int)blocks, count);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
