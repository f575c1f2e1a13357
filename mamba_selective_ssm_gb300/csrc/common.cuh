// Device and host helpers shared by the libssscan kernels (sm_103a).
//
// - scalar math built on the ex2 / rcp hardware approximations (exp(x) as
//   2^(x*log2 e), sigmoid as 1/(1+2^(-z*log2 e)));
// - bf16 <-> fp32 conversion (bf16 -> fp32 is a 16-bit shift; fp32 -> bf16
//   rounds to nearest even with the cvt.rn instruction);
// - packed f32x2 arithmetic (one issue slot for two FP32 lanes);
// - mbarrier / TMA (cp.async.bulk.tensor) primitives with bounded waits:
//   a wait that runs out sets the library's device error word and the kernel
//   drains and returns instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssscan.h"

namespace ssk {

// SMs of the current device (0 when the query fails).
inline int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

// CTAs of `kern` that fit on one SM at `threads` threads and `smem` dynamic
// shared-memory bytes, counted from the kernel's registers and shared memory
// and the device's per-SM limits (registers allocated per warp in 256s, 1 KB of
// shared memory reserved per CTA).  The runtime occupancy query returns 1 for
// kernels that use tensor memory, which is not what the hardware schedules.
template <typename K>
inline int resident_ctas(K kern, int threads, size_t smem) {
  cudaFuncAttributes fa;
  int dev = 0, smem_sm = 0, regs_sm = 0, thr_sm = 0, blk_sm = 0;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&blk_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev) != cudaSuccess)
    return 0;
  const int warps = (threads + 31) / 32;
  const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
  int n = blk_sm;
  if (regs_warp > 0 && regs_sm / (regs_warp * warps) < n) n = regs_sm / (regs_warp * warps);
  if (thr_sm / (warps * 32) < n) n = thr_sm / (warps * 32);
  const size_t per_cta = smem + fa.sharedSizeBytes + 1024;
  if ((int)((size_t)smem_sm / per_cta) < n) n = (int)((size_t)smem_sm / per_cta);
  return n;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- math

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid(z) = 1 / (1 + exp(-z)); saturates cleanly to 0 / 1 for large |z|.
__device__ __forceinline__ float sigmoid(float z) { return rcp(1.0f + ex2(-z * kLog2e)); }

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 bc2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 ex2_2(float2 u) { return make_float2(ex2(u.x), ex2(u.y)); }

// ---------------------------------------------------------------- dtypes

// the low bf16 of a pair: the 16-bit shift written as an integer multiply, which issues on the FMA pipe rather
// than the ALU pipe the other half's mask and the pair packing already load (RMSNorm forward 15.3 -> 15.0 us)
__device__ __forceinline__ float bf16_lo(uint32_t w) {
  uint32_t r;
  asm("mul.lo.u32 %0, %1, 65536;" : "=r"(r) : "r"(w));
  return __uint_as_float(r);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
struct ActT;

template <>
struct ActT<float> {
  static constexpr int kBytes = 4;
  static constexpr CUtensorMapDataType kTma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  __device__ __forceinline__ static float ld(const float* p) { return *p; }
  // 8 consecutive elements -> fp32 (p 16-byte aligned)
  __device__ __forceinline__ static void ld8(const float* p, float* o) {
    float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
  }
  __device__ __forceinline__ static void ld4(const float* p, float* o) {
    float4 a = *reinterpret_cast<const float4*>(p);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  }
  __device__ __forceinline__ static void st8(float* p, const float* v) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  // 2 consecutive elements (p 8-byte aligned) as a packed pair
  __device__ __forceinline__ static float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
  // 4 consecutive elements (p 16-byte aligned) as two packed pairs
  __device__ __forceinline__ static void ld4x2(const float* p, float2& a, float2& b) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    a = make_float2(v.x, v.y);
    b = make_float2(v.z, v.w);
  }
  __device__ __forceinline__ static void st1(float* p, float v) { *p = v; }
  __device__ __forceinline__ static void st2(float* p, float a, float b) { *reinterpret_cast<float2*>(p) = make_float2(a, b); }
};

template <>
struct ActT<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr CUtensorMapDataType kTma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  __device__ __forceinline__ static float ld(const __nv_bfloat16* p) {
    return __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  __device__ __forceinline__ static void ld8(const __nv_bfloat16* p, float* o) {
    uint4 w = *reinterpret_cast<const uint4*>(p);
    o[0] = bf16_lo(w.x); o[1] = bf16_hi(w.x); o[2] = bf16_lo(w.y); o[3] = bf16_hi(w.y);
    o[4] = bf16_lo(w.z); o[5] = bf16_hi(w.z); o[6] = bf16_lo(w.w); o[7] = bf16_hi(w.w);
  }
  __device__ __forceinline__ static void ld4(const __nv_bfloat16* p, float* o) {
    uint2 w = *reinterpret_cast<const uint2*>(p);
    o[0] = bf16_lo(w.x); o[1] = bf16_hi(w.x); o[2] = bf16_lo(w.y); o[3] = bf16_hi(w.y);
  }
  __device__ __forceinline__ static uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static void st8(__nv_bfloat16* p, const float* v) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
  }
  __device__ __forceinline__ static float2 ld2(const __nv_bfloat16* p) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(bf16_lo(w), bf16_hi(w));
  }
  __device__ __forceinline__ static void ld4x2(const __nv_bfloat16* p, float2& a, float2& b) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    a = make_float2(bf16_lo(w.x), bf16_hi(w.x));
    b = make_float2(bf16_lo(w.y), bf16_hi(w.y));
  }
  __device__ __forceinline__ static void st1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
  __device__ __forceinline__ static void st2(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<uint32_t*>(p) = pack2(a, b);
  }
};

// 8 consecutive activations as loaded (16 bytes of bf16, 32 of fp32) and their widening
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  using V = uint4;
  static __device__ __forceinline__ V ld(const __nv_bfloat16* p) { return *reinterpret_cast<const uint4*>(p); }
  static __device__ __forceinline__ V zero() { return make_uint4(0u, 0u, 0u, 0u); }
  static __device__ __forceinline__ void wide(const V& v, float* o) {
    o[0] = bf16_lo(v.x); o[1] = bf16_hi(v.x); o[2] = bf16_lo(v.y); o[3] = bf16_hi(v.y);
    o[4] = bf16_lo(v.z); o[5] = bf16_hi(v.z); o[6] = bf16_lo(v.w); o[7] = bf16_hi(v.w);
  }
};
template <>
struct Raw8<float> {
  struct V {
    float4 a, b;
  };
  static __device__ __forceinline__ V ld(const float* p) {
    return V{reinterpret_cast<const float4*>(p)[0], reinterpret_cast<const float4*>(p)[1]};
  }
  static __device__ __forceinline__ V zero() { return V{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)}; }
  static __device__ __forceinline__ void wide(const V& v, float* o) {
    o[0] = v.a.x; o[1] = v.a.y; o[2] = v.a.z; o[3] = v.a.w; o[4] = v.b.x; o[5] = v.b.y; o[6] = v.b.z; o[7] = v.b.w;
  }
};

// ---------------------------------------------------------------- smem / mbarrier / TMA

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Issued by the thread that is about to refill a shared-memory slot with an
// async-proxy copy (TMA, bulk copy), after the barrier that follows the CTA's
// last generic-proxy reads of that slot: it orders those reads before the
// copy's writes.  Without it a refill can land while reads issued before the
// barrier are still queued (seen as stale rows in a 4-slot TMA ring).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`
// nanoseconds.  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t addr = smem_u32(bar);
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63u) == 0) {
      const uint64_t now = globaltimer_ns();
      if (it == 0) t0 = now;
      else if (now - t0 > limit_ns) return false;
    }
  }
}

// 3-D tiled TMA load: box at coordinates (c0 innermost, c1, c2).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk copy global -> shared, completing on an mbarrier: both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tensor memory
// TMEM serves as per-thread scratch: thread i of warp w owns TMEM lane
// 32 * (w % 4) + i and addresses its columns with the 32x32b access shape.

// Allocate `ncols` columns (a power of two >= 32); the whole warp executes it
// and the base address lands in *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
// Give up the right to allocate: another CTA of a TMEM-using kernel is only
// placed on this SM beside us once we have done so, so every CTA of such a
// kernel executes it early, whether or not it allocated.
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Store 8 floats into 8 consecutive columns of the thread's lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, float4 a, float4 b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(__float_as_uint(a.x)), "r"(__float_as_uint(a.y)), "r"(__float_as_uint(a.z)), "r"(__float_as_uint(a.w)),
               "r"(__float_as_uint(b.x)), "r"(__float_as_uint(b.y)), "r"(__float_as_uint(b.z)), "r"(__float_as_uint(b.w))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Load 8 floats from 8 consecutive columns of the thread's lane and wait for
// them (load and wait in one statement so no use can move above the wait).
__device__ __forceinline__ void tmem_ld8_wait(uint32_t taddr, float4& a, float4& b) {
  uint32_t r0, r1, r2, r3, r4, r5, r6, r7;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7)
      : "r"(taddr)
      : "memory");
  a = make_float4(__uint_as_float(r0), __uint_as_float(r1), __uint_as_float(r2), __uint_as_float(r3));
  b = make_float4(__uint_as_float(r4), __uint_as_float(r5), __uint_as_float(r6), __uint_as_float(r7));
}

// Time a kernel waits on its own TMA copies before declaring failure.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Device error word codes (or-ed together).
constexpr unsigned kErrTmaTimeout = 1u;

// Column sums of a [rows, ncols] fp32 partial array in a fixed order:
// out(i) = sum_{g < rows} part[g * ncols + i], delivered to Store::put(i, v).
// Block (32, RG): thread (x, y) adds rows g = y, y+RG, ... in ascending order
// (loads issued four at a time, adds in that order), then the RG partial sums
// are added y = 0..RG-1; deterministic run to run.  RG = 32 when the columns
// alone give too few blocks to fill the GPU.
// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with launch_dependent() may be scheduled while the kernel
// before it in the stream is still running; it must call pdl_wait() before it
// reads anything that kernel writes (the wait returns once that grid has
// completed and its writes are visible; it returns at once for a kernel
// launched the ordinary way).  pdl_trigger() in the kernel before lets the
// dependent launch start early; without it the dependent starts when it exits.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <class Store, int RG>
__global__ void __launch_bounds__(32 * RG) colsum_kernel(const float* __restrict__ part, long long ncols, int rows, Store st) {
  __shared__ float red[RG][33];
  const long long i = (long long)blockIdx.x * 32 + threadIdx.x;
  float acc = 0.f;
  pdl_wait();  // the partials come from the kernel before
  if (i < ncols) {
    int g = threadIdx.y;
    for (; g + 3 * RG < rows; g += 4 * RG) {
      const float v0 = part[(size_t)g * ncols + i], v1 = part[(size_t)(g + RG) * ncols + i];
      const float v2 = part[(size_t)(g + 2 * RG) * ncols + i], v3 = part[(size_t)(g + 3 * RG) * ncols + i];
      acc += v0;
      acc += v1;
      acc += v2;
      acc += v3;
    }
    for (; g < rows; g += RG) acc += part[(size_t)g * ncols + i];
  }
  red[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && i < ncols) {
    float v = red[0][threadIdx.x];
#pragma unroll
    for (int y = 1; y < RG; ++y) v += red[y][threadIdx.x];
    st.put(i, v);
  }
}

template <class Store>
inline cudaError_t colsum(const float* part, long long ncols, int rows, Store st, cudaStream_t s) {
  const long long blocks = (ncols + 31) / 32;
  if (blocks < 4ll * device_sm_count() && rows >= 64)
    return launch_dependent(colsum_kernel<Store, 32>, dim3((unsigned)blocks), dim3(32, 32), 0, s, part, ncols, rows, st);
  return launch_dependent(colsum_kernel<Store, 8>, dim3((unsigned)blocks), dim3(32, 8), 0, s, part, ncols, rows, st);
}

}  // namespace ssk

// ---------------------------------------------------------------- host side

namespace ssh {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Encode a tiled tensor map (driver entry point fetched through the runtime,
// so the library needs no link against libcuda).  Returns false on failure.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace ssh
