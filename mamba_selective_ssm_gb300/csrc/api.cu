// Host-side glue of libssscan: status strings, TMA descriptor encoding and the
// device error word query.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace ssh {

int read_clear_fwd_err(cudaStream_t s, unsigned* out);
int read_clear_bwd_err(cudaStream_t s, unsigned* out);
int read_clear_rms_err(cudaStream_t s, unsigned* out);
int read_clear_rmsf_err(cudaStream_t s, unsigned* out);

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  const CUresult r = g_encode(map, dt, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ssh

extern "C" const char* ss_strerror(int code) {
  switch (code) {
    case SS_OK: return "ok";
    case SS_ERR_NULL: return "a required pointer is NULL";
    case SS_ERR_DIM: return "a size is non-positive or out of the supported range";
    case SS_ERR_UNSUPPORTED:
      return "unsupported configuration (N must be 4, 8 or 16; dtype SS_F32 or SS_BF16; d_conv 1..4; chunk 8 or a multiple "
             "of 16, at most 512 in the backward)";
    case SS_ERR_ALIGN: return "misaligned buffer (pointers must be 16-byte aligned; D and dim multiples of 8; bf16 with N=4 needs even L)";
    case SS_ERR_WORKSPACE: return "workspace missing or smaller than the *_workspace_size() query";
    case SS_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case SS_ERR_DEVICE: return "a kernel gave up waiting on its own asynchronous copies; its outputs are invalid";
    default: return "unknown status code";
  }
}

extern "C" int ss_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned a = 0, b = 0, c = 0, d = 0;
  if (ssh::read_clear_fwd_err(s, &a) != SS_OK) return SS_ERR_CUDA;
  if (ssh::read_clear_bwd_err(s, &b) != SS_OK) return SS_ERR_CUDA;
  if (ssh::read_clear_rms_err(s, &c) != SS_OK) return SS_ERR_CUDA;
  if (ssh::read_clear_rmsf_err(s, &d) != SS_OK) return SS_ERR_CUDA;
  return (a | b | c | d) ? SS_ERR_DEVICE : SS_OK;
}
