// Host-side plumbing shared by the entry points: status strings, version,
// device queries and the tensor-map encoder.
#include <mutex>

#include "common.cuh"

namespace scout {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, void* addr, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t* estr,
                      CUtensorMapSwizzle swz) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  if (g_encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  return g_encode(map, dt, rank, addr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace scout

extern "C" const char* scout_status_string(int status) {
  switch (status) {
    case SCOUT_OK: return "SCOUT_OK";
    case SCOUT_ERR_INVALID_ARG: return "SCOUT_ERR_INVALID_ARG: null pointer or inconsistent size";
    case SCOUT_ERR_UNSUPPORTED: return "SCOUT_ERR_UNSUPPORTED: shape, dtype or alignment not supported";
    case SCOUT_ERR_WORKSPACE: return "SCOUT_ERR_WORKSPACE: workspace missing or too small";
    case SCOUT_ERR_CUDA: return "SCOUT_ERR_CUDA: the CUDA runtime rejected a launch or copy";
    case SCOUT_ERR_TIMEOUT: return "SCOUT_ERR_TIMEOUT: a bounded wait expired";
    default: return "unknown scout status";
  }
}

extern "C" int scout_version(void) { return 1 * 10000 + 0 * 100 + 0; }
