// tmap.cu -- TMA tensor-map encoding through the driver entry point (no link against
// libcuda; the runtime resolves the symbol).
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"

namespace dm {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;
static std::string g_encode_err;

bool tma_encoder_ready(std::string* err) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
      g_encode_err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(e);
      return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr && err) *err = g_encode_err;
  return g_encode != nullptr;
}

bool make_map(CUtensorMap* map, int elem_bytes, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, std::string* err, int swizzle_bytes) {
  if (!tma_encoder_ready(err)) return false;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = g_encode(map, dt, static_cast<cuuint32_t>(rank),
                              const_cast<void*>(base), gdim, gstride, bdim, estride,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (err) {
      *err = "cuTensorMapEncodeTiled failed (code " + std::to_string(static_cast<int>(r)) + "), rank " +
             std::to_string(rank);
      for (int i = 0; i < rank; ++i)
        *err += " dim" + std::to_string(i) + "=" + std::to_string(dims[i]) + "/box" +
                std::to_string(box[i]);
    }
    return false;
  }
  return true;
}

}  // namespace dm
