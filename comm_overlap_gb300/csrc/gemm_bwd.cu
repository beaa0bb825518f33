// gemm_bwd.cu -- backward GEMM instantiations: output-gradient GEMM with the activation
// backward fused in its epilogue, input-gradient partials (or fused with their shard-sum), and
// fp32-accumulating weight gradients.
#include "gemm.cuh"

namespace dm {

cudaError_t launch_gemm_bwd(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const GemmArgs& args, cudaStream_t st) {
  switch (variant) {
    case GV_BWD_ACT: return launch_gemm_t<EPI_ACT_BWD, false, true>(ta, tb, em, args, st);
    case GV_BWD_GLU: return launch_gemm_t<EPI_GLU_BWD, false, true>(ta, tb, em, args, st);
    case GV_BWD_PARTIAL: return launch_gemm_t<EPI_F32_STORE, false, true>(ta, tb, em, args, st);
    case GV_BWD_REDUCE: return launch_gemm_t<EPI_F32_REDUCE, false, true>(ta, tb, em, args, st);
    case GV_WGRAD: return launch_gemm_t<EPI_F32_ACCUM, true, true>(ta, tb, em, args, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_gemm_bwd_error(int* code) { return take_error_word(code); }

}  // namespace dm
