// gemm_fp8.cu -- FP8 (E4M3) instantiations of the persistent GEMM: the first linear with the
// activation and the E4M3 re-quantisation of its output, and the second linear into fp32 shard
// partials (or fused with their shard-sum).  The reduction stays in fp32 ("04 · TP/SP 的通信-计算
// overlap 与工程优化", section 4: FP8 for what moves, higher precision for what is summed).
#include "gemm.cuh"

namespace dm {

cudaError_t launch_gemm_fp8(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const GemmArgs& args, cudaStream_t st) {
  switch (variant) {
    case GV_F8_FWD_ACT: return launch_gemm_t<EPI_ACT_F8, false, false, true>(ta, tb, em, args, st);
    case GV_F8_FWD_GLU: return launch_gemm_t<EPI_GLU_F8, false, false, true>(ta, tb, em, args, st);
    case GV_F8_FWD_PARTIAL: return launch_gemm_t<EPI_F32_STORE, false, false, true>(ta, tb, em, args, st);
    case GV_F8_FWD_REDUCE: return launch_gemm_t<EPI_F32_REDUCE, false, false, true>(ta, tb, em, args, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_gemm_fp8_error(int* code) { return take_error_word(code); }

}  // namespace dm
