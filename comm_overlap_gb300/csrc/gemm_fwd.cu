// gemm_fwd.cu -- forward GEMM instantiations: first linear (+activation) and second linear
// (-> fp32 shard partials).
#include "gemm.cuh"

namespace dm {

int gemm_out_tile_n(int variant) { return variant == GV_FWD_GLU ? 128 : kBN; }

cudaError_t launch_gemm_fwd(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                            const GemmArgs& args, cudaStream_t st) {
  switch (variant) {
    case GV_FWD_ACT: return launch_gemm_t<EPI_ACT_BF16, false, false>(ta, tb, tc, args, st);
    case GV_FWD_GLU: return launch_gemm_t<EPI_GLU_BF16, false, false>(ta, tb, tc, args, st);
    case GV_FWD_PARTIAL: return launch_gemm_t<EPI_F32_STORE, false, false>(ta, tb, tc, args, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_gemm_fwd_error(int* code) { return take_error_word(code); }

}  // namespace dm
