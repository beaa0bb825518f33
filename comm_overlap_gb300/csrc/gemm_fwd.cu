// gemm_fwd.cu -- forward GEMM instantiations: first linear (+activation) and second linear
// (-> fp32 shard partials, or fused with their shard-sum).
#include "gemm.cuh"

namespace dm {

int gemm_out_tile_n(int variant) { return (variant == GV_FWD_GLU || variant == GV_F8_FWD_GLU) ? 128 : kBN; }

cudaError_t launch_gemm_fwd(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const GemmArgs& args, cudaStream_t st) {
  switch (variant) {
    case GV_FWD_ACT: return launch_gemm_t<EPI_ACT_BF16, false, false>(ta, tb, em, args, st);
    case GV_FWD_GLU: return launch_gemm_t<EPI_GLU_BF16, false, false>(ta, tb, em, args, st);
    case GV_FWD_PARTIAL: return launch_gemm_t<EPI_F32_STORE, false, false>(ta, tb, em, args, st);
    case GV_FWD_REDUCE: return launch_gemm_t<EPI_F32_REDUCE, false, false>(ta, tb, em, args, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_gemm_fwd_error(int* code) { return take_error_word(code); }

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait gives up after
// `timeout_ns`, records `site` in the error word and the kernel returns.
__global__ void wait_selftest_kernel(uint64_t timeout_ns, int site) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(b, 0, &abort_flag, &g_gemm_err, site, timeout_ns);
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int site, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns, site);
  return cudaGetLastError();
}

}  // namespace dm
