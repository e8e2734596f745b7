// Kernel K1 with the per-head qk-norm finished in the epilogue (RMS_NORM / LAYER_NORM
// and RoPE as each tile leaves TMEM; no second pass; tiles hold whole heads), one
// instantiation per tile width and GEMM form. The templates are in qkv_gemm_mxf8.cuh;
// kernel_kinds.cuh instantiates one epilogue kind for every tile width and form.
#include "qkv_gemm_mxf8.cuh"
#include "kernel_kinds.cuh"

namespace qkvcte {

cudaError_t launch_gemm_stats(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                              const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms);

cudaError_t launch_gemm_head(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                             const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms) {
  if (a.head_norm != 0) return launch_kind<kEpiHead>(g, tmA, tmW, tmSF, a, s, num_sms);
  return launch_gemm_stats(g, tmA, tmW, tmSF, a, s, num_sms);
}

}  // namespace qkvcte
