// Kernel K1 with the per-head statistics epilogue (RMS: sums of squares per row and
// head; LayerNorm: each tile part's mean and centred M2, values handed over centred)
// for the norm/RoPE pass to finish the per-head norm from. The templates are in
// qkv_gemm_mxf8.cuh.
#include "qkv_gemm_mxf8.cuh"
#include "kernel_kinds.cuh"

namespace qkvcte {

cudaError_t launch_gemm_stats(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                              const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms) {
  if (a.stats_kind == 2) return launch_kind<kEpiStatsRms>(g, tmA, tmW, tmSF, a, s, num_sms);
  return launch_kind<kEpiStatsLayer>(g, tmA, tmW, tmSF, a, s, num_sms);
}

}  // namespace qkvcte
