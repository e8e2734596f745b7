// Kernel K1 with the per-head qk-norm epilogue (RMS_NORM / LAYER_NORM and RoPE
// finished as each tile leaves TMEM; no second pass), one instantiation per tile
// width and GEMM form. The templates are in qkv_gemm_mxf8.cuh.
#include "qkv_gemm_mxf8.cuh"

namespace qkvcte {

cudaError_t launch_gemm_head(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                             const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms) {
  const NormRopeArgs none{};
  if (g.cta_pair) {
    switch (g.tile_n) {
      case 128: return launch_gemm_pair_t<128, true, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 192: return launch_gemm_pair_t<192, true, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 240: return launch_gemm_pair_t<240, true, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 256: return launch_gemm_pair_t<256, true, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.tile_n) {
    case 128: return launch_gemm_t<128, true>(g, tmA, tmW, a, s, num_sms);
    case 192: return launch_gemm_t<192, true>(g, tmA, tmW, a, s, num_sms);
    case 240: return launch_gemm_t<240, true>(g, tmA, tmW, a, s, num_sms);
    case 256: return launch_gemm_t<256, true>(g, tmA, tmW, a, s, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvcte
