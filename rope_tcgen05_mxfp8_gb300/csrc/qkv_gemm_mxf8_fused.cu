// Kernel K1 (CTA-pair form) whose epilogue warps also run the norm/RoPE tasks
// between tiles, so the whole path is one GEMM launch after the scale repack; one
// instantiation per tile width. The templates are in qkv_gemm_mxf8.cuh, the tasks in
// qk_norm_rope.cuh.
#include "qkv_gemm_mxf8.cuh"

namespace qkvcte {

cudaError_t launch_gemm_fused(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                              const CUtensorMap& tmSF, const GemmArgs& a, const NormRopeArgs& nr, cudaStream_t s,
                              int num_sms) {
  switch (g.tile_n) {
    case 128: return launch_gemm_pair_t<128, kEpiPlain, true>(g, tmA, tmW, tmSF, a, nr, s, num_sms);
    case 192: return launch_gemm_pair_t<192, kEpiPlain, true>(g, tmA, tmW, tmSF, a, nr, s, num_sms);
    case 240: return launch_gemm_pair_t<240, kEpiPlain, true>(g, tmA, tmW, tmSF, a, nr, s, num_sms);
    case 256: return launch_gemm_pair_t<256, kEpiPlain, true>(g, tmA, tmW, tmSF, a, nr, s, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvcte
