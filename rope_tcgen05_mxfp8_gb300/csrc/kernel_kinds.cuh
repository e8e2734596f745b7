// Launch one epilogue kind of K1 for the plan's tile width and GEMM form (used by the
// translation units that instantiate the per-head kinds).
#pragma once

#include "qkv_gemm_mxf8.cuh"

namespace qkvcte {
namespace {

template <int kEpi>
cudaError_t launch_kind(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW, const CUtensorMap& tmSF,
                        const GemmArgs& a, cudaStream_t s, int num_sms) {
  const NormRopeArgs none{};
  if (g.cta_pair) {
    switch (g.tile_n) {
      case 128: return launch_gemm_pair_t<128, kEpi, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 192: return launch_gemm_pair_t<192, kEpi, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 240: return launch_gemm_pair_t<240, kEpi, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 256: return launch_gemm_pair_t<256, kEpi, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.tile_n) {
    case 128: return launch_gemm_t<128, kEpi>(g, tmA, tmW, a, s, num_sms);
    case 192: return launch_gemm_t<192, kEpi>(g, tmA, tmW, a, s, num_sms);
    case 240: return launch_gemm_t<240, kEpi>(g, tmA, tmW, a, s, num_sms);
    case 256: return launch_gemm_t<256, kEpi>(g, tmA, tmW, a, s, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace qkvcte
