// Internal interfaces between the C-ABI front end and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace qkvcte {

// Device status word bits (workspace word 0): which bounded wait ran out.
enum : uint32_t {
  kErrProducerEmptyWait = 1u << 0,
  kErrMmaFullWait = 1u << 1,
  kErrMmaTmemEmptyWait = 1u << 2,
  kErrEpilogueTmemFullWait = 1u << 3,
  kErrDrainWait = 1u << 4,
};

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)                 status words
//   [256, 256 + ss_bytes)    fp32 [T, 2] sum-of-squares accumulator (used when the
//                            caller passes no sumsq buffer)
//   [.., + sf_bytes)         W's UE8M0 scales repacked per (N tile, K stage) in the
//                            order the MMA's scale-factor copy consumes them
//   [.., + qk_bytes)         fp32 [T, I_q + I_k]: the un-normalised Q and K columns,
//                            handed from K1 to K2 (only when a norm/RoPE pass runs)
struct WorkspaceLayout {
  size_t status_off, sumsq_off, sf_off, qk_off, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// GEMM (kernel K1) configuration chosen at plan time.
struct GemmShape {
  int T, H, I;
  int tile_n;       // N tile (columns of O per tile)
  int m_tiles, n_tiles, k_stages;
  int sf_chunks;    // 128-column scale-factor chunks per N tile
};

struct GemmArgs {
  const float* a_scale;
  const float* w_col_scale;  // may be null
  const uint16_t* bias;      // may be null
  const uint8_t* sf_packed;
  uint16_t* O;
  float* qk;                 // fp32 [T, k_end] Q/K hand-off, or null: Q/K go to O as bf16
  float* sumsq;              // may be null: then no sum of squares is accumulated
  uint32_t* status;
  int q_end, k_end;          // Q = [0, q_end), K = [q_end, k_end), V = [k_end, I)
  uint32_t flags;
};

struct NormRopeArgs {
  int T, I, n_q, n_kv, d_head;
  int norm, rope;
  float eps;
  const float* sumsq;
  const float* qk;           // fp32 [T, (n_q + n_kv) * d_head] un-normalised Q and K
  const uint16_t* gamma_q;
  const uint16_t* gamma_k;
  const float* cos_t;
  const float* sin_t;
  uint16_t* O;
  float* inv_rms;            // may be null
};

// Supported N tiles (compile-time instantiations of K1).
bool gemm_tile_supported(int tile_n);
int gemm_sf_chunks(int tile_n);
size_t gemm_smem_bytes(int tile_n);

// Launchers. Each returns cudaSuccess or the launch error.
cudaError_t launch_prep(const GemmShape& g, const uint8_t* w_sf, uint8_t* sf_packed, float* sumsq,
                        size_t sumsq_count, uint32_t* status, cudaStream_t s, int num_sms);
cudaError_t launch_gemm(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                        const GemmArgs& a, cudaStream_t s, int num_sms);
cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s, int num_sms);

}  // namespace qkvcte
