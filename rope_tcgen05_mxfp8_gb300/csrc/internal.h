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
  kErrNormReadyWait = 1u << 5,
  kErrTileIdWait = 1u << 6,
};

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)                 status word (offset 0); at kStampOffset four uint64
//                            %globaltimer stamps: K1 first start, K1 last end, norm/RoPE
//                            first start, norm/RoPE last end; at kTaskCounterOffset the
//                            counter the norm/RoPE tasks are claimed from, and after it
//                            the counter the CTA-pair GEMM claims its tiles from
//   [256, 256 + ss_bytes)    fp32 [T, 2] sum-of-squares accumulator (used when the
//                            caller passes no sumsq buffer)
//   [.., + sf_bytes)         W's UE8M0 scales repacked per (N tile, K stage) in the
//                            order the MMA's scale-factor copy consumes them
//   [.., + ready_bytes)      uint32 [blocks128]: per 128-row block, how many epilogue
//                            warp-tiles of K1's Q/K tiles have finished (4 per tile)
//   [.., + 4 * kSmTable)     uint32 per SM (%smid): the mask of SM sub-partitions
//                            (%warpid & 3) K1's TMA-load and MMA-issue warps occupy while
//                            K1's CTA there runs, 0 otherwise (a scheduling hint for
//                            the norm/RoPE pass)
//   [.., + qk_bytes)         the un-normalised Q and K columns handed from K1 to K2
//                            (only when a norm/RoPE pass runs) in block floating
//                            point: per row and 16-column chunk, one power-of-two
//                            exponent byte E and 16 fp16 values f with
//                            value = f * 2^(E-127), |f| < 2. Tile-major: for row t and
//                            chunk k < k_end/16, idx = (t/128 * k_end/16 + k) * 128
//                            + t%128; the 16 fp16 sit at qk_val[idx*16 ..] (32 bytes)
//                            and the exponent at qk_exp[idx]
//   [.., + stats_bytes)      only for a per-head norm finished by the norm/RoPE pass: the
//                            per-(row, head) statistics (see GemmArgs::stats_kind)
//   [.., + T*H), [.., + 4T)  only for a packed or bf16 input: the e4m3 codes [T, H] and
//                            fp32 row scales [T] the producer step writes for the GEMM
constexpr size_t kStampOffset = 64;
constexpr size_t kTaskCounterOffset = 128;  // uint32: the next unclaimed norm/RoPE task
constexpr size_t kTileCounterOffset = 132;  // uint32: the next unclaimed CTA-pair GEMM tile
static_assert(kTileCounterOffset == kTaskCounterOffset + 4, "prep clears both counters as one pair of words");
constexpr int kSmTable = 1024;              // entries of the per-SM sub-partition table

struct WorkspaceLayout {
  size_t status_off, sumsq_off, sf_off, ready_off, sm_busy_off, qk_off, qk_exp_off, stats_off, act_off, act_scale_off,
      total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kMaxBands = 16;

// The CTA-pair GEMM takes its last kClaimedWaves waves of tiles from a counter.
constexpr int kClaimedWaves = 6;

// The static part of a CTA pair's tile sequence: its tile number seq < n_static is
// pair + seq * pairs; the tiles from dyn_base on are claimed from the counter
// (dyn_base + the counter's value, while below num_tiles).
struct PairSchedule {
  int pair, pairs, n_static, dyn_base, num_tiles;

  __host__ __device__ PairSchedule(int num_tiles_, int pair_, int pairs_)
      : pair(pair_), pairs(pairs_), num_tiles(num_tiles_) {
    const int waves = num_tiles_ / pairs_;
    n_static = waves > kClaimedWaves ? waves - kClaimedWaves : 0;
    dyn_base = n_static * pairs_;
  }
  __host__ __device__ bool is_static(int seq) const { return seq < n_static; }
  __host__ __device__ int static_tile(int seq) const { return pair + seq * pairs; }
};

// GEMM (kernel K1) configuration chosen at plan time.
//
// Tile order: the N tiles are cut into bands (contiguous runs of N tiles). The
// persistent grid walks the bands one after the other and, inside a band, row panel
// by row panel (m outer, n inner), so the CTAs running at any moment share one band's
// slab of W, which stays resident in L2 while A streams through. The bands of tiles
// holding Q or K columns come first and the V-only bands last: the norm/RoPE pass
// waits only for a panel's Q/K tiles, so it overlaps the V bands.
struct GemmShape {
  int T, H, I;
  int tile_n;       // N tile (columns of O per tile)
  int cta_pair;     // 1: tiles of 256 rows computed by a CTA pair (M = 256 MMA)
  int blocks128;    // ceil(T / 128): 128-row blocks (counters, hand-off rows)
  int m_tiles, n_tiles, k_stages;
  int sf_chunks;    // 128-column scale-factor chunks per N tile
  int n_qk_tiles;   // N tiles holding at least one Q or K column: [0, n_qk_tiles)
  int n_bands;                     // segments: a band's N tiles over a range of row panels
  int band_n0[kMaxBands];          // first N tile of each segment
  int band_nc[kMaxBands];          // N tiles in each segment
  int band_m0[kMaxBands];          // first row panel (m) of each segment
  int band_tile0[kMaxBands + 1];   // linear index of each segment's first tile
};

// (m, n) of linear tile `tile` in the banded order.
__host__ __device__ inline void tile_coords(const GemmShape& g, int tile, int& m, int& n) {
  int b = 0;
  while (b + 1 < g.n_bands && tile >= g.band_tile0[b + 1]) ++b;
  const int local = tile - g.band_tile0[b];
  const int nc = g.band_nc[b];
  const int ml = local / nc;
  m = g.band_m0[b] + ml;
  n = g.band_n0[b] + (local - ml * nc);
}

// Cut [0, n_tiles) into bands of at most `band_tiles` N tiles, Q/K tiles first. With
// m_chunks > 1 the Q/K bands take turns over m_chunks ranges of row panels (every Q/K
// band over the first range, then over the next, ...), so row panels complete from
// early on; the V bands follow over all row panels.
inline void make_bands(GemmShape& g, int band_tiles, int m_chunks = 1) {
  if (band_tiles < 1) band_tiles = 1;
  const int qk_run = g.n_qk_tiles;
  const int runs[2][2] = {{0, qk_run}, {qk_run, g.n_tiles - qk_run}};
  int need = 0;
  for (const auto& r : runs) need += (r[1] + band_tiles - 1) / band_tiles;
  while (need > kMaxBands) {
    ++band_tiles;
    need = 0;
    for (const auto& r : runs) need += (r[1] + band_tiles - 1) / band_tiles;
  }
  const int qk_bands = (qk_run + band_tiles - 1) / band_tiles;
  if (m_chunks > g.m_tiles) m_chunks = g.m_tiles;
  while (m_chunks > 1 && need - qk_bands + qk_bands * m_chunks > kMaxBands) --m_chunks;
  if (m_chunks < 1 || qk_bands == 0) m_chunks = 1;
  const int per_chunk = (g.m_tiles + m_chunks - 1) / m_chunks;
  g.n_bands = 0;
  int tile0 = 0;
  auto add = [&](int n0, int nc, int m0, int mc) {
    if (nc <= 0 || mc <= 0) return;
    g.band_n0[g.n_bands] = n0;
    g.band_nc[g.n_bands] = nc;
    g.band_m0[g.n_bands] = m0;
    g.band_tile0[g.n_bands] = tile0;
    tile0 += nc * mc;
    ++g.n_bands;
  };
  for (int m0 = 0; m0 < g.m_tiles; m0 += per_chunk) {
    const int mc = g.m_tiles - m0 < per_chunk ? g.m_tiles - m0 : per_chunk;
    for (int n0 = 0; n0 < qk_run; n0 += band_tiles) add(n0, qk_run - n0 < band_tiles ? qk_run - n0 : band_tiles, m0, mc);
  }
  for (int n0 = qk_run; n0 < g.n_tiles; n0 += band_tiles)
    add(n0, g.n_tiles - n0 < band_tiles ? g.n_tiles - n0 : band_tiles, 0, g.m_tiles);
  g.band_tile0[g.n_bands] = tile0;
}

struct GemmArgs {
  const float* a_scale;
  const float* w_col_scale;  // may be null
  const uint16_t* bias;      // may be null
  const uint8_t* sf_packed;
  uint16_t* O;
  uint16_t* qk_val;          // Q/K hand-off fp16 values, or null: Q/K go to O as bf16
  uint8_t* qk_exp;           // Q/K hand-off exponent bytes
  float* sumsq;              // may be null: then no sum of squares is accumulated
  uint32_t* ready;           // per-panel completion counters (K2 overlaps K1 on them)
  uint32_t* sm_busy;         // [kSmTable] sub-partitions of this kernel's load and MMA warps, per SM
  unsigned long long* stamps;  // [0] first CTA start (min), [1] last CTA end (max)
  uint32_t* tile_next;       // the CTA-pair form's tile counter (zeroed by prep)
  uint32_t* status;
  int q_end, k_end;          // Q = [0, q_end), K = [q_end, k_end), V = [k_end, I)
  int d_head;
  int nbsd;                  // O layout: 0 = BSD [T, I]; 1 = NBSd [I/d_head, T, d_head]
  uint32_t flags;
  // Per-head qk-norm finished in the epilogue (every tile holds whole heads):
  // 0 = off (Q/K go to the hand-off, or to O as projected), 2 = RMS, 3 = LayerNorm.
  int head_norm;
  int rope;                  // rotate-half RoPE in the epilogue (head_norm != 0 only)
  float eps;
  const uint16_t* gamma_q;   // [d_head] bf16 (head_norm != 0)
  const uint16_t* gamma_k;   // [d_head] bf16, or null without a K segment
  const float* cos_t;        // [T, d_head] fp32 (rope)
  const float* sin_t;
  // Per-head norm finished by the norm/RoPE pass: the epilogue writes per-(row, head)
  // statistics of the un-normalised Q/K. stats_kind 2 (RMS): sum(o^2) per (row, head),
  // accumulated with atomics (zeroed by prep). stats_kind 3 (LayerNorm): for each of
  // the stat_parts tiles a head's columns can span, the part's (shift, mean, M2, 0) as
  // a float4 at ((row * heads + head) * stat_parts + part); the part's Q/K values are
  // handed over as o - shift (shift: the part's first value in the row).
  int stats_kind;
  float* head_stats;
  int stat_parts;
};

// Element (row t, column c) of O in either layout (c and the 16 columns after it
// lie in one head: d_head and every chunk start are multiples of 16).
__host__ __device__ inline size_t out_index(int nbsd, int T, int I, int d_head, int t, int c) {
  if (nbsd) {
    const int h = c / d_head;
    return (static_cast<size_t>(h) * T + t) * d_head + (c - h * d_head);
  }
  return static_cast<size_t>(t) * I + c;
}

struct NormRopeArgs {
  int T, I, n_q, n_kv, d_head;
  int norm, rope;
  float eps;
  const float* sumsq;
  const uint16_t* qk_val;    // block floating point hand-off of the un-normalised Q/K
  const uint8_t* qk_exp;
  const uint16_t* gamma_q;
  const uint16_t* gamma_k;
  const float* cos_t;
  const float* sin_t;
  uint16_t* O;
  float* inv_rms;            // may be null
  int nbsd;                  // O layout (see GemmArgs)
  const uint32_t* ready;     // per 128-row panel: K1 epilogue warp-tiles finished
  const uint32_t* sm_busy;   // [kSmTable] K1's load/MMA sub-partitions per SM (0: no K1 CTA there)
  int claim;                 // 1: claim tasks from task_next, off K1's load/MMA sub-partitions; 0: stride
  uint32_t ready_target;     // 4 * K1's Q/K tiles: the panel's Q and K are final
  unsigned long long* stamps;  // [0] first block start (min), [1] last block end (max)
  uint32_t* status;
  uint32_t* task_next;       // next unclaimed task (claimed by K2's warps, or by the fused GEMM's epilogue warps)
  // The CTA-pair GEMM's claimed-tile counter and the count at which every pair has
  // reached the claimed tail: from then on no warp of the pass holds back (or null).
  const uint32_t* gemm_claims;
  uint32_t release_at;
  // per-head norm (norm 2 RMS / 3 LayerNorm) from the GEMM's per-(row, head)
  // statistics (see GemmArgs); 0: the across-heads norm or none
  int head_kind;
  const float* head_stats;
  int stat_parts;
  int tile_n;
  int head_group;            // heads per task of the standalone pass (set at its launch)
};

// Supported N tiles (compile-time instantiations of K1).
bool gemm_tile_supported(int tile_n);
int gemm_sf_chunks(int tile_n);
// Bytes of the repacked scales of one N tile for one 128-byte K block, and the row
// size in which the scale tensor map addresses them (a box row holds at most 256
// uint32).
constexpr int kSfBlockBytesPerChunk = 2048;
constexpr int kSfRowBytes = 1024;
size_t gemm_smem_bytes(int tile_n);

// Launchers. Each returns cudaSuccess or the launch error.
cudaError_t launch_prep(const GemmShape& g, const uint8_t* w_sf, uint8_t* sf_packed, float* sumsq,
                        size_t sumsq_count, uint32_t* ready, uint32_t* sm_busy, uint32_t* status,
                        unsigned long long* stamps,
                        uint32_t* task_next, float* zero_extra, size_t zero_extra_count, cudaStream_t s,
                        int num_sms, bool after_producer);
// K1. tmSF: the repacked scales as a uint32 map of kSfRowBytes-byte rows, one K block's
// image (sf_chunks * 2048 bytes) per box (used by the CTA-pair kernel). With `fused` (CTA-pair form only)
// the epilogue warps also run the norm/RoPE tasks of `*fused` between tiles, and no
// separate pass is launched.
cudaError_t launch_gemm(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                        const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms,
                        const NormRopeArgs* fused);
// K1 with the per-head qk-norm epilogue, or with the per-head statistics epilogue
// (qkv_gemm_mxf8_head.cu); launch_gemm calls it when a.head_norm or a.stats_kind is set.
cudaError_t launch_gemm_head(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                             const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms);
// K1 (CTA-pair form) with the norm/RoPE tasks run by its epilogue warps
// (qkv_gemm_mxf8_fused.cu); launch_gemm calls it when given `fused`.
cudaError_t launch_gemm_fused(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                              const CUtensorMap& tmSF, const GemmArgs& a, const NormRopeArgs& nr, cudaStream_t s,
                              int num_sms);
// K2, the norm/RoPE pass as its own kernel. With `overlap` it is launched right after
// K1 on the same stream as a programmatic dependent launch, so its blocks start while
// K1 runs and take each row panel as soon as K1 marks it ready.
cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s, int num_sms, bool overlap);

// Device address (on the current device) of the allocation-free entry point's scratch
// array (qkv_gemm_mxf8.cu); cudaGetSymbolAddress's status.
cudaError_t noalloc_scratch_address(void** out);

// dst |= src on the stream (qkv_gemm_mxf8.cu): the status of a run made of chunks.
cudaError_t launch_status_or(const uint32_t* src, uint32_t* dst, cudaStream_t s);

// The producer step (row_quant.cu): bf16 [T, H] -> e4m3 codes [T, H] + fp32 scales [T]
// and/or packed [T, H + 4] rows (either output may be null, not both); H % 16 == 0.
cudaError_t launch_row_quantize(const uint16_t* X, int T, int H, uint8_t* codes, float* scale, uint8_t* packed,
                                cudaStream_t s, int num_sms);
// Interleaved -> rotate-half lane order of the first qk_rows rows (whole heads of
// d_head rows), the rest copied (rope_permute.cu); src and dst do not overlap.
cudaError_t launch_permute_rows(const void* src, void* dst, long long rows, long long row_bytes, long long qk_rows,
                                int d_head, cudaStream_t s, int num_sms);
// Packed [T, H + 4] -> codes [T, H] + scales [T]; H % 16 == 0.
cudaError_t launch_unpack_rows(const uint8_t* packed, int T, int H, uint8_t* codes, float* scale, cudaStream_t s,
                               int num_sms);

}  // namespace qkvcte
