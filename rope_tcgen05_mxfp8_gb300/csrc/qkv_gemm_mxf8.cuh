// Kernel K1 templates, instantiated by qkv_gemm_mxf8.cu (plain epilogue) and
// qkv_gemm_mxf8_head.cu (per-head qk-norm epilogue).
//
// Kernel K1: O = dequant(A_fp8 @ W_fp8^T) * a_scale[t] * w_col_scale[i] + bias[i] -> bf16,
// plus the per-token sum of o^2 over the Q and the K columns.
//
// Follows the `qkv_cte` kernel reference page: the projection O[S, I] = A[S, H] @ W[H, I]
// (+ bias) ("Upstream behavior"), dequantised, bias-added and stored as each output
// tile leaves the accumulator, with the across-heads norm's step a (a per-token
// sum(x^2) over the whole Q segment and K segment of the un-normalised output,
// "Design" 1) folded into that same copy-out.
//
// GB300 design (not the page's Trainium schedule):
//   * persistent grid, one CTA per SM, tiles of 128 rows x tile_n columns, walked in
//     bands of N tiles (those holding Q or K columns first, V-only tiles last),
//     row-panel-major inside a band, so the band's slab of W stays resident in L2
//     while A streams;
//   * warp 0: TMA producer. Per K stage it loads a 128x128-byte A tile and a
//     tile_n x 128-byte W tile (128-byte swizzle) plus the stage's repacked UE8M0
//     block scales, all counted on one mbarrier;
//   * warp 1: one thread issues tcgen05.cp for the block scales and four
//     tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 each, one UE8M0 scale per row of
//     B per MMA, selected by the scale-factor byte id) into a TMEM fp32 accumulator;
//   * warps 2-5: epilogue. tcgen05.ld the accumulator (one TMEM lane = one row per
//     thread), apply the row scale / column scale / bias, accumulate the Q and K sums
//     of squares in fp32 and add them to sumsq[T, 2] with one atomic per row and
//     segment. V columns are stored as final bf16. Q and K columns go to a
//     tile-major workspace hand-off when the norm/RoPE pass follows, in block
//     floating point (fp16 with a power-of-two exponent per row and 16 columns: 11
//     significant bits, any range), so the bf16 rounding happens once, at the end,
//     and the stores coalesce whatever row a thread owns; else as bf16. With two accumulator stages
//     the epilogue of tile j overlaps the MMAs of tile j+1. After each tile every
//     epilogue warp fences its stores and bumps its row panel's ready counter; the
//     norm/RoPE pass, launched as a programmatic dependent of this grid, starts on a
//     panel once all its tiles are in.
//   * A carries no MX scale of its own (its only scale is the fp32 row scale), so the
//     A-side scale factors are the constant 2^0 (UE8M0 127), copied to TMEM once.
// Every mbarrier wait is bounded; a wait that runs out records its role in the
// status word and the CTA unwinds, waiting for its own copies and MMAs before it
// releases TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "fp32x2.cuh"
#include "qk_norm_rope.cuh"

namespace qkvcte {

namespace {

constexpr int kBM = 128;       // rows per tile (the MMA's M)
constexpr int kBK = 128;       // K elements (bytes of e4m3) per pipeline stage
constexpr int kThreads = 192;  // producer warp, MMA warp, 4 epilogue warps
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kFlagTestStall = 0x1u;

// W's block scales for one 128-byte K block as the GEMM copies them into TMEM: 128 rows
// (TMEM lanes) x 16 bytes (4 columns) per 128-column chunk of the N tile, lane q*32 + r,
// column c holding the four K-scales of tile column 128*chunk + 32*c + r (the scale
// layout of an M = 128 block-scaled MMA, which wants the same 32 rows in each lane
// quarter, so the image holds them four times). Stored as 8-row x 16-byte core
// matrices, the chunks of one 8-row group side by side: core matrix (group g, chunk j)
// at byte 128 * (g * SF_CHUNKS + j). Every read of a descriptor over this image stays
// inside it whichever way its two offsets are taken.
static_assert(kSfBlockBytesPerChunk == 128 * 16, "128 lanes x 4 scale columns per chunk");

// One tcgen05.cp of one K block's scales (the image above) into TMEM columns
// taddr + 4 * chunk. One copy per K block rather than one quarter-replicating copy per
// chunk: with 256-byte K stages, four 32x128b.warpx4 copies after each full-barrier
// wait cost about a tenth of the tensor pipe's time; two 128x256b copies cost nothing
// measurable.
template <int SF_CHUNKS, bool kPair>
__device__ __forceinline__ void copy_block_scales(uint32_t taddr, uint32_t sf_smem) {
  static_assert(SF_CHUNKS == 1 || SF_CHUNKS == 2, "one or two 128-column chunks");
  if constexpr (SF_CHUNKS == 2) {
    const uint64_t d = smem_desc_plain_lbo_sbo(sf_smem, 128, 256);
    if constexpr (kPair) tc_copy_128x256b_pair(taddr, d); else tc_copy_128x256b(taddr, d);
  } else {
    const uint64_t d = smem_desc_plain_lbo_sbo(sf_smem, 128, 128);
    if constexpr (kPair) tc_copy_128x128b_pair(taddr, d); else tc_copy_128x128b(taddr, d);
  }
}

template <int BN>
struct K1Cfg {
  static constexpr int SF_CHUNKS = (BN + 127) / 128;
  static constexpr int A_BYTES = kBM * kBK;
  static constexpr int B_BYTES = BN * kBK;
  static constexpr int SFB_BYTES = SF_CHUNKS * kSfBlockBytesPerChunk;
  static constexpr int SFB_COLS = SF_CHUNKS * 4;
  static constexpr int ACC_STAGES = (2 * BN + 4 + SFB_COLS <= 512) ? 2 : 1;
  static constexpr int SFA_COL = ACC_STAGES * BN;
  static constexpr int SFB_COL = SFA_COL + 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFB_BYTES;
  static constexpr int SMEM_LIMIT = 232448;          // 227 KB opt-in per block
  static constexpr int FIXED = 1024 + 512 + 256;      // alignment slack, A scales, barriers
  static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr size_t SMEM = FIXED + static_cast<size_t>(STAGES) * STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128 is a multiple of 16 up to 256");
  static_assert(SFB_COL + SFB_COLS <= 512, "TMEM columns");
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert(B_BYTES % 1024 == 0, "swizzle atoms");
};

__device__ __forceinline__ void record_failure(uint32_t* status, volatile int* abort_flag, uint32_t code) {
  atomicOr(status, code);
  *abort_flag = 1;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// Epilogue, shared by the single-CTA and CTA-pair kernels.
//
// One warp drains 32 rows (its TMEM lane quarter, one row per thread) of one
// accumulator tile. Per 16 columns: o = acc * (a_scale * w_col_scale) + bias, the
// Q/K sum of squares (a 16-column chunk never straddles a segment boundary: both
// are multiples of 16), then one 32-byte store. Q/K chunks go to the hand-off in
// block floating point (16 fp16 scaled by the chunk's power-of-two exponent,
// tile-major, so the warp's store writes 1 KB of consecutive memory); V goes to O
// as final bf16 (one full 32-byte sector per row), BSD or NBSd.
// ---------------------------------------------------------------------------
// Per-column dequant scale (a_scale * w_col_scale) and bias of the 16 columns at col0.
__device__ __forceinline__ void scale_bias16(const GemmArgs& a, float ascale, int col0, float* sc, float* bias) {
  if (a.w_col_scale != nullptr) {
    const float4* p = reinterpret_cast<const float4*>(a.w_col_scale + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v4 = __ldg(p + q);
      sc[4 * q + 0] = ascale * v4.x;
      sc[4 * q + 1] = ascale * v4.y;
      sc[4 * q + 2] = ascale * v4.z;
      sc[4 * q + 3] = ascale * v4.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) sc[j] = ascale;
  }
  if (a.bias != nullptr) {
    const uint4* p = reinterpret_cast<const uint4*>(a.bias + col0);
    const uint4 b0 = __ldg(p), b1 = __ldg(p + 1);
    const uint32_t w[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      bias[2 * j] = bf16_bits_to_float(w[j] & 0xFFFFu);
      bias[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) bias[j] = 0.0f;
  }
}

// o = acc * scale + bias for the 16 accumulator columns at TMEM address taddr.
__device__ __forceinline__ void projected16(const GemmArgs& a, uint32_t taddr, float ascale, int col0, float* v) {
  uint32_t r[16];
  tmem_ld_32x32b_x16(taddr, r);
  float sc[16], bias[16];
  scale_bias16(a, ascale, col0, sc, bias);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = fmaf(__uint_as_float(r[j]), sc[j], bias[j]);
}

__device__ __forceinline__ void store16_bf16(uint16_t* dst, const float* v, uint64_t pol) {
  uint32_t packed[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
  st_global_v8_b32_hint(dst, packed, pol);
}

// ---------------------------------------------------------------------------
// Epilogue with the per-head qk-norm of the upstream kernel: each head's slice is
// normalised by its own statistics, then rotated, while the accumulator is still in
// TMEM ([qkv_cte] "Upstream behavior": per-head RMS_NORM / LAYER_NORM and RoPE
// applied as the finished matmul result is copied out, with the dequant scale and
// the bias). Every tile holds whole heads (tile_n % d_head == 0), so nothing is
// handed to a second pass. Per Q/K head and row (one thread): pass 1 reads the
// head's columns from TMEM for sum(o) and sum(o^2) (the latter also feeds the
// segment sums); LayerNorm takes a second pass for sum((o - mean)^2); the last pass
// reads the two halves of the head together, applies (o - mean) * inv * gamma and
// the rotate-half rotation, and stores bf16. V heads are stored as projected.
// ---------------------------------------------------------------------------
template <int BN>
__device__ __forceinline__ void epilogue_drain_head(const GemmShape& g, const GemmArgs& a, uint32_t t_acc,
                                                    int block128, int row_in_block, int col_base, uint64_t pol_out,
                                                    float& ss_q, float& ss_k) {
  const int row = block128 * 128 + row_in_block;
  const bool row_ok = row < g.T;
  const int tr = row_ok ? row : g.T - 1;  // in-bounds row for table loads
  const float ascale = row_ok ? a.a_scale[row] : 0.0f;
  const int d = a.d_head;
  const int half = d >> 1;
  const float inv_d = 1.0f / static_cast<float>(d);
  ss_q = 0.0f;
  ss_k = 0.0f;
  for (int hc = 0; hc < BN; hc += d) {
    const int colh = col_base + hc;
    if (colh >= g.I) break;  // ragged last tile: whole heads only (uniform across the warp)
    const uint32_t th = t_acc + static_cast<uint32_t>(hc);
    if (colh >= a.k_end) {  // a V head
      for (int c = 0; c < d; c += 16) {
        float v[16];
        projected16(a, th + static_cast<uint32_t>(c), ascale, colh + c, v);
        if (row_ok) store16_bf16(a.O + out_index(a.nbsd, g.T, g.I, d, row, colh + c), v, pol_out);
      }
      continue;
    }
    const bool is_q = colh < a.q_end;
    float s1 = 0.0f, s2 = 0.0f;
    for (int c = 0; c < d; c += 16) {
      float v[16];
      projected16(a, th + static_cast<uint32_t>(c), ascale, colh + c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        s1 += v[j];
        s2 = fmaf(v[j], v[j], s2);
      }
    }
    if (is_q) ss_q += s2; else ss_k += s2;
    float mean = 0.0f, var = s2 * inv_d;
    if (a.head_norm == 3) {  // LayerNorm: centred second pass
      mean = s1 * inv_d;
      float s3 = 0.0f;
      for (int c = 0; c < d; c += 16) {
        float v[16];
        projected16(a, th + static_cast<uint32_t>(c), ascale, colh + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float dv = v[j] - mean;
          s3 = fmaf(dv, dv, s3);
        }
      }
      var = s3 * inv_d;
    }
    const float inv = 1.0f / sqrtf(var + a.eps);
    const uint16_t* gamma = is_q ? a.gamma_q : a.gamma_k;
    for (int c = 0; c < half; c += 16) {
      float lo[16], hi[16];
      projected16(a, th + static_cast<uint32_t>(c), ascale, colh + c, lo);
      projected16(a, th + static_cast<uint32_t>(c + half), ascale, colh + c + half, hi);
      float g_lo[16], g_hi[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 gl = __ldg(reinterpret_cast<const uint4*>(gamma + c) + q);
        const uint4 gh = __ldg(reinterpret_cast<const uint4*>(gamma + c + half) + q);
        const uint32_t wl[4] = {gl.x, gl.y, gl.z, gl.w}, wh[4] = {gh.x, gh.y, gh.z, gh.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          g_lo[8 * q + 2 * j] = bf16_bits_to_float(wl[j] & 0xFFFFu);
          g_lo[8 * q + 2 * j + 1] = bf16_bits_to_float(wl[j] >> 16);
          g_hi[8 * q + 2 * j] = bf16_bits_to_float(wh[j] & 0xFFFFu);
          g_hi[8 * q + 2 * j + 1] = bf16_bits_to_float(wh[j] >> 16);
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        lo[j] = (lo[j] - mean) * inv * g_lo[j];
        hi[j] = (hi[j] - mean) * inv * g_hi[j];
      }
      if (a.rope) {
        const float* cr = a.cos_t + static_cast<size_t>(tr) * d + c;
        const float* sr = a.sin_t + static_cast<size_t>(tr) * d + c;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 cl = __ldg(reinterpret_cast<const float4*>(cr) + q);
          const float4 ch = __ldg(reinterpret_cast<const float4*>(cr + half) + q);
          const float4 sl = __ldg(reinterpret_cast<const float4*>(sr) + q);
          const float4 sh = __ldg(reinterpret_cast<const float4*>(sr + half) + q);
          const float cl4[4] = {cl.x, cl.y, cl.z, cl.w}, ch4[4] = {ch.x, ch.y, ch.z, ch.w};
          const float sl4[4] = {sl.x, sl.y, sl.z, sl.w}, sh4[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float x = lo[4 * q + j], y = hi[4 * q + j];
            lo[4 * q + j] = x * cl4[j] - y * sl4[j];
            hi[4 * q + j] = y * ch4[j] + x * sh4[j];
          }
        }
      }
      if (row_ok) {
        store16_bf16(a.O + out_index(a.nbsd, g.T, g.I, d, row, colh + c), lo, pol_out);
        store16_bf16(a.O + out_index(a.nbsd, g.T, g.I, d, row, colh + c + half), hi, pol_out);
      }
    }
  }
}

// Block-float hand-off of 16 values: the chunk's exponent E = floor(log2 max|v|)
// (clamped; 0 for zero or non-finite maxima) and v * 2^-E in fp16, so every value
// keeps 11 significant bits relative to the chunk maximum whatever its range.
__device__ __forceinline__ void store_handoff16(const GemmArgs& a, size_t idx, const float* v) {
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
  const int field = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu);
  int e = (field == 0 || field == 255) ? 0 : field - 127;
  e = e < -126 ? -126 : (e > 126 ? 126 : e);
  const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
  uint32_t hv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 x = fmul2(make_float2(v[2 * j], v[2 * j + 1]), make_float2(down, down));
    hv[j] = pack_f16x2(x.x, x.y);
  }
  st_global_v8_b32(a.qk_val + idx * 16, hv);
  a.qk_exp[idx] = static_cast<uint8_t>(e + 127);
}

// Close one part of a Q/K head (its columns c0..c1 in this tile) for the per-head
// statistics. RMS adds the part's sum of squares to the (row, head) total. LayerNorm:
// the drain has taken the part in one pass, centred on the part's first value `shift`
// (s1 = sum(o - shift), s2 = sum((o - shift)^2)) and has handed the values over
// centred the same way, so a large common offset cannot push the deviations LayerNorm
// amplifies below the hand-off's resolution, and the part's M2 = s2 - s1^2/n loses
// only the bits of (mean - shift)^2 / variance. The part's (shift, mean, M2) go to the
// statistics; the norm/RoPE pass combines the parts with Chan et al.'s pairwise update
// (no large sums subtracted) and adds shift - mean_head back.
__device__ __forceinline__ void stats_flush(const GemmArgs& a, int row, bool row_ok, int head, int part, int c0,
                                            int c1, float s1, float s2, float shift) {
  if (!row_ok) return;
  const int heads = a.k_end / a.d_head;
  if (a.stats_kind == 2) {
    atomicAdd(&a.head_stats[static_cast<size_t>(row) * heads + head], s2);
    return;
  }
  const float n = static_cast<float>(c1 - c0);
  const float dm = s1 / n;  // mean - shift
  const float m2 = fmaxf(fmaf(-s1, dm, s2), 0.0f);
  reinterpret_cast<float4*>(a.head_stats)[(static_cast<size_t>(row) * heads + head) * a.stat_parts + part] =
      make_float4(shift, shift + dm, m2, 0.0f);
}

// kStats: 0 none, 2 per-head RMS statistics, 3 per-head LayerNorm statistics.
template <int BN, int kStats>
__device__ __forceinline__ void epilogue_drain_plain(const GemmShape& g, const GemmArgs& a, uint32_t t_acc,
                                                     int block128, int row_in_block, int col_base, uint64_t pol_out,
                                                     float& ss_q, float& ss_k) {
  const int row = block128 * 128 + row_in_block;
  const bool row_ok = row < g.T;
  const float ascale = row_ok ? a.a_scale[row] : 0.0f;
  const int qk_chunks = a.k_end >> 4;
  const size_t qk_row_idx = static_cast<size_t>(block128) * qk_chunks * 128 + row_in_block;
  ss_q = 0.0f;
  ss_k = 0.0f;
  int st_head = -1, st_c0 = 0, st_c1 = 0;  // the open head part (kStats)
  float st_s1 = 0.0f, st_s2 = 0.0f, st_shift = 0.0f;
#pragma unroll
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t r[32];
    const uint32_t taddr = t_acc + static_cast<uint32_t>(c0);
    if (c0 + 32 <= BN)
      tmem_ld_32x32b_x32(taddr, r);
    else
      tmem_ld_32x32b_x16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (c0 + 16 * h >= BN) break;
      const int col0 = col_base + c0 + 16 * h;
      if (col0 >= g.I) break;  // ragged last N tile (uniform across the warp)
      float sc[16];
      if (a.w_col_scale != nullptr) {
        const float4* p = reinterpret_cast<const float4*>(a.w_col_scale + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v4 = __ldg(p + q);
          sc[4 * q + 0] = ascale * v4.x;
          sc[4 * q + 1] = ascale * v4.y;
          sc[4 * q + 2] = ascale * v4.z;
          sc[4 * q + 3] = ascale * v4.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) sc[j] = ascale;
      }
      float bias[16];
      if (a.bias != nullptr) {
        const uint4* p = reinterpret_cast<const uint4*>(a.bias + col0);
        const uint4 b0 = __ldg(p), b1 = __ldg(p + 1);
        const uint32_t w[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          bias[2 * j] = bf16_bits_to_float(w[j] & 0xFFFFu);
          bias[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) bias[j] = 0.0f;
      }
      float v[16];
      float2 sq2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 o = ffma2(make_float2(__uint_as_float(r[16 * h + 2 * j]), __uint_as_float(r[16 * h + 2 * j + 1])),
                               make_float2(sc[2 * j], sc[2 * j + 1]), make_float2(bias[2 * j], bias[2 * j + 1]));
        v[2 * j] = o.x;
        v[2 * j + 1] = o.y;
        sq2 = ffma2(o, o, sq2);
      }
      const float sq = sq2.x + sq2.y;
      if (col0 < a.q_end) ss_q += sq; else if (col0 < a.k_end) ss_k += sq;
      if constexpr (kStats != 0) {
        if (col0 < a.k_end) {
          const int hh = col0 / a.d_head;  // uniform across the warp
          if (hh != st_head) {
            if (st_head >= 0)
              stats_flush(a, row, row_ok, st_head, col_base / BN - (st_head * a.d_head) / BN, st_c0, st_c1, st_s1,
                          st_s2, st_shift);
            st_head = hh;
            st_c0 = col0;
            st_s1 = st_s2 = 0.0f;
            if constexpr (kStats == 3) st_shift = v[0];
          }
          if constexpr (kStats == 3) {  // LayerNorm: centred on the part's first value
            float2 s1 = make_float2(0.0f, 0.0f), s2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 dv = make_float2(v[2 * j] - st_shift, v[2 * j + 1] - st_shift);
              v[2 * j] = dv.x;
              v[2 * j + 1] = dv.y;
              s1 = make_float2(s1.x + dv.x, s1.y + dv.y);
              s2 = ffma2(dv, dv, s2);
            }
            st_s1 += s1.x + s1.y;
            st_s2 += s2.x + s2.y;
          } else {
            st_s2 += sq;
          }
          st_c1 = col0 + 16;
        }
      }
      if (a.qk_val != nullptr && col0 < a.k_end) {
        // Q/K columns the norm/RoPE pass will finish (centred for the LayerNorm statistics)
        store_handoff16(a, qk_row_idx + static_cast<size_t>(col0 >> 4) * 128, v);
      } else if (row_ok) {
        uint32_t packed[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) packed[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        // final values nothing here reads again: first out of L2
        st_global_v8_b32_hint(a.O + out_index(a.nbsd, g.T, g.I, a.d_head, row, col0), packed, pol_out);
      }
    }
  }
  if constexpr (kStats != 0) {
    if (st_head >= 0)
      stats_flush(a, row, row_ok, st_head, col_base / BN - (st_head * a.d_head) / BN, st_c0, st_c1, st_s1, st_s2,
                  st_shift);
  }
}

// Epilogue kinds, each a separate instantiation of the kernels (the per-head ones need
// more registers per thread, which would otherwise leave no room on an SM
// sub-partition for a norm/RoPE warp beside the GEMM's two warps there):
//   kEpiPlain : Q/K to the norm/RoPE hand-off (or as projected), V to O
//   kEpiHead  : the per-head norm and RoPE finished here (tiles hold whole heads)
//   kEpiStatsRms / kEpiStatsLayer : as plain, plus the per-head statistics (RMS: sums of
//               squares; LayerNorm: each part's mean and centred M2, values handed over
//               centred) the norm/RoPE pass finishes from
constexpr int kEpiPlain = 0, kEpiHead = 1, kEpiStatsRms = 2, kEpiStatsLayer = 3;

template <int BN, int kEpi>
__device__ __forceinline__ void epilogue_drain(const GemmShape& g, const GemmArgs& a, uint32_t t_acc, int block128,
                                               int row_in_block, int col_base, uint64_t pol_out, float& ss_q,
                                               float& ss_k) {
  if constexpr (kEpi == kEpiHead)
    epilogue_drain_head<BN>(g, a, t_acc, block128, row_in_block, col_base, pol_out, ss_q, ss_k);
  else
    epilogue_drain_plain<BN, kEpi == kEpiStatsRms ? 2 : (kEpi == kEpiStatsLayer ? 3 : 0)>(
        g, a, t_acc, block128, row_in_block, col_base, pol_out, ss_q, ss_k);
}

// After the accumulator is released: add this warp's rows' sums of squares and, for
// a tile holding Q/K columns, publish its 32 rows on the 128-row block's counter
// once its stores and sums are visible.
template <int BN>
__device__ __forceinline__ void epilogue_publish(const GemmShape& g, const GemmArgs& a, int block128,
                                                 int row_in_block, int col_base, bool qk_tile, float ss_q,
                                                 float ss_k, int lane) {
  const int row = block128 * 128 + row_in_block;
  if (row < g.T && a.sumsq != nullptr) {
    if (col_base < a.q_end) atomicAdd(&a.sumsq[2 * static_cast<size_t>(row)], ss_q);
    if (col_base + BN > a.q_end && col_base < a.k_end) atomicAdd(&a.sumsq[2 * static_cast<size_t>(row) + 1], ss_k);
  }
  if (qk_tile) {
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(a.ready + block128, 1u);
  }
}

// Record in the per-SM table which sub-partitions this CTA's TMA-load and MMA-issue
// warps occupy (0 when the CTA is done). The norm/RoPE pass, running beside the GEMM,
// keeps its warps off those two while the CTA runs: sharing a scheduler with them slows
// the GEMM three times as much as running on the other two. Only a hint: nothing waits
// for it to be exact. Called by thread 0 after prep (which clears the table).
__device__ __forceinline__ void publish_busy(const GemmArgs& a, uint32_t mask) {
  if (threadIdx.x != 0 || a.sm_busy == nullptr) return;
  a.sm_busy[nrp::sm_id() & (kSmTable - 1)] = mask;
  __threadfence();
}

template <int BN, int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_mxf8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                         const GemmShape g, const GemmArgs a) {
  using C = K1Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::STAGES * C::A_BYTES;
  uint8_t* sSFB = sB + C::STAGES * C::B_BYTES;
  uint8_t* sSFA = sSFB + C::STAGES * C::SFB_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFA + 512);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* busy_slot = tmem_slot + 2;  // [2]: sub-partition bits of the load and MMA warps

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&tfull[s]), 1);
      mbar_init(smem_u32(&tempty[s]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp >= 2) {
    // A-side block scales: UE8M0 127 (= 1.0) for every row and K block.
    reinterpret_cast<uint32_t*>(sSFA)[threadIdx.x - 64] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
  }
  if (warp <= 1 && lane == 0) busy_slot[warp] = 1u << (nrp::warp_slot() & 3);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The set-up above overlaps the prep kernel (a programmatic dependency): everything
  // below reads its scale image or its cleared sums, counters and stamps.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  publish_busy(a, busy_slot[0] | busy_slot[1]);
  // Every CTA of this persistent grid is resident: let the norm/RoPE pass launch now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) atomicMin(&a.stamps[0], globaltimer_ns());

  const int num_tiles = g.m_tiles * g.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      // A's row panel is read by every CTA working on the band at about the same time:
      // evict-first let it go before the last reader came (1.70 GB of DRAM reads per
      // 480p launch instead of 0.64 GB) and cost ~1 % of the GEMM's time
      const uint64_t pol_stream = policy_evict_normal();
      const uint64_t pol_keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = (a.flags & kFlagTestStall) == 0;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int m_blk, n_blk;
        tile_coords(g, tile, m_blk, n_blk);
        for (int kb = 0; kb < g.k_stages; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            record_failure(a.status, abort_flag, kErrProducerEmptyWait);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          tma_load_2d(smem_u32(sA + stage * C::A_BYTES), &tmA, kb * kBK, m_blk * kBM, fb, pol_stream);
          tma_load_2d(smem_u32(sB + stage * C::B_BYTES), &tmW, kb * kBK, n_blk * BN, fb, pol_keep);
          bulk_load(smem_u32(sSFB + stage * C::SFB_BYTES),
                    a.sf_packed + (static_cast<size_t>(n_blk) * g.k_stages + kb) * C::SFB_BYTES,
                    C::SFB_BYTES, fb);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Do not leave while our own copies may still be landing in shared memory:
      // wait for the (at most STAGES) most recent loads.
      const int pending = issued < C::STAGES ? issued : C::STAGES;
      int s = stage;
      uint32_t ph = phase;
      for (int i = 0; i < pending; ++i) {
        if (s == 0) {
          s = C::STAGES - 1;
          ph ^= 1u;
        } else {
          --s;
        }
        if (!mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, kWaitLimitNs)) {
          record_failure(a.status, abort_flag, kErrDrainWait);
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = idesc_mxf8_e4m3(kBM, BN);
      const uint32_t sfa_t = tmem_base + C::SFA_COL;
      const uint32_t sfb_t = tmem_base + C::SFB_COL;
      tc_copy_32x128b_x4(sfa_t, smem_desc_plain(smem_u32(sSFA)));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          record_failure(a.status, abort_flag, kErrMmaTmemEmptyWait);
          break;
        }
        tc_fence_after();
        const uint32_t d_t = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < g.k_stages; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            record_failure(a.status, abort_flag, kErrMmaFullWait);
            ok = false;
            break;
          }
          tc_fence_after();
          copy_block_scales<C::SF_CHUNKS, false>(sfb_t, smem_u32(sSFB + stage * C::SFB_BYTES));
          const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * C::A_BYTES));
          const uint64_t bd = smem_desc_sw128(smem_u32(sB + stage * C::B_BYTES));
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k) {
            // +32 bytes along K inside the swizzle atom = +2 in the 16-byte address field
            mma_mxf8(d_t, ad + 2 * k, bd + 2 * k, idesc_with_sf_id(idesc, 0, k), sfa_t, sfb_t,
                     (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[acc]));
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every tcgen05 operation issued above completes before TMEM is released.
      tc_commit(smem_u32(drain));
      if (!mbar_wait_bounded(smem_u32(drain), 0, nullptr, kWaitLimitNs))
        record_failure(a.status, abort_flag, kErrDrainWait);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const uint64_t pol_out = policy_evict_first();
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_block = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int m_blk, n_blk;
      tile_coords(g, tile, m_blk, n_blk);
      bool ok = mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) record_failure(a.status, abort_flag, kErrEpilogueTmemFullWait);
        break;
      }
      tc_fence_after();
      float ss_q, ss_k;
      epilogue_drain<BN, kEpi>(g, a, t_lane + static_cast<uint32_t>(acc * BN), m_blk, row_in_block, n_blk * BN, pol_out,
                         ss_q, ss_k);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
      epilogue_publish<BN>(g, a, m_blk, row_in_block, n_blk * BN, n_blk < g.n_qk_tiles, ss_q, ss_k, lane);
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    atomicMax(&a.stamps[1], globaltimer_ns());
    publish_busy(a, 0u);  // this SM's sub-partitions are free for the norm/RoPE pass
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant: tiles of 256 rows x BN columns computed by a cluster of two CTAs
// with M = 256 MMAs (tcgen05 cta_group::2). Each CTA loads its 128 rows of A, its
// half of the W tile (BN/2 rows) and the scales of all BN columns; all loads count on
// the leader's (rank 0) barrier. The leader's MMA thread copies the scales into both
// CTAs' TMEM and issues the MMAs for both; commits arrive on both CTAs' barriers.
// Each CTA's epilogue drains its own TMEM rows and releases the accumulator on the
// leader's barrier. Per SM this halves the W bytes staged and read from shared
// memory and the scale-factor copies per FLOP.
// ---------------------------------------------------------------------------
// Stage depth. A ring stage holds two 128-byte K blocks (K = 256 per stage: eight MMAs
// and two scale-factor copies per barrier wait). The tensor pipe runs the MMAs of
// a continuously fed issue stream at the full rate, but every stage boundary (the
// wait for the stage's operands and the copy of its block scales into TMEM, which is
// ordered against the MMAs in flight) opens a bubble. Measured on GB300 with the
// 480p tile stream and real TMA traffic, M = 256, N = 240: 1.50 ms per launch with
// 128-byte stages against 1.20 ms with 256-byte stages (1.06 ms with no stage
// boundaries at all), so the boundaries are made half as frequent. A K length that
// is an odd number of 128-byte blocks ends on a half stage.
//
// Ring depth: as many stages as fit (three at tile_n 192 to 256: 192 to 216 KB). Measured at
// the Wan 480p shape with the norm/RoPE pass overlapped: 1.616 ms per step with three
// 256-byte stages against 2.094 ms with two (which left more L1 for the pass beside
// the GEMM, but cannot cover the load latency).
// The CTA-pair form's tile sequence: whole waves first, pair p taking tiles p, p + P,
// p + 2P, ... (P pairs), then the last kClaimedWaves waves' worth from a counter, so
// that pairs slowed by other work on their SMs (the norm/RoPE pass beside the GEMM)
// take fewer of them instead of finishing last. Claiming every tile cost about 4 % of
// the GEMM's cycles at the Wan 480p shape; claiming the last six waves only keeps that
// to the tail. Once every pair has claimed a tile the norm/RoPE pass stops holding its
// warps back (the counter is its signal), so that it ends with the now even tail.
//
// A claimed tile is claimed by the leader's load thread one tile ahead (the atomic's
// latency hides behind the current tile's loads) and published to both CTAs through a
// ring of kTileRing slots with one mbarrier each (one arrival per publication; -1 ends
// the sequence). A slot is rewritten kTileRing tiles later; by then every reader has
// read it: the load thread publishes tile s only after it has loaded tile s - 1, which
// needs the MMA issuer to have finished tile s - 1 - STAGES, which needs the epilogue to
// have drained tile s - 1 - STAGES - ACC_STAGES.
constexpr int kTileRing = 8;


struct PairTileRing {
  int* ids;        // [kTileRing]
  uint64_t* full;  // [kTileRing]

  // Leader's load thread: claimed tile (or -1) number `d` of the pair (counted from
  // the pair's first claimed tile), to both CTAs.
  __device__ __forceinline__ void publish(int d, int tile, uint32_t peer) const {
    const int r = d & (kTileRing - 1);
    ids[r] = tile;
    st_shared_cluster_s32(mapa_shared(smem_u32(&ids[r]), peer), tile);
    mbar_arrive(smem_u32(&full[r]));
    mbar_arrive_cluster(mapa_shared(smem_u32(&full[r]), peer));
  }

  // Any reader: claimed tile number `d` (false if the bounded wait ran out, or if the
  // slot holds neither a tile below num_tiles nor -1).
  __device__ __forceinline__ bool fetch(int d, int& tile, const volatile int* abort, int num_tiles) const {
    const int r = d & (kTileRing - 1);
    if (!mbar_wait_bounded_cluster(smem_u32(&full[r]), static_cast<uint32_t>(d / kTileRing) & 1u, abort,
                                   kWaitLimitNs))
      return false;
    tile = ids[r];
    return tile >= -1 && tile < num_tiles;
  }
};

template <int BN>
struct K1PairCfg {
  static constexpr int HALF_N = BN / 2;
  static constexpr int SF_CHUNKS = (BN + 127) / 128;
  static constexpr int KW = 2;                           // 128-byte K blocks per stage
  static constexpr int A_HALF = kBM * kBK;               // one 128-byte K block of A
  static constexpr int B_HALF = HALF_N * kBK;            // ... of this CTA's half of W
  static constexpr int SF_HALF = SF_CHUNKS * kSfBlockBytesPerChunk;  // ... of the tile's scales
  static constexpr int A_BYTES = KW * A_HALF;
  static constexpr int B_BYTES = KW * B_HALF;
  static constexpr int SFB_BYTES = KW * SF_HALF;
  static constexpr int SFB_COLS = KW * SF_CHUNKS * 4;
  static constexpr int ACC_STAGES = (2 * BN + 4 + SFB_COLS <= 512) ? 2 : 1;
  static constexpr int SFA_COL = ACC_STAGES * BN;
  static constexpr int SFB_COL = SFA_COL + 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFB_BYTES;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int FIXED = 1024 + 512 + 256;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr size_t SMEM = FIXED + static_cast<size_t>(STAGES) * STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "pair MMA N");
  static_assert(HALF_N % 8 == 0, "W half tile in whole 8-row swizzle atoms");
  static_assert(B_HALF % 1024 == 0 && A_HALF % 1024 == 0, "K blocks on swizzle-atom boundaries");
  static_assert(SFB_COL + SFB_COLS <= 512, "TMEM columns");
  static_assert(STAGES >= 2, "pipeline depth");
};

// ---------------------------------------------------------------------------
// Norm/RoPE tasks run by the epilogue warps of the fused kernel (the work of K2,
// qk_norm_rope.cuh). A warp claims tasks from a grid-wide counter in panel order and
// runs one only once K1's counter shows its panel complete; it does this only while
// its next accumulator is not ready, so draining a tile always comes first and the
// MMAs never wait for norm work (a task is a few microseconds, a tile's MMAs about
// thirteen). When its tiles are done the warp finishes the tasks left. Used on
// request (QKV_CTE_FLAG_NORM_IN_GEMM): the norm work slows the GEMM as much from
// inside it as from a kernel of its own beside it, and adds a tail.
// ---------------------------------------------------------------------------
// Heads per fused task: short, so a drain is never held up long, yet long enough to
// spread a row's cos/sin loads over several heads (measured at the 480p shape: 4 heads
// 2.04 ms, 10 heads 1.93 ms, 20 heads 2.04 ms per call).
constexpr int kFusedHeadGroup = 10;

struct FusedWork {
  long long pending = -1;  // claimed, not yet run
  bool done = false;       // the counter is exhausted
  bool started = false;
};

__device__ __forceinline__ void fused_claim(const NormRopeArgs& nr, long long n_tasks, FusedWork& w) {
  uint32_t t = 0;
  if ((threadIdx.x & 31) == 0) t = atomicAdd(nr.task_next, 1u);
  t = __shfl_sync(0xffffffffu, t, 0);
  if (static_cast<long long>(t) >= n_tasks) {
    w.done = true;
    w.pending = -1;
  } else {
    w.pending = static_cast<long long>(t);
  }
}

// Run the pending task if its panel is complete; returns whether it ran.
__device__ __forceinline__ bool fused_try(const NormRopeArgs& nr, FusedWork& w, uint64_t once) {
  const int panel = nrp::task_panel(nr, w.pending, kFusedHeadGroup);
  int ready = 0;
  if ((threadIdx.x & 31) == 0) ready = nrp::ld_acquire(nr.ready + panel) >= nr.ready_target ? 1 : 0;
  ready = __shfl_sync(0xffffffffu, ready, 0);
  if (!ready) return false;
  if (!w.started) {
    w.started = true;
    if ((threadIdx.x & 31) == 0) atomicMin(&nr.stamps[0], globaltimer_ns());
  }
  nrp::run_task<false>(nr, w.pending, kFusedHeadGroup, once);
  w.pending = -1;
  return true;
}

// Lane 0's value of `v`, for a decision the whole warp takes together: the task
// helpers use full-warp shuffles, so no lane may leave a loop the others stay in (a
// lane that read the abort flag before lane 0 had set it would otherwise wait in a
// shuffle for lanes that have left).
__device__ __forceinline__ bool warp_uniform(bool v) {
  return __shfl_sync(0xffffffffu, v ? 1 : 0, 0) != 0;
}

// Wait (bounded) for the accumulator barrier, running norm tasks meanwhile.
__device__ __forceinline__ bool fused_wait_acc(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               const NormRopeArgs& nr, long long n_tasks, FusedWork& w,
                                               uint64_t once) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    int ready = 0;
    if ((threadIdx.x & 31) == 0) ready = mbar_test_wait(bar, parity) ? 1 : 0;
    ready = __shfl_sync(0xffffffffu, ready, 0);
    if (ready) return mbar_wait_bounded(bar, parity, abort_flag, kWaitLimitNs);  // completes at once, per lane
    if (warp_uniform(*abort_flag != 0)) return false;
    bool ran = false;
    if (!w.done) {
      if (w.pending < 0) fused_claim(nr, n_tasks, w);
      if (w.pending >= 0) ran = fused_try(nr, w, once);
    }
    if (!ran) {
      if (warp_uniform(globaltimer_ns() - t0 > kWaitLimitNs)) return false;
      __nanosleep(64);
    }
  }
}

// After the warp's last tile: the tasks left (each panel wait bounded).
__device__ __forceinline__ void fused_finish(const NormRopeArgs& nr, long long n_tasks, FusedWork& w,
                                             volatile int* abort_flag, uint32_t* status, uint64_t once) {
  uint64_t t0 = globaltimer_ns();
  while (!w.done && !warp_uniform(*abort_flag != 0)) {
    if (w.pending < 0) {
      fused_claim(nr, n_tasks, w);
      if (w.done) break;
    }
    if (fused_try(nr, w, once)) {
      t0 = globaltimer_ns();
      continue;
    }
    if (warp_uniform(globaltimer_ns() - t0 > kWaitLimitNs)) {
      if ((threadIdx.x & 31) == 0) atomicOr(status, kErrNormReadyWait);
      break;
    }
    __nanosleep(256);
  }
  if (w.started && (threadIdx.x & 31) == 0) atomicMax(&nr.stamps[1], globaltimer_ns());
}

template <int BN, int kEpi, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_mxf8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                              const __grid_constant__ CUtensorMap tmSF, const GemmShape g, const GemmArgs a,
                              const __grid_constant__ NormRopeArgs nr) {
  using C = K1PairCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::STAGES * C::A_BYTES;
  uint8_t* sSFB = sB + C::STAGES * C::B_BYTES;
  uint8_t* sSFA = sSFB + C::STAGES * C::SFB_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFA + 512);  // used in the leader
  uint64_t* empty = full + C::STAGES;                         // both
  uint64_t* tfull = empty + C::STAGES;                        // both
  uint64_t* tempty = tfull + 2;                               // leader: 4 warps x 2 CTAs
  uint64_t* drain = tempty + 2;                               // leader
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* busy_slot = tmem_slot + 2;  // [2]: sub-partition bits of the load and MMA warps
  const PairTileRing ring{reinterpret_cast<int*>(busy_slot + 2), reinterpret_cast<uint64_t*>(busy_slot + 2 + kTileRing)};
  static_assert((2 * C::STAGES + 5) * 8 + 16 + kTileRing * (4 + 8) <= 256, "barrier area");
  static_assert(C::STAGES + C::ACC_STAGES + 1 < kTileRing, "a tile-id slot is reread only after every reader");
  const PairSchedule sched(g.m_tiles * g.n_tiles, static_cast<int>(blockIdx.x >> 1), static_cast<int>(gridDim.x >> 1));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // rank in the pair
  constexpr uint32_t lead = 0u;             // cluster rank of the pair's leader
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&tfull[s]), 1);
      mbar_init(smem_u32(&tempty[s]), 8);
    }
    mbar_init(smem_u32(drain), 1);
    for (int r = 0; r < kTileRing; ++r) mbar_init(smem_u32(&ring.full[r]), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmSF);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp >= 2) {
    reinterpret_cast<uint32_t*>(sSFA)[threadIdx.x - 64] = 0x7F7F7F7Fu;  // A-side scales: 2^0
    fence_proxy_async_smem();
  }
  // the load warp's sub-partition, and the MMA issuer's (the leader's MMA warp only)
  if (warp <= 1 && lane == 0) busy_slot[warp] = (warp == 0 || leader) ? 1u << (nrp::warp_slot() & 3) : 0u;
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers, TMEM and A-side scales of both CTAs are ready
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // prep complete (as above)
  publish_busy(a, busy_slot[0] | busy_slot[1]);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) atomicMin(&a.stamps[0], globaltimer_ns());

  const int num_tiles = g.m_tiles * g.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      // A's row panel is read by every CTA working on the band at about the same time:
      // evict-first let it go before the last reader came (1.70 GB of DRAM reads per
      // 480p launch instead of 0.64 GB) and cost ~1 % of the GEMM's time
      const uint64_t pol_stream = policy_evict_normal();
      const uint64_t pol_keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      // test hook: hand out the first tile, then load nothing (every wait downstream runs out)
      const bool stall = (a.flags & kFlagTestStall) != 0;
      bool ok = true;
      const int n_stages = (g.k_stages + C::KW - 1) / C::KW;
      uint32_t claimed = (leader && sched.n_static == 0) ? atomicAdd(a.tile_next, 1u) : 0u;
      for (int seq = 0; ok; ++seq) {
        int tile;
        if (sched.is_static(seq)) {
          tile = sched.static_tile(seq);
          if (leader && seq + 1 == sched.n_static) claimed = atomicAdd(a.tile_next, 1u);  // the first claimed
        } else if (leader) {
          const long long t = static_cast<long long>(sched.dyn_base) + claimed;
          tile = t < num_tiles ? static_cast<int>(t) : -1;
          ring.publish(seq - sched.n_static, tile, lead ^ 1u);
          if (tile >= 0) claimed = atomicAdd(a.tile_next, 1u);
        } else if (!ring.fetch(seq - sched.n_static, tile, abort_flag, num_tiles)) {
          record_failure(a.status, abort_flag, kErrTileIdWait);
          break;
        }
        if (tile < 0 || stall) break;
        int m_blk, n_blk;
        tile_coords(g, tile, m_blk, n_blk);
        for (int ks = 0; ks < n_stages; ++ks) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, kWaitLimitNs)) {
            record_failure(a.status, abort_flag, kErrProducerEmptyWait);
            ok = false;
            break;
          }
          const int kb0 = ks * C::KW;  // first 128-byte K block of the stage
          const int halves = g.k_stages - kb0 < C::KW ? g.k_stages - kb0 : C::KW;
          const uint32_t fb_local = smem_u32(&full[stage]);
          if (leader)
            mbar_arrive_expect_tx(fb_local, 2u * static_cast<uint32_t>(halves) * (C::A_HALF + C::B_HALF + C::SF_HALF));
          const uint32_t fb = mapa_shared(fb_local, lead);
          for (int h = 0; h < halves; ++h) {
            const int kb = kb0 + h;
            tma_load_2d_pair(smem_u32(sA + stage * C::A_BYTES + h * C::A_HALF), &tmA, kb * kBK,
                             m_blk * 2 * kBM + static_cast<int>(rank) * kBM, fb, pol_stream);
            tma_load_2d_pair(smem_u32(sB + stage * C::B_BYTES + h * C::B_HALF), &tmW, kb * kBK,
                             n_blk * BN + static_cast<int>(rank) * C::HALF_N, fb, pol_keep);
            tma_load_2d_pair(smem_u32(sSFB + stage * C::SFB_BYTES + h * C::SF_HALF), &tmSF, 0,
                             (n_blk * g.k_stages + kb) * (C::SF_HALF / kSfRowBytes), fb, pol_keep);
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // The leader's barrier counts both CTAs' copies: before leaving, the leader
      // waits for the most recent ones to land (the peer's too).
      if (leader) {
        const int pending = issued < C::STAGES ? issued : C::STAGES;
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < pending; ++i) {
          if (s == 0) {
            s = C::STAGES - 1;
            ph ^= 1u;
          } else {
            --s;
          }
          if (!mbar_wait_bounded(smem_u32(&full[s]), ph, nullptr, kWaitLimitNs)) {
            record_failure(a.status, abort_flag, kErrDrainWait);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader only, for both CTAs) ----------------
      const uint32_t idesc = idesc_mxf8_e4m3(2 * kBM, BN);
      const uint32_t sfa_t = tmem_base + C::SFA_COL;
      const uint32_t sfb_t = tmem_base + C::SFB_COL;
      const int n_stages = (g.k_stages + C::KW - 1) / C::KW;
      tc_copy_32x128b_x4_pair(sfa_t, smem_desc_plain(smem_u32(sSFA)));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        int tile;
        if (sched.is_static(seq)) {
          tile = sched.static_tile(seq);
        } else if (!ring.fetch(seq - sched.n_static, tile, abort_flag, num_tiles)) {
          record_failure(a.status, abort_flag, kErrTileIdWait);
          break;
        }
        if (tile < 0) break;
        if (!mbar_wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          record_failure(a.status, abort_flag, kErrMmaTmemEmptyWait);
          break;
        }
        tc_fence_after();
        const uint32_t d_t = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int ks = 0; ks < n_stages; ++ks) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
            record_failure(a.status, abort_flag, kErrMmaFullWait);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_smem = smem_u32(sSFB + stage * C::SFB_BYTES);
          const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * C::A_BYTES));
          const uint64_t bd = smem_desc_sw128(smem_u32(sB + stage * C::B_BYTES));
          // The block scales of the stage's K blocks first, then their MMAs back to back,
          // as straight-line code: the tensor pipe idles whenever the issue stream stalls.
          if (g.k_stages - ks * C::KW >= C::KW) {
#pragma unroll
            for (int h = 0; h < C::KW; ++h)
              copy_block_scales<C::SF_CHUNKS, true>(sfb_t + 4 * h * C::SF_CHUNKS, sf_smem + h * C::SF_HALF);
#pragma unroll
            for (int h = 0; h < C::KW; ++h)
#pragma unroll
              for (int k = 0; k < kBK / 32; ++k)
                mma_mxf8_pair(d_t, ad + (h * C::A_HALF >> 4) + 2 * k, bd + (h * C::B_HALF >> 4) + 2 * k,
                              idesc_with_sf_id(idesc, 0, k), sfa_t, sfb_t + 4 * h * C::SF_CHUNKS,
                              (ks | h | k) != 0 ? 1u : 0u);
          } else {  // the last stage of an odd number of 128-byte K blocks: one block
            copy_block_scales<C::SF_CHUNKS, true>(sfb_t, sf_smem);
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
              mma_mxf8_pair(d_t, ad + 2 * k, bd + 2 * k, idesc_with_sf_id(idesc, 0, k), sfa_t, sfb_t,
                            (ks | k) != 0 ? 1u : 0u);
          }
          // the stage is free once every CTA that wrote into it sees this pair done
          tc_commit_pair_multicast(smem_u32(&empty[stage]), static_cast<uint16_t>(0x3u << lead));
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(smem_u32(&tfull[acc]), static_cast<uint16_t>(0x3u << lead));
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      tc_commit_pair(smem_u32(drain));
      if (!mbar_wait_bounded(smem_u32(drain), 0, nullptr, kWaitLimitNs))
        record_failure(a.status, abort_flag, kErrDrainWait);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5, both CTAs) ----------------
    const uint64_t pol_out = policy_evict_first();
    const int quarter = warp & 3;
    const int row_in_block = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    FusedWork fw;
    const long long n_tasks = kFused ? nrp::task_count(nr, kFusedHeadGroup) : 0;
    const uint64_t once = kFused ? nrp::evict_first_policy() : 0;
    for (int seq = 0;; ++seq) {
      int tile = -1, got = 1;
      if (sched.is_static(seq)) {
        tile = sched.static_tile(seq);
      } else {
        if (lane == 0) got = ring.fetch(seq - sched.n_static, tile, abort_flag, num_tiles) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        tile = __shfl_sync(0xffffffffu, tile, 0);
      }
      if (!got) {
        if (lane == 0) record_failure(a.status, abort_flag, kErrTileIdWait);
        break;
      }
      if (tile < 0) break;
      int m_blk, n_blk;
      tile_coords(g, tile, m_blk, n_blk);
      bool ok;
      if constexpr (kFused)
        ok = fused_wait_acc(smem_u32(&tfull[acc]), acc_phase, abort_flag, nr, n_tasks, fw, once);
      else
        ok = mbar_wait_bounded(smem_u32(&tfull[acc]), acc_phase, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) record_failure(a.status, abort_flag, kErrEpilogueTmemFullWait);
        break;
      }
      tc_fence_after();
      const int block128 = m_blk * 2 + static_cast<int>(rank);
      // A 128-row half wholly past T (T mod 256 in (0, 128]) has nothing to store.
      const bool live = block128 * kBM < g.T;
      float ss_q = 0.0f, ss_k = 0.0f;
      if (live)
        epilogue_drain<BN, kEpi>(g, a, t_lane + static_cast<uint32_t>(acc * BN), block128, row_in_block, n_blk * BN,
                           pol_out, ss_q, ss_k);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), lead));
      if (live)
        epilogue_publish<BN>(g, a, block128, row_in_block, n_blk * BN, n_blk < g.n_qk_tiles, ss_q, ss_k, lane);
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (kFused) fused_finish(nr, n_tasks, fw, abort_flag, a.status, once);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no MMA, copy or remote arrive still targets either CTA
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    atomicMax(&a.stamps[1], globaltimer_ns());
    publish_busy(a, 0u);  // this SM's sub-partitions are free for the norm/RoPE pass
  }
}

template <int BN, int kEpi>
cudaError_t launch_gemm_t(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                          const GemmArgs& a, cudaStream_t s, int num_sms) {
  using C = K1Cfg<BN>;
  auto kern = qkv_gemm_mxf8_kernel<BN, kEpi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  const int tiles = g.m_tiles * g.n_tiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  // a programmatic dependent of the prep kernel: the prologue overlaps it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmW, g, a);
}

// The launch of the CTA-pair GEMM: clusters of one pair, one pair per two SMs.
template <int BN, int kEpi, bool kFused>
cudaError_t launch_gemm_pair_t(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                               const CUtensorMap& tmSF, const GemmArgs& a, const NormRopeArgs& nr, cudaStream_t s,
                               int num_sms) {
  using C = K1PairCfg<BN>;
  auto kern = qkv_gemm_mxf8_pair_kernel<BN, kEpi, kFused>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  const int tiles = g.m_tiles * g.n_tiles;
  const int pairs = num_sms / 2;
  const int grid = 2 * (tiles < pairs ? tiles : pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the prep kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmW, tmSF, g, a, nr);
}

}  // namespace

}  // namespace qkvcte
