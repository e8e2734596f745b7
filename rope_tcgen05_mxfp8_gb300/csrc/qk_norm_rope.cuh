// The norm/RoPE work on the Q/K hand-off, shared by the standalone pass (K2,
// qk_norm_rope.cu) and the GEMM whose epilogue warps run it between tiles
// (qkv_gemm_mxf8_fused.cu).
//
// Follows the `qkv_cte` kernel reference page, "Design" 1 (steps b and c: finish
// inv_rms = 1/sqrt(sum(o^2) / (n_heads * d_head) + eps) per token and segment, re-read
// each token's Q and K, multiply by the segment-wide gamma) and "Design" 2 (RoPE in
// the same pass, inv_rms folded into it, out = y*cos + [-y_hi, y_lo]*sin with
// position-only cos/sin broadcast over the heads).
//
// On one GPU every head is local, so the page's cross-rank AllReduce of the sums is
// the identity: K1 already summed over every column tile of the row. K1 hands Q/K over
// in block floating point (fp16 with a power-of-two exponent per row and 16 columns,
// in a tile-major workspace buffer), so the result is rounded to bf16 once, here.
//
// Work is cut into warp tasks: task_rows(d) consecutive rows x the whole low half of
// a group of heads. Lane (r, q) owns row r and the 16-column chunk q of the low half
// (plus its partner d/2 away, the rotate-half pair), so the lanes of one row store
// whole 128-byte lines of O (d = 128) and read the tile-major hand-off in 256-byte
// runs; four heads' loads are in flight at once, and each lane keeps its cos/sin chunk
// and inv_rms in registers across the group's heads. A task may run once K1's counter
// for its 128-row panel shows every Q/K tile published; tasks are numbered panel by
// panel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fp32x2.cuh"
#include "internal.h"

namespace qkvcte {
namespace nrp {

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kHeadBatch = 4;  // default: heads whose hand-off loads are in flight together

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The SM this thread runs on, and its warp's hardware slot there: the slot's low two
// bits name the SM sub-partition (the warp scheduler) the warp issues from. Both are
// where the warp is now; they serve as scheduling hints only.
__device__ __forceinline__ uint32_t sm_id() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
  return v;
}

__device__ __forceinline__ uint32_t warp_slot() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%warpid;" : "=r"(v));
  return v;
}

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

// One hand-off chunk of a row, raw: 16 fp16 (32 bytes) and the chunk's exponent
// byte, read through L2 (the GEMM writes them while this work runs).
struct RawChunk {
  uint32_t w[8];
  uint16_t e;
};

__device__ __forceinline__ void load_raw(const uint16_t* val, const uint8_t* ex, RawChunk& r, uint64_t policy) {
  asm volatile("ld.global.cg.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
                 "=r"(r.w[6]), "=r"(r.w[7])
               : "l"(val), "l"(policy)
               : "memory");
  asm volatile("ld.global.cg.u8 %0, [%1];" : "=h"(r.e) : "l"(ex) : "memory");
}

__device__ __forceinline__ void decode16(const RawChunk& r, float* f) {
  const float up = __uint_as_float(static_cast<uint32_t>(r.e) << 23);  // 2^(e - 127)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 p = fmul2(__half22float2(*reinterpret_cast<const __half2*>(&r.w[j])), make_float2(up, up));
    f[2 * j] = p.x;
    f[2 * j + 1] = p.y;
  }
}

__device__ __forceinline__ void load8_nc(const float* p, float* v) {
  asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}

__device__ __forceinline__ void store16_bf16(uint16_t* dst, const float* f, uint64_t policy) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t*>(&v);
  }
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "l"(policy)
               : "memory");
}

// Rows per warp task: the low half of a head is d/32 chunks of 16 columns, one lane
// each, and a task takes the largest power of two of rows that fits 32 lanes (so a
// task never crosses a 128-row panel). Lanes past rows * chunks idle.
__host__ __device__ inline int task_rows(int d_head) {
  const int per_row = d_head / 32;
  int r = 32 / per_row;
  while (r & (r - 1)) r &= r - 1;
  return r;
}

__host__ __device__ inline long long task_count(const NormRopeArgs& p, int group_heads) {
  const int rows = task_rows(p.d_head);
  const int groups = (p.n_q + p.n_kv + group_heads - 1) / group_heads;
  return static_cast<long long>((p.T + rows - 1) / rows) * groups;
}

// The 128-row panel whose completion task `task` waits for.
__device__ __forceinline__ int task_panel(const NormRopeArgs& p, long long task, int group_heads) {
  const int groups = (p.n_q + p.n_kv + group_heads - 1) / group_heads;
  return static_cast<int>(task / groups) * task_rows(p.d_head) >> 7;
}

// Wait (bounded) until K1 has finished every Q/K tile of the row panel.
__device__ __forceinline__ bool wait_panel_ready(const uint32_t* flag, uint32_t target) {
  if (ld_acquire(flag) >= target) return true;
  const unsigned long long t0 = now_ns();
  while (true) {
    __nanosleep(500);
    if (ld_acquire(flag) >= target) return true;
    if (now_ns() - t0 > kWaitLimitNs) return false;
  }
}

// This lane's share of the GEMM's statistics for head `hg` of row `t`, loaded with the
// head's hand-off chunks so the loads are in flight together. RMS: the head's sum of
// squares in .x. LayerNorm: the (shift, mean, M2, -) of the head's tile part c (the
// lane's chunk index), when the head has that part; the lanes of a row share them in
// head_factors. Read through L2: the GEMM writes them while this runs.
__device__ __forceinline__ float4 head_stats_share(const NormRopeArgs& p, int t, int hg, int c) {
  const int heads = p.n_q + p.n_kv;
  if (p.head_kind == 2) return make_float4(__ldcg(p.head_stats + static_cast<size_t>(t) * heads + hg), 0.f, 0.f, 0.f);
  const float4* st = reinterpret_cast<const float4*>(p.head_stats) + (static_cast<size_t>(t) * heads + hg) * p.stat_parts;
  return c < p.stat_parts ? __ldcg(st + c) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// The per-head norm factors of head `hg` for row `t`. RMS: from the head's sum of
// squares. LayerNorm: the parts' (mean, M2) are combined in part order with Chan,
// Golub and LeVeque's pairwise update (no large sums subtracted); part i comes from
// lane row_base + i of the row (its head_stats_share), or is loaded here when the row
// has fewer lanes than parts. The hand-off holds each part's values centred on the
// part's shift, so `shift_lo` / `shift_hi` (shift_part - mean_head of the parts holding
// this lane's low and high chunk) turn them into deviations from the head's mean.
// Called by the whole warp (the shuffles; the head is the same for every lane). Every
// lane of a row repeats this per head, so it uses the fast reciprocal square root and
// quotient (a few ulp, far below the bf16 rounding of the result).
__device__ __forceinline__ void head_factors(const NormRopeArgs& p, int t, int hg, int col_lo, int col_hi, float4 share,
                                             int row_base, int per_row, float inv_d, float& inv, float& shift_lo,
                                             float& shift_hi) {
  const int d = p.d_head;
  if (p.head_kind == 2) {
    inv = rsqrtf(fmaf(share.x, inv_d, p.eps));
    shift_lo = shift_hi = 0.0f;
    return;
  }
  const int heads = p.n_q + p.n_kv;
  const int hs = hg * d;
  const int t0 = hs / p.tile_n;
  const int part_lo = col_lo / p.tile_n - t0, part_hi = col_hi / p.tile_n - t0;
  const float4* st = reinterpret_cast<const float4*>(p.head_stats) + (static_cast<size_t>(t) * heads + hg) * p.stat_parts;
  float n = 0.0f, m = 0.0f, m2 = 0.0f, c_lo = 0.0f, c_hi = 0.0f;
  for (int i = 0; i < p.stat_parts; ++i) {
    const int lo = max(hs, (t0 + i) * p.tile_n);
    const int hi = min(hs + d, (t0 + i + 1) * p.tile_n);
    if (lo >= hi) break;  // the same for the whole warp
    float4 part;
    if (i < per_row) {
      part.x = __shfl_sync(0xffffffffu, share.x, row_base + i);
      part.y = __shfl_sync(0xffffffffu, share.y, row_base + i);
      part.z = __shfl_sync(0xffffffffu, share.z, row_base + i);
    } else {
      part = __ldcg(st + i);
    }
    const float ni = static_cast<float>(hi - lo);
    const float nn = n + ni;
    const float w = __fdividef(ni, nn);
    const float delta = part.y - m;
    m = fmaf(delta, w, m);
    m2 += part.z + delta * delta * (n * w);
    n = nn;
    if (i == part_lo) c_lo = part.x;
    if (i == part_hi) c_hi = part.x;
  }
  inv = rsqrtf(fmaf(m2, inv_d, p.eps));
  shift_lo = c_lo - m;
  shift_hi = c_hi - m;
}

// One task, called by a whole warp once its panel is known to be complete. kHeadStats:
// the per-head norm from the GEMM's statistics (a separate instantiation, so the
// across-heads form keeps its lower register count). kBatch: heads whose loads are in
// flight together (more per warp, or fewer registers and so more warps per SM).
template <bool kHeadStats, int kBatch = kHeadBatch>
__device__ __forceinline__ void run_task(const NormRopeArgs& p, long long task, int group_heads, uint64_t once) {
  const int lane = threadIdx.x & 31;
  const int d = p.d_head;
  const int half = d / 2;
  const int per_row = d / 32;  // lanes per row: the 16-column chunks of the low half
  const int rows = task_rows(d);
  const int lr = lane / per_row;       // this lane's row inside the task
  const int c = lane - lr * per_row;   // this lane's chunk of the low half
  const bool lane_on = lr < rows;
  const int heads = p.n_q + p.n_kv;
  const int qk_chunks = heads * d / 16;
  const int groups = (heads + group_heads - 1) / group_heads;
  const int u = static_cast<int>(task / groups);
  const int grp = static_cast<int>(task - static_cast<long long>(u) * groups);
  const int h_begin = grp * group_heads;
  const int h_end = min(heads, h_begin + group_heads);
  const int row0 = u * rows;
  const int t = lane_on ? row0 + lr : row0;  // idle lanes shadow the task's first row
  const bool row_ok = lane_on && t < p.T;
  const int panel = row0 >> 7;
  (void)ld_acquire(p.ready + panel);  // each lane acquires the panel's publication
  const int tr = t < p.T ? t : p.T - 1;

  const float inv_d = 1.0f / static_cast<float>(d);  // per-head norms
  float inv_q = 1.0f, inv_k = 1.0f;
  if (p.norm && !kHeadStats) {
    if (p.n_q > 0)
      inv_q = 1.0f / sqrtf(p.sumsq[2 * static_cast<size_t>(tr)] / static_cast<float>(p.n_q * d) + p.eps);
    if (p.n_kv > 0)
      inv_k = 1.0f / sqrtf(p.sumsq[2 * static_cast<size_t>(tr) + 1] / static_cast<float>(p.n_kv * d) + p.eps);
  }
  float cl[16], ch[16], sl[16], sh[16];
  if (p.rope) {
    const float* cr = p.cos_t + static_cast<size_t>(tr) * d + c * 16;
    const float* sr = p.sin_t + static_cast<size_t>(tr) * d + c * 16;
    load8_nc(cr, cl);
    load8_nc(cr + 8, cl + 8);
    load8_nc(cr + half, ch);
    load8_nc(cr + half + 8, ch + 8);
    load8_nc(sr, sl);
    load8_nc(sr + 8, sl + 8);
    load8_nc(sr + half, sh);
    load8_nc(sr + half + 8, sh + 8);
  }
  const size_t idx0 = static_cast<size_t>(panel) * qk_chunks * 128 + (t & 127);
  for (int hg0 = h_begin; hg0 < h_end; hg0 += kBatch) {
    RawChunk raw_lo[kBatch], raw_hi[kBatch];
    float4 share[kBatch];  // per-head norms: this lane's share of the statistics
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int hg = hg0 + k;
      if (hg >= h_end) break;
      const int seg = hg >= p.n_q ? 1 : 0;
      const int col = (seg ? p.n_q * d : 0) + (seg ? hg - p.n_q : hg) * d + c * 16;
      const size_t i_lo = idx0 + static_cast<size_t>(col >> 4) * 128;
      const size_t i_hi = idx0 + static_cast<size_t>((col + half) >> 4) * 128;
      load_raw(p.qk_val + i_lo * 16, p.qk_exp + i_lo, raw_lo[k], once);
      load_raw(p.qk_val + i_hi * 16, p.qk_exp + i_hi, raw_hi[k], once);
      if constexpr (kHeadStats) share[k] = head_stats_share(p, tr, hg, c);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int hg = hg0 + k;
      if (hg >= h_end) break;
      const int seg = hg >= p.n_q ? 1 : 0;
      const int off = (seg ? hg - p.n_q : hg) * d + c * 16;  // column inside the segment
      const int col = (seg ? p.n_q * d : 0) + off;            // column of O (low half)
      float lo[16], hi[16];
      decode16(raw_lo[k], lo);
      decode16(raw_hi[k], hi);
      if constexpr (kHeadStats) {  // per-head norm: (y - mean) * inv * gamma[d_head]
        float inv, shift_lo, shift_hi;
        head_factors(p, tr, hg, col, col + half, share[k], lane - c, per_row, inv_d, inv, shift_lo, shift_hi);
        const uint16_t* gamma = (seg ? p.gamma_k : p.gamma_q) + c * 16;
        float g[8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          unpack8(__ldg(reinterpret_cast<const uint4*>(gamma) + q), g);
#pragma unroll
          for (int j = 0; j < 8; ++j) lo[8 * q + j] = (lo[8 * q + j] + shift_lo) * (inv * g[j]);
          unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + half) + q), g);
#pragma unroll
          for (int j = 0; j < 8; ++j) hi[8 * q + j] = (hi[8 * q + j] + shift_hi) * (inv * g[j]);
        }
      } else if (p.norm) {  // across heads
        const uint16_t* gamma = seg ? p.gamma_k : p.gamma_q;
        const float inv = seg ? inv_k : inv_q;
        const float2 inv2 = make_float2(inv, inv);
        float g[8];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + off) + q), g);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 y = fmul2(make_float2(lo[8 * q + 2 * j], lo[8 * q + 2 * j + 1]),
                                   fmul2(inv2, make_float2(g[2 * j], g[2 * j + 1])));
            lo[8 * q + 2 * j] = y.x;
            lo[8 * q + 2 * j + 1] = y.y;
          }
          unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + off + half) + q), g);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 y = fmul2(make_float2(hi[8 * q + 2 * j], hi[8 * q + 2 * j + 1]),
                                   fmul2(inv2, make_float2(g[2 * j], g[2 * j + 1])));
            hi[8 * q + 2 * j] = y.x;
            hi[8 * q + 2 * j + 1] = y.y;
          }
        }
      }
      if (p.rope) {
        // a = lo*cos_lo - hi*sin_lo, b = hi*cos_hi + lo*sin_hi, two lanes per instruction
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 l2 = make_float2(lo[2 * j], lo[2 * j + 1]);
          const float2 h2 = make_float2(hi[2 * j], hi[2 * j + 1]);
          const float2 a = ffma2(h2, make_float2(-sl[2 * j], -sl[2 * j + 1]),
                                 fmul2(l2, make_float2(cl[2 * j], cl[2 * j + 1])));
          const float2 b = ffma2(l2, make_float2(sh[2 * j], sh[2 * j + 1]),
                                 fmul2(h2, make_float2(ch[2 * j], ch[2 * j + 1])));
          lo[2 * j] = a.x;
          lo[2 * j + 1] = a.y;
          hi[2 * j] = b.x;
          hi[2 * j + 1] = b.y;
        }
      }
      if (row_ok) {
        store16_bf16(p.O + out_index(p.nbsd, p.T, p.I, d, t, col), lo, once);
        store16_bf16(p.O + out_index(p.nbsd, p.T, p.I, d, t, col + half), hi, once);
      }
    }
  }
  if (!kHeadStats && c == 0 && grp == 0 && row_ok && p.norm && p.inv_rms != nullptr) {
    p.inv_rms[2 * static_cast<size_t>(t)] = p.n_q > 0 ? inv_q : 0.0f;
    p.inv_rms[2 * static_cast<size_t>(t) + 1] = p.n_kv > 0 ? inv_k : 0.0f;
  }
}

}  // namespace nrp
}  // namespace qkvcte
