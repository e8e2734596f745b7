// Kernel K2: across-heads RMSNorm apply + rotate-half RoPE of the Q and K columns,
// written into O; V is never read.
//
// Follows the `qkv_cte` kernel reference page, "Design" 1 (steps b and c: finish
// inv_rms = 1/sqrt(sum(o^2) / (n_heads * d_head) + eps) per token and segment, re-read
// each token's Q and K, multiply by the segment-wide gamma) and "Design" 2 (RoPE in
// the same pass, inv_rms folded into it, out = y*cos + [-y_hi, y_lo]*sin with
// position-only cos/sin broadcast over the heads).
//
// On one GPU every head is local, so the page's cross-rank AllReduce of the sums is
// the identity: K1 already summed over every column tile of the row. The pass is
// launched as a programmatic dependent of K1: its blocks run beside K1's persistent
// CTAs and take each task's rows once K1's counter says their 128-row panel is
// complete (a bounded acquire wait), so it mostly hides under the GEMM. The page writes
// the un-normalised Q/K into the output and re-reads it; here K1 hands them over in
// block floating point (fp16 with a power-of-two exponent per row and 16 columns, in
// a tile-major workspace buffer), so the result is rounded to bf16 once, here. This
// pass is HBM-bound. A warp covers a few rows and the whole low half of a head: lane
// (r, q) owns row r and the 16-column chunk q of the low half (plus its partner d/2
// away), so the lanes of one row store whole 128-byte lines of O (d = 128) and read
// the tile-major hand-off in 256-byte runs; four heads' loads are in flight at once,
// each lane keeps its cos/sin chunk and inv_rms in registers across all heads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace qkvcte {

namespace {

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}




constexpr int kThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait (bounded) until K1 has finished every Q/K tile of the row panel.
__device__ bool wait_panel_ready(const uint32_t* flag, uint32_t target) {
  if (ld_acquire(flag) >= target) return true;
  const unsigned long long t0 = now_ns();
  while (true) {
    __nanosleep(500);
    if (ld_acquire(flag) >= target) return true;
    if (now_ns() - t0 > kWaitLimitNs) return false;
  }
}


// One hand-off chunk of a row, raw: 16 fp16 (32 bytes) and the chunk's exponent
// byte, read through L2 (the GEMM writes them while this kernel runs).
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
    const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&r.w[j]));
    f[2 * j] = p.x * up;
    f[2 * j + 1] = p.y * up;
  }
}

__device__ __forceinline__ void load8_nc(const float* p, float* v) {
  asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}

__device__ __forceinline__ void st_global_v8_b32(void* p, const uint32_t* w, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void store16_bf16(uint16_t* dst, const float* f, uint64_t policy) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t*>(&v);
  }
  st_global_v8_b32(dst, w, policy);
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

constexpr int kHeadBatch = 4;   // heads whose hand-off loads are in flight together
constexpr int kHeadGroup = 20;  // heads per warp task (a multiple of kHeadBatch)

// Rows per warp task: the low half of a head is d/32 chunks of 16 columns, one lane
// each, and a task takes the largest power of two of rows that fits 32 lanes (so a
// task never crosses a 128-row panel). Lanes past rows * chunks idle.
__host__ __device__ inline int task_rows(int d_head) {
  const int per_row = d_head / 32;
  int r = 32 / per_row;
  while (r & (r - 1)) r &= r - 1;
  return r;
}

// One warp task = task_rows(d) consecutive rows x the whole low half of up to
// kHeadGroup heads, each lane with its chunk's partner d/2 away (the rotation pairs
// lane j with lane j + d/2 inside each head). Small tasks keep the warps evenly
// loaded to the end.
__global__ void __launch_bounds__(kThreads) qk_norm_rope_kernel(const NormRopeArgs p) {
  if (threadIdx.x == 0) atomicMin(&p.stamps[0], now_ns());
  const int lane = threadIdx.x & 31;
  const int d = p.d_head;
  const int half = d / 2;
  const int per_row = d / 32;  // lanes per row: the 16-column chunks of the low half
  const int rows = task_rows(d);
  const int lr = lane / per_row;          // this lane's row inside the task
  const int c = lane - lr * per_row;      // this lane's chunk of the low half
  const bool lane_on = lr < rows;
  const int heads = p.n_q + p.n_kv;
  const int qk_chunks = heads * d / 16;
  const int groups = (heads + kHeadGroup - 1) / kHeadGroup;
  const long long units = (p.T + rows - 1) / rows;
  const long long tasks = units * groups;
  const long long warps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  // Read-once hand-off and write-once output: first out of L2, so the GEMM's
  // L2-resident weight band running beside this pass keeps its place.
  const uint64_t once = evict_first_policy();
  for (long long task = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); task < tasks;
       task += warps) {
    const int u = static_cast<int>(task / groups);
    const int grp = static_cast<int>(task - static_cast<long long>(u) * groups);
    const int h_begin = grp * kHeadGroup;
    const int h_end = min(heads, h_begin + kHeadGroup);
    const int row0 = u * rows;
    const int t = lane_on ? row0 + lr : row0;  // idle lanes shadow the task's first row
    const bool row_ok = lane_on && t < p.T;
    const int panel = row0 >> 7;
    int ok = 1;
    if (lane == 0) ok = wait_panel_ready(p.ready + panel, p.ready_target) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) atomicOr(p.status, kErrNormReadyWait);
      break;
    }
    (void)ld_acquire(p.ready + panel);  // each lane acquires the panel's publication
    const int tr = t < p.T ? t : p.T - 1;

    float inv_q = 1.0f, inv_k = 1.0f;
    if (p.norm) {
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
    for (int hg0 = h_begin; hg0 < h_end; hg0 += kHeadBatch) {
      RawChunk raw_lo[kHeadBatch], raw_hi[kHeadBatch];
#pragma unroll
      for (int k = 0; k < kHeadBatch; ++k) {
        const int hg = hg0 + k;
        if (hg >= h_end) break;
        const int seg = hg >= p.n_q ? 1 : 0;
        const int col = (seg ? p.n_q * d : 0) + (seg ? hg - p.n_q : hg) * d + c * 16;
        const size_t i_lo = idx0 + static_cast<size_t>(col >> 4) * 128;
        const size_t i_hi = idx0 + static_cast<size_t>((col + half) >> 4) * 128;
        load_raw(p.qk_val + i_lo * 16, p.qk_exp + i_lo, raw_lo[k], once);
        load_raw(p.qk_val + i_hi * 16, p.qk_exp + i_hi, raw_hi[k], once);
      }
#pragma unroll
      for (int k = 0; k < kHeadBatch; ++k) {
        const int hg = hg0 + k;
        if (hg >= h_end) break;
        const int seg = hg >= p.n_q ? 1 : 0;
        const int off = (seg ? hg - p.n_q : hg) * d + c * 16;  // column inside the segment
        const int col = (seg ? p.n_q * d : 0) + off;            // column of O (low half)
        float lo[16], hi[16];
        decode16(raw_lo[k], lo);
        decode16(raw_hi[k], hi);
        if (p.norm) {
          const uint16_t* gamma = seg ? p.gamma_k : p.gamma_q;
          const float inv = seg ? inv_k : inv_q;
          float g[8];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + off) + q), g);
#pragma unroll
            for (int j = 0; j < 8; ++j) lo[8 * q + j] *= inv * g[j];
            unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + off + half) + q), g);
#pragma unroll
            for (int j = 0; j < 8; ++j) hi[8 * q + j] *= inv * g[j];
          }
        }
        if (p.rope) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a = lo[j] * cl[j] - hi[j] * sl[j];
            const float b = hi[j] * ch[j] + lo[j] * sh[j];
            lo[j] = a;
            hi[j] = b;
          }
        }
        if (row_ok) {
          store16_bf16(p.O + out_index(p.nbsd, p.T, p.I, d, t, col), lo, once);
          store16_bf16(p.O + out_index(p.nbsd, p.T, p.I, d, t, col + half), hi, once);
        }
      }
    }
    if (c == 0 && grp == 0 && row_ok && p.norm && p.inv_rms != nullptr) {
      p.inv_rms[2 * static_cast<size_t>(t)] = inv_q;
      p.inv_rms[2 * static_cast<size_t>(t) + 1] = p.n_kv > 0 ? inv_k : 0.0f;
    }
  }
  if (threadIdx.x == 0) atomicMax(&p.stamps[1], now_ns());
}

}  // namespace

cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s, int num_sms, bool overlap) {
  if (!a.norm && !a.rope) return cudaSuccess;
  if (a.d_head < 32 || a.d_head % 32 != 0) return cudaErrorInvalidValue;
  const int rows = task_rows(a.d_head);
  const long long tasks = static_cast<long long>((a.T + rows - 1) / rows) *
                          ((a.n_q + a.n_kv + kHeadGroup - 1) / kHeadGroup);
  if (tasks == 0) return cudaSuccess;
  // Overlapped with the GEMM, the grid is kept to what fits beside each GEMM CTA
  // (registers are the limit) so every block finds its units as their panels
  // complete. That sizing only affects speed: the GEMM never waits for this kernel.
  // Alone, the pass takes every SM it can hold.
  int per_sm = 1;
  if (!overlap) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, qk_norm_rope_kernel, kThreads, 0) == cudaSuccess &&
        occ > per_sm)
      per_sm = occ;
  }
  long long blocks = (tasks + kThreads / 32 - 1) / (kThreads / 32);
  if (blocks > static_cast<long long>(per_sm) * num_sms) blocks = static_cast<long long>(per_sm) * num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qk_norm_rope_kernel, a);
}

}  // namespace qkvcte
