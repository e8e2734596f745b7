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
// CTAs and take each 16-row unit once K1's counter says the unit's 128-row panel is
// complete (a bounded acquire wait), so it mostly hides under the GEMM. The page writes
// the un-normalised Q/K into the output and re-reads it; here K1 hands them over in
// fp32 (a workspace buffer) so the result is rounded to bf16 once, here. This pass
// is HBM-bound: each thread reads 8 lanes of the low half of a head and the 8
// partner lanes d/2 away (2 x 32 bytes of fp32) and writes 2 x 16 bytes of bf16 to
// O, with the per-position cos/sin and the gamma vectors served from L1/L2.
#include <cuda_bf16.h>

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

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void load8f(const float* p, float (&f)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Data another kernel wrote while this one runs: read through L2 (not L1).
__device__ __forceinline__ void load8f_l2(const float* p, float (&f)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

constexpr int kUnitRows = 16;                       // rows per work unit (divides 128)
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait (bounded) until K1 has finished every tile of the row panel.
__device__ bool wait_panel_ready(const uint32_t* flag, uint32_t target) {
  if (ld_acquire(flag) >= target) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (true) {
    __nanosleep(500);
    if (ld_acquire(flag) >= target) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const NormRopeArgs p) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) atomicMin(&p.stamps[0], now_ns());
  const int chunks = p.d_head / 16;  // 8-lane chunks in the low half of one head
  const int half = p.d_head / 2;
  const int qk_width = (p.n_q + p.n_kv) * p.d_head;
  const int per_row = (p.n_q + p.n_kv) * chunks;
  const int n_units = (p.T + kUnitRows - 1) / kUnitRows;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int row0 = u * kUnitRows;
    const int rows = min(kUnitRows, p.T - row0);
    if (threadIdx.x == 0) {
      const bool ok = wait_panel_ready(p.ready + row0 / 128, p.ready_target);
      if (!ok) atomicOr(p.status, kErrNormReadyWait);
      s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) break;  // uniform across the block
    const int items = rows * per_row;
#pragma unroll 2
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int tr = it / per_row;
      const int rem = it - tr * per_row;
      const int t = row0 + tr;
      const int hg = rem / chunks;
      const int c = rem - hg * chunks;
      const int seg = hg >= p.n_q ? 1 : 0;
      const int h = seg ? hg - p.n_q : hg;
      const int n_heads = seg ? p.n_kv : p.n_q;
      const int off = h * p.d_head + c * 8;  // column inside the segment
      const int seg_base = seg ? p.n_q * p.d_head : 0;
      uint16_t* row = p.O + static_cast<size_t>(t) * p.I + seg_base;
      const float* src = p.qk + static_cast<size_t>(t) * qk_width + seg_base + off;

      float lo[8], hi[8];
      load8f_l2(src, lo);
      load8f_l2(src + half, hi);

      if (p.norm) {
        const float ss = p.sumsq[2 * static_cast<size_t>(t) + seg];
        const float inv = 1.0f / sqrtf(ss / static_cast<float>(n_heads * p.d_head) + p.eps);
        const uint16_t* gamma = seg ? p.gamma_k : p.gamma_q;
        float glo[8], ghi[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + off)), glo);
        unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + off + half)), ghi);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          lo[j] = lo[j] * inv * glo[j];
          hi[j] = hi[j] * inv * ghi[j];
        }
        if (p.inv_rms != nullptr && h == 0 && c == 0) {
          p.inv_rms[2 * static_cast<size_t>(t) + seg] = inv;
          if (p.n_kv == 0) p.inv_rms[2 * static_cast<size_t>(t) + 1] = 0.0f;
        }
      }
      if (p.rope) {
        const float* cr = p.cos_t + static_cast<size_t>(t) * p.d_head + c * 8;
        const float* sr = p.sin_t + static_cast<size_t>(t) * p.d_head + c * 8;
        float cl[8], ch[8], sl[8], sh[8];
        load8f(cr, cl);
        load8f(cr + half, ch);
        load8f(sr, sl);
        load8f(sr + half, sh);
        float olo[8], ohi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          olo[j] = lo[j] * cl[j] - hi[j] * sl[j];
          ohi[j] = hi[j] * ch[j] + lo[j] * sh[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          lo[j] = olo[j];
          hi[j] = ohi[j];
        }
      }
      *reinterpret_cast<uint4*>(row + off) = pack8(lo);
      *reinterpret_cast<uint4*>(row + off + half) = pack8(hi);
    }
    __syncthreads();  // s_ok is rewritten for the next unit
  }
  if (threadIdx.x == 0) atomicMax(&p.stamps[1], now_ns());
}

}  // namespace

cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s, int num_sms, bool overlap) {
  if (!a.norm && !a.rope) return cudaSuccess;
  const int n_units = (a.T + kUnitRows - 1) / kUnitRows;
  if (n_units == 0) return cudaSuccess;
  const int blocks = n_units < 2 * num_sms ? n_units : 2 * num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
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
