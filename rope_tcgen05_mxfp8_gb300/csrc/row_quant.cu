// The producer step before the projection: bf16 activations -> ROW_MX rows (per-row
// e4m3 codes plus one fp32 dequant scale), and the packed [T, H + 4] row layout
// (each row's H codes, then the four bytes of its scale). [qkv_cte] "Interface"
// table, packed_hidden row (the projection takes row-quantised FP8; its producer
// quantises) and "Upstream behavior" (the packed H + 4 activation layout).
//
// Both kernels are HBM-bound streams:
//   quantise: read 2H bytes, write H + 4 (codes + scale, or the packed row);
//   unpack:   read H + 4 bytes, write H + 4.
// The GEMM reads its A operand with TMA, which needs a 16-byte row pitch; the
// packed pitch H + 4 is 4 mod 16, so a packed input is unpacked first.

#include "internal.h"
#include "ptx.cuh"

namespace qkvcte {

namespace {

constexpr int kThreads = 256;       // unpack: 8 warps, a warp owns one row at a time
constexpr int kQuantThreads = 128;  // quantise: a CTA of 4 warps owns one row at a time
constexpr int kRegChunks = 5;       // 16-byte chunks per thread kept in registers: rows of up to
                                    // 5 * 128 * 8 = 5120 elements are read from HBM once (longer
                                    // rows read their remainder a second time, from L2)

__device__ __forceinline__ uint4 ld_once_v4(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ uint32_t ld_once_u32(const void* p, uint64_t pol) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

// |x| of two bf16 values at once: clear both sign bits. Finite bf16 magnitudes
// order like their bit patterns, so the row maximum is an integer maximum.
__device__ __forceinline__ uint32_t abs_max_pairs(uint32_t acc, const uint4& v) {
  acc = __vmaxu2(acc, v.x & 0x7fff7fffu);
  acc = __vmaxu2(acc, v.y & 0x7fff7fffu);
  acc = __vmaxu2(acc, v.z & 0x7fff7fffu);
  return __vmaxu2(acc, v.w & 0x7fff7fffu);
}

// Scales at or above this use the multiply-and-correct quotient below; smaller ones
// (rows whose largest magnitude is under 448 * 2^-90) divide.
constexpr float kFastQuotientMinScale = 0x1p-90f;

// The correctly rounded fp32 quotient x / s from r = RN(1/s), by Markstein's
// correction step (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(x * r) is
// within one ulp of x / s, the remainder e = x - s * q0 is exact in one fma, and
// RN(q0 + e * r) is RN(x / s). The remainder stays exact while it is a normal
// number, which holds for every quotient that can reach an e4m3 code (|q| >= 2^-11)
// once s >= 2^-90; smaller quotients all give a zero code whatever their last bits.
// A zero x gives a zero of x's sign, as a division does.
__device__ __forceinline__ float quotient_corrected(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-s, q0, x);
  return copysignf(__fmaf_rn(e, r, q0), x);
}

// Two bf16 (one 32-bit word, element 0 in the low half) -> two e4m3 codes, element
// 0 in the low byte: each is the fp32 quotient x / s, correctly rounded, converted
// with round-to-nearest-even and saturation to +-448.
template <bool kCorrected>
__device__ __forceinline__ uint32_t quantise_pair(uint32_t w, float s, float r) {
  const float x0 = __uint_as_float(w << 16);
  const float x1 = __uint_as_float(w & 0xffff0000u);
  const float q0 = kCorrected ? quotient_corrected(x0, s, r) : __fdiv_rn(x0, s);
  const float q1 = kCorrected ? quotient_corrected(x1, s, r) : __fdiv_rn(x1, s);
  uint16_t c;
  // the first source operand lands in the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(q1), "f"(q0));
  return c;
}

template <bool kCorrected>
__device__ __forceinline__ void emit_chunk(const uint4& v, float s, float r, uint8_t* code_row,
                                           uint8_t* packed_row, int col) {
  const uint32_t w0 = quantise_pair<kCorrected>(v.x, s, r) | (quantise_pair<kCorrected>(v.y, s, r) << 16);
  const uint32_t w1 = quantise_pair<kCorrected>(v.z, s, r) | (quantise_pair<kCorrected>(v.w, s, r) << 16);
  if (code_row != nullptr) *reinterpret_cast<uint2*>(code_row + col) = make_uint2(w0, w1);
  if (packed_row != nullptr) {
    // packed rows are only 4-byte aligned (pitch H + 4)
    reinterpret_cast<uint32_t*>(packed_row + col)[0] = w0;
    reinterpret_cast<uint32_t*>(packed_row + col)[1] = w1;
  }
}

// One CTA of kQuantThreads per row at a time (grid-stride over rows): each thread
// holds kRegChunks 16-byte chunks of the row in registers, so the registers per
// thread stay low and many CTAs per SM keep enough loads in flight; the four warps
// combine their row maxima through shared memory (one barrier per row: the slot
// alternates between rows, and a warp reuses a slot only after the barrier of the
// row in between).
__global__ void __launch_bounds__(kQuantThreads, 10) row_quantize_kernel(const uint16_t* __restrict__ X, int T,
                                                                         int H, uint8_t* __restrict__ codes,
                                                                         float* __restrict__ scale,
                                                                         uint8_t* __restrict__ packed) {
  __shared__ uint32_t warp_max[2][kQuantThreads / 32];
  // Inside a run the next kernel (the scale repack and clears) does not read what this
  // one writes before it waits for it: it may start now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int chunks = H >> 3;  // 8 bf16 = 16 bytes per chunk
  const uint64_t once = policy_evict_first();
  int parity = 0;
  for (int row = blockIdx.x; row < T; row += gridDim.x, parity ^= 1) {
    const uint16_t* xr = X + static_cast<size_t>(row) * H;
    uint4 v[kRegChunks];
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < kRegChunks; ++i) {
      const int c = i * kQuantThreads + tid;
      if (c < chunks) v[i] = ld_once_v4(xr + static_cast<size_t>(c) * 8, once);
    }
#pragma unroll
    for (int i = 0; i < kRegChunks; ++i)
      if (i * kQuantThreads + tid < chunks) m2 = abs_max_pairs(m2, v[i]);
    for (int c = kRegChunks * kQuantThreads + tid; c < chunks; c += kQuantThreads)  // rows longer than
      m2 = abs_max_pairs(m2, ld_once_v4(xr + static_cast<size_t>(c) * 8, once));    // the registers hold
    const uint32_t wm = __reduce_max_sync(0xffffffffu, max(m2 & 0xffffu, m2 >> 16));
    if (lane == 0) warp_max[parity][warp] = wm;
    __syncthreads();
    uint32_t m = warp_max[parity][0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) m = max(m, warp_max[parity][w]);
    const float amax = __uint_as_float(m << 16);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint8_t* code_row = codes != nullptr ? codes + static_cast<size_t>(row) * H : nullptr;
    uint8_t* packed_row = packed != nullptr ? packed + static_cast<size_t>(row) * (H + 4) : nullptr;
    if (s >= kFastQuotientMinScale) {  // uniform over the CTA: s is the row's
      const float r = __frcp_rn(s);
#pragma unroll
      for (int i = 0; i < kRegChunks; ++i) {
        const int c = i * kQuantThreads + tid;
        if (c < chunks) emit_chunk<true>(v[i], s, r, code_row, packed_row, c * 8);
      }
      for (int c = kRegChunks * kQuantThreads + tid; c < chunks; c += kQuantThreads)
        emit_chunk<true>(ld_once_v4(xr + static_cast<size_t>(c) * 8, once), s, r, code_row, packed_row, c * 8);
    } else {
#pragma unroll
      for (int i = 0; i < kRegChunks; ++i) {
        const int c = i * kQuantThreads + tid;
        if (c < chunks) emit_chunk<false>(v[i], s, 0.0f, code_row, packed_row, c * 8);
      }
      for (int c = kRegChunks * kQuantThreads + tid; c < chunks; c += kQuantThreads)
        emit_chunk<false>(ld_once_v4(xr + static_cast<size_t>(c) * 8, once), s, 0.0f, code_row, packed_row,
                          c * 8);
    }
    if (tid == 0) {
      if (scale != nullptr) scale[row] = s;
      if (packed_row != nullptr) *reinterpret_cast<float*>(packed_row + H) = s;
    }
  }
}

// Packed [T, H + 4] -> codes [T, H] + scales [T]. A lane moves 16 bytes: four
// 4-byte loads (the packed row is only 4-byte aligned) and one 16-byte store.
__global__ void __launch_bounds__(kThreads) unpack_rows_kernel(const uint8_t* __restrict__ packed, int T, int H,
                                                               uint8_t* __restrict__ codes,
                                                               float* __restrict__ scale) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // as in row_quantize_kernel
  const int lane = threadIdx.x & 31;
  const int warp = static_cast<int>((blockIdx.x * static_cast<unsigned>(kThreads) + threadIdx.x) >> 5);
  const int n_warps = static_cast<int>((gridDim.x * static_cast<unsigned>(kThreads)) >> 5);
  const int chunks = H >> 4;
  const uint64_t once = policy_evict_first();
  for (int row = warp; row < T; row += n_warps) {
    const uint8_t* pr = packed + static_cast<size_t>(row) * (H + 4);
    uint8_t* cr = codes + static_cast<size_t>(row) * H;
    for (int c0 = 0; c0 < chunks; c0 += 4 * 32) {
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + k * 32 + lane;
        if (c < chunks) {
          const uint8_t* p = pr + static_cast<size_t>(c) * 16;
          v[k] = make_uint4(ld_once_u32(p, once), ld_once_u32(p + 4, once), ld_once_u32(p + 8, once),
                            ld_once_u32(p + 12, once));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + k * 32 + lane;
        if (c < chunks) *reinterpret_cast<uint4*>(cr + static_cast<size_t>(c) * 16) = v[k];
      }
    }
    if (lane == 0) scale[row] = __uint_as_float(ld_once_u32(pr + H, once));
  }
}

template <typename K>
int resident_blocks(K kernel, int threads, int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm * num_sms;
}

}  // namespace

cudaError_t launch_row_quantize(const uint16_t* X, int T, int H, uint8_t* codes, float* scale, uint8_t* packed,
                                cudaStream_t s, int num_sms) {
  if (T <= 0) return cudaSuccess;
  const int grid = min(resident_blocks(row_quantize_kernel, kQuantThreads, num_sms), T);
  row_quantize_kernel<<<grid, kQuantThreads, 0, s>>>(X, T, H, codes, scale, packed);
  return cudaGetLastError();
}

cudaError_t launch_unpack_rows(const uint8_t* packed, int T, int H, uint8_t* codes, float* scale, cudaStream_t s,
                               int num_sms) {
  if (T <= 0) return cudaSuccess;
  const int rows_per_block = kThreads / 32;
  int grid = resident_blocks(unpack_rows_kernel, kThreads, num_sms);
  grid = min(grid, (T + rows_per_block - 1) / rows_per_block);
  unpack_rows_kernel<<<grid, kThreads, 0, s>>>(packed, T, H, codes, scale);
  return cudaGetLastError();
}

}  // namespace qkvcte
