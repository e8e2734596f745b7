// Offline conversion of an interleaved-RoPE checkpoint to the rotate-half lane order
// this library applies ([qkv_cte] "Design" 2: the caller permutes the Q/K weights,
// bias, gamma and cos/sin caches once, so the kernel never sees the interleaved
// form). Within every Q and K head, output lane i takes input lane perm[i] with
// perm[j] = 2j and perm[d/2 + j] = 2j + 1 (pair (2j, 2j+1) becomes (j, j + d/2));
// rows past the Q/K heads (the V channels) are copied unchanged. A row is whatever
// one output channel owns: a row of W's codes, of its block scales, one bias or
// per-column scale entry, one gamma entry, one cos/sin table entry.

#include "internal.h"

namespace qkvcte {

namespace {

template <typename E>
__global__ void permute_rows_kernel(const E* __restrict__ src, E* __restrict__ dst, long long rows,
                                    long long row_elems, long long qk_rows, int d_head) {
  const long long total = rows * row_elems;
  const int half = d_head >> 1;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / row_elems;
    const long long e = i - r * row_elems;
    long long from = r;
    if (r < qk_rows) {
      const long long head0 = r - r % d_head;
      const int lane = static_cast<int>(r - head0);
      from = head0 + (lane < half ? 2 * lane : 2 * (lane - half) + 1);
    }
    dst[i] = src[from * row_elems + e];
  }
}

template <typename E>
cudaError_t launch_t(const void* src, void* dst, long long rows, long long row_bytes, long long qk_rows, int d_head,
                     cudaStream_t s, int num_sms) {
  const long long elems = rows * (row_bytes / static_cast<long long>(sizeof(E)));
  const int threads = 256;
  long long blocks = (elems + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  permute_rows_kernel<E><<<static_cast<int>(blocks), threads, 0, s>>>(
      static_cast<const E*>(src), static_cast<E*>(dst), rows, row_bytes / static_cast<long long>(sizeof(E)), qk_rows,
      d_head);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute_rows(const void* src, void* dst, long long rows, long long row_bytes, long long qk_rows,
                                int d_head, cudaStream_t s, int num_sms) {
  if (rows <= 0 || row_bytes <= 0) return cudaSuccess;
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (row_bytes % 16 == 0 && a % 16 == 0) return launch_t<uint4>(src, dst, rows, row_bytes, qk_rows, d_head, s, num_sms);
  if (row_bytes % 4 == 0 && a % 4 == 0) return launch_t<uint32_t>(src, dst, rows, row_bytes, qk_rows, d_head, s, num_sms);
  if (row_bytes % 2 == 0 && a % 2 == 0) return launch_t<uint16_t>(src, dst, rows, row_bytes, qk_rows, d_head, s, num_sms);
  return launch_t<uint8_t>(src, dst, rows, row_bytes, qk_rows, d_head, s, num_sms);
}

}  // namespace qkvcte
