// Kernel K1 with the plain epilogue (Q/K to the norm/RoPE hand-off or as projected),
// the scale repack / clear kernel, and the GEMM dispatch. The kernel templates and
// their design notes are in qkv_gemm_mxf8.cuh.
#include "qkv_gemm_mxf8.cuh"

namespace qkvcte {

namespace {

// Repack W's UE8M0 scales [I, H/32] into, per (N tile, K stage), SF_CHUNKS blocks of
// 512 bytes: byte 16*r + 4*c + kb of block `chunk` is the scale of output column
// n = tile*tile_n + 128*chunk + 32*c + r for K block 4*stage + kb. That is the
// 32-row x 16-byte shared-memory image tcgen05.cp 32x128b.warpx4 turns into the
// TMEM scale-factor layout of an M=128 block-scaled MMA. Columns past I (or past
// the tile) get 127. Also clears the status word, the panel counters, the timing
// stamps and the sum-of-squares buffer.
__global__ void qkv_prep_kernel(const uint8_t* __restrict__ w_sf, uint32_t* __restrict__ packed, int I,
                                int k_blocks, int tile_n, int n_tiles, int k_stages, int sf_chunks,
                                float* __restrict__ sumsq, size_t sumsq_count, uint32_t* __restrict__ ready,
                                int m_tiles, uint32_t* status, unsigned long long* stamps,
                                uint32_t* task_next, float* __restrict__ zero_extra, size_t zero_extra_count) {
  const size_t words = static_cast<size_t>(n_tiles) * k_stages * sf_chunks * 128;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t first = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t w = first; w < words; w += stride) {
    const int within = static_cast<int>(w & 127);
    const int r = within >> 2;
    const int c = within & 3;
    size_t rest = w >> 7;
    const int chunk = static_cast<int>(rest % sf_chunks);
    rest /= sf_chunks;
    const int kst = static_cast<int>(rest % k_stages);
    const int nt = static_cast<int>(rest / k_stages);
    const int n_local = chunk * 128 + c * 32 + r;
    const int n = nt * tile_n + n_local;
    uint32_t v = 0x7F7F7F7Fu;
    if (n_local < tile_n && n < I)
      v = __ldg(reinterpret_cast<const uint32_t*>(w_sf + static_cast<size_t>(n) * k_blocks + kst * 4));
    packed[w] = v;
  }
  for (size_t i = first; i < sumsq_count; i += stride) sumsq[i] = 0.0f;
  for (size_t i = first; i < zero_extra_count; i += stride) zero_extra[i] = 0.0f;
  for (size_t i = first; i < static_cast<size_t>(m_tiles); i += stride) ready[i] = 0u;
  if (first == 0) {
    status[0] = 0u;
    *task_next = 0u;
    stamps[0] = stamps[2] = ~0ull;
    stamps[1] = stamps[3] = 0ull;
  }
}

// dst |= src: one chunk's status word into the status word of a run made of chunks.
__global__ void status_or_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst) {
  if (threadIdx.x == 0) *dst |= *src;
}

}  // namespace

cudaError_t launch_status_or(const uint32_t* src, uint32_t* dst, cudaStream_t s) {
  status_or_kernel<<<1, 32, 0, s>>>(src, dst);
  return cudaGetLastError();
}

bool gemm_tile_supported(int tile_n) {
  return tile_n == 128 || tile_n == 192 || tile_n == 240 || tile_n == 256;
}

int gemm_sf_chunks(int tile_n) { return (tile_n + 127) / 128; }

size_t gemm_smem_bytes(int tile_n) {
  switch (tile_n) {
    case 128: return K1Cfg<128>::SMEM;
    case 192: return K1Cfg<192>::SMEM;
    case 240: return K1Cfg<240>::SMEM;
    case 256: return K1Cfg<256>::SMEM;
    default: return 0;
  }
}

cudaError_t launch_prep(const GemmShape& g, const uint8_t* w_sf, uint8_t* sf_packed, float* sumsq,
                        size_t sumsq_count, uint32_t* ready, uint32_t* status, unsigned long long* stamps,
                        uint32_t* task_next, float* zero_extra, size_t zero_extra_count, cudaStream_t s,
                        int num_sms) {
  const size_t words = static_cast<size_t>(g.n_tiles) * g.k_stages * g.sf_chunks * 128;
  size_t work = words > sumsq_count ? words : sumsq_count;
  if (zero_extra_count > work) work = zero_extra_count;
  size_t blocks = (work + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  qkv_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      w_sf, reinterpret_cast<uint32_t*>(sf_packed), g.I, g.H / 32, g.tile_n, g.n_tiles, g.k_stages,
      g.sf_chunks, sumsq, sumsq_count, ready, g.blocks128, status, stamps, task_next, zero_extra, zero_extra_count);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmShape& g, const CUtensorMap& tmA, const CUtensorMap& tmW,
                        const CUtensorMap& tmSF, const GemmArgs& a, cudaStream_t s, int num_sms,
                        const NormRopeArgs* fused) {
  if (a.head_norm != 0 || a.stats_kind != 0) return launch_gemm_head(g, tmA, tmW, tmSF, a, s, num_sms);
  if (fused != nullptr) {
    if (!g.cta_pair) return cudaErrorInvalidValue;
    return launch_gemm_fused(g, tmA, tmW, tmSF, a, *fused, s, num_sms);
  }
  const NormRopeArgs none{};
  if (g.cta_pair) {
    switch (g.tile_n) {
      case 128: return launch_gemm_pair_t<128, kEpiPlain, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 192: return launch_gemm_pair_t<192, kEpiPlain, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 240: return launch_gemm_pair_t<240, kEpiPlain, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      case 256: return launch_gemm_pair_t<256, kEpiPlain, false>(g, tmA, tmW, tmSF, a, none, s, num_sms);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.tile_n) {
    case 128: return launch_gemm_t<128, kEpiPlain>(g, tmA, tmW, a, s, num_sms);
    case 192: return launch_gemm_t<192, kEpiPlain>(g, tmA, tmW, a, s, num_sms);
    case 240: return launch_gemm_t<240, kEpiPlain>(g, tmA, tmW, a, s, num_sms);
    case 256: return launch_gemm_t<256, kEpiPlain>(g, tmA, tmW, a, s, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvcte
