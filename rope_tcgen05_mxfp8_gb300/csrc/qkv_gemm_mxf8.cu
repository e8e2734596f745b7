// Kernel K1 with the plain epilogue (Q/K to the norm/RoPE hand-off or as projected),
// the scale repack / clear kernel, and the GEMM dispatch. The kernel templates and
// their design notes are in qkv_gemm_mxf8.cuh.
#include "qkv_gemm_mxf8.cuh"
#include "qkv_cte.h"

namespace qkvcte {

namespace {

// Repack W's UE8M0 scales [I, H/32] into, per (N tile, 128-byte K block), the image
// one tcgen05.cp turns into the TMEM scale-factor layout of an M=128 block-scaled MMA
// (sf_chunks * 2048 bytes; qkv_gemm_mxf8.cuh describes it): byte kb of word c of
// image row l = 32*q + r, chunk j is the scale of output column
// n = tile*tile_n + 128*j + 32*c + r for K element group 4*block + kb, for each of the
// four lane quarters q. Columns past I (or past the tile) get 127.
//
// The first n_tiles * stage_groups blocks each repack one N tile for up to
// kPrepStages K stages: they read the tile's rows of w_sf (consecutive threads,
// consecutive rows: 4 * kPrepStages contiguous bytes each) into shared memory and
// write the blocks from there, so both sides are coalesced. Every block then takes a
// share of the clears: the sum-of-squares buffer, the extra statistics, the panel
// counters, the per-SM sub-partition table, the status word, the task counter and the
// timing stamps. Launched as a
// programmatic dependent of a producer kernel (bf16 or packed activations), this
// kernel does its own work beside it and waits for it before it ends, so the GEMM,
// which waits for this kernel, also finds the producer's output complete.
constexpr int kPrepThreads = 256;
constexpr int kPrepStages = 8;

__global__ void __launch_bounds__(kPrepThreads) qkv_prep_kernel(
    const uint8_t* __restrict__ w_sf, uint32_t* __restrict__ packed, int I, int k_blocks, int tile_n, int n_tiles,
    int k_stages, int sf_chunks, float* __restrict__ sumsq, size_t sumsq_count, uint32_t* __restrict__ ready,
    int m_tiles, uint32_t* __restrict__ sm_busy, uint32_t* status, unsigned long long* stamps, uint32_t* task_next,
    float* __restrict__ zero_extra, size_t zero_extra_count) {
  __shared__ uint32_t rows[256][kPrepStages + 1];  // +1: the column reads below hit 32 banks
  const int groups = (k_stages + kPrepStages - 1) / kPrepStages;
  if (static_cast<int>(blockIdx.x) < n_tiles * groups) {
    const int nt = static_cast<int>(blockIdx.x) / groups;
    const int kst0 = (static_cast<int>(blockIdx.x) - nt * groups) * kPrepStages;
    const int n_st = min(kPrepStages, k_stages - kst0);
    const int i = threadIdx.x;  // tile_n <= 256 = kPrepThreads
    const int n = nt * tile_n + i;
    const bool live = i < tile_n && n < I;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(w_sf + static_cast<size_t>(live ? n : 0) * k_blocks) + kst0;
#pragma unroll
    for (int k = 0; k < kPrepStages; ++k) rows[i][k] = (live && k < n_st) ? __ldg(src + k) : 0x7F7F7F7Fu;
    __syncthreads();
    // The image's four lane quarters are the same 32-row block (sf_chunks * 512 bytes):
    // each thread builds one 16-byte row of a core matrix of that block and stores it
    // four times.
    const int per_stage = sf_chunks * (kSfBlockBytesPerChunk / 4);  // words per K block
    const int quarter16 = per_stage / 16;                          // 16-byte rows per lane quarter
    uint4* dst = reinterpret_cast<uint4*>(packed + (static_cast<size_t>(nt) * k_stages + kst0) * per_stage);
    for (int v = threadIdx.x; v < n_st * quarter16; v += kPrepThreads) {
      const int ks = v / quarter16;
      const int row16 = v - ks * quarter16;
      const int core = row16 >> 3;  // 8-row x 16-byte core matrix: (row group, chunk)
      const int chunk = core % sf_chunks;
      const int lane = (core / sf_chunks) * 8 + (row16 & 7);  // TMEM lane within the quarter
      const int n0 = chunk * 128 + lane;                      // word c holds column n0 + 32 c
      const uint4 q = make_uint4(rows[n0][ks], rows[n0 + 32][ks], rows[n0 + 64][ks], rows[n0 + 96][ks]);
      uint4* d = dst + static_cast<size_t>(ks) * (per_stage / 4) + row16;
#pragma unroll
      for (int r = 0; r < 4; ++r) d[r * quarter16] = q;
    }
  }
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t first = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (size_t i = first; i < sumsq_count; i += stride) sumsq[i] = 0.0f;
  if ((zero_extra_count & 3) == 0 && (reinterpret_cast<uintptr_t>(zero_extra) & 15) == 0) {
    float4* z4 = reinterpret_cast<float4*>(zero_extra);
    for (size_t i = first; i < zero_extra_count / 4; i += stride) z4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  } else {
    for (size_t i = first; i < zero_extra_count; i += stride) zero_extra[i] = 0.0f;
  }
  for (size_t i = first; i < static_cast<size_t>(m_tiles); i += stride) ready[i] = 0u;
  for (size_t i = first; i < static_cast<size_t>(kSmTable); i += stride) sm_busy[i] = 0u;
  if (first == 0) {
    status[0] = 0u;
    task_next[0] = 0u;  // norm/RoPE tasks
    task_next[1] = 0u;  // CTA-pair GEMM tiles (kTileCounterOffset)
    stamps[0] = stamps[2] = ~0ull;
    stamps[1] = stamps[3] = 0ull;
  }
  // With a programmatic predecessor (the producer step), end only after it has.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The scratch of the allocation-free entry point: QKV_CTE_NOALLOC_SCRATCH_BYTES on every
// GPU that loads the library, held until the process exits. It sits in the same
// translation unit (one CUDA module) as the prep kernel, which every run launches
// first: whatever call first runs on a device maps the module and the array together,
// so a later lookup of the array's address maps nothing.
static __device__ __align__(256) uint8_t g_noalloc_scratch[QKV_CTE_NOALLOC_SCRATCH_BYTES];

// dst |= src: one chunk's status word into the status word of a run made of chunks.
__global__ void status_or_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst) {
  if (threadIdx.x == 0) *dst |= *src;
}

}  // namespace

cudaError_t noalloc_scratch_address(void** out) { return cudaGetSymbolAddress(out, g_noalloc_scratch); }

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
                        size_t sumsq_count, uint32_t* ready, uint32_t* sm_busy, uint32_t* status,
                        unsigned long long* stamps, uint32_t* task_next, float* zero_extra, size_t zero_extra_count,
                        cudaStream_t s, int num_sms, bool after_producer) {
  if (g.tile_n > kPrepThreads) return cudaErrorInvalidValue;
  const size_t repack = static_cast<size_t>(g.n_tiles) * ((g.k_stages + kPrepStages - 1) / kPrepStages);
  size_t clear = sumsq_count > zero_extra_count / 4 ? sumsq_count : zero_extra_count / 4;
  if (clear < static_cast<size_t>(g.blocks128)) clear = static_cast<size_t>(g.blocks128);
  if (clear < static_cast<size_t>(kSmTable)) clear = static_cast<size_t>(kSmTable);
  size_t blocks = (clear + kPrepThreads - 1) / kPrepThreads;
  const size_t cap = static_cast<size_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < repack) blocks = repack;
  if (blocks == 0) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kPrepThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_producer ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qkv_prep_kernel, w_sf, reinterpret_cast<uint32_t*>(sf_packed), g.I, g.H / 32,
                            g.tile_n, g.n_tiles, g.k_stages, g.sf_chunks, sumsq, sumsq_count, ready, g.blocks128,
                            sm_busy, status, stamps, task_next, zero_extra, zero_extra_count);
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
