// C-ABI front end: plan validation, workspace layout, TMA descriptors and the launch
// sequence prep -> K1 (GEMM + epilogue) -> K2 (norm + RoPE) on the caller's stream.
// The argument set follows the `qkv_cte` kernel reference page's "Interface" table,
// with the differences listed in qkv_cte.h.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "internal.h"
#include "qkv_cte.h"

using namespace qkvcte;

struct qkv_cte_plan_s {
  qkv_cte_desc d;
  GemmShape g;
  WorkspaceLayout ws;
  int q_end, k_end;
  // QKV_CTE_FLAG_PROFILE: events before the prep kernel, after it, and after the last
  // kernel of the latest run (no event between K1 and K2: it would serialise them)
  cudaEvent_t ev[2] = {nullptr, nullptr};
  int ev_device = -1;
  bool ran = false;
  bool has_norm_pass = false;
  bool second_pass = false;  // the norm/RoPE work runs (across-heads norm, or RoPE alone)
  bool fused_norm = false;   // ... inside the CTA-pair GEMM's epilogue warps
  const void* last_workspace = nullptr;
  // qkv_cte_run_host: plans for one chunk and for the shorter last chunk, the copy
  // streams and the events that order staging buffers (created on first use)
  qkv_cte_plan_s* chunk_plan = nullptr;
  qkv_cte_plan_s* tail_plan = nullptr;
  int chunk_rows = 0;
  int host_device = -1;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_done[2] = {nullptr, nullptr}, ev_out[2] = {nullptr, nullptr};
};

namespace {

thread_local char g_last_error[512] = "";

__attribute__((format(printf, 2, 3))) int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_last_error[0] = '\0';
  return QKV_CTE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
  bool init = false;
  int major = 0, minor = 0, sms = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(QKV_CTE_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail(QKV_CTE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    d.init = true;
  }
  *out = d;
  return QKV_CTE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D K-major uint8 operand [rows, cols], tiles of box_rows x 128 bytes, 128-byte swizzle.
int encode_operand(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   const char* what) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return fail(QKV_CTE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QKV_CTE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, int(r));
  return QKV_CTE_OK;
}

// The repacked scales as uint32 rows of kSfRowBytes: one N tile's image for one
// 128-byte K block (sf_chunks * kSfBlockBytesPerChunk bytes, whole rows) per TMA box.
int encode_scales(CUtensorMap* m, void* base, const GemmShape& g) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return fail(QKV_CTE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint32_t words = kSfRowBytes / 4;
  const cuuint32_t rows_per_block = (cuuint32_t)(g.sf_chunks * kSfBlockBytesPerChunk / kSfRowBytes);
  cuuint64_t dims[2] = {words, (cuuint64_t)g.n_tiles * (cuuint64_t)g.k_stages * rows_per_block};
  cuuint64_t strides[1] = {(cuuint64_t)kSfRowBytes};
  cuuint32_t box[2] = {words, rows_per_block};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QKV_CTE_ERR_CUDA, "cuTensorMapEncodeTiled(scales) failed: %d", int(r));
  return QKV_CTE_OK;
}

// N tiles per band: the band's W slab (tile_n * H bytes per N tile) is kept to about
// 28 MB so that it stays resident in the 129 MB L2 beside the streaming traffic
// (measured at the Wan 480p shape: 28 MB bands beat 56 MB, 110 MB and one band).
// QKV_CTE_BAND_MB overrides the budget (for tuning sweeps).
int band_tiles(const GemmShape& g) {
  double mb = 28.0;
  if (const char* e = getenv("QKV_CTE_BAND_MB")) {
    const double v = atof(e);
    if (v > 0) mb = v;
  }
  const double per_tile = (double)g.tile_n * (double)g.H;
  int n = (int)(mb * 1048576.0 / per_tile);
  return n < 1 ? 1 : n;
}

// Row-panel ranges the Q/K bands take turns over (1: each Q/K band over all panels).
// QKV_CTE_M_CHUNKS overrides it (for tuning sweeps).
int band_m_chunks() {
  int c = 1;
  if (const char* e = getenv("QKV_CTE_M_CHUNKS")) {
    const int v = atoi(e);
    if (v > 0) c = v;
  }
  return c;
}

bool per_head_norm(const qkv_cte_desc& d) {
  return d.norm == QKV_CTE_NORM_HEAD_RMS || d.norm == QKV_CTE_NORM_HEAD_LAYER;
}

// Per-head norm finished in the GEMM's epilogue (tiles of whole heads, no second pass)
// rather than from per-head statistics by the norm/RoPE pass (the default).
bool head_norm_in_epilogue(const qkv_cte_desc& d) {
  return per_head_norm(d) && (d.flags & QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE) != 0;
}

// Tiles a head's columns can touch: the statistics keep one part per tile.
int stat_parts(int d_head, int tile_n) { return (d_head + tile_n - 2) / tile_n + 1; }

int choose_tile_n(const qkv_cte_desc& d, int I) {
  if (d.tile_n != 0) return d.tile_n;
  (void)I;
  if (head_norm_in_epilogue(d)) {
    // The per-head epilogue needs whole heads in every tile: the widest built tile
    // with two TMEM accumulator stages that d_head divides, else 256 (one stage).
    for (int t : {240, 192, 128})
      if (t % d.d_head == 0) return t;
    return 256;
  }
  return 240;  // two TMEM accumulator stages: the epilogue overlaps the next tile's MMAs
}

}  // namespace

extern "C" {

int qkv_cte_version(void) { return QKV_CTE_ABI_VERSION; }

const char* qkv_cte_last_error(void) { return g_last_error; }

int qkv_cte_plan(qkv_cte_plan_t* out, const qkv_cte_desc* desc, size_t* workspace_bytes) {
  if (out == nullptr || desc == nullptr || workspace_bytes == nullptr)
    return fail(QKV_CTE_ERR_INVALID, "qkv_cte_plan: null argument");
  *out = nullptr;
  const qkv_cte_desc& d = *desc;
  if (d.tokens < 0) return fail(QKV_CTE_ERR_INVALID, "tokens must be >= 0 (got %lld)", (long long)d.tokens);
  if (d.tokens > INT32_MAX) return fail(QKV_CTE_ERR_UNSUPPORTED, "tokens > INT32_MAX");
  if (d.hidden <= 0) return fail(QKV_CTE_ERR_INVALID, "hidden must be > 0");
  if (d.hidden % 128 != 0) return fail(QKV_CTE_ERR_UNSUPPORTED, "hidden %d is not a multiple of 128", d.hidden);
  if (d.n_q_heads < 0) return fail(QKV_CTE_ERR_INVALID, "n_q_heads must be >= 0");
  if (d.n_kv_heads < 0) return fail(QKV_CTE_ERR_INVALID, "n_kv_heads must be >= 0");
  if (d.d_head <= 0) return fail(QKV_CTE_ERR_INVALID, "d_head must be > 0");
  if (d.d_head % 16 != 0) return fail(QKV_CTE_ERR_UNSUPPORTED, "d_head %d is not a multiple of 16", d.d_head);
  if (d.mode == QKV_CTE_MODE_FUSED) {
    if (d.n_kv_heads < 1) return fail(QKV_CTE_ERR_INVALID, "fused mode needs n_kv_heads >= 1");
  } else if (d.mode == QKV_CTE_MODE_SEPARATE) {
    if (d.n_kv_heads != 0) return fail(QKV_CTE_ERR_INVALID, "separate mode needs n_kv_heads == 0");
    if (d.n_q_heads < 1) return fail(QKV_CTE_ERR_INVALID, "separate mode needs n_q_heads >= 1");
  } else {
    return fail(QKV_CTE_ERR_INVALID, "unknown mode %d", d.mode);
  }
  if (d.norm < QKV_CTE_NORM_NONE || d.norm > QKV_CTE_NORM_HEAD_LAYER)
    return fail(QKV_CTE_ERR_INVALID, "unknown norm %d", d.norm);
  if (d.rope != 0 && d.rope != 1) return fail(QKV_CTE_ERR_INVALID, "rope must be 0 or 1");
  if (!(d.eps >= 0.0f) || d.eps > 1e30f) return fail(QKV_CTE_ERR_INVALID, "eps must be finite and >= 0");
  if (d.output_layout != QKV_CTE_LAYOUT_BSD && d.output_layout != QKV_CTE_LAYOUT_NBSD)
    return fail(QKV_CTE_ERR_INVALID, "unknown output layout");
  const uint32_t known_flags = QKV_CTE_FLAG_TEST_STALL | QKV_CTE_FLAG_PROFILE | QKV_CTE_FLAG_SERIAL_PASSES |
                               QKV_CTE_FLAG_GEMM_CTA_PAIR | QKV_CTE_FLAG_GEMM_SINGLE_CTA |
                               QKV_CTE_FLAG_NORM_IN_GEMM | QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE;
  if ((d.flags & ~known_flags) != 0) return fail(QKV_CTE_ERR_INVALID, "unknown flags 0x%x", d.flags);
  if ((d.flags & QKV_CTE_FLAG_GEMM_CTA_PAIR) && (d.flags & QKV_CTE_FLAG_GEMM_SINGLE_CTA))
    return fail(QKV_CTE_ERR_INVALID, "QKV_CTE_FLAG_GEMM_CTA_PAIR and QKV_CTE_FLAG_GEMM_SINGLE_CTA exclude each other");
  if (d.input_layout != QKV_CTE_INPUT_ROW_FP8 && d.input_layout != QKV_CTE_INPUT_PACKED &&
      d.input_layout != QKV_CTE_INPUT_BF16)
    return fail(QKV_CTE_ERR_INVALID, "unknown input layout %d", d.input_layout);
  const long long I = (long long)(d.n_q_heads + 2LL * d.n_kv_heads) * d.d_head;
  if (I > INT32_MAX / 2) return fail(QKV_CTE_ERR_UNSUPPORTED, "output width too large");
  // The norm/RoPE pass and the per-head epilogue work on 16-column chunks paired with
  // the chunk d_head/2 away (the rotate-half partner), so d_head/2 must be a multiple
  // of 16 whenever either of them runs.
  if ((d.norm != QKV_CTE_NORM_NONE || d.rope) && d.d_head % 32 != 0)
    return fail(QKV_CTE_ERR_UNSUPPORTED, "a norm or RoPE needs d_head %% 32 == 0 (got %d)", d.d_head);
  const int tile_n = choose_tile_n(d, (int)I);
  if (!gemm_tile_supported(tile_n)) return fail(QKV_CTE_ERR_UNSUPPORTED, "tile_n %d not built", tile_n);
  if (head_norm_in_epilogue(d) && tile_n % d.d_head != 0)
    return fail(QKV_CTE_ERR_UNSUPPORTED, "per-head norm needs whole heads per tile: tile_n %d, d_head %d", tile_n,
                d.d_head);

  qkv_cte_plan_s* p = new (std::nothrow) qkv_cte_plan_s();
  if (p == nullptr) return fail(QKV_CTE_ERR_INVALID, "out of host memory");
  p->d = d;
  GemmShape& g = p->g;
  g.T = (int)d.tokens;
  g.H = d.hidden;
  g.I = (int)I;
  g.tile_n = tile_n;
  // The pair form is the default once there is more than one 128-row block: it stages
  // half of each W tile per SM and issues the MMAs for two SMs from one thread;
  // measured ~1% faster at 480p.
  if (d.flags & QKV_CTE_FLAG_GEMM_CTA_PAIR)
    g.cta_pair = 1;
  else if (d.flags & QKV_CTE_FLAG_GEMM_SINGLE_CTA)
    g.cta_pair = 0;
  else
    g.cta_pair = d.tokens > 128 ? 1 : 0;
  g.blocks128 = (g.T + 127) / 128;
  g.m_tiles = g.cta_pair ? (g.T + 255) / 256 : g.blocks128;
  g.n_tiles = (g.I + tile_n - 1) / tile_n;
  g.k_stages = g.H / 128;
  if ((long long)g.m_tiles * g.n_tiles > INT32_MAX) {
    delete p;
    return fail(QKV_CTE_ERR_UNSUPPORTED, "%d x %d output tiles exceed INT32_MAX", g.m_tiles, g.n_tiles);
  }
  g.sf_chunks = gemm_sf_chunks(tile_n);
  p->q_end = d.n_q_heads * d.d_head;
  p->k_end = p->q_end + d.n_kv_heads * d.d_head;
  g.n_qk_tiles = (p->k_end + tile_n - 1) / tile_n;
  if (g.n_qk_tiles > g.n_tiles) g.n_qk_tiles = g.n_tiles;
  // The norm/RoPE pass (and its hand-off) runs for the across-heads norm, or RoPE
  // without a norm; the per-head norms finish in the GEMM's epilogue.
  const bool second_pass = !head_norm_in_epilogue(d) && (d.norm != QKV_CTE_NORM_NONE || d.rope);
  p->second_pass = second_pass;
  p->fused_norm = second_pass && g.cta_pair && !per_head_norm(d) && (d.flags & QKV_CTE_FLAG_NORM_IN_GEMM) &&
                  !(d.flags & QKV_CTE_FLAG_SERIAL_PASSES);
  make_bands(g, band_tiles(g), band_m_chunks());
  WorkspaceLayout& w = p->ws;
  w.status_off = 0;
  w.sumsq_off = 256;
  w.sf_off = w.sumsq_off + align_up((size_t)g.T * 2 * sizeof(float), 256);
  w.ready_off = w.sf_off + align_up((size_t)g.n_tiles * g.k_stages * g.sf_chunks * kSfBlockBytesPerChunk, 256);
  w.sm_busy_off = w.ready_off + align_up((size_t)g.blocks128 * sizeof(uint32_t), 256);
  w.qk_off = w.sm_busy_off + align_up((size_t)kSmTable * sizeof(uint32_t), 256);
  const size_t hand_rows = second_pass ? (size_t)g.blocks128 * 128 : 0;
  w.qk_exp_off = w.qk_off + align_up(hand_rows * p->k_end * sizeof(uint16_t), 256);
  w.stats_off = w.qk_exp_off + align_up(hand_rows * (p->k_end / 16), 256);
  const size_t qk_heads = (size_t)(d.n_q_heads + d.n_kv_heads);
  size_t stats_bytes = 0;
  if (per_head_norm(d) && !head_norm_in_epilogue(d))
    stats_bytes = hand_rows * qk_heads *
                  (d.norm == QKV_CTE_NORM_HEAD_RMS ? sizeof(float) : 4 * sizeof(float) * stat_parts(d.d_head, tile_n));
  w.act_off = w.stats_off + align_up(stats_bytes, 256);
  const bool produced = d.input_layout != QKV_CTE_INPUT_ROW_FP8;
  w.act_scale_off = w.act_off + (produced ? align_up((size_t)g.T * g.H, 256) : 0);
  w.total = w.act_scale_off + (produced ? align_up((size_t)g.T * sizeof(float), 256) : 0);
  *workspace_bytes = w.total;
  *out = p;
  return ok();
}

int qkv_cte_get_plan_info(qkv_cte_plan_t plan, qkv_cte_plan_info* info) {
  if (plan == nullptr || info == nullptr) return fail(QKV_CTE_ERR_INVALID, "null argument");
  info->tile_n = plan->g.tile_n;
  info->m_tiles = plan->g.m_tiles;
  info->n_tiles = plan->g.n_tiles;
  info->n_bands = plan->g.n_bands;
  info->cta_pair = plan->g.cta_pair;
  info->norm_in_gemm = plan->fused_norm ? 1 : 0;
  info->workspace_bytes = (int64_t)plan->ws.total;
  return ok();
}

void qkv_cte_destroy(qkv_cte_plan_t plan) {
  if (plan == nullptr) return;
  for (cudaEvent_t e : plan->ev)
    if (e != nullptr) cudaEventDestroy(e);
  qkv_cte_destroy(plan->chunk_plan);
  qkv_cte_destroy(plan->tail_plan);
  for (cudaEvent_t e : {plan->ev_start, plan->ev_in[0], plan->ev_in[1], plan->ev_done[0], plan->ev_done[1],
                        plan->ev_out[0], plan->ev_out[1]})
    if (e != nullptr) cudaEventDestroy(e);
  if (plan->h2d != nullptr) cudaStreamDestroy(plan->h2d);
  if (plan->d2h != nullptr) cudaStreamDestroy(plan->d2h);
  delete plan;
}

int qkv_cte_pass_times(qkv_cte_plan_t plan, float* ms) {
  if (plan == nullptr || ms == nullptr) return fail(QKV_CTE_ERR_INVALID, "null argument");
  if (!(plan->d.flags & QKV_CTE_FLAG_PROFILE)) return fail(QKV_CTE_ERR_INVALID, "plan made without QKV_CTE_FLAG_PROFILE");
  if (!plan->ran) return fail(QKV_CTE_ERR_INVALID, "plan has not run");
  cudaError_t e = cudaEventSynchronize(plan->ev[1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms[3], plan->ev[0], plan->ev[1]);
  unsigned long long st[4] = {0, 0, 0, 0};
  if (e == cudaSuccess)
    e = cudaMemcpy(st, static_cast<const uint8_t*>(plan->last_workspace) + kStampOffset, sizeof(st),
                   cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "pass times: %s", cudaGetErrorString(e));
  ms[1] = st[1] > st[0] ? (float)((st[1] - st[0]) * 1e-6) : 0.0f;
  ms[2] = (plan->has_norm_pass && st[3] > st[2]) ? (float)((st[3] - st[2]) * 1e-6) : 0.0f;
  // The rest of the run: the producer step, the scale repack and clears, launch gaps.
  // The GEMM starts its timed span once that work is complete (it waits for it).
  const unsigned long long last = plan->has_norm_pass && st[3] > st[1] ? st[3] : st[1];
  const float spans = last > st[0] ? (float)((last - st[0]) * 1e-6) : 0.0f;
  ms[0] = ms[3] > spans ? ms[3] - spans : 0.0f;
  return ok();
}

int qkv_cte_run(qkv_cte_plan_t plan, const uint8_t* A, const float* a_scale, const uint8_t* W,
                const uint8_t* w_sf, const float* w_col_scale, const uint16_t* bias, const uint16_t* gamma_q,
                const uint16_t* gamma_k, const float* cos_table, const float* sin_table, uint16_t* O,
                float* sumsq, float* inv_rms, void* workspace, size_t workspace_bytes, void* stream) {
  if (plan == nullptr) return fail(QKV_CTE_ERR_INVALID, "null plan");
  const qkv_cte_desc& d = plan->d;
  const GemmShape& g = plan->g;
  if (g.T == 0) {
    // An empty problem reads and writes no tensor; it only resets the status word.
    if (workspace != nullptr) {
      cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
    }
    return ok();
  }
  const bool produced = d.input_layout != QKV_CTE_INPUT_ROW_FP8;
  if (!A || !W || !w_sf || !O || !workspace)
    return fail(QKV_CTE_ERR_INVALID, "A, W, w_sf, O and workspace are required");
  if (!produced && !a_scale) return fail(QKV_CTE_ERR_INVALID, "a_scale is required with separate FP8 rows");
  if (produced && a_scale)
    return fail(QKV_CTE_ERR_INVALID, "a_scale must be NULL with a packed or bf16 input (the scales come from it)");
  if (d.norm && d.n_q_heads > 0 && !gamma_q) return fail(QKV_CTE_ERR_INVALID, "norm with a Q segment needs gamma_q");
  if (d.norm && d.n_kv_heads > 0 && !gamma_k) return fail(QKV_CTE_ERR_INVALID, "norm with a K segment needs gamma_k");
  if (gamma_k && !(d.norm && d.n_kv_heads > 0))
    return fail(QKV_CTE_ERR_INVALID, "gamma_k given but the call has no normalised K segment");
  if (gamma_q && !(d.norm && d.n_q_heads > 0))
    return fail(QKV_CTE_ERR_INVALID, "gamma_q given but the call has no normalised Q segment");
  if (inv_rms && per_head_norm(d))
    return fail(QKV_CTE_ERR_INVALID, "inv_rms is an output of the across-heads norm only (per-head norm: NULL)");
  if (d.rope && (!cos_table || !sin_table)) return fail(QKV_CTE_ERR_INVALID, "rope needs cos and sin tables");
  if (!d.rope && (cos_table || sin_table)) return fail(QKV_CTE_ERR_INVALID, "cos/sin given but rope is off");
  if (!aligned(A, d.input_layout == QKV_CTE_INPUT_PACKED ? 4 : 16) || !aligned(W, 16) || !aligned(O, 32))
    return fail(QKV_CTE_ERR_UNSUPPORTED,
                "A must be 16-byte aligned (4-byte for packed rows), W 16-byte and O 32-byte aligned");
  if ((a_scale && !aligned(a_scale, 4)) || !aligned(w_sf, 4) || (sumsq && !aligned(sumsq, 4)) || (inv_rms && !aligned(inv_rms, 4)))
    return fail(QKV_CTE_ERR_UNSUPPORTED, "a_scale, w_sf, sumsq and inv_rms must be 4-byte aligned");
  if ((w_col_scale && !aligned(w_col_scale, 16)) || (bias && !aligned(bias, 16)) ||
      (gamma_q && !aligned(gamma_q, 16)) || (gamma_k && !aligned(gamma_k, 16)))
    return fail(QKV_CTE_ERR_UNSUPPORTED, "w_col_scale, bias and gamma must be 16-byte aligned");
  if ((cos_table && !aligned(cos_table, 32)) || (sin_table && !aligned(sin_table, 32)))
    return fail(QKV_CTE_ERR_UNSUPPORTED, "cos and sin tables must be 32-byte aligned");
  if (!aligned(workspace, 256)) return fail(QKV_CTE_ERR_UNSUPPORTED, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->ws.total)
    return fail(QKV_CTE_ERR_INVALID, "workspace of %zu bytes is smaller than the planned %zu",
                workspace_bytes, plan->ws.total);

  DeviceInfo dev;
  int rc = device_info(&dev);
  if (rc != QKV_CTE_OK) return rc;
  if (!(dev.major == 10 && dev.minor == 3))
    return fail(QKV_CTE_ERR_ARCH, "device is sm_%d%d; this library is built for sm_103a", dev.major, dev.minor);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // With a packed or bf16 input the GEMM reads the codes and scales the producer
  // step writes into the workspace.
  const uint8_t* A_codes = produced ? ws + plan->ws.act_off : A;
  const float* A_scale = produced ? reinterpret_cast<const float*>(ws + plan->ws.act_scale_off) : a_scale;
  CUtensorMap tmA, tmW;
  if ((rc = encode_operand(&tmA, A_codes, (uint64_t)g.T, (uint64_t)g.H, 128u, "A")) != QKV_CTE_OK) return rc;
  const uint32_t w_box_rows = g.cta_pair ? (uint32_t)g.tile_n / 2 : (uint32_t)g.tile_n;
  if ((rc = encode_operand(&tmW, W, (uint64_t)g.I, (uint64_t)g.H, w_box_rows, "W")) != QKV_CTE_OK) return rc;

  uint32_t* status = reinterpret_cast<uint32_t*>(ws + plan->ws.status_off);
  const bool need_ss = d.norm || sumsq != nullptr;
  float* ss = sumsq ? sumsq : reinterpret_cast<float*>(ws + plan->ws.sumsq_off);
  uint8_t* sf_packed = ws + plan->ws.sf_off;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool prof = (d.flags & QKV_CTE_FLAG_PROFILE) != 0;
  cudaError_t e = cudaSuccess;
  if (prof) {
    int cur = 0;
    cudaGetDevice(&cur);
    if (plan->ev[0] != nullptr && plan->ev_device != cur)
      return fail(QKV_CTE_ERR_INVALID, "a profiled plan must stay on one device");
    for (int i = 0; i < 2 && plan->ev[i] == nullptr; ++i)
      if ((e = cudaEventCreate(&plan->ev[i])) != cudaSuccess)
        return fail(QKV_CTE_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
    plan->ev_device = cur;
    if ((e = cudaEventRecord(plan->ev[0], s)) != cudaSuccess)
      return fail(QKV_CTE_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
  }

  if (d.input_layout == QKV_CTE_INPUT_PACKED)
    e = launch_unpack_rows(A, g.T, g.H, ws + plan->ws.act_off, reinterpret_cast<float*>(ws + plan->ws.act_scale_off),
                           s, dev.sms);
  else if (d.input_layout == QKV_CTE_INPUT_BF16)
    e = launch_row_quantize(reinterpret_cast<const uint16_t*>(A), g.T, g.H, ws + plan->ws.act_off,
                            reinterpret_cast<float*>(ws + plan->ws.act_scale_off), nullptr, s, dev.sms);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "producer launch: %s", cudaGetErrorString(e));

  uint32_t* ready = reinterpret_cast<uint32_t*>(ws + plan->ws.ready_off);
  uint32_t* sm_busy = reinterpret_cast<uint32_t*>(ws + plan->ws.sm_busy_off);
  unsigned long long* stamps = reinterpret_cast<unsigned long long*>(ws + kStampOffset);
  uint32_t* task_next = reinterpret_cast<uint32_t*>(ws + kTaskCounterOffset);
  const bool head_stats = per_head_norm(d) && !head_norm_in_epilogue(d);
  float* stats = head_stats ? reinterpret_cast<float*>(ws + plan->ws.stats_off) : nullptr;
  // the RMS statistics are sums accumulated with atomics: they start at zero
  const size_t zero_stats =
      head_stats && d.norm == QKV_CTE_NORM_HEAD_RMS ? (size_t)g.blocks128 * 128 * (d.n_q_heads + d.n_kv_heads) : 0;
  e = launch_prep(g, w_sf, sf_packed, need_ss ? ss : nullptr, need_ss ? (size_t)g.T * 2 : 0, ready, sm_busy, status,
                  stamps, task_next, stats, zero_stats, s, dev.sms, produced);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "prep launch: %s", cudaGetErrorString(e));

  GemmArgs ga;
  ga.a_scale = A_scale;
  ga.w_col_scale = w_col_scale;
  ga.bias = bias;
  ga.sf_packed = sf_packed;
  ga.O = O;
  uint16_t* qk_val = plan->second_pass ? reinterpret_cast<uint16_t*>(ws + plan->ws.qk_off) : nullptr;
  uint8_t* qk_exp = plan->second_pass ? ws + plan->ws.qk_exp_off : nullptr;
  ga.qk_val = qk_val;
  ga.qk_exp = qk_exp;
  ga.sumsq = need_ss ? ss : nullptr;
  ga.ready = ready;
  ga.sm_busy = sm_busy;
  ga.stamps = stamps;
  ga.tile_next = reinterpret_cast<uint32_t*>(ws + kTileCounterOffset);
  ga.status = status;
  ga.q_end = plan->q_end;
  ga.k_end = plan->k_end;
  ga.flags = d.flags;
  ga.d_head = d.d_head;
  ga.nbsd = d.output_layout == QKV_CTE_LAYOUT_NBSD ? 1 : 0;
  ga.head_norm = head_norm_in_epilogue(d) ? d.norm : 0;
  ga.rope = head_norm_in_epilogue(d) ? d.rope : 0;
  ga.stats_kind = head_stats ? d.norm : 0;
  ga.head_stats = stats;
  ga.stat_parts = stat_parts(d.d_head, g.tile_n);
  ga.eps = d.eps;
  ga.gamma_q = gamma_q;
  ga.gamma_k = gamma_k;
  ga.cos_t = cos_table;
  ga.sin_t = sin_table;
  NormRopeArgs na{};
  na.T = g.T;
  na.I = g.I;
  na.n_q = d.n_q_heads;
  na.n_kv = d.n_kv_heads;
  na.d_head = d.d_head;
  na.norm = d.norm;
  na.rope = d.rope;
  na.eps = d.eps;
  na.sumsq = ss;
  na.qk_val = qk_val;
  na.qk_exp = qk_exp;
  na.gamma_q = gamma_q;
  na.gamma_k = gamma_k;
  na.cos_t = cos_table;
  na.sin_t = sin_table;
  na.O = O;
  na.inv_rms = inv_rms;
  na.nbsd = d.output_layout == QKV_CTE_LAYOUT_NBSD ? 1 : 0;
  na.ready = ready;
  na.sm_busy = sm_busy;
  na.ready_target = 4u * (uint32_t)g.n_qk_tiles;
  na.status = status;
  na.stamps = stamps + 2;
  na.task_next = task_next;
  {
    // every pair has claimed its first tail tile: the pass's held-back warps join in
    const long long tiles = (long long)g.m_tiles * g.n_tiles;
    const long long pairs = std::min<long long>(tiles, dev.sms / 2);
    const bool tail = g.cta_pair && pairs > 0 && tiles / pairs > kClaimedWaves;
    na.gemm_claims = tail ? ga.tile_next : nullptr;
    na.release_at = tail ? (uint32_t)pairs : 0xFFFFFFFFu;
  }
  na.head_kind = head_stats ? d.norm : 0;
  na.head_stats = stats;
  na.stat_parts = stat_parts(d.d_head, g.tile_n);
  na.tile_n = g.tile_n;
  CUtensorMap tmSF;
  if ((rc = encode_scales(&tmSF, sf_packed, g)) != QKV_CTE_OK) return rc;
  // On request the norm/RoPE tasks run inside the CTA-pair GEMM's epilogue warps;
  // otherwise as their own kernel, overlapped with the GEMM (or after it, serialised).
  const bool fused = plan->second_pass && plan->fused_norm;
  e = launch_gemm(g, tmA, tmW, tmSF, ga, s, dev.sms, fused ? &na : nullptr);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));

  if (plan->second_pass && !fused) {
    e = launch_norm_rope(na, s, dev.sms, (d.flags & QKV_CTE_FLAG_SERIAL_PASSES) == 0);
    if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "norm/rope launch: %s", cudaGetErrorString(e));
  }
  if (prof) {
    cudaEventRecord(plan->ev[1], s);
    plan->ran = true;
    plan->has_norm_pass = plan->second_pass;
    plan->last_workspace = workspace;
  }
  return ok();
}

int qkv_cte_status(void* workspace, void* stream) {
  if (workspace == nullptr) return fail(QKV_CTE_ERR_INVALID, "null workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (word == 0) return ok();
  const uint32_t known = kErrProducerEmptyWait | kErrMmaFullWait | kErrMmaTmemEmptyWait |
                         kErrEpilogueTmemFullWait | kErrDrainWait | kErrNormReadyWait | kErrTileIdWait;
  if (word & ~known)
    return fail(QKV_CTE_ERR_INVALID,
                "workspace status word holds 0x%x, which no run wrote: zero the workspace before its first use",
                word);
  const uint32_t zero = 0;
  e = cudaMemcpyAsync(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
  return fail(QKV_CTE_ERR_DEVICE_TIMEOUT,
              "device wait ran out (status 0x%x:%s%s%s%s%s%s%s)", word,
              (word & kErrProducerEmptyWait) ? " load-stage-free" : "",
              (word & kErrMmaFullWait) ? " mma-operands-ready" : "",
              (word & kErrMmaTmemEmptyWait) ? " mma-accumulator-free" : "",
              (word & kErrEpilogueTmemFullWait) ? " epilogue-accumulator-ready" : "",
              (word & kErrDrainWait) ? " drain" : "",
              (word & kErrNormReadyWait) ? " norm-panel-ready" : "",
              (word & kErrTileIdWait) ? " tile-id" : "");
}

namespace {

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_rows(int64_t tokens, int32_t hidden, const char* who) {
  if (tokens < 0) return fail(QKV_CTE_ERR_INVALID, "%s: tokens must be >= 0", who);
  if (tokens > INT32_MAX) return fail(QKV_CTE_ERR_UNSUPPORTED, "%s: tokens > INT32_MAX", who);
  if (hidden <= 0) return fail(QKV_CTE_ERR_INVALID, "%s: hidden must be > 0", who);
  if (hidden % 16 != 0) return fail(QKV_CTE_ERR_UNSUPPORTED, "%s: hidden %d is not a multiple of 16", who, hidden);
  return QKV_CTE_OK;
}

int check_device(DeviceInfo* dev) {
  int rc = device_info(dev);
  if (rc != QKV_CTE_OK) return rc;
  if (!(dev->major == 10 && dev->minor == 3))
    return fail(QKV_CTE_ERR_ARCH, "device is sm_%d%d; this library is built for sm_103a", dev->major, dev->minor);
  return QKV_CTE_OK;
}

}  // namespace

int qkv_cte_row_quantize(const uint16_t* X, int64_t tokens, int32_t hidden, uint8_t* A, float* a_scale,
                         uint8_t* packed, void* stream) {
  int rc = check_rows(tokens, hidden, "qkv_cte_row_quantize");
  if (rc != QKV_CTE_OK) return rc;
  if (tokens == 0) return ok();  // empty tensors may come as null pointers
  if ((A == nullptr) != (a_scale == nullptr))
    return fail(QKV_CTE_ERR_INVALID, "qkv_cte_row_quantize: give both A and a_scale, or neither");
  if (A == nullptr && packed == nullptr)
    return fail(QKV_CTE_ERR_INVALID, "qkv_cte_row_quantize: no output (A + a_scale and/or packed)");
  if (X == nullptr) return fail(QKV_CTE_ERR_INVALID, "qkv_cte_row_quantize: null X");
  if (!aligned(X, 16) || (A && !aligned(A, 16)) || (a_scale && !aligned(a_scale, 4)) || (packed && !aligned(packed, 4)))
    return fail(QKV_CTE_ERR_UNSUPPORTED,
                "qkv_cte_row_quantize: X and A must be 16-byte aligned, a_scale and packed 4-byte aligned");
  const size_t T = (size_t)tokens, H = (size_t)hidden;
  if (overlaps(X, T * H * 2, A, T * H) || overlaps(X, T * H * 2, a_scale, T * 4) ||
      overlaps(X, T * H * 2, packed, T * (H + 4)) || overlaps(A, T * H, packed, T * (H + 4)) ||
      overlaps(a_scale, T * 4, packed, T * (H + 4)) || overlaps(A, T * H, a_scale, T * 4))
    return fail(QKV_CTE_ERR_INVALID, "qkv_cte_row_quantize: buffers overlap");
  DeviceInfo dev;
  if ((rc = check_device(&dev)) != QKV_CTE_OK) return rc;
  cudaError_t e = launch_row_quantize(X, (int)tokens, hidden, A, a_scale, packed, static_cast<cudaStream_t>(stream),
                                      dev.sms);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "row quantise launch: %s", cudaGetErrorString(e));
  return ok();
}

int qkv_cte_unpack_rows(const uint8_t* packed, int64_t tokens, int32_t hidden, uint8_t* A, float* a_scale,
                        void* stream) {
  int rc = check_rows(tokens, hidden, "qkv_cte_unpack_rows");
  if (rc != QKV_CTE_OK) return rc;
  if (tokens == 0) return ok();
  if (packed == nullptr || A == nullptr || a_scale == nullptr)
    return fail(QKV_CTE_ERR_INVALID, "qkv_cte_unpack_rows: packed, A and a_scale are required");
  if (!aligned(packed, 4) || !aligned(A, 16) || !aligned(a_scale, 4))
    return fail(QKV_CTE_ERR_UNSUPPORTED,
                "qkv_cte_unpack_rows: packed and a_scale must be 4-byte aligned, A 16-byte aligned");
  const size_t T = (size_t)tokens, H = (size_t)hidden;
  if (overlaps(packed, T * (H + 4), A, T * H) || overlaps(packed, T * (H + 4), a_scale, T * 4) ||
      overlaps(A, T * H, a_scale, T * 4))
    return fail(QKV_CTE_ERR_INVALID, "qkv_cte_unpack_rows: buffers overlap");
  DeviceInfo dev;
  if ((rc = check_device(&dev)) != QKV_CTE_OK) return rc;
  cudaError_t e = launch_unpack_rows(packed, (int)tokens, hidden, A, a_scale, static_cast<cudaStream_t>(stream),
                                     dev.sms);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "unpack launch: %s", cudaGetErrorString(e));
  return ok();
}

int qkv_cte_interleaved_to_rotate_half(const void* src, void* dst, int64_t rows, int64_t row_bytes,
                                       int32_t n_q_heads, int32_t n_kv_heads, int32_t d_head, void* stream) {
  const char* who = "qkv_cte_interleaved_to_rotate_half";
  if (rows < 0 || row_bytes <= 0) return fail(QKV_CTE_ERR_INVALID, "%s: rows must be >= 0, row_bytes > 0", who);
  if (d_head <= 0 || d_head % 2 != 0) return fail(QKV_CTE_ERR_INVALID, "%s: d_head must be even and > 0", who);
  if (n_q_heads < 0 || n_kv_heads < 0) return fail(QKV_CTE_ERR_INVALID, "%s: negative head count", who);
  const long long qk_rows = (long long)(n_q_heads + (long long)n_kv_heads) * d_head;
  if (qk_rows > rows) return fail(QKV_CTE_ERR_INVALID, "%s: %lld Q/K rows exceed the %lld rows given", who,
                                  qk_rows, (long long)rows);
  if (rows > 0 && row_bytes > INT64_MAX / rows) return fail(QKV_CTE_ERR_UNSUPPORTED, "%s: size overflow", who);
  if (rows == 0) return ok();
  if (src == nullptr || dst == nullptr) return fail(QKV_CTE_ERR_INVALID, "%s: null buffer", who);
  if (overlaps(src, (size_t)(rows * row_bytes), dst, (size_t)(rows * row_bytes)))
    return fail(QKV_CTE_ERR_INVALID, "%s: src and dst overlap (the permutation is not in place)", who);
  DeviceInfo dev;
  int rc = check_device(&dev);
  if (rc != QKV_CTE_OK) return rc;
  cudaError_t e = launch_permute_rows(src, dst, rows, row_bytes, qk_rows, d_head, static_cast<cudaStream_t>(stream),
                                      dev.sms);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "permute launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Host-streaming entry point
//
// The activations come from (and the output goes to) pinned host memory. Rows are
// independent, so the call cuts them into chunks and pipelines three streams: the
// upload of chunk i+1, the path on chunk i (on the caller's stream) and the readback
// of chunk i-1, with two staging slots on the device ordered by events. On Grace the
// link moves ~0.2 TB/s each way, so at the Wan shapes the readback of O bounds the
// call and the upload and the computation hide under it.
// ---------------------------------------------------------------------------

namespace {

int input_row_bytes(const qkv_cte_desc& d) {
  if (d.input_layout == QKV_CTE_INPUT_PACKED) return d.hidden + 4;
  if (d.input_layout == QKV_CTE_INPUT_BF16) return 2 * d.hidden;
  return d.hidden;
}

int effective_chunk_rows(const qkv_cte_plan_s* p, int32_t chunk_rows) {
  // default: 2048 rows (measured at 480p: 5.55 ms per call, against 5.68 with 4096 and
  // 5.96 with 8192; the readback of O alone takes ~5.2 ms)
  long long r = chunk_rows > 0 ? chunk_rows : 2048;
  r = (r + 255) / 256 * 256;  // whole 256-row tiles of the CTA-pair GEMM
  if (r > p->g.T) r = p->g.T;
  return static_cast<int>(r);
}

struct HostScratch {
  size_t status, a[2], s[2], o[2], ws, total;
};

HostScratch host_scratch_layout(const qkv_cte_plan_s* p, int rows, size_t chunk_ws) {
  HostScratch h;
  h.status = 0;
  size_t off = 256;
  const size_t a_bytes = align_up((size_t)rows * input_row_bytes(p->d), 256);
  const size_t s_bytes = align_up((size_t)rows * sizeof(float), 256);
  const size_t o_bytes = align_up((size_t)rows * p->g.I * sizeof(uint16_t), 256);
  for (int i = 0; i < 2; ++i) {
    h.a[i] = off;
    off += a_bytes;
    h.s[i] = off;
    off += s_bytes;
    h.o[i] = off;
    off += o_bytes;
  }
  h.ws = off;
  h.total = off + align_up(chunk_ws, 256);
  return h;
}

// The plans for chunks of `rows` tokens (and the tail), created once per chunk size.
int ensure_chunk_plans(qkv_cte_plan_s* p, int rows) {
  if (p->chunk_plan != nullptr && p->chunk_rows == rows) return QKV_CTE_OK;
  qkv_cte_destroy(p->chunk_plan);
  qkv_cte_destroy(p->tail_plan);
  p->chunk_plan = p->tail_plan = nullptr;
  p->chunk_rows = 0;
  qkv_cte_desc cd = p->d;
  cd.flags &= ~QKV_CTE_FLAG_PROFILE;
  cd.tokens = rows;
  size_t ws = 0;
  int rc = qkv_cte_plan(&p->chunk_plan, &cd, &ws);
  if (rc != QKV_CTE_OK) return rc;
  const int tail = p->g.T % rows;
  if (tail != 0) {
    cd.tokens = tail;
    rc = qkv_cte_plan(&p->tail_plan, &cd, &ws);
    if (rc != QKV_CTE_OK) return rc;
  }
  p->chunk_rows = rows;
  return QKV_CTE_OK;
}

int ensure_host_streams(qkv_cte_plan_s* p) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (p->h2d != nullptr) {
    if (p->host_device != dev) return fail(QKV_CTE_ERR_INVALID, "a plan used with host buffers must stay on one device");
    return QKV_CTE_OK;
  }
  e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&p->ev_start, &p->ev_in[0], &p->ev_in[1], &p->ev_done[0], &p->ev_done[1], &p->ev_out[0],
                          &p->ev_out[1]})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "stream/event creation: %s", cudaGetErrorString(e));
  p->host_device = dev;
  return QKV_CTE_OK;
}

bool pinned_host(const void* ptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" int qkv_cte_host_scratch_bytes(qkv_cte_plan_t plan, int32_t chunk_rows, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return fail(QKV_CTE_ERR_INVALID, "null argument");
  *bytes = 0;
  if (plan->g.T == 0) return ok();
  const int rows = effective_chunk_rows(plan, chunk_rows);
  const int rc = ensure_chunk_plans(plan, rows);
  if (rc != QKV_CTE_OK) return rc;
  *bytes = host_scratch_layout(plan, rows, plan->chunk_plan->ws.total).total;
  return ok();
}

extern "C" int qkv_cte_run_host(qkv_cte_plan_t plan, const void* A_host, const float* a_scale_host, const uint8_t* W,
                                const uint8_t* w_sf, const float* w_col_scale, const uint16_t* bias,
                                const uint16_t* gamma_q, const uint16_t* gamma_k, const float* cos_table,
                                const float* sin_table, uint16_t* O_host, float* sumsq, float* inv_rms, void* scratch,
                                size_t scratch_bytes, int32_t chunk_rows, void* stream) {
  if (plan == nullptr) return fail(QKV_CTE_ERR_INVALID, "null plan");
  const qkv_cte_desc& d = plan->d;
  const int T = plan->g.T;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (scratch != nullptr) {
      cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);
      if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
    }
    return ok();
  }
  const bool row_fp8 = d.input_layout == QKV_CTE_INPUT_ROW_FP8;
  if (!A_host || !O_host || !scratch) return fail(QKV_CTE_ERR_INVALID, "A_host, O_host and scratch are required");
  if (row_fp8 != (a_scale_host != nullptr))
    return fail(QKV_CTE_ERR_INVALID, "a_scale_host is required with separate FP8 rows and must be NULL otherwise");
  if (!pinned_host(A_host) || !pinned_host(O_host) || (a_scale_host && !pinned_host(a_scale_host)))
    return fail(QKV_CTE_ERR_UNSUPPORTED,
                "A_host, a_scale_host and O_host must be pinned host memory (cudaHostAlloc / cudaHostRegister)");
  if (!aligned(scratch, 256)) return fail(QKV_CTE_ERR_UNSUPPORTED, "scratch must be 256-byte aligned");
  const int rows = effective_chunk_rows(plan, chunk_rows);
  int rc = ensure_chunk_plans(plan, rows);
  if (rc != QKV_CTE_OK) return rc;
  const HostScratch hs = host_scratch_layout(plan, rows, plan->chunk_plan->ws.total);
  if (scratch_bytes < hs.total)
    return fail(QKV_CTE_ERR_INVALID, "scratch of %zu bytes is smaller than the %zu this chunk size needs",
                scratch_bytes, hs.total);
  if ((rc = ensure_host_streams(plan)) != QKV_CTE_OK) return rc;

  uint8_t* sc = static_cast<uint8_t*>(scratch);
  uint32_t* status = reinterpret_cast<uint32_t*>(sc + hs.status);
  const size_t in_row = (size_t)input_row_bytes(d);
  const int I = plan->g.I;
  const int dh = d.d_head;
  const bool nbsd = d.output_layout == QKV_CTE_LAYOUT_NBSD;
  const int heads = I / dh;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaEventRecord(plan->ev_start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->h2d, plan->ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->d2h, plan->ev_start, 0);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "stream ordering: %s", cudaGetErrorString(e));
  const int chunks = (T + rows - 1) / rows;
  for (int i = 0; i < chunks; ++i) {
    const int slot = i & 1;
    const int r0 = i * rows;
    const int n = T - r0 < rows ? T - r0 : rows;
    qkv_cte_plan_s* cp = n == rows ? plan->chunk_plan : plan->tail_plan;
    uint8_t* a_dev = sc + hs.a[slot];
    float* s_dev = reinterpret_cast<float*>(sc + hs.s[slot]);
    uint16_t* o_dev = reinterpret_cast<uint16_t*>(sc + hs.o[slot]);
    // upload: the slot is free once the path on chunk i-2 has read it
    if (i >= 2) e = cudaStreamWaitEvent(plan->h2d, plan->ev_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(a_dev, static_cast<const uint8_t*>(A_host) + (size_t)r0 * in_row, (size_t)n * in_row,
                          cudaMemcpyHostToDevice, plan->h2d);
    if (e == cudaSuccess && row_fp8)
      e = cudaMemcpyAsync(s_dev, a_scale_host + r0, (size_t)n * sizeof(float), cudaMemcpyHostToDevice, plan->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(plan->ev_in[slot], plan->h2d);
    // the path on this chunk, on the caller's stream, once its rows are in and the
    // output slot's previous readback (chunk i-2) is done
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, plan->ev_in[slot], 0);
    if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(s, plan->ev_out[slot], 0);
    if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "chunk %d upload: %s", i, cudaGetErrorString(e));
    rc = qkv_cte_run(cp, a_dev, row_fp8 ? s_dev : nullptr, W, w_sf, w_col_scale, bias, gamma_q, gamma_k,
                     cos_table ? cos_table + (size_t)r0 * dh : nullptr, sin_table ? sin_table + (size_t)r0 * dh : nullptr,
                     o_dev, sumsq ? sumsq + 2 * (size_t)r0 : nullptr, inv_rms ? inv_rms + 2 * (size_t)r0 : nullptr,
                     sc + hs.ws, hs.total - hs.ws, s);
    if (rc != QKV_CTE_OK) return rc;
    e = launch_status_or(reinterpret_cast<const uint32_t*>(sc + hs.ws), status, s);
    if (e == cudaSuccess) e = cudaEventRecord(plan->ev_done[slot], s);
    // readback of the chunk's output
    if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->d2h, plan->ev_done[slot], 0);
    if (e == cudaSuccess) {
      if (!nbsd) {
        e = cudaMemcpyAsync(O_host + (size_t)r0 * I, o_dev, (size_t)n * I * sizeof(uint16_t), cudaMemcpyDeviceToHost,
                            plan->d2h);
      } else {  // NBSd: each head's rows of this chunk go to that head's block of O
        e = cudaMemcpy2DAsync(O_host + (size_t)r0 * dh, (size_t)T * dh * sizeof(uint16_t), o_dev,
                              (size_t)n * dh * sizeof(uint16_t), (size_t)n * dh * sizeof(uint16_t), heads,
                              cudaMemcpyDeviceToHost, plan->d2h);
      }
    }
    if (e == cudaSuccess) e = cudaEventRecord(plan->ev_out[slot], plan->d2h);
    if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "chunk %d readback: %s", i, cudaGetErrorString(e));
  }
  // the caller's stream resumes once every readback is done
  e = cudaStreamWaitEvent(s, plan->ev_out[(chunks - 1) & 1], 0);
  if (e == cudaSuccess && chunks > 1) e = cudaStreamWaitEvent(s, plan->ev_out[chunks & 1], 0);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "stream ordering: %s", cudaGetErrorString(e));
  return ok();
}

// ---------------------------------------------------------------------------
// Allocation-free entry point
//
// Some callers cannot allocate device memory at the moment they want to run this
// projection: a serving process that allocates everything at start-up and forbids
// cudaMalloc afterwards (it can stall or fragment a pool other work relies on), a
// plug-in inside a framework whose allocator owns all device memory, or code on a
// latency-critical path where an allocation may synchronise the device. For them
// this entry point runs the same kernels with their scratch in a fixed array that
// is part of the library image instead of a caller-provided workspace.
// ---------------------------------------------------------------------------

namespace {

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch on the current device, looked up once per device.
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(QKV_CTE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(QKV_CTE_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = noalloc_scratch_address(&p);
    if (e != cudaSuccess || p == nullptr)
      return fail(QKV_CTE_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return QKV_CTE_OK;
}

}  // namespace

extern "C" int qkv_cte_run_noalloc(qkv_cte_plan_t plan, const uint8_t* A, const float* a_scale, const uint8_t* W,
                                   const uint8_t* w_sf, const float* w_col_scale, const uint16_t* bias,
                                   const uint16_t* gamma_q, const uint16_t* gamma_k, const float* cos_table,
                                   const float* sin_table, uint16_t* O, float* sumsq, float* inv_rms,
                                   void* stream) {
  if (plan == nullptr) return fail(QKV_CTE_ERR_INVALID, "null plan");
  if (plan->ws.total > (size_t)QKV_CTE_NOALLOC_SCRATCH_BYTES)
    return fail(QKV_CTE_ERR_UNSUPPORTED,
                "this problem needs %zu bytes of scratch; qkv_cte_run_noalloc holds %zu "
                "(use qkv_cte_run with a workspace)",
                plan->ws.total, (size_t)QKV_CTE_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (plan->g.T > 0) {
    const int rc = noalloc_scratch(&scratch);
    if (rc != QKV_CTE_OK) return rc;
  }
  // qkv_cte_run clears everything that must start at zero (status word, sums of
  // squares, panel counters) in its first kernel, on the same stream.
  return qkv_cte_run(plan, A, a_scale, W, w_sf, w_col_scale, bias, gamma_q, gamma_k, cos_table, sin_table, O,
                     sumsq, inv_rms, scratch, (size_t)QKV_CTE_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int qkv_cte_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != QKV_CTE_OK) return rc;
  return qkv_cte_status(scratch, stream);
}
