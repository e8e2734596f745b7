/*
 * qkv_cte.h - C ABI of the GB300 (sm_103a) fused QKV context-encoding projection.
 *
 * The operation is the one described on the `qkv_cte` kernel reference page
 * ("Kernel reference: qkv_cte - Wan2.2 additions to the NKI Library QKV CTE MXFP8
 * projection", vllm-omni-neuron docs, kernels/qkv-cte), cited below as [qkv_cte]
 * with the page's section headings:
 *
 *   O[T, I] = dequant(A_fp8[T, H] @ W_fp8[H, I]) (+ bias),  I = (n_q + 2 n_kv) * d_head,
 *             stored as BSD [T, I] or NBSd [I/d_head, T, d_head] ([qkv_cte] "Upstream
 *             behavior" output layouts; "Interface" output_layout)
 *             ([qkv_cte] "Upstream behavior", first bullet; "Interface" argument table)
 *   Q, K   : across-heads RMSNorm - one RMS per token over the whole Q (or K) segment,
 *            inv_rms = 1/sqrt(sum(o^2) / (n_heads * d_head) + eps), times a segment-wide
 *            per-channel gamma ([qkv_cte] "Design" 1, steps a-c), then rotate-half RoPE
 *            out = y*cos + [-y_hi, y_lo]*sin with position-only cos/sin tables broadcast
 *            over heads ([qkv_cte] "Design" 2)
 *   V      : left as projected ([qkv_cte] "Design" 1, step c)
 *   n_kv_heads == 0: one segment, normalised as Q - the separate Q / K / V calls of
 *            cross-attention ([qkv_cte] "Design" 5)
 *
 * Number formats
 *   A      : FP8 e4m3 ("fn") codes, one fp32 dequant scale per row (ROW_MX activations).
 *   W      : FP8 e4m3 codes with one UE8M0 scale (2^(e-127)) per 32 consecutive H
 *            elements of each output channel (MXFP8 weights).
 *   bias, gamma : bfloat16 bit patterns. cos/sin : fp32. O : bfloat16 bit patterns,
 *            round-to-nearest-even. sumsq / inv_rms : fp32.
 *
 * Memory and ownership
 *   Every tensor pointer is a DEVICE pointer owned by the caller; the library never
 *   frees or keeps it past the call. The plan owns only host-side state. The workspace
 *   is caller-allocated device memory of the size qkv_cte_plan reports; it holds the
 *   per-call scratch (repacked weight scales, the sum-of-squares accumulator, a device
 *   status word, per-panel completion counters, timing stamps and, when a norm or RoPE
 *   pass runs, the un-normalised Q and K columns in block floating point: about
 *   2.06*ceil(T/128)*128*(n_q + n_kv)*d_head bytes; with a packed or bf16 input also
 *   the e4m3 codes and row scales the producer step writes, T*(H + 4) bytes) and must
 *   not be shared by calls that overlap on the GPU. The norm/RoPE
 *   kernel is launched as a programmatic dependent of the GEMM so the two overlap. qkv_cte_run is stream-ordered and asynchronous: it never
 *   synchronises. O must not alias any input.
 *
 * Errors
 *   Every entry point returns 0 on success or a negative QKV_CTE_ERR_* code, never
 *   throws, and records a message readable with qkv_cte_last_error() (thread-local).
 *   Argument checks happen before any launch: a call that returns an error launched
 *   nothing. Device-side waits are bounded; a wait that runs out sets the workspace's
 *   status word and the kernel returns. qkv_cte_status() reports it.
 */
#ifndef QKV_CTE_H
#define QKV_CTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QKV_CTE_ABI_VERSION 4

#define QKV_CTE_OK 0
#define QKV_CTE_ERR_INVALID (-1)        /* null / inconsistent argument, mode-segment mismatch */
#define QKV_CTE_ERR_UNSUPPORTED (-2)    /* shape, layout or alignment this build does not take */
#define QKV_CTE_ERR_CUDA (-3)           /* a CUDA runtime / launch error */
#define QKV_CTE_ERR_ARCH (-4)           /* current device is not sm_103 */
#define QKV_CTE_ERR_DEVICE_TIMEOUT (-5) /* a bounded device wait ran out (see qkv_cte_status) */

enum { QKV_CTE_MODE_FUSED = 0, QKV_CTE_MODE_SEPARATE = 1 };

/* qk-norm of Q and K (desc.norm):
 *   NONE         : no norm;
 *   ACROSS_HEADS : one RMS per token over the whole Q (or K) segment, gamma [n_heads*d_head]
 *                  per segment ([qkv_cte] "Design" 1; Wan's RMS_NORM_ACROSS_HEADS);
 *   HEAD_RMS     : per head, x / sqrt(mean(x^2) + eps) * gamma, gamma [d_head] shared by the
 *                  segment's heads;
 *   HEAD_LAYER   : per head, (x - mean) / sqrt(mean((x - mean)^2) + eps) * gamma, gamma
 *                  [d_head], no bias ([qkv_cte] "Upstream behavior": the per-head RMS_NORM /
 *                  LAYER_NORM fused into the matmul's copy-out).
 * The per-head kinds are finished by the norm/RoPE pass from per-(row, head) statistics
 * the GEMM writes (or, with QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE, in the GEMM's epilogue
 * with tiles of whole heads); RoPE is applied after the norm in every kind. */
enum { QKV_CTE_NORM_NONE = 0, QKV_CTE_NORM_ACROSS_HEADS = 1, QKV_CTE_NORM_HEAD_RMS = 2, QKV_CTE_NORM_HEAD_LAYER = 3 };
enum { QKV_CTE_LAYOUT_BSD = 0, QKV_CTE_LAYOUT_NBSD = 1 };

/* What `A` of qkv_cte_run holds ([qkv_cte] "Interface" table, packed_hidden row, and
 * its producer):
 *   ROW_FP8: e4m3 codes [T, H] (16-byte aligned) with the fp32 row scales in a_scale;
 *   PACKED : the packed rows [T, H + 4] (each row's H codes, then its fp32 scale,
 *            little-endian; 4-byte aligned); a_scale must be NULL. The run first
 *            unpacks them into the workspace (their pitch is not 16-byte aligned, so
 *            the GEMM's TMA loads cannot read them in place);
 *   BF16   : bf16 activations [T, H] (16-byte aligned); a_scale must be NULL. The run
 *            first quantises them per row into the workspace, exactly as
 *            qkv_cte_row_quantize does. */
enum { QKV_CTE_INPUT_ROW_FP8 = 0, QKV_CTE_INPUT_PACKED = 1, QKV_CTE_INPUT_BF16 = 2 };

/* Test hook: the GEMM's load warp issues nothing, so every bounded wait downstream
 * runs out and the kernel exits through its error path (status word set). */
#define QKV_CTE_FLAG_TEST_STALL 0x1u
/* Record a CUDA event before and after each run so qkv_cte_pass_times() can report
 * per-pass device times (nothing is recorded between the run's launches, which
 * overlap). */
#define QKV_CTE_FLAG_PROFILE 0x2u
/* Launch the norm/RoPE pass as its own kernel after the GEMM has finished instead of
 * overlapping the two (same results; used to time each pass on its own). */
#define QKV_CTE_FLAG_SERIAL_PASSES 0x4u
/* GEMM form: tiles of 256 rows on a pair of SMs (M = 256 MMAs; each SM stages half
 * of the weight tile), or tiles of 128 rows on one SM. Neither flag: the library
 * chooses. Both: -1. */
#define QKV_CTE_FLAG_GEMM_CTA_PAIR 0x8u
#define QKV_CTE_FLAG_GEMM_SINGLE_CTA 0x10u
/* Run the norm/RoPE work inside the CTA-pair GEMM's epilogue warps, between tiles (one
 * kernel), instead of as a kernel of its own overlapped with the GEMM through a
 * programmatic dependent launch (the default). Same results; measured slower at the Wan
 * shapes (the norm work slows the GEMM just as much from inside it, and what is left
 * when the tiles are done runs as a tail). Ignored without the pair form or with
 * QKV_CTE_FLAG_SERIAL_PASSES. */
#define QKV_CTE_FLAG_NORM_IN_GEMM 0x20u
/* Per-head norms (QKV_CTE_NORM_HEAD_RMS / _LAYER): finish the norm and RoPE in the GEMM's
 * epilogue while each tile is in TMEM (tiles of whole heads, no second pass) instead
 * of the default: the GEMM writes per-(row, head) statistics (RMS: sum of squares;
 * LayerNorm: each tile part's shift, mean and centred sum of squares) and the norm/RoPE pass
 * finishes from them, which keeps the GEMM's wide tiles. Same results to rounding. */
#define QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE 0x40u
/* Problem description ([qkv_cte] "Interface" argument table, flattened to scalars). */
typedef struct {
    int64_t tokens;        /* T = B*S rows; 0 is allowed (nothing is launched); <= INT32_MAX */
    int32_t hidden;        /* H, contraction length; multiple of 128 */
    int32_t n_q_heads;     /* Q heads in this call (>= 1; 0 in fused mode: a K|V call, e.g. the
                              cross-attention K and V projections of the context tokens as one
                              launch, W = [W_k; W_v], K normalised with gamma_k, V as projected) */
    int32_t n_kv_heads;    /* K/V heads; 0 for a single-segment (separate) call */
    int32_t d_head;        /* head dim; multiple of 16, of 32 when a norm or RoPE runs */
    int32_t mode;          /* QKV_CTE_MODE_FUSED (n_kv >= 1, n_q >= 0) or QKV_CTE_MODE_SEPARATE
                              (n_kv == 0, n_q >= 1) */
    int32_t norm;          /* QKV_CTE_NORM_*: 0 none, 1 across heads, 2 per-head RMS, 3 per-head LayerNorm */
    int32_t rope;          /* 1: rotate-half RoPE on Q (and K); needs cos/sin */
    int32_t output_layout; /* QKV_CTE_LAYOUT_BSD: O[T, I]; QKV_CTE_LAYOUT_NBSD: O[I/d_head, T, d_head]
                              (heads in column order: Q heads, then K, then V) */
    float eps;             /* norm epsilon, >= 0 */
    uint32_t flags;        /* 0 or QKV_CTE_FLAG_* bits */
    int32_t tile_n;        /* GEMM N tile: 0 = automatic, else 128, 192, 240 or 256 */
    int32_t input_layout;  /* QKV_CTE_INPUT_*: what A holds (0 = e4m3 codes + separate scales) */
} qkv_cte_desc;

typedef struct qkv_cte_plan_s* qkv_cte_plan_t;

/* What a plan chose (host only). */
typedef struct {
    int32_t tile_n;          /* GEMM N tile (columns of O per tile) */
    int32_t m_tiles;         /* GEMM row tiles (128 rows, or 256 with a CTA pair) */
    int32_t n_tiles;         /* N tiles */
    int32_t n_bands;         /* bands of N tiles in the GEMM's tile order */
    int32_t cta_pair;        /* 1: 256-row tiles on SM pairs; 0: 128-row tiles */
    int32_t norm_in_gemm;    /* 1: the norm/RoPE work runs inside the GEMM's epilogue warps (one
                                kernel); 0: as a kernel of its own, or there is none */
    int64_t workspace_bytes; /* as returned by qkv_cte_plan */
} qkv_cte_plan_info;

/* Validate `desc` (host only, no CUDA call) and create a plan.
 * out            : receives the plan (set to NULL on error).
 * workspace_bytes: receives the device workspace size qkv_cte_run needs.
 * Returns 0, -1 (null pointer, bad head counts, mode/segment mismatch, flag values,
 * unknown input layout) or
 * -2 (H % 128, d_head % 16, d_head % 32 with a norm or RoPE, T > INT32_MAX, unknown tile_n,
 * a per-head norm in the epilogue with a tile_n that d_head does not divide). */
int qkv_cte_plan(qkv_cte_plan_t* out, const qkv_cte_desc* desc, size_t* workspace_bytes);

/* Fill `info` for `plan`. Returns 0 or -1 (null pointer). */
int qkv_cte_get_plan_info(qkv_cte_plan_t plan, qkv_cte_plan_info* info);

/* Run the whole path on `stream` (a cudaStream_t; NULL = legacy default stream).
 *
 * A          : per desc.input_layout (QKV_CTE_INPUT_*): uint8 [T, H] e4m3 codes, row-major,
 *              16-byte aligned; or packed uint8 [T, H + 4] rows, 4-byte aligned; or bf16
 *              [T, H], 16-byte aligned
 * a_scale    : fp32   [T]         per-row dequant scale (ROW_FP8 input only; NULL otherwise)
 * W          : uint8  [I, H]      e4m3 codes, K-major (row i = output channel i); 16-byte aligned
 * w_sf       : uint8  [I, H/32]   UE8M0 block scales, row-major; 4-byte aligned
 * w_col_scale: fp32   [I] or NULL per-output-channel multiplier ("weight_scales"); 16-byte aligned
 * bias       : bf16   [I] or NULL; 16-byte aligned
 * gamma_q    : bf16   Q gamma, required iff norm != NONE and n_q > 0: [n_q*d_head] (across heads)
 *              or [d_head] (per head), else NULL; 16-byte aligned
 * gamma_k    : bf16   K gamma, [n_kv*d_head] or [d_head]; required iff norm != NONE and n_kv > 0,
 *              else NULL
 * cos_table, sin_table: fp32 [T, d_head] rotate-half tables; required iff rope, else NULL;
 *              32-byte aligned
 * O          : bf16 output, [T, I] (BSD) or [I/d_head, T, d_head] (NBSd: element (h, t, j)
 *              is column h*d_head + j of token t); 32-byte aligned; must not alias any input
 * sumsq      : fp32   [T, 2] or NULL: per-token sum of o^2 over the un-normalised Q and K
 *              segments ([qkv_cte] "Design" 1 step a; column 1 is 0 when n_kv == 0, column 0
 *              when n_q == 0)
 * inv_rms    : fp32   [T, 2] or NULL: the rsqrt factors of step b (written iff norm is
 *              ACROSS_HEADS; must be NULL with a per-head norm; the column of an absent
 *              segment is 0)
 * workspace  : device scratch of at least the planned size; 256-byte aligned
 * With tokens == 0 every tensor pointer may be NULL: no kernel is launched and only
 * the workspace's status word is reset (when a workspace is given).
 * Returns 0 or -1/-2/-3/-4 (nothing launched on -1/-2/-4). */
int qkv_cte_run(qkv_cte_plan_t plan, const uint8_t* A, const float* a_scale, const uint8_t* W,
                const uint8_t* w_sf, const float* w_col_scale, const uint16_t* bias,
                const uint16_t* gamma_q, const uint16_t* gamma_k, const float* cos_table,
                const float* sin_table, uint16_t* O, float* sumsq, float* inv_rms,
                void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise `stream`, then read and clear the device status word in `workspace`.
 * Each run clears the word before its kernels start, so this reports the most recent
 * run that used `workspace`; before the first run the workspace must hold zeros.
 * Returns 0, -5 if one of its bounded device waits ran out (the message names the
 * wait), -1 if the word holds bits no run writes (an uninitialised workspace), or -3
 * on a CUDA error. */
int qkv_cte_status(void* workspace, void* stream);

/* Device times in milliseconds of the most recent run of `plan`, which must have been
 * created with QKV_CTE_FLAG_PROFILE. ms must hold 4 floats:
 *   ms[0] the rest of the run: the input's unpack or quantise step when it is packed
 *         or bf16, the scale repack and clears, and launch gaps (ms[3] less the span
 *         from the GEMM's start to the last end of the GEMM or the norm/RoPE work);
 *   ms[1] GEMM with its fused epilogue (including the norm/RoPE work when it runs in
 *         the GEMM's epilogue warps), and ms[2] norm + RoPE (0 when the call has
 *         neither): first start to last end of that work, from %globaltimer stamps the
 *         kernels write into the workspace (the two overlap, so no CUDA event can
 *         separate them);
 *   ms[3] the whole run, from CUDA events.
 * Blocks until that run has finished; its workspace must still be valid. Returns 0, -1
 * (no flag, never run, null pointer) or -3. */
int qkv_cte_pass_times(qkv_cte_plan_t plan, float* ms);

/* The producer step on its own: bf16 activations -> ROW_MX rows ([qkv_cte] "Interface"
 * table, packed_hidden row: per-row FP8 codes plus one fp32 dequant scale, made by the
 * projection's producer; "Upstream behavior": the packed H + 4 layout).
 *
 * Per row t: amax = max_h |X[t, h]|; s = amax / 448 (1.0 for an all-zero row); code
 * = e4m3(X[t, h] / s), the quotient an IEEE fp32 division, converted with round to
 * nearest even and saturation to +-448 (the row's largest element maps to 448). X
 * must be finite.
 *
 * X       : bf16 [T, H], 16-byte aligned
 * A       : uint8 [T, H] e4m3 codes or NULL; 16-byte aligned
 * a_scale : fp32 [T] dequant scales or NULL (given together with A); 4-byte aligned
 * packed  : uint8 [T, H + 4] packed rows (codes, then the scale's 4 bytes,
 *           little-endian) or NULL; 4-byte aligned
 * At least one of A / packed; no output may overlap X or another output. H % 16 == 0.
 * Stream-ordered and asynchronous. Returns 0, -1 (null or overlapping buffers, no
 * output), -2 (H % 16, alignment, T > INT32_MAX), -3 or -4. tokens == 0 checks only
 * tokens and hidden, launches nothing and returns 0 (every pointer may be NULL). */
int qkv_cte_row_quantize(const uint16_t* X, int64_t tokens, int32_t hidden, uint8_t* A, float* a_scale,
                         uint8_t* packed, void* stream);

/* Packed rows [T, H + 4] (4-byte aligned) -> e4m3 codes A [T, H] (16-byte aligned) and
 * fp32 scales a_scale [T] (4-byte aligned): the layout qkv_cte_run reads with
 * QKV_CTE_INPUT_ROW_FP8. Byte-exact. H % 16 == 0; buffers must not overlap.
 * Returns 0, -1, -2, -3 or -4 as qkv_cte_row_quantize (tokens == 0 likewise). */
int qkv_cte_unpack_rows(const uint8_t* packed, int64_t tokens, int32_t hidden, uint8_t* A, float* a_scale,
                        void* stream);

/* Offline conversion of an interleaved-RoPE checkpoint (lanes 2j, 2j+1 of a head form
 * pair j, as in Wan's checkpoint) to the rotate-half lane order qkv_cte_run applies
 * ([qkv_cte] "Design" 2: the caller permutes the Q/K weights, bias, gamma and cos/sin
 * caches once). Copies `rows` rows of `row_bytes` bytes from src to dst; within each of
 * the first (n_q_heads + n_kv_heads) heads of d_head rows, row i of the head takes
 * row perm[i] with perm[j] = 2j, perm[d/2 + j] = 2j + 1; the remaining rows (V) are
 * copied as they are. Byte-exact. Apply it to every per-output-channel tensor:
 *   W codes  [I, H]     : rows = I, row_bytes = H
 *   w_sf     [I, H/32]  : rows = I, row_bytes = H/32
 *   bias, w_col_scale   : rows = I, row_bytes = 2 / 4
 *   gamma               : across heads: rows = n*d, heads (n, 0); per head: rows = d, heads (1, 0)
 *   cos/sin [T, d] fp32 : rows = T*d, row_bytes = 4, heads (T, 0) (each table row is one "head")
 * src, dst: device buffers of rows*row_bytes bytes that do not overlap (not in place).
 * Stream-ordered and asynchronous. Returns 0, -1 (bad counts, d_head odd, Q/K rows
 * beyond `rows`, null or overlapping buffers), -2, -3 or -4. rows == 0 launches nothing. */
int qkv_cte_interleaved_to_rotate_half(const void* src, void* dst, int64_t rows, int64_t row_bytes,
                                       int32_t n_q_heads, int32_t n_kv_heads, int32_t d_head, void* stream);

/* qkv_cte_run on activations in pinned HOST memory, writing O to pinned host memory,
 * with the copies overlapped with the computation. Rows are independent, so the
 * tokens are cut into chunks of `chunk_rows` (0: 2048; rounded up to a multiple of
 * 256) and three streams are pipelined: the upload of chunk i+1 (an internal stream),
 * the path on chunk i (on `stream`) and the readback of chunk i-1 (an internal
 * stream), through two staging slots in `scratch`. The call is stream-ordered: work
 * enqueued on `stream` afterwards sees all of O written to the host.
 *
 * A_host       : pinned host, [T, H] e4m3 codes, [T, H+4] packed rows or [T, H] bf16 (desc.input_layout)
 * a_scale_host : pinned host fp32 [T] with separate FP8 rows, else NULL
 * W .. sin_table: DEVICE tensors as for qkv_cte_run (weights and tables stay resident)
 * O_host       : pinned host output, [T, I] or [I/d_head, T, d_head] (desc.output_layout)
 * sumsq, inv_rms: DEVICE [T, 2] or NULL, as for qkv_cte_run
 * scratch      : device memory of qkv_cte_host_scratch_bytes(plan, chunk_rows); 256-byte
 *                aligned; its first word is the status word qkv_cte_status reads (the OR of
 *                every chunk's status)
 * Returns 0, -1, -2 (host memory not pinned, alignment), -3 or -4. A plan used here
 * keeps two streams and a plan per chunk size until qkv_cte_destroy; calls on one plan
 * must not overlap. */
int qkv_cte_run_host(qkv_cte_plan_t plan, const void* A_host, const float* a_scale_host, const uint8_t* W,
                     const uint8_t* w_sf, const float* w_col_scale, const uint16_t* bias,
                     const uint16_t* gamma_q, const uint16_t* gamma_k, const float* cos_table,
                     const float* sin_table, uint16_t* O_host, float* sumsq, float* inv_rms, void* scratch,
                     size_t scratch_bytes, int32_t chunk_rows, void* stream);

/* Device scratch bytes qkv_cte_run_host needs for `plan` and `chunk_rows` (0 for an
 * empty problem). Host only (creates the per-chunk plans). Returns 0 or -1/-2. */
int qkv_cte_host_scratch_bytes(qkv_cte_plan_t plan, int32_t chunk_rows, size_t* bytes);

/* Size of the scratch array behind qkv_cte_run_noalloc: 24 MiB on every GPU that
 * loads the library, held until the process exits. */
#define QKV_CTE_NOALLOC_SCRATCH_BYTES (24u << 20)

/* qkv_cte_run without a workspace, for callers that cannot allocate device memory
 * when they run the projection (a server that forbids allocation after start-up, a
 * plug-in whose host framework owns all device memory, a latency-critical path where
 * an allocation could synchronise the device). The page this library follows has no
 * counterpart: it is an addition of this library.
 *
 * Arguments, layouts and return codes are those of qkv_cte_run without `workspace`
 * and `workspace_bytes`: the scratch is a fixed array of QKV_CTE_NOALLOC_SCRATCH_BYTES
 * inside the library. The call allocates nothing (no cudaMalloc, no allocating
 * library routine). A problem whose planned workspace exceeds the array is rejected
 * with QKV_CTE_ERR_UNSUPPORTED before any launch. With the fused Wan layout (H=5120,
 * 40+40 heads of 128) up to 640 tokens fit; so do the separate cross-attention K and
 * V calls on 512 context tokens.
 *
 * The array is part of the library's device code. CUDA maps code and array on a device
 * the first time the library launches a kernel there (the first run of any entry point
 * on that device), which is a one-time allocation by the driver; the first
 * qkv_cte_run_noalloc on a device also looks up the array's address
 * (cudaGetSymbolAddress). A caller that must not allocate at all therefore makes one
 * call at start-up on each device it uses (this entry point or qkv_cte_run), before
 * allocation is forbidden and before any stream capture; every later call allocates
 * nothing.
 * Every call shares the one array and each call clears the parts that must start at
 * zero, so calls that overlap on the GPU (different streams, or other host threads)
 * race and corrupt each other's results: serialise them. Bounded-wait timeouts are
 * recorded in the array's status word: read it with qkv_cte_noalloc_status. */
int qkv_cte_run_noalloc(qkv_cte_plan_t plan, const uint8_t* A, const float* a_scale, const uint8_t* W,
                        const uint8_t* w_sf, const float* w_col_scale, const uint16_t* bias,
                        const uint16_t* gamma_q, const uint16_t* gamma_k, const float* cos_table,
                        const float* sin_table, uint16_t* O, float* sumsq, float* inv_rms, void* stream);

/* qkv_cte_status for the array behind qkv_cte_run_noalloc on the current device: waits
 * for `stream`, returns 0, or QKV_CTE_ERR_DEVICE_TIMEOUT (and clears the word) when a
 * bounded wait of an earlier allocation-free call ran out, or -3 on a CUDA error.
 * Allocates nothing. Like qkv_cte_run_noalloc it has no counterpart on the page this
 * library follows. */
int qkv_cte_noalloc_status(void* stream);

/* Release a plan. NULL is a no-op. */
void qkv_cte_destroy(qkv_cte_plan_t plan);

/* Message for the last non-zero return on this thread ("" if none). */
const char* qkv_cte_last_error(void);

/* QKV_CTE_ABI_VERSION of the loaded library. */
int qkv_cte_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QKV_CTE_H */
