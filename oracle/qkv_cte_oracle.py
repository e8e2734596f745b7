"""Oracle for the fused QKV context-encoding projection (test infrastructure).

THIS IS TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH. Only the tests, the
package's ``smoke()`` check and the benchmark's CPU-baseline / reference leg may
import it. It shares no code with the CUDA library: it decodes every FP8, UE8M0
and bf16 bit pattern itself and computes in float64.

What it computes is the method of the ``qkv_cte`` kernel reference page
("Kernel reference: qkv_cte - Wan2.2 additions to the NKI Library QKV CTE MXFP8
projection", vllm-omni-neuron docs, kernels/qkv-cte), cited below as [qkv_cte]
with the page's own section headings:

  1. O[S, I] = A[S, H] @ W[H, I] (+ bias), I = (n_q + 2 n_kv) * d_head
     ([qkv_cte] "Upstream behavior", first bullet), with ROW_MX activations
     (per-row FP8 codes plus one fp32 dequant scale per row) and MXFP8 weights
     ([qkv_cte] "Upstream behavior", quantization-modes bullet; "Interface"
     argument table, rows packed_hidden / weight / weight_scales / bias).
  2. Across-heads RMSNorm of Q and of K: a per-token sum(x^2) over the whole
     un-normalised Q (and K) segment, inv_rms = rsqrt(sum / (n_heads * d_head * tp)
     + eps), then multiplication by the segment-wide per-channel gamma
     ([qkv_cte] "Design", "1) Across-heads QK RMSNorm with a single cross-rank
     AllReduce", steps a, b, c).
  3. Rotate-half RoPE after the norm, pairing lanes (i, i + d/2) within each head,
     with position-only cos/sin tables broadcast over heads:
     out = y * cos + [-y_hi, y_lo] * sin ([qkv_cte] "Design", "2) Bundled
     rotate-half RoPE in the same pass").
  4. V is never normalised ([qkv_cte] "Design" 1, step c); with n_kv_heads = 0 the
     whole projection is one segment, normalised as Q ([qkv_cte] "Design",
     "5) Individual QKV projections for cross-attention").
  5. The producer step before the projection: bf16 activations quantised per row
     to FP8 codes plus one fp32 dequant scale, optionally packed as [T, H + 4]
     rows (codes, then the scale's four bytes) ([qkv_cte] "Upstream behavior",
     packed H + 4 layout; "Interface" table, packed_hidden row).
  6. The per-head qk-norm of the upstream kernel (RMS_NORM / LAYER_NORM with a
     [d_head] gamma) as an alternative to the across-heads norm, and the offline
     interleaved -> rotate-half lane permutation of the Q/K channels ([qkv_cte]
     "Upstream behavior", per-head qk-norm bullet; "Design" 2, last paragraphs).

Readings of points the page leaves open (each also listed in the design notes):

  * MX block: one UE8M0 scale per 32 consecutive H elements of each weight row
    (the OCP MX block); the page only says "MXFP8" / "MX weight".
  * weight_scales [1, I] fp32 ("Interface" table) is an optional per-output-column
    multiplier applied with the activation row scale; absent means 1.
  * The activation carries no MX block scale of its own: its only scale is the
    per-row fp32 dequant scale (ROW_MX, "Interface" table, packed_hidden row).
  * sum(x^2) is taken over the bias-included, un-normalised projection before any
    rounding ("Design" 1, step a: the sum of the output copied out of the matmul).
  * tp = 1: this call holds every head of the segment.
  * gamma multiplies before the rotation, and inv_rms folds into it:
    y = x * inv_rms * gamma, then the rotate-half combination ("Design" 1 step c
    with "Design" 2).
  * norm off leaves gamma unused (gamma belongs to the norm); RoPE off leaves y.
  * Row quantisation: s = amax / 448 (1 for an all-zero row), code = e4m3(x / s)
    rounded to nearest-even with saturation, both divisions in fp32; the packed
    scale tail is little-endian.

Pins: every function here is checked in tests/test_oracle_pins.py against
something other than itself - an exhaustive comparison with torch's float8 codecs,
exact rational brute force on tiny shapes, torch's fp64 rms_norm, the complex
closed form of the rotation, and the invariants the method implies. No function
is parity-unpinned.
"""
from __future__ import annotations

import numpy as np

SEG_Q, SEG_K, SEG_V = 0, 1, 2

# qk-norm kinds: none; the across-heads RMSNorm ([qkv_cte] "Design" 1); the per-head
# RMS_NORM / LAYER_NORM of the upstream kernel ([qkv_cte] "Upstream behavior").
NORM_NONE, NORM_ACROSS_HEADS, NORM_HEAD_RMS, NORM_HEAD_LAYER = 0, 1, 2, 3


# ---------------------------------------------------------------------------
# codecs
# ---------------------------------------------------------------------------

def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """FP8 E4M3 ("fn": no infinities) bit patterns -> float64.

    Layout s.eeee.mmm with exponent bias 7. e == 0 encodes subnormals
    m * 2^-9; e == 15 with m == 7 is NaN; every other pattern is
    (1 + m/8) * 2^(e-7). This is the FP8 element type of both the packed
    activation codes and the MX weight ([qkv_cte] "Interface" table).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    mag = np.where(e == 0, sub, normal)
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    """UE8M0 block-scale bytes -> float64: 2^(e - 127); 0xFF is NaN."""
    e = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    return np.where(e == 255, np.nan, np.exp2(e - 127.0))


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64 (exact: bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# step 1: the projection
# ---------------------------------------------------------------------------

def dequant_activations(A: np.ndarray, a_scale: np.ndarray) -> np.ndarray:
    """ROW_MX activations: a[t, h] = e4m3(A[t, h]) * a_scale[t].

    [qkv_cte] "Upstream behavior" (packed H + 4 layout: per-row FP8 codes plus a
    4-byte fp32 dequant scale) and "Interface" table, packed_hidden row.
    """
    return decode_e4m3(A) * np.asarray(a_scale, dtype=np.float64)[:, None]


def dequant_weights(W: np.ndarray, w_sf: np.ndarray) -> np.ndarray:
    """MXFP8 weights: w[i, h] = e4m3(W[i, h]) * 2^(w_sf[i, h // 32] - 127).

    W is stored K-major as [I, H] (row i = output channel i); w_sf is [I, H/32].
    [qkv_cte] "Upstream behavior" (MXFP8 quantization mode) and "Design" 3
    (nc_matmul_mx applies the MX scales inside the matmul).
    """
    I, H = W.shape
    scale = decode_ue8m0(w_sf)                       # [I, H/32]
    block = np.arange(H) // 32                       # the block each h belongs to
    return decode_e4m3(W) * scale[:, block]


def project(A, a_scale, W, w_sf, w_col_scale=None, bias=None) -> np.ndarray:
    """O = A @ W (+ bias) in float64: o[t, i] = sum_h a[t, h] * w[i, h] * cs[i] + b[i].

    [qkv_cte] "Upstream behavior", first bullet; weight_scales and bias from the
    "Interface" table (cs = weight_scales, 1 when absent; b = bias, 0 when absent).
    """
    a = dequant_activations(A, a_scale)
    w = dequant_weights(W, w_sf)
    o = a @ w.T
    if w_col_scale is not None:
        o = o * np.asarray(w_col_scale, dtype=np.float64)[None, :]
    if bias is not None:
        o = o + decode_bf16(bias)[None, :]
    return o


# ---------------------------------------------------------------------------
# step 2: across-heads RMSNorm
# ---------------------------------------------------------------------------

def segments(n_q_heads: int, n_kv_heads: int, d_head: int):
    """Column ranges of the Q, K and V segments of O: I = (n_q + 2 n_kv) * d_head.

    With n_kv_heads == 0 there is one segment and it is treated as Q
    ([qkv_cte] "Design" 5). With n_q_heads == 0 (and n_kv_heads > 0) the Q segment is
    empty: the call projects K and V only (the cross-attention K and V calls of
    "Design" 5 run as one).
    """
    q = (0, n_q_heads * d_head)
    k = (q[1], q[1] + n_kv_heads * d_head)
    v = (k[1], k[1] + n_kv_heads * d_head)
    return q, k, v


def segment_sumsq(o: np.ndarray, n_q_heads: int, n_kv_heads: int, d_head: int) -> np.ndarray:
    """Per-token sum(x^2) over the whole un-normalised Q segment and K segment.

    Returns [rows, 2] (column 1 is 0 when there is no K segment).
    [qkv_cte] "Design" 1, step a (accumulate).
    """
    q, k, _ = segments(n_q_heads, n_kv_heads, d_head)
    ss = np.zeros((o.shape[0], 2), dtype=np.float64)
    ss[:, SEG_Q] = np.sum(o[:, q[0]:q[1]] ** 2, axis=1)
    if n_kv_heads > 0:
        ss[:, SEG_K] = np.sum(o[:, k[0]:k[1]] ** 2, axis=1)
    return ss


def inv_rms(sumsq: np.ndarray, n_q_heads: int, n_kv_heads: int, d_head: int, eps: float,
            tp: int = 1) -> np.ndarray:
    """inv_rms = 1 / sqrt(sumsq / (n_heads * d_head * tp) + eps), per token and segment.

    [qkv_cte] "Design" 1, step b (reduce). With one GPU holding every head, tp = 1
    and the cross-rank AllReduce is the identity. The K column is 0 when the call
    has no K segment (its rsqrt is skipped, "Design" 5); likewise the Q column when
    the call has no Q heads (a K|V call).
    """
    out = np.zeros_like(sumsq)
    if n_q_heads > 0:
        out[:, SEG_Q] = 1.0 / np.sqrt(sumsq[:, SEG_Q] / (n_q_heads * d_head * tp) + eps)
    if n_kv_heads > 0:
        out[:, SEG_K] = 1.0 / np.sqrt(sumsq[:, SEG_K] / (n_kv_heads * d_head * tp) + eps)
    return out


# ---------------------------------------------------------------------------
# step 3: norm apply + rotate-half RoPE on one segment
# ---------------------------------------------------------------------------

def head_norm(x: np.ndarray, gamma, d_head: int, kind: int, eps: float) -> np.ndarray:
    """Per-head qk-norm of one segment: every head's d_head lanes are normalised by
    their own statistics, then multiplied by the per-head gamma [d_head] that all the
    segment's heads share.

      RMS_NORM:   y = x / sqrt(mean(x^2) + eps) * gamma
      LAYER_NORM: y = (x - mean(x)) / sqrt(mean((x - mean(x))^2) + eps) * gamma

    [qkv_cte] "Upstream behavior" (optional fused per-head qk-norm, RMS_NORM /
    LAYER_NORM) and "Design" 1 (the per-head gamma is [1, d_head]; each head's slice
    normalised by its own RMS). The page gives LAYER_NORM no bias term.
    """
    rows, width = x.shape
    h = x.reshape(rows, width // d_head, d_head)
    if kind == NORM_HEAD_LAYER:
        h = h - h.mean(axis=2, keepdims=True)
    inv = 1.0 / np.sqrt(np.mean(h ** 2, axis=2, keepdims=True) + eps)
    return (h * inv * decode_bf16(gamma)[None, None, :]).reshape(rows, width)


def rope_interleaved(y: np.ndarray, cos, sin, d_head: int) -> np.ndarray:
    """RoPE in the interleaved-lane convention of Wan's checkpoint: lanes (2j, 2j+1)
    of each head form pair j ([qkv_cte] "Design" 2: the caller converts it offline).
    Tables are [rows, d_head] in the same convention (entries 2j and 2j+1 hold pair
    j's cos / sin):
      out[2j]   = y[2j]   * cos[2j]   - y[2j+1] * sin[2j]
      out[2j+1] = y[2j+1] * cos[2j+1] + y[2j]   * sin[2j+1]
    """
    rows, width = y.shape
    heads = width // d_head
    h = y.reshape(rows, heads, d_head)
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s_ = np.asarray(sin, dtype=np.float64)[:, None, :]
    swapped = np.empty_like(h)
    swapped[:, :, 0::2] = -h[:, :, 1::2]
    swapped[:, :, 1::2] = h[:, :, 0::2]
    return (h * c + swapped * s_).reshape(rows, width)


def interleaved_to_rotate_half(d_head: int) -> np.ndarray:
    """The lane permutation that turns the interleaved convention into rotate-half:
    new lane i takes old lane perm[i], with perm[j] = 2j and perm[d/2 + j] = 2j + 1
    for j < d/2, so pair (2j, 2j+1) becomes pair (j, j + d/2). [qkv_cte] "Design" 2
    (the caller permutes the Q/K weights, bias, gamma and cos/sin caches once)."""
    half = d_head // 2
    perm = np.empty(d_head, dtype=np.int64)
    perm[:half] = 2 * np.arange(half)
    perm[half:] = 2 * np.arange(half) + 1
    return perm


def permute_qk_rows(x: np.ndarray, n_q_heads: int, n_kv_heads: int, d_head: int) -> np.ndarray:
    """Apply ``interleaved_to_rotate_half`` to every Q and K head along axis 0 of x
    (one entry per output channel: W [I, H], w_sf [I, H/32], bias [I], w_col_scale
    [I]); the V channels are copied unchanged. A gamma of one segment is a call with
    that segment's heads and n_kv_heads = 0; a cos/sin table [T, d] is permuted along
    its columns (pass the transpose)."""
    x = np.asarray(x)
    perm = interleaved_to_rotate_half(d_head)
    n_qk = n_q_heads + n_kv_heads
    idx = np.arange(x.shape[0])
    for h in range(n_qk):
        idx[h * d_head:(h + 1) * d_head] = h * d_head + perm
    return x[idx]


def rotate_half(y: np.ndarray, d_head: int) -> np.ndarray:
    """[-y_hi, y_lo] per head: lane i pairs with lane i + d/2 ([qkv_cte] "Design" 2)."""
    rows, width = y.shape
    h = y.reshape(rows, width // d_head, d_head)
    lo = h[:, :, : d_head // 2]
    hi = h[:, :, d_head // 2:]
    return np.concatenate([-hi, lo], axis=2).reshape(rows, width)


def apply_norm_rope(x: np.ndarray, inv: np.ndarray, gamma, cos, sin, d_head: int,
                    norm: int, rope: int) -> np.ndarray:
    """One segment (all its heads) of one set of tokens.

    y = x * inv_rms * gamma when the norm is on ("Design" 1, step c), else y = x;
    out = y * cos + rotate_half(y) * sin when RoPE is on ("Design" 2), where cos/sin
    are the per-position [rows, d_head] tables broadcast over the heads.
    """
    rows, width = x.shape
    y = x
    if norm == NORM_ACROSS_HEADS:
        y = x * inv[:, None] * decode_bf16(gamma)[None, :]
    if rope:
        heads = width // d_head
        c = np.tile(np.asarray(cos, dtype=np.float64), (1, heads))
        s = np.tile(np.asarray(sin, dtype=np.float64), (1, heads))
        y = y * c + rotate_half(y, d_head) * s
    return y


# ---------------------------------------------------------------------------
# the whole path
# ---------------------------------------------------------------------------

def qkv_cte(A, a_scale, W, w_sf, bias, gamma_q, gamma_k, cos, sin, *, n_q_heads: int,
            n_kv_heads: int, d_head: int, norm: int, rope: int, eps: float,
            w_col_scale=None, rows=None, rope_layout: str = "rotate_half"):
    """The fused projection for the given rows (all rows when ``rows`` is None).

    norm is one of NORM_NONE, NORM_ACROSS_HEADS (gamma [n_heads * d_head] per
    segment), NORM_HEAD_RMS or NORM_HEAD_LAYER (gamma [d_head] per segment).
    rope_layout "interleaved" applies RoPE in the interleaved-lane convention
    (``rope_interleaved``) instead of rotate-half, for checking the permutation.
    Rows are independent, so a row subset gives exactly the rows of the full
    result. Returns a dict of float64 arrays: O [rows, I] (Q/K normalised and
    rotated, V as projected), sumsq [rows, 2] (of the un-normalised projection, in
    every mode), inv_rms [rows, 2] (zeros unless the norm is across heads).
    """
    if rows is not None:
        rows = np.asarray(rows)
        A = A[rows]
        a_scale = a_scale[rows]
        if cos is not None:
            cos = cos[rows]
            sin = sin[rows]
    o = project(A, a_scale, W, w_sf, w_col_scale, bias)
    ss = segment_sumsq(o, n_q_heads, n_kv_heads, d_head)
    across = norm == NORM_ACROSS_HEADS
    inv = inv_rms(ss, n_q_heads, n_kv_heads, d_head, eps) if across else np.zeros_like(ss)
    out = o.copy()
    q, k, _ = segments(n_q_heads, n_kv_heads, d_head)
    parts = ([(q, SEG_Q, gamma_q)] if n_q_heads > 0 else []) + ([(k, SEG_K, gamma_k)] if n_kv_heads > 0 else [])
    for (c0, c1), seg, gamma in parts:
        x = o[:, c0:c1]
        if norm in (NORM_HEAD_RMS, NORM_HEAD_LAYER):
            x = head_norm(x, gamma, d_head, norm, eps)
        if rope_layout == "interleaved":
            y = apply_norm_rope(x, inv[:, seg], gamma, None, None, d_head, norm if across else 0, 0)
            out[:, c0:c1] = rope_interleaved(y, cos, sin, d_head) if rope else y
        else:
            out[:, c0:c1] = apply_norm_rope(x, inv[:, seg], gamma, cos, sin, d_head, norm if across else 0,
                                            rope)
    return dict(O=out, sumsq=ss, inv_rms=inv, projected=o)


def to_nbsd(O: np.ndarray, d_head: int) -> np.ndarray:
    """BSD [T, I] -> NBSd [n_heads, T, d_head] with n_heads = I / d_head: element (h, t, j)
    is O[t, h*d_head + j], heads in column order (Q heads, then K, then V).

    [qkv_cte] "Upstream behavior" (BSD and NBSd output layouts) and "Interface" table
    (output_layout: NBSd [num_heads, B, S, d_head]; B*S is the token axis here).
    """
    T, I = O.shape
    return O.reshape(T, I // d_head, d_head).transpose(1, 0, 2)


# ---------------------------------------------------------------------------
# the producer step: bf16 -> ROW_MX rows, and the packed H + 4 row layout
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def encode_e4m3(v) -> np.ndarray:
    """Real values -> FP8 E4M3 ("fn") codes: the nearest point of the e4m3 grid,
    ties to the even code (mantissa LSB 0), magnitudes above 448 clamped to 448
    (a saturating conversion: finite in, finite out), the sign kept (a negative value
    that rounds to zero gives -0, code 0x80). NaN gives 0x7F.

    The grid is whatever ``decode_e4m3`` says the 127 non-negative finite codes are;
    codes are ascending in magnitude, so neighbours on the grid are neighbouring codes.
    """
    v = np.asarray(v, dtype=np.float64)
    mags = decode_e4m3(np.arange(0x7F, dtype=np.uint8))      # codes 0x00..0x7E, ascending
    a = np.minimum(np.abs(v), E4M3_MAX)
    a = np.where(np.isnan(a), 0.0, a)
    hi = np.minimum(np.searchsorted(mags, a, side="left"), 0x7E)  # mags[hi - 1] < a <= mags[hi]
    lo = np.maximum(hi - 1, 0)
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo).astype(np.uint8)
    code = code | (np.signbit(v).astype(np.uint8) << 7)
    return np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)


def row_quantise(x_bits: np.ndarray):
    """bf16 activations [T, H] (bit patterns) -> ROW_MX rows: (codes uint8 [T, H],
    dequant scale float32 [T]).

    Per row: amax = max |x| (exact); s = amax / 448 (1 for an all-zero row); each
    code is x / s rounded to e4m3 by ``encode_e4m3``, so code * s reproduces x to
    FP8 precision and the row's largest element maps to 448. [qkv_cte] "Interface"
    table, packed_hidden row (per-row FP8 codes plus an fp32 dequant scale; the
    projection does not quantise bf16 itself, its producer does) and "Upstream
    behavior" (the ROW_MX quantization mode).

    The page fixes no precision for this step. A code is an integer that a floating
    point quotient decides, so the two divisions are taken in IEEE fp32 (numpy
    float32, correctly rounded, subnormals kept), the precision of the scale the
    page stores; the CUDA producer divides the same way.
    """
    x = decode_bf16(x_bits).astype(np.float32)             # exact: bf16 is a truncated fp32
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        q = (x / s[:, None]).astype(np.float32)
    return encode_e4m3(q.astype(np.float64)), s


def pack_rows(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """ROW_MX rows -> the packed layout [T, H + 4]: each row's H codes, then the four
    bytes of its fp32 dequant scale, little-endian. [qkv_cte] "Upstream behavior"
    (the packed H + 4 activation layout) and "Interface" table, packed_hidden."""
    codes = np.asarray(codes, dtype=np.uint8)
    T, H = codes.shape
    tail = np.asarray(scale, dtype="<f4").reshape(T, 1).view(np.uint8)
    return np.concatenate([codes, tail], axis=1)


def unpack_rows(packed: np.ndarray):
    """Packed [T, H + 4] -> (codes uint8 [T, H], scale float32 [T]); the inverse of
    ``pack_rows``."""
    packed = np.asarray(packed, dtype=np.uint8)
    H = packed.shape[1] - 4
    codes = np.ascontiguousarray(packed[:, :H])
    scale = np.ascontiguousarray(packed[:, H:]).view("<f4").reshape(-1).astype(np.float32)
    return codes, scale


def qkv_cte_from_inputs(call, inp, rows=None):
    """Convenience wrapper over :func:`qkv_cte` for a ``workloads.Call`` and its inputs."""
    from workloads import as_numpy_bits

    n = {k: as_numpy_bits(v) for k, v in inp.items()}
    return qkv_cte(n["A"], n["a_scale"], n["W"], n["w_sf"], n["bias"], n["gamma_q"],
                   n["gamma_k"], n["cos"], n["sin"], n_q_heads=call.n_q_heads,
                   n_kv_heads=call.n_kv_heads, d_head=call.d_head, norm=call.norm,
                   rope=call.rope, eps=call.eps, w_col_scale=n["w_col_scale"], rows=rows)
