"""Seeded synthetic workloads for the fused QKV context-encoding projection.

This module is shared by the tests, the benchmark and the oracle checks. It
produces *inputs only*: row-quantised FP8 activations, MX-quantised FP8 weights,
bias, gamma and rotate-half RoPE tables with the shapes and value distributions
of the Wan2.2 DiT attention projections. It holds none of the projection's
arithmetic (no GEMM, no norm, no RoPE application).

Quantisation happens here because, on the `qkv_cte` kernel reference page
(vllm-omni-neuron docs, kernels/qkv-cte, Interface table, ``packed_hidden``
row), the kernel consumes already-quantised activations produced by a separate
AdaLN/row-quantise kernel; the projection itself never quantises.

Everything is generated on the CPU with ``torch.Generator`` seeds so that the
GPU path and the oracle see bit-identical inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Call:
    """One projection call: shapes, mode and the synthetic-input recipe."""

    name: str
    tokens: int            # T = B*S rows
    hidden: int            # H (contraction)
    n_q_heads: int
    n_kv_heads: int        # 0 => separate (single-segment) mode
    d_head: int
    norm: int              # 1 = across-heads RMSNorm on Q (and K)
    rope: int              # 1 = rotate-half RoPE on Q and K
    rope_grid: Optional[Sequence[int]]  # (F, Hg, Wg) latent grid, or None for 1D positions
    outlier_frac: float    # fraction of rows carrying 20x outlier channels
    seed: int
    eps: float = 1e-6
    w_std: float = 0.02
    bias_std: float = 0.02
    gamma_std: float = 0.1
    has_w_col_scale: bool = False

    @property
    def width(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.d_head

    @property
    def mode(self) -> int:
        return 0 if self.n_kv_heads > 0 else 1

    @property
    def flops(self) -> float:
        return 2.0 * self.tokens * self.hidden * self.width


def _fused(name, tokens, hidden, nq, nkv, d, grid, outliers, seed=0):
    return Call(name, tokens, hidden, nq, nkv, d, norm=1, rope=1, rope_grid=grid,
                outlier_frac=outliers, seed=seed)


# The workloads. Shapes follow the Wan2.2 A14B attention projections: 40
# heads of 128, hidden 5120, latent-patch grids of 21 frames.
WORKLOADS: Dict[str, List[Call]] = {
    "tiny": [_fused("tiny", 256, 512, 4, 4, 128, None, 0.0)],
    "short": [_fused("short", 4096, 5120, 40, 40, 128, (21, 14, 14), 0.0)],
    "wan480p": [_fused("wan480p", 32760, 5120, 40, 40, 128, (21, 30, 52), 0.001)],
    # the first 16384 tokens of the 480p layout: inputs above L2, a few GB on the
    # device in all, for profiler captures that replay a kernel many times
    "half480p": [_fused("half480p", 16384, 5120, 40, 40, 128, (21, 30, 52), 0.001)],
    "wan720p": [_fused("wan720p", 75600, 5120, 40, 40, 128, (21, 45, 80), 0.001)],
    "cross": [
        Call("cross_q", 32760, 5120, 40, 0, 128, norm=1, rope=0, rope_grid=None,
             outlier_frac=0.0, seed=100),
        Call("cross_k", 512, 5120, 40, 0, 128, norm=1, rope=0, rope_grid=None,
             outlier_frac=0.0, seed=200),
        Call("cross_v", 512, 5120, 40, 0, 128, norm=0, rope=0, rope_grid=None,
             outlier_frac=0.0, seed=300),
    ],
    # the cross-attention K and V projections of the 512 context tokens as one call:
    # no Q heads, W = [W_k; W_v], K normalised across heads, V as projected
    "cross_kv": [Call("cross_kv", 512, 5120, 0, 40, 128, norm=1, rope=0, rope_grid=None,
                      outlier_frac=0.0, seed=400)],
}


def workload(name: str) -> List[Call]:
    return WORKLOADS[name]


def custom_call(name="custom", tokens=256, hidden=512, n_q_heads=4, n_kv_heads=4, d_head=128,
                norm=1, rope=1, rope_grid=None, outlier_frac=0.0, seed=0, eps=1e-6,
                has_w_col_scale=False, w_std=0.02) -> Call:
    return Call(name, tokens, hidden, n_q_heads, n_kv_heads, d_head, norm=norm, rope=rope,
                rope_grid=rope_grid, outlier_frac=outlier_frac, seed=seed, eps=eps,
                has_w_col_scale=has_w_col_scale, w_std=w_std)


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------

def _gen(seed: int, sub: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed * 1000 + sub)
    return g


def _to_e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """float32 -> e4m3fn bit patterns, round-to-nearest-even, saturated at +-448."""
    x = x.clamp(-E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def row_quantise(a_bf16: torch.Tensor):
    """Per-row FP8 quantisation (the producer kernel's job, outside the path).

    scale = amax/448 (1 for an all-zero row); codes = RNE-saturated e4m3(a/scale).
    Returns (codes uint8 [T,H], scale float32 [T]).
    """
    a = a_bf16.float()
    amax = a.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = _to_e4m3_codes(a / scale[:, None])
    return codes, scale.contiguous()


def mx_quantise(w: torch.Tensor):
    """MX quantisation of a [I,H] weight along H in blocks of 32.

    The block exponent is E = clamp(ceil(log2(amax/448)) + 127, 1, 254) (127 for an
    all-zero block), so that amax / 2^(E-127) <= 448 and no code clips.
    Returns (codes uint8 [I,H], w_sf uint8 [I,H/32]).
    """
    I, H = w.shape
    blocks = w.float().reshape(I, H // 32, 32)
    amax = blocks.abs().amax(dim=2).double()
    ratio = amax / E4M3_MAX
    mant, expo = torch.frexp(ratio)            # ratio = mant * 2^expo, mant in [0.5, 1)
    ceil_log2 = torch.where(mant == 0.5, expo - 1, expo)
    e = torch.clamp(ceil_log2 + 127, 1, 254)
    e = torch.where(amax > 0, e, torch.full_like(e, 127))
    scale = torch.pow(2.0, (e - 127).double()).float()
    codes = _to_e4m3_codes(blocks / scale[:, :, None]).reshape(I, H)
    return codes.contiguous(), e.to(torch.uint8).contiguous()


def _bf16_bits(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).contiguous()


def rope_positions(call: Call, rows: int) -> torch.Tensor:
    """Per-token rotation angles [rows, d_head/2] in float64 (input recipe only).

    1D (no grid): pair j of token s has angle s * 1e4^(-2j/d_head).
    3D grid (F, Hg, Wg): tokens map t-major to (f, h, w); the d_head/2 rotation
    pairs are split over the three axes (22/21/21 for d_head=128, i.e. the first
    axis takes the remainder) and axis a of width d_a = 2*pairs_a uses frequencies
    1e4^(-2j/d_a) times that axis' position. Token s beyond F*Hg*Wg never occurs;
    a grid larger than the token count uses its first `rows` positions.
    """
    d = call.d_head
    half = d // 2
    s = torch.arange(rows, dtype=torch.float64)
    if call.rope_grid is None:
        j = torch.arange(half, dtype=torch.float64)
        inv = torch.pow(torch.tensor(1e4, dtype=torch.float64), -2.0 * j / d)
        return s[:, None] * inv[None, :]
    F, Hg, Wg = call.rope_grid
    p_h = half // 3
    p_w = half // 3
    p_t = half - p_h - p_w
    f_pos = torch.div(s, Hg * Wg, rounding_mode="floor")
    h_pos = torch.remainder(torch.div(s, Wg, rounding_mode="floor"), Hg)
    w_pos = torch.remainder(s, Wg)
    parts = []
    for pos, pairs in ((f_pos, p_t), (h_pos, p_h), (w_pos, p_w)):
        j = torch.arange(pairs, dtype=torch.float64)
        inv = torch.pow(torch.tensor(1e4, dtype=torch.float64), -2.0 * j / (2 * pairs))
        parts.append(pos[:, None] * inv[None, :])
    return torch.cat(parts, dim=1)


def rope_tables(call: Call, rows: int):
    """Rotate-half cos/sin tables float32 [rows, d_head]; lanes j and j+d/2 share an angle."""
    ang = rope_positions(call, rows)
    cos = torch.cos(ang).float()
    sin = torch.sin(ang).float()
    return torch.cat([cos, cos], dim=1).contiguous(), torch.cat([sin, sin], dim=1).contiguous()


def make_activations(call: Call) -> torch.Tensor:
    """The bf16 activations [T, H] of a call (the producer's input): N(0, 1), with
    round(outlier_frac * T) seeded rows carrying a seeded set of 64 channels x20."""
    T, H, s = call.tokens, call.hidden, call.seed
    a = torch.randn(T, H, generator=_gen(s, 0), dtype=torch.float32).to(torch.bfloat16)
    n_out = int(round(call.outlier_frac * T))
    if n_out > 0:
        rows = torch.randperm(T, generator=_gen(s, 4))[:n_out]
        chans = torch.randperm(H, generator=_gen(s, 5))[:64]
        block = a[rows][:, chans].float() * 20.0
        sub = a[rows]
        sub[:, chans] = block.to(torch.bfloat16)
        a[rows] = sub
    return a


def bf16_bits(x: torch.Tensor):
    """A bf16 tensor's bit patterns as a numpy uint16 array (for the oracle)."""
    return x.contiguous().view(torch.int16).numpy().view("uint16")


def make_inputs(call: Call) -> Dict[str, Optional[torch.Tensor]]:
    """All inputs of one call as CPU tensors.

    Keys: A (uint8 [T,H] e4m3 codes), a_scale (float32 [T]), W (uint8 [I,H] e4m3
    codes, K-major), w_sf (uint8 [I,H/32] UE8M0), w_col_scale (float32 [I] or None),
    bias (bfloat16 [I]), gamma_q (bfloat16 [n_q*d], or None without Q heads), gamma_k
    (bfloat16 [n_kv*d] or None), cos/sin (float32 [T,d] or None).
    """
    T, H, I, d = call.tokens, call.hidden, call.width, call.d_head
    s = call.seed
    a = make_activations(call)
    A, a_scale = row_quantise(a)
    del a
    w = torch.randn(I, H, generator=_gen(s, 1), dtype=torch.float32) * call.w_std
    W, w_sf = mx_quantise(w)
    del w
    bias = _bf16_bits(torch.randn(I, generator=_gen(s, 2)) * call.bias_std)
    g = torch.randn(I, generator=_gen(s, 3)) * call.gamma_std + 1.0
    nq = call.n_q_heads * d
    nk = call.n_kv_heads * d
    if call.norm in (2, 3):  # per-head norms: one [d_head] gamma per segment
        gq = g[:d] if call.n_q_heads > 0 else g[:0]
        gk = g[nq:nq + d] if call.n_kv_heads > 0 else g[:0]
        g = torch.cat([gq, gk])
        nq, nk = gq.numel(), gk.numel()
    gamma_q = _bf16_bits(g[:nq]) if nq > 0 else None
    gamma_k = _bf16_bits(g[nq:nq + nk]) if nk > 0 else None
    w_col_scale = None
    if call.has_w_col_scale:
        w_col_scale = (torch.rand(I, generator=_gen(s, 6)) * 1.5 + 0.25).float()
    cos = sin = None
    if call.rope:
        cos, sin = rope_tables(call, T)
    return dict(A=A, a_scale=a_scale, W=W, w_sf=w_sf, w_col_scale=w_col_scale, bias=bias,
                gamma_q=gamma_q, gamma_k=gamma_k, cos=cos, sin=sin)


def sample_rows(call: Call, count: int, seed: int = 12345) -> torch.Tensor:
    """Seeded sorted sample of distinct row indices (always includes the last row)."""
    if count >= call.tokens:
        return torch.arange(call.tokens)
    g = torch.Generator()
    g.manual_seed(seed)
    idx = torch.randperm(call.tokens - 1, generator=g)[:count - 1]
    idx = torch.cat([idx, torch.tensor([call.tokens - 1])])
    return torch.sort(idx).values


def as_numpy_bits(t: Optional[torch.Tensor]):
    """CPU tensor -> numpy array of its raw bits (bfloat16 -> uint16)."""
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view("uint16")
    return t.contiguous().numpy()
