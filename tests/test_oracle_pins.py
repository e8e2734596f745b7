"""Pins of the float64 oracle to things other than itself (CPU only).

Every oracle function is checked against an independent source:
  * the FP8 / UE8M0 / bf16 codecs exhaustively against torch's own dtypes and the
    OFP8 specification's code points (tests/golden/ofp8_e4m3_values.txt);
  * the whole path against an exact brute force written with pure-Python loops and
    rational arithmetic on tiny shapes, and against a hand-worked closed-form case
    (tests/golden/hand_example.json);
  * the across-heads norm against torch's fp64 ``rms_norm`` over the whole segment;
  * the rotate-half RoPE against the complex-multiplication closed form;
  * invariants from the qkv_cte page's definitions: unit-RMS rows for an all-ones
    gamma with zero angle, per-pair norm preservation, V equal to the plain
    dequantised projection, the separate-mode Q call equal to the fused Q slice,
    and row subsets equal to the rows of the full result.

``test_planted_mistakes_are_caught`` plants plausible mistakes in the oracle (on the
CPU, through monkeypatch) and checks that at least one pin fails for each.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import qkv_cte_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers (independent decoders from torch)
# ---------------------------------------------------------------------------

def _torch_e4m3(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def _torch_bf16(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy()).view(
        torch.bfloat16).to(torch.float64).numpy()


def _rand_codes(rng, shape):
    c = rng.integers(0, 254, size=shape).astype(np.uint8)
    c[c == 0x7F] = 0x7E   # no NaN codes
    return c


def _rand_bf16_bits(rng, shape, mean=0.0, std=1.0):
    x = torch.from_numpy(rng.normal(mean, std, size=shape).astype(np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def _tiny_case(seed=0, T=3, H=96, nq=2, nkv=1, d=4, col_scale=True, distinct_halves=True):
    rng = np.random.default_rng(seed)
    I = (nq + 2 * nkv) * d
    c = dict(
        A=_rand_codes(rng, (T, H)),
        a_scale=rng.uniform(0.01, 0.2, size=T).astype(np.float32),
        W=_rand_codes(rng, (I, H)),
        w_sf=rng.integers(118, 136, size=(I, H // 32)).astype(np.uint8),
        w_col_scale=(rng.uniform(0.5, 2.0, size=I).astype(np.float32) if col_scale else None),
        bias=_rand_bf16_bits(rng, I, 0.0, 0.5),
        gamma_q=_rand_bf16_bits(rng, nq * d, 1.0, 0.3) if nq else None,
        gamma_k=_rand_bf16_bits(rng, nkv * d, 1.0, 0.3) if nkv else None,
    )
    ang = rng.uniform(-math.pi, math.pi, size=(T, d))
    if not distinct_halves:
        ang[:, d // 2:] = ang[:, : d // 2]
    c["cos"] = np.cos(ang).astype(np.float32)
    c["sin"] = np.sin(ang).astype(np.float32)
    shape = dict(n_q_heads=nq, n_kv_heads=nkv, d_head=d)
    return c, shape


def _run(c, shape, norm=1, rope=1, eps=1e-6, rows=None):
    return O.qkv_cte(c["A"], c["a_scale"], c["W"], c["w_sf"], c["bias"], c["gamma_q"],
                     c["gamma_k"], c["cos"] if rope else None, c["sin"] if rope else None,
                     norm=norm, rope=rope, eps=eps, w_col_scale=c["w_col_scale"], rows=rows,
                     **shape)


def _brute_force(c, nq, nkv, d, norm, rope, eps):
    """The whole path with Python loops: exact rationals for the projection and the
    sums of squares, floats for rsqrt and the rotation. Decoders come from torch."""
    A = _torch_e4m3(c["A"])
    W = _torch_e4m3(c["W"])
    T, H = A.shape
    I = W.shape[0]
    sf = [[Fraction(2) ** (int(e) - 127) for e in row] for row in c["w_sf"]]
    bias = _torch_bf16(c["bias"])
    cs = c["w_col_scale"]
    o = []
    for t in range(T):
        row = []
        for i in range(I):
            acc = Fraction(0)
            for h in range(H):
                acc += Fraction(float(A[t, h])) * Fraction(float(W[i, h])) * sf[i][h // 32]
            acc *= Fraction(float(c["a_scale"][t]))
            if cs is not None:
                acc *= Fraction(float(cs[i]))
            acc += Fraction(float(bias[i]))
            row.append(acc)
        o.append(row)
    segs = []
    if nq:
        segs.append((0, 0, nq * d, _torch_bf16(c["gamma_q"]), nq))
    if nkv:
        segs.append((1, nq * d, (nq + nkv) * d, _torch_bf16(c["gamma_k"]), nkv))
    out = [[float(v) for v in row] for row in o]
    ss = [[0.0, 0.0] for _ in range(T)]
    inv = [[0.0, 0.0] for _ in range(T)]
    for t in range(T):
        for s_idx, lo, hi, gamma, nh in segs:
            exact = sum((o[t][i] ** 2 for i in range(lo, hi)), Fraction(0))
            ss[t][s_idx] = float(exact)
            r = 1.0 / math.sqrt(float(exact / (nh * d)) + eps) if norm else 0.0
            inv[t][s_idx] = r
            y = []
            for i in range(lo, hi):
                v = float(o[t][i])
                y.append(v * r * float(gamma[i - lo]) if norm else v)
            for head in range(nh):
                base = head * d
                for j in range(d):
                    yj = y[base + j]
                    if rope:
                        if j < d // 2:
                            partner = -y[base + j + d // 2]
                        else:
                            partner = y[base + j - d // 2]
                        val = yj * float(c["cos"][t][j]) + partner * float(c["sin"][t][j])
                    else:
                        val = yj
                    out[t][lo + base + j] = val
    return np.array(out), np.array(ss), np.array(inv)


def _close(a, b, rel=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    tol = rel * (np.abs(b) + np.max(np.abs(b)) * 1e-3 + 1e-300)
    assert np.all(err <= tol), f"{what}: max err {err.max():.3e}"


# ---------------------------------------------------------------------------
# pins (plain functions so the planted-mistake test can run them all)
# ---------------------------------------------------------------------------

def pin_e4m3_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    got = O.decode_e4m3(codes)
    ref = _torch_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def pin_e4m3_spec_values():
    with open(os.path.join(GOLDEN, "ofp8_e4m3_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, value = line.split()[:2]
            got = float(O.decode_e4m3(np.array([int(code, 16)], dtype=np.uint8))[0])
            if value == "nan":
                assert math.isnan(got), code
            else:
                want = float(eval(value))  # exact expressions such as 7*2**-9
                assert got == want, (code, got, want)
                if value.startswith("-"):
                    assert math.copysign(1.0, got) < 0, code


def pin_ue8m0_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    got = O.decode_ue8m0(codes)
    for e in range(255):
        assert got[e] == math.ldexp(1.0, e - 127), e
    assert math.isnan(got[255])
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(got[:255], ref[:255])


def pin_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = O.decode_bf16(bits)
    ref = _torch_bf16(bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def pin_full_bruteforce():
    for seed, (norm, rope) in enumerate([(1, 1), (1, 0), (0, 1), (0, 0)]):
        c, shape = _tiny_case(seed=seed)
        res = _run(c, shape, norm=norm, rope=rope)
        out, ss, inv = _brute_force(c, shape["n_q_heads"], shape["n_kv_heads"], shape["d_head"],
                                    norm, rope, 1e-6)
        _close(res["O"], out, what=f"O norm={norm} rope={rope}")
        _close(res["sumsq"], ss, what="sumsq")
        if norm:
            _close(res["inv_rms"], inv, what="inv_rms")


def pin_separate_bruteforce():
    c, shape = _tiny_case(seed=7, nq=3, nkv=0, d=4, col_scale=False)
    res = _run(c, shape, norm=1, rope=0)
    out, ss, inv = _brute_force(c, 3, 0, 4, 1, 0, 1e-6)
    _close(res["O"], out, what="separate O")
    _close(res["sumsq"], ss, what="separate sumsq")
    _close(res["inv_rms"], inv, what="separate inv")


def pin_kv_call_bruteforce():
    """A call with no Q heads (the K|V form): K normalised across its heads, V as projected."""
    for seed, rope in ((13, 0), (14, 1)):
        c, shape = _tiny_case(seed=seed, nq=0, nkv=2, d=4)
        res = _run(c, shape, norm=1, rope=rope)
        out, ss, inv = _brute_force(c, 0, 2, 4, 1, rope, 1e-6)
        _close(res["O"], out, what=f"K|V O rope={rope}")
        _close(res["sumsq"], ss, what="K|V sumsq")
        _close(res["inv_rms"], inv, what="K|V inv")
        assert np.all(res["sumsq"][:, 0] == 0) and np.all(res["inv_rms"][:, 0] == 0)


def pin_kv_call_equals_separate_k_and_v_calls():
    """The K|V call on W = [W_k; W_v] gives the separate K call (normalised as its only
    segment, gamma_k as its gamma) on the K columns and the separate plain V call on the
    V columns, as the cross-attention's three separate calls would."""
    c, shape = _tiny_case(seed=15, T=3, H=64, nq=0, nkv=2, d=8)
    kv = _run(c, shape, norm=1, rope=0)
    k = 16
    sep_k = dict(c, W=c["W"][:k], w_sf=c["w_sf"][:k], bias=c["bias"][:k], w_col_scale=c["w_col_scale"][:k],
                 gamma_q=c["gamma_k"], gamma_k=None)
    sep_v = dict(c, W=c["W"][k:], w_sf=c["w_sf"][k:], bias=c["bias"][k:], w_col_scale=c["w_col_scale"][k:],
                 gamma_q=None, gamma_k=None)
    one = dict(n_q_heads=2, n_kv_heads=0, d_head=8)
    rk = _run(sep_k, one, norm=1, rope=0)
    rv = _run(sep_v, one, norm=0, rope=0)
    _close(kv["O"][:, :k], rk["O"], rel=1e-14, what="K|V vs separate K")
    _close(kv["O"][:, k:], rv["O"], rel=0, what="K|V vs separate V")
    _close(kv["inv_rms"][:, 1], rk["inv_rms"][:, 0], rel=1e-14, what="K|V inv vs separate K")
    _close(kv["sumsq"][:, 1], rk["sumsq"][:, 0], rel=1e-14, what="K|V sumsq vs separate K")


def pin_hand_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    H = g["hidden"]
    I = (g["n_q_heads"] + 2 * g["n_kv_heads"]) * g["d_head"]
    hx = lambda xs: np.array([int(x, 16) for x in xs], dtype=np.uint16)
    res = O.qkv_cte(
        np.full((1, H), int(g["A_code"], 16), dtype=np.uint8),
        np.array([g["a_scale"]], dtype=np.float32),
        np.full((I, H), int(g["W_code"], 16), dtype=np.uint8),
        np.repeat(np.array(g["w_sf"], dtype=np.uint8)[:, None], H // 32, axis=1),
        hx(g["bias_bf16"]), hx(g["gamma_q_bf16"]), hx(g["gamma_k_bf16"]),
        np.array([g["cos"]], dtype=np.float32), np.array([g["sin"]], dtype=np.float32),
        n_q_heads=g["n_q_heads"], n_kv_heads=g["n_kv_heads"], d_head=g["d_head"], norm=1, rope=1,
        eps=g["eps"])
    ev = lambda xs: np.array([eval(x, {"math": math}) for x in xs], dtype=np.float64)
    _close(res["sumsq"][0], ev(g["expected"]["sumsq"]), rel=1e-15, what="hand sumsq")
    _close(res["inv_rms"][0], ev(g["expected"]["inv_rms"]), rel=1e-14, what="hand inv")
    _close(res["O"][0], ev(g["expected"]["O"]), rel=1e-14, what="hand O")


def pin_norm_vs_torch_rms_norm():
    c, shape = _tiny_case(seed=3, T=5, H=64, nq=3, nkv=2, d=8)
    res = _run(c, shape, norm=1, rope=0, eps=1e-3)
    o = torch.from_numpy(res["projected"])
    for lo, hi, g in ((0, 24, c["gamma_q"]), (24, 40, c["gamma_k"])):
        ref = torch.nn.functional.rms_norm(o[:, lo:hi], (hi - lo,),
                                           weight=torch.from_numpy(_torch_bf16(g)), eps=1e-3)
        _close(res["O"][:, lo:hi], ref.numpy(), rel=1e-12, what="rms_norm")
    _close(res["O"][:, 40:], res["projected"][:, 40:], rel=0, what="V untouched")


def pin_rope_complex_closed_form():
    rng = np.random.default_rng(11)
    rows, heads, d = 4, 3, 16
    y = rng.normal(size=(rows, heads * d))
    ang = rng.uniform(-10, 10, size=(rows, d // 2))
    cos = np.concatenate([np.cos(ang)] * 2, axis=1)
    sin = np.concatenate([np.sin(ang)] * 2, axis=1)
    got = O.apply_norm_rope(y, None, None, cos, sin, d, norm=0, rope=1)
    h = y.reshape(rows, heads, d)
    z = (h[:, :, : d // 2] + 1j * h[:, :, d // 2:]) * np.exp(1j * ang)[:, None, :]
    ref = np.concatenate([z.real, z.imag], axis=2).reshape(rows, heads * d)
    _close(got, ref, rel=1e-13, what="rope closed form")


def pin_unit_rms_invariant():
    c, shape = _tiny_case(seed=5, T=4, H=64, nq=2, nkv=2, d=8, distinct_halves=False)
    c["gamma_q"] = np.full(16, 0x3F80, dtype=np.uint16)
    c["gamma_k"] = np.full(16, 0x3F80, dtype=np.uint16)
    c["cos"] = np.ones_like(c["cos"])
    c["sin"] = np.zeros_like(c["sin"])
    eps = 1e-2
    res = _run(c, shape, norm=1, rope=1, eps=eps)
    for lo, hi, col in ((0, 16, 0), (16, 32, 1)):
        ms = res["sumsq"][:, col] / 16
        rms = np.sqrt(np.mean(res["O"][:, lo:hi] ** 2, axis=1))
        _close(rms, np.sqrt(ms / (ms + eps)), rel=1e-13, what="unit rms")


def pin_pair_norm_invariant():
    c, shape = _tiny_case(seed=6, T=4, H=64, nq=2, nkv=1, d=8, distinct_halves=False)
    # float64 tables: the invariant needs cos^2 + sin^2 == 1 to rounding of fp64
    ang = np.random.default_rng(60).uniform(-math.pi, math.pi, size=(4, 4))
    c["cos"] = np.cos(np.concatenate([ang, ang], axis=1))
    c["sin"] = np.sin(np.concatenate([ang, ang], axis=1))
    normed = _run(c, shape, norm=1, rope=0)["O"]
    roped = _run(c, shape, norm=1, rope=1)["O"]
    for lo, hi in ((0, 16), (16, 24)):
        a = normed[:, lo:hi].reshape(4, -1, 8)
        b = roped[:, lo:hi].reshape(4, -1, 8)
        na = a[:, :, :4] ** 2 + a[:, :, 4:] ** 2
        nb = b[:, :, :4] ** 2 + b[:, :, 4:] ** 2
        _close(nb, na, rel=1e-12, what="pair norm")


def pin_v_is_plain_projection():
    c, shape = _tiny_case(seed=8, T=2, H=64, nq=1, nkv=2, d=4)
    res = _run(c, shape, norm=1, rope=1)
    out, _, _ = _brute_force(dict(c), 1, 2, 4, 0, 0, 1e-6)   # plain projection
    _close(res["O"][:, 12:], out[:, 12:], what="V")


def pin_separate_equals_fused_slice():
    c, shape = _tiny_case(seed=9, T=3, H=64, nq=2, nkv=2, d=8, distinct_halves=False)
    fused = _run(c, shape, norm=1, rope=1)
    q = 16
    sep = dict(c, W=c["W"][:q], w_sf=c["w_sf"][:q], bias=c["bias"][:q],
               w_col_scale=c["w_col_scale"][:q], gamma_k=None)
    res = _run(sep, dict(n_q_heads=2, n_kv_heads=0, d_head=8), norm=1, rope=1)
    _close(res["O"], fused["O"][:, :q], rel=1e-14, what="separate vs fused")
    _close(res["inv_rms"][:, 0], fused["inv_rms"][:, 0], rel=1e-14, what="separate inv")


def pin_rows_subset():
    c, shape = _tiny_case(seed=10, T=6, H=64, nq=1, nkv=1, d=8)
    full = _run(c, shape)
    rows = np.array([0, 3, 5])
    sub = _run(c, shape, rows=rows)
    for k in ("O", "sumsq", "inv_rms"):
        _close(sub[k], full[k][rows], rel=0, what=k)


def pin_nbsd_layout():
    rng = np.random.default_rng(12)
    T, heads, d = 5, 3, 4
    o = rng.normal(size=(T, heads * d))
    n = O.to_nbsd(o, d)
    assert n.shape == (heads, T, d)
    for h in range(heads):
        for t in range(T):
            for j in range(d):
                assert n[h, t, j] == o[t, h * d + j]


# --- the producer step: e4m3 encoder, row quantiser, packed rows ------------------

def _e4m3_grid():
    return _torch_e4m3(np.arange(0x7F, dtype=np.uint8))      # ascending magnitudes 0 .. 448


def pin_encode_e4m3_vs_torch():
    """The encoder against torch's float32 -> float8_e4m3fn cast (round to nearest,
    ties to even) on every grid point, every midpoint (the ties), one fp32 ulp either
    side of each midpoint, and random values over the whole range, both signs.
    torch does not saturate, so this covers |v| <= 448; saturation has its own pin."""
    g = _e4m3_grid()
    mid = (g[1:] + g[:-1]) / 2
    m32 = mid.astype(np.float32)
    assert np.all(m32.astype(np.float64) == mid)              # the ties are exact in fp32
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(0))
    rng = np.random.default_rng(60)
    rnd = np.exp2(rng.uniform(-14, np.log2(448.0), size=20000)).astype(np.float32)
    v = np.concatenate([g.astype(np.float32), m32, up[up <= 448], dn, rnd, np.float32([0.0])])
    v = np.concatenate([v, -v])
    got = O.encode_e4m3(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} codes differ from torch's cast"
    assert O.encode_e4m3(np.float64(-0.0)) == 0x80 and O.encode_e4m3(np.float64(0.0)) == 0x00


def pin_encode_e4m3_saturation():
    """Saturating conversion: every finite magnitude above 448 (including those past
    the would-be next binade, and infinity) gives the largest finite code, 0x7E /
    0xFE (S.1111.110 = 448 by the OFP8 table); NaN stays NaN (0x7F)."""
    v = np.array([448.0, 455.9, 464.0, 470.0, 480.0, 1e4, 3.0e38, np.inf])
    assert np.all(O.encode_e4m3(v) == 0x7E)
    assert np.all(O.encode_e4m3(-v) == 0xFE)
    assert O.encode_e4m3(np.float64(np.nan)) == 0x7F
    assert _torch_e4m3(np.uint8([0x7E]))[0] == 448.0


def _quant_rows():
    """bf16 rows covering the method's cases: Gaussian, heavy outliers, values in the
    bf16 subnormal range, an all-zero row, a one-hot row, a row of negative zeros and
    tiny negatives, and one row per exponent band."""
    rng = np.random.default_rng(61)
    H = 64
    rows = [rng.normal(0, 1, H), rng.normal(0, 1, H) * np.where(rng.random(H) < 0.05, 300.0, 1.0),
            rng.normal(0, 1, H) * 1e-39, np.zeros(H), np.eye(1, H, 17)[0] * -3.5,
            np.concatenate([[-0.0] * (H // 2), -np.abs(rng.normal(0, 1e-6, H // 2))]),
            rng.normal(0, 1, H) * 1e30, rng.normal(0, 1, H) * 2.0 ** -100]
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def pin_row_quantise_invariants():
    bits = _quant_rows()
    x = _torch_bf16(bits)
    codes, s = O.row_quantise(bits)
    assert codes.dtype == np.uint8 and codes.shape == x.shape and s.dtype == np.float32
    val = _torch_e4m3(codes)
    amax = np.abs(x).max(axis=1)
    for t in range(x.shape[0]):
        if amax[t] == 0:
            assert s[t] == 1.0 and np.all(val[t] == 0), "all-zero row: scale 1, zero codes"
            continue
        # the scale is the row's amax over 448 to fp32 precision (subnormal scales
        # keep only their absolute precision)
        assert abs(float(s[t]) * 448.0 - amax[t]) <= 2.0 ** -23 * amax[t] + 448.0 * 2.0 ** -150
        q = x[t] / float(s[t])
        # the largest element lands on the top of the grid
        assert np.max(np.abs(val[t])) == 448.0
        # nearest grid point: error at most half an e4m3 step at |q| (plus the fp32
        # rounding of the quotient, and the relative slack of a subnormal scale)
        e = np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6)))
        half_step = 2.0 ** (e - 4)
        slack = 2.0 ** -22 * np.abs(q) + (2.0 ** -7 * np.abs(q) if s[t] < 2.0 ** -126 else 0.0)
        assert np.all(np.abs(val[t] - q) <= half_step + slack), f"row {t}: not the nearest code"
        # sign kept (zeros included), order kept
        assert np.array_equal(codes[t] >> 7, np.signbit(x[t]).astype(np.uint8))
        order = np.argsort(x[t], kind="stable")
        assert np.all(np.diff(val[t][order]) >= 0)


def pin_row_quantise_exact_power_of_two():
    """Closed form: a row whose elements are e4m3 grid points times 2^j, with 448*2^j
    present, has scale exactly 2^j and quantises without error."""
    rng = np.random.default_rng(62)
    g = _e4m3_grid()
    for j in (-20, -3, 0, 5, 40):
        vals = rng.choice(g, size=32) * rng.choice([-1.0, 1.0], size=32)
        vals[7] = 448.0
        x = vals * 2.0 ** j
        bits = torch.tensor(x[None, :], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.all(_torch_bf16(bits)[0] == x)               # exact in bf16
        codes, s = O.row_quantise(bits)
        assert s[0] == 2.0 ** j
        assert np.all(_torch_e4m3(codes)[0] * 2.0 ** j == x)


def pin_row_quantise_vs_torch_route():
    """The special case the method reduces to in torch: fp32 amax / 448, fp32
    division, then torch's e4m3 cast (torch does not saturate, but every quotient here
    is below 464, where rounding alone already gives 448)."""
    bits = _quant_rows()
    xt = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float()
    amax = xt.abs().amax(dim=1)
    st = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    qt = xt / st[:, None]
    assert float(qt.abs().max()) < 464.0
    ref = qt.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    codes, s = O.row_quantise(bits)
    assert np.array_equal(s, st.numpy())
    assert np.array_equal(codes, ref)


def pin_packed_rows_layout():
    """Byte layout by brute force: row t of the packed tensor is the row's H codes
    followed by struct.pack('<f', scale); unpacking inverts packing exactly."""
    import struct

    rng = np.random.default_rng(63)
    T, H = 3, 8
    codes = _rand_codes(rng, (T, H))
    scale = np.float32([0.015625, 3.0e-5, 2.5])
    p = O.pack_rows(codes, scale)
    assert p.dtype == np.uint8 and p.shape == (T, H + 4)
    flat = p.reshape(-1)
    for t in range(T):
        row = bytes(codes[t].tolist()) + struct.pack("<f", float(scale[t]))
        assert bytes(flat[t * (H + 4):(t + 1) * (H + 4)].tolist()) == row
    c2, s2 = O.unpack_rows(p)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scale) and s2.dtype == np.float32


# --- per-head qk-norm and the interleaved -> rotate-half permutation ----------------

def _head_case(seed, nq=3, nkv=2, d=8, T=4, H=64):
    c, shape = _tiny_case(seed=seed, T=T, H=H, nq=nq, nkv=nkv, d=d)
    rng = np.random.default_rng(seed + 500)
    c["gamma_q"] = _rand_bf16_bits(rng, d, 1.0, 0.3)
    c["gamma_k"] = _rand_bf16_bits(rng, d, 1.0, 0.3) if nkv else None
    return c, shape


def pin_head_norm_vs_torch():
    """Per-head RMS_NORM and LAYER_NORM against torch's own fp64 rms_norm / layer_norm
    over each head's d_head lanes with the [d_head] gamma as weight (no bias)."""
    import torch.nn.functional as F

    for kind in (O.NORM_HEAD_RMS, O.NORM_HEAD_LAYER):
        c, shape = _head_case(seed=70 + kind)
        nq, nkv, d = shape["n_q_heads"], shape["n_kv_heads"], shape["d_head"]
        eps = 1e-5
        res = _run(c, shape, norm=kind, rope=0, eps=eps)
        o = torch.from_numpy(res["projected"])
        T = o.shape[0]
        for lo, hi, g in ((0, nq * d, c["gamma_q"]), (nq * d, (nq + nkv) * d, c["gamma_k"])):
            x = o[:, lo:hi].reshape(T, -1, d)
            w = torch.from_numpy(_torch_bf16(g))
            ref = F.rms_norm(x, (d,), w, eps) if kind == O.NORM_HEAD_RMS else F.layer_norm(x, (d,), w, None, eps)
            _close(res["O"][:, lo:hi], ref.reshape(T, -1).numpy(), rel=1e-12, what=f"head norm {kind}")
        _close(res["O"][:, (nq + nkv) * d:], res["projected"][:, (nq + nkv) * d:], rel=0, what="V untouched")
        _close(res["inv_rms"], np.zeros_like(res["inv_rms"]), rel=0, what="no across-heads inv_rms")


def pin_head_norm_invariants():
    """gamma = 1, no rotation: every head of Q and K has RMS 1 (RMS_NORM), or mean 0
    and mean square 1 (LAYER_NORM), up to eps; one head per segment makes the per-head
    RMS_NORM the across-heads norm (with the same gamma)."""
    eps = 1e-9
    for kind in (O.NORM_HEAD_RMS, O.NORM_HEAD_LAYER):
        c, shape = _head_case(seed=80 + kind)
        d = shape["d_head"]
        ones = np.full(d, 0x3F80, dtype=np.uint16)
        c["gamma_q"], c["gamma_k"] = ones, ones
        res = _run(c, shape, norm=kind, rope=0, eps=eps)
        qk = (shape["n_q_heads"] + shape["n_kv_heads"]) * d
        h = res["O"][:, :qk].reshape(res["O"].shape[0], -1, d)
        assert np.allclose(np.mean(h ** 2, axis=2), 1.0, rtol=1e-6)
        if kind == O.NORM_HEAD_LAYER:
            assert np.allclose(np.mean(h, axis=2), 0.0, atol=1e-9)
    c, shape = _tiny_case(seed=85, T=5, H=64, nq=1, nkv=1, d=8)
    per_head = _run(c, shape, norm=O.NORM_HEAD_RMS, rope=1)
    across = _run(c, shape, norm=O.NORM_ACROSS_HEADS, rope=1)
    _close(per_head["O"], across["O"], rel=1e-12, what="one head per segment")


def pin_rope_interleaved_complex():
    """Interleaved RoPE is the complex product of each lane pair (2j, 2j+1) with
    e^{i theta_j} (tables carry theta_j at lanes 2j and 2j+1)."""
    rng = np.random.default_rng(90)
    T, heads, d = 3, 2, 8
    y = rng.normal(size=(T, heads * d))
    th = rng.uniform(-math.pi, math.pi, size=(T, d // 2))
    cos, sin = np.repeat(np.cos(th), 2, axis=1), np.repeat(np.sin(th), 2, axis=1)
    got = O.rope_interleaved(y, cos, sin, d).reshape(T, heads, d)
    z = y.reshape(T, heads, d // 2, 2)
    zc = (z[..., 0] + 1j * z[..., 1]) * np.exp(1j * th)[:, None, :]
    _close(got[..., 0::2], zc.real, rel=1e-13, what="interleaved re")
    _close(got[..., 1::2], zc.imag, rel=1e-13, what="interleaved im")


def pin_permutation_layout():
    """The permutation by hand for d = 8, and its application to labelled channels:
    Q and K heads permuted head by head, V channels in place."""
    assert O.interleaved_to_rotate_half(8).tolist() == [0, 2, 4, 6, 1, 3, 5, 7]
    nq, nkv, d = 2, 1, 4
    lab = np.arange((nq + 2 * nkv) * d)
    got = O.permute_qk_rows(lab, nq, nkv, d).tolist()
    assert got == [0, 2, 1, 3, 4, 6, 5, 7, 8, 10, 9, 11, 12, 13, 14, 15]


def pin_interleaved_checkpoint_equivalence():
    """The offline conversion the page prescribes: an interleaved-convention model
    (weights, scales, bias, gamma, cos/sin in interleaved lane order, interleaved RoPE)
    equals the rotate-half path run on the permuted tensors, up to the same
    permutation of the Q/K output columns - for every norm kind."""
    for norm in (O.NORM_ACROSS_HEADS, O.NORM_HEAD_RMS, O.NORM_HEAD_LAYER, O.NORM_NONE):
        c, shape = (_head_case(seed=95 + norm) if norm in (O.NORM_HEAD_RMS, O.NORM_HEAD_LAYER)
                    else _tiny_case(seed=95 + norm, T=4, H=64, nq=3, nkv=2, d=8))
        nq, nkv, d = shape["n_q_heads"], shape["n_kv_heads"], shape["d_head"]
        rng = np.random.default_rng(99 + norm)
        th = rng.uniform(-math.pi, math.pi, size=(c["A"].shape[0], d // 2))
        cos_il = np.repeat(np.cos(th), 2, axis=1).astype(np.float32)
        sin_il = np.repeat(np.sin(th), 2, axis=1).astype(np.float32)
        il = O.qkv_cte(c["A"], c["a_scale"], c["W"], c["w_sf"], c["bias"], c["gamma_q"], c["gamma_k"], cos_il,
                       sin_il, norm=norm, rope=1, eps=1e-6, w_col_scale=c["w_col_scale"], rope_layout="interleaved",
                       **shape)
        per_head = norm in (O.NORM_HEAD_RMS, O.NORM_HEAD_LAYER)
        pg = (lambda g, n: O.permute_qk_rows(g, 1, 0, d)) if per_head else (lambda g, n: O.permute_qk_rows(g, n, 0, d))
        rh = O.qkv_cte(c["A"], c["a_scale"],
                       O.permute_qk_rows(c["W"], nq, nkv, d), O.permute_qk_rows(c["w_sf"], nq, nkv, d),
                       O.permute_qk_rows(c["bias"], nq, nkv, d), pg(c["gamma_q"], nq), pg(c["gamma_k"], nkv),
                       O.permute_qk_rows(cos_il.T, 1, 0, d).T, O.permute_qk_rows(sin_il.T, 1, 0, d).T,
                       norm=norm, rope=1, eps=1e-6, w_col_scale=O.permute_qk_rows(c["w_col_scale"], nq, nkv, d),
                       **shape)
        expect = O.permute_qk_rows(il["O"].T, nq, nkv, d).T
        _close(rh["O"], expect, rel=1e-12, what=f"interleaved equivalence, norm {norm}")


PINS = [pin_head_norm_vs_torch, pin_head_norm_invariants, pin_rope_interleaved_complex, pin_permutation_layout,
        pin_interleaved_checkpoint_equivalence, pin_nbsd_layout, pin_encode_e4m3_vs_torch, pin_encode_e4m3_saturation, pin_row_quantise_invariants,
        pin_row_quantise_exact_power_of_two, pin_row_quantise_vs_torch_route, pin_packed_rows_layout, pin_e4m3_exhaustive, pin_e4m3_spec_values, pin_ue8m0_exhaustive, pin_bf16_exhaustive,
        pin_full_bruteforce, pin_separate_bruteforce, pin_hand_example, pin_norm_vs_torch_rms_norm,
        pin_rope_complex_closed_form, pin_unit_rms_invariant, pin_pair_norm_invariant,
        pin_v_is_plain_projection, pin_separate_equals_fused_slice, pin_rows_subset,
        pin_kv_call_bruteforce, pin_kv_call_equals_separate_k_and_v_calls]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

_orig = {name: getattr(O, name) for name in
         ("decode_e4m3", "decode_ue8m0", "decode_bf16", "dequant_activations", "dequant_weights",
          "project", "segments", "segment_sumsq", "inv_rms", "rotate_half", "apply_norm_rope",
          "qkv_cte", "to_nbsd", "encode_e4m3", "row_quantise", "pack_rows", "unpack_rows", "head_norm",
          "rope_interleaved", "interleaved_to_rotate_half", "permute_qk_rows")}


def _e4m3_bias8(codes):
    return _orig["decode_e4m3"](codes) * 0.5


def _e4m3_subnormal_as_normal(codes):
    c = np.asarray(codes, dtype=np.uint8)
    v = _orig["decode_e4m3"](c)
    sub = ((c >> 3) & 0xF) == 0
    return np.where(sub & ((c & 7) > 0), np.sign(v + 0.0) * (1 + (c & 7) / 8.0) * 2.0 ** -6, v)


def _e4m3_unsigned(codes):
    return np.abs(_orig["decode_e4m3"](codes))


def _ue8m0_bias128(codes):
    return _orig["decode_ue8m0"](codes) * 0.5


def _bf16_wrong_shift(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 15
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def _weights_block16(W, w_sf):
    I, H = W.shape
    scale = O.decode_ue8m0(w_sf)
    return O.decode_e4m3(W) * scale[:, np.minimum(np.arange(H) // 16, H // 32 - 1)]


def _weights_block_transposed(W, w_sf):
    I, H = W.shape
    scale = O.decode_ue8m0(w_sf)
    return O.decode_e4m3(W) * scale[:, np.arange(H) % (H // 32)]


def _act_scale_ignored(A, a_scale):
    return O.decode_e4m3(A)


def _project_no_bias(A, a_scale, W, w_sf, w_col_scale=None, bias=None):
    return _orig["project"](A, a_scale, W, w_sf, w_col_scale, None)


def _project_no_colscale(A, a_scale, W, w_sf, w_col_scale=None, bias=None):
    return _orig["project"](A, a_scale, W, w_sf, None, bias)


def _project_transposed(A, a_scale, W, w_sf, w_col_scale=None, bias=None):
    a = O.dequant_activations(A, a_scale)
    w = O.dequant_weights(W, w_sf)
    o = a @ w[:, ::-1].T          # output columns reversed (a wrong index map)
    if w_col_scale is not None:
        o = o * np.asarray(w_col_scale, dtype=np.float64)[None, :]
    if bias is not None:
        o = o + O.decode_bf16(bias)[None, :]
    return o


def _sumsq_mean(o, nq, nkv, d):
    ss = _orig["segment_sumsq"](o, nq, nkv, d)
    ss[:, 0] /= nq * d
    return ss


def _sumsq_k_includes_v(o, nq, nkv, d):
    ss = _orig["segment_sumsq"](o, nq, nkv, d)
    if nkv:
        ss[:, 1] = np.sum(o[:, nq * d:] ** 2, axis=1)
    return ss


def _inv_eps_outside(ss, nq, nkv, d, eps, tp=1):
    out = _orig["inv_rms"](ss, nq, nkv, d, 0.0, tp)
    return out + eps


def _inv_heads_only(ss, nq, nkv, d, eps, tp=1):
    out = np.zeros_like(ss)
    out[:, 0] = 1.0 / np.sqrt(ss[:, 0] / nq + eps)
    if nkv:
        out[:, 1] = 1.0 / np.sqrt(ss[:, 1] / nkv + eps)
    return out


def _inv_k_uses_nq(ss, nq, nkv, d, eps, tp=1):
    out = _orig["inv_rms"](ss, nq, nkv, d, eps, tp)
    if nkv:
        out[:, 1] = 1.0 / np.sqrt(ss[:, 1] / (nq * d) + eps)
    return out


def _rotate_sign(y, d):
    return -_orig["rotate_half"](y, d)


def _rotate_interleaved(y, d):
    rows, width = y.shape
    h = y.reshape(rows, width // 2, 2)
    return np.stack([-h[:, :, 1], h[:, :, 0]], axis=2).reshape(rows, width)


def _gamma_after_rope(x, inv, gamma, cos, sin, d, norm, rope):
    y = _orig["apply_norm_rope"](x, inv, None, cos, sin, d, 0, rope)
    if norm:
        y = y * inv[:, None] * O.decode_bf16(gamma)[None, :]
    return y


def _cos_sin_swapped(x, inv, gamma, cos, sin, d, norm, rope):
    return _orig["apply_norm_rope"](x, inv, gamma, sin, cos, d, norm, rope)


def _gamma_ignored(x, inv, gamma, cos, sin, d, norm, rope):
    ones = np.full(x.shape[1], 0x3F80, dtype=np.uint16)
    return _orig["apply_norm_rope"](x, inv, ones, cos, sin, d, norm, rope)


def _v_normalised(*args, **kw):
    res = _orig["qkv_cte"](*args, **kw)
    nq, nkv, d = kw["n_q_heads"], kw["n_kv_heads"], kw["d_head"]
    if nkv and kw["norm"]:
        v = res["projected"][:, (nq + nkv) * d:]
        res["O"][:, (nq + nkv) * d:] = v / np.sqrt(np.mean(v ** 2, axis=1, keepdims=True) + kw["eps"])
    return res


def _nbsd_heads_swapped(O_, d):
    T, I = O_.shape
    return O_.reshape(T, d, I // d).transpose(2, 0, 1)


def _k_uses_gamma_q(*args, **kw):
    args = list(args)
    if args[6] is not None:
        args[6] = args[5][: len(args[6])]
    return _orig["qkv_cte"](*args, **kw)


def _encode_truncate(v):
    v = np.asarray(v, dtype=np.float64)
    g = _e4m3_grid()
    a = np.minimum(np.abs(v), 448.0)
    idx = np.searchsorted(g, a, side="right") - 1
    return (idx.astype(np.uint8) | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)


def _encode_ties_away(v):
    v = np.asarray(v, dtype=np.float64)
    g = _e4m3_grid()
    a = np.minimum(np.abs(v), 448.0)
    hi = np.minimum(np.searchsorted(g, a, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    code = np.where(g[hi] - a <= a - g[lo], hi, lo).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << 7)


def _encode_no_saturation(v):
    v = np.asarray(v, dtype=np.float64)
    c = _orig["encode_e4m3"](v)
    return np.where(np.abs(v) > 464.0, np.uint8(0x7F), c).astype(np.uint8)


def _encode_drops_sign(v):
    return _orig["encode_e4m3"](np.abs(np.asarray(v, dtype=np.float64)))


def _quant_scale_127(x_bits):
    x = O.decode_bf16(x_bits).astype(np.float32)
    amax = np.abs(x).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    return O.encode_e4m3((x / s[:, None]).astype(np.float64)), s


def _quant_amax_whole_tensor(x_bits):
    x = O.decode_bf16(x_bits).astype(np.float32)
    amax = np.full(x.shape[0], np.abs(x).max(), dtype=np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)
    return O.encode_e4m3((x / s[:, None]).astype(np.float64)), s


def _quant_multiply_by_448_over_amax(x_bits):
    x = O.decode_bf16(x_bits).astype(np.float32)
    amax = np.abs(x).max(axis=1)
    with np.errstate(divide="ignore", over="ignore"):
        r = np.where(amax > 0, np.float32(448.0) / amax, np.float32(1.0)).astype(np.float32)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    with np.errstate(invalid="ignore"):
        q = (x * r[:, None]).astype(np.float32)
    return O.encode_e4m3(q.astype(np.float64)), s


def _pack_scale_first(codes, scale):
    p = _orig["pack_rows"](codes, scale)
    H = p.shape[1] - 4
    return np.concatenate([p[:, H:], p[:, :H]], axis=1)


def _pack_big_endian(codes, scale):
    codes = np.asarray(codes, dtype=np.uint8)
    tail = np.asarray(scale, dtype=">f4").reshape(-1, 1).view(np.uint8)
    return np.concatenate([codes, tail], axis=1)


def _head_norm_segment_stats(x, gamma, d, kind, eps):
    rows, width = x.shape
    h = x.reshape(rows, width // d, d)
    if kind == O.NORM_HEAD_LAYER:
        h = h - h.mean(axis=(1, 2), keepdims=True)
    inv = 1.0 / np.sqrt(np.mean(h ** 2, axis=(1, 2), keepdims=True) + eps)
    return (h * inv * O.decode_bf16(gamma)[None, None, :]).reshape(rows, width)


def _head_norm_unbiased(x, gamma, d, kind, eps):
    rows, width = x.shape
    h = x.reshape(rows, width // d, d)
    if kind == O.NORM_HEAD_LAYER:
        h = h - h.mean(axis=2, keepdims=True)
        inv = 1.0 / np.sqrt(np.sum(h ** 2, axis=2, keepdims=True) / (d - 1) + eps)
    else:
        inv = 1.0 / np.sqrt(np.mean(h ** 2, axis=2, keepdims=True) + eps)
    return (h * inv * O.decode_bf16(gamma)[None, None, :]).reshape(rows, width)


def _head_norm_layer_uncentred(x, gamma, d, kind, eps):
    return _orig["head_norm"](x, gamma, d, O.NORM_HEAD_RMS, eps)


def _rope_interleaved_sign(y, cos, sin, d):
    return _orig["rope_interleaved"](y, cos, -np.asarray(sin), d)


def _perm_odd_first(d):
    half = d // 2
    return np.concatenate([2 * np.arange(half) + 1, 2 * np.arange(half)])


def _permute_v_too(x, nq, nkv, d):
    return _orig["permute_qk_rows"](x, nq + nkv, nkv, d) if nkv else _orig["permute_qk_rows"](x, nq, nkv, d)


MUTANTS = {
    "head_norm_segment_stats": ("head_norm", _head_norm_segment_stats),
    "head_norm_unbiased_var": ("head_norm", _head_norm_unbiased),
    "head_norm_layer_uncentred": ("head_norm", _head_norm_layer_uncentred),
    "rope_interleaved_sign": ("rope_interleaved", _rope_interleaved_sign),
    "perm_odd_first": ("interleaved_to_rotate_half", _perm_odd_first),
    "permute_v_too": ("permute_qk_rows", _permute_v_too),
    "encode_truncate": ("encode_e4m3", _encode_truncate),
    "encode_ties_away": ("encode_e4m3", _encode_ties_away),
    "encode_no_saturation": ("encode_e4m3", _encode_no_saturation),
    "encode_drops_sign": ("encode_e4m3", _encode_drops_sign),
    "quant_scale_127": ("row_quantise", _quant_scale_127),
    "quant_amax_whole_tensor": ("row_quantise", _quant_amax_whole_tensor),
    "quant_multiply_by_reciprocal": ("row_quantise", _quant_multiply_by_448_over_amax),
    "pack_scale_first": ("pack_rows", _pack_scale_first),
    "pack_big_endian": ("pack_rows", _pack_big_endian),
    "e4m3_bias8": ("decode_e4m3", _e4m3_bias8),
    "e4m3_subnormal_as_normal": ("decode_e4m3", _e4m3_subnormal_as_normal),
    "e4m3_unsigned": ("decode_e4m3", _e4m3_unsigned),
    "ue8m0_bias128": ("decode_ue8m0", _ue8m0_bias128),
    "bf16_wrong_shift": ("decode_bf16", _bf16_wrong_shift),
    "weights_block16": ("dequant_weights", _weights_block16),
    "weights_block_transposed": ("dequant_weights", _weights_block_transposed),
    "act_scale_ignored": ("dequant_activations", _act_scale_ignored),
    "project_no_bias": ("project", _project_no_bias),
    "project_no_colscale": ("project", _project_no_colscale),
    "project_column_map": ("project", _project_transposed),
    "sumsq_mean": ("segment_sumsq", _sumsq_mean),
    "sumsq_k_includes_v": ("segment_sumsq", _sumsq_k_includes_v),
    "inv_eps_outside": ("inv_rms", _inv_eps_outside),
    "inv_heads_only": ("inv_rms", _inv_heads_only),
    "inv_k_uses_nq": ("inv_rms", _inv_k_uses_nq),
    "rotate_sign": ("rotate_half", _rotate_sign),
    "rotate_interleaved": ("rotate_half", _rotate_interleaved),
    "gamma_after_rope": ("apply_norm_rope", _gamma_after_rope),
    "cos_sin_swapped": ("apply_norm_rope", _cos_sin_swapped),
    "gamma_ignored": ("apply_norm_rope", _gamma_ignored),
    "v_normalised": ("qkv_cte", _v_normalised),
    "k_uses_gamma_q": ("qkv_cte", _k_uses_gamma_q),
    "nbsd_heads_swapped": ("to_nbsd", _nbsd_heads_swapped),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except Exception:  # any failure (assertion, shape error) counts as caught
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"
