"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on seeded
inputs and compare with the float64 oracle on the same inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import workloads as wl
from oracle import qkv_cte_oracle as O
from rope_tcgen05_mxfp8_gb300 import QkvCte

# Tolerances: per bf16 output element |err| <= REL*|ref| + ABS; sums of squares and
# inv_rms within SS_REL relative.
REL = 1e-2
ABS = 1e-2
SS_REL = 1e-4


def to_device(inp, dev):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def run_path(call, g, tile_n=0, flags=0, want_sumsq=True, want_inv=True, stream=None, out=None, nbsd=False,
             input_layout=0, A_in=None):
    """Run through the C ABI; the returned O is always viewed as BSD [T, I] (an NBSd
    result is permuted back, so the comparison sees every element where the oracle
    puts it). With a packed or bf16 input layout, A_in is that input on the device."""
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_LAYOUT_BSD, QKV_CTE_LAYOUT_NBSD

    dev = g["A"].device
    op = QkvCte(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, norm=call.norm,
                rope=call.rope, eps=call.eps, tile_n=tile_n, flags=flags, device=dev,
                output_layout=QKV_CTE_LAYOUT_NBSD if nbsd else QKV_CTE_LAYOUT_BSD, input_layout=input_layout)
    sumsq = torch.full((call.tokens, 2), float("nan"), dtype=torch.float32, device=dev) if want_sumsq else None
    # inv_rms is an output of the across-heads norm only
    inv = (torch.full((call.tokens, 2), float("nan"), dtype=torch.float32, device=dev)
           if want_inv and call.norm in (0, 1) else None)
    heads = call.width // call.d_head
    if out is None:
        shape = (heads, call.tokens, call.d_head) if nbsd else (call.tokens, call.width)
        out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev)
    A, a_scale = (g["A"], g["a_scale"]) if input_layout == 0 else (A_in, None)
    op(A, a_scale, g["W"], g["w_sf"], g["bias"], g["gamma_q"] if call.norm else None,
       g["gamma_k"] if call.norm else None, g["cos"], g["sin"], out=out, w_col_scale=g["w_col_scale"],
       sumsq=sumsq, inv_rms=inv, stream=stream)
    if nbsd:
        out = out.permute(1, 0, 2).reshape(call.tokens, call.width)
    return op, out, sumsq, inv


def _diag(name, got, ref, bad):
    d = os.environ.get("QKV_DIAG_DIR")
    if not d:
        return ""
    os.makedirs(d, exist_ok=True)
    path = os.path.join(d, f"{name}.npz")
    rows = np.unique(np.nonzero(bad)[0])[:16]
    np.savez_compressed(path, got=got[rows], ref=ref[rows], rows=rows)
    return f" (diagnostics in {path})"


def check_outputs(call, inp, out, sumsq, inv, rows=None, name="case"):
    """Compare the GPU outputs with the oracle on `rows` (all rows when None)."""
    ref = O.qkv_cte_from_inputs(call, inp, rows=rows)
    idx = torch.arange(call.tokens) if rows is None else torch.as_tensor(rows)
    got = out.index_select(0, idx.to(out.device)).float().cpu().double().numpy()
    r = ref["O"]
    err = np.abs(got - r)
    bad = ~(err <= REL * np.abs(r) + ABS)      # NaN in got counts as bad
    if bad.any():
        br, bc = np.nonzero(bad)
        msg = (f"{name}: {int(bad.sum())}/{bad.size} outputs outside tolerance; first at row "
               f"{int(idx[br[0]])} col {int(bc[0])}: got {got[br[0], bc[0]]!r} ref {r[br[0], bc[0]]!r}; "
               f"bad rows {len(np.unique(br))}, bad cols {len(np.unique(bc))} "
               f"(cols mod 128 {sorted(set((bc % 128).tolist()))[:8]}...)")
        raise AssertionError(msg + _diag(name, got, r, bad))
    # segments the call has (Q unless it is a K|V call, K unless it is a separate call);
    # the columns of an absent segment must be exactly 0
    segs = ([0] if call.n_q_heads > 0 else []) + ([1] if call.n_kv_heads > 0 else [])
    absent = [c for c in (0, 1) if c not in segs]
    if sumsq is not None:
        s = sumsq.index_select(0, idx.to(sumsq.device)).cpu().double().numpy()
        for c in segs:
            rel = np.abs(s[:, c] - ref["sumsq"][:, c]) / np.maximum(np.abs(ref["sumsq"][:, c]), 1e-30)
            assert np.all(rel <= SS_REL), f"{name}: sumsq[{c}] max rel err {np.nanmax(rel):.3e}"
        for c in absent:
            assert np.all(s[:, c] == 0), f"{name}: sumsq column {c} should be 0 without that segment"
    if inv is not None and call.norm == 1:
        v = inv.index_select(0, idx.to(inv.device)).cpu().double().numpy()
        for c in segs:
            rel = np.abs(v[:, c] - ref["inv_rms"][:, c]) / np.abs(ref["inv_rms"][:, c])
            assert np.all(rel <= SS_REL), f"{name}: inv_rms[{c}] max rel err {np.nanmax(rel):.3e}"
        for c in absent:
            assert np.all(v[:, c] == 0), f"{name}: inv_rms column {c} should be 0 without that segment"
    return float(np.max(err)) if err.size else 0.0


def assert_same_to_rounding(call, a, b, name="runs"):
    """Two runs of the same inputs through the same kernels (BSD views [T, I]).

    V columns must be bit-identical: nothing in their arithmetic depends on order.
    Q/K depend on inv_rms, whose fp32 sum of squares is built from atomics in a
    run-dependent order, so it may differ in its last bits. The fp32 values before
    rounding then differ by a few 2^-24 of |lo|+|hi| of the rotated pair, and the
    rotation keeps the pair's norm, so that is at most 2 * the row's largest |O|.
    Bound: one bf16 ulp of the larger value (a flipped rounding) + 2^-18 of the
    row's largest magnitude (the pre-rounding drift, with margin), where the
    rotation cancels."""
    assert a.shape == b.shape == (call.tokens, call.width)
    assert bool(torch.isfinite(a).all()) and bool(torch.isfinite(b).all()), f"{name}: non-finite output"
    k_end = (call.n_q_heads + call.n_kv_heads) * call.d_head  # the Q/K columns (and V after them)
    assert torch.equal(a[:, k_end:], b[:, k_end:]), f"{name}: V columns differ"
    fa, fb = a[:, :k_end].float(), b[:, :k_end].float()
    mag = torch.maximum(fa.abs(), fb.abs())
    rowmax = mag.amax(dim=1, keepdim=True)
    tol = 2 ** -7 * mag + 2 ** -18 * rowmax
    bad = (fa - fb).abs() > tol
    nbad = int(bad.sum())
    assert nbad == 0, f"{name}: {nbad} Q/K outputs differ by more than rounding"


def sampled_rows(call, count=4096):
    return wl.sample_rows(call, count).numpy()
