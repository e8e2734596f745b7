"""GPU parity of the per-head qk-norm (RMS_NORM / LAYER_NORM finished in the GEMM
epilogue) and of the interleaved -> rotate-half checkpoint permutation, against the
oracle."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import qkv_cte_oracle as O
from rope_tcgen05_mxfp8_gb300 import (QKV_CTE_FLAG_GEMM_CTA_PAIR, QKV_CTE_FLAG_GEMM_SINGLE_CTA,
                                      QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE, qkv_cte_interleaved_to_rotate_half)

from gpu_harness import check_outputs, run_path, sampled_rows, to_device

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
RMS, LAYER = O.NORM_HEAD_RMS, O.NORM_HEAD_LAYER


FORMS = {"stats": 0, "epilogue": QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE}


def _case(call, flags=0, tile_n=0, rows=None, nbsd=False, name=None, form="stats", inp=None):
    inp = inp if inp is not None else wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, tile_n=tile_n, flags=flags | FORMS[form], nbsd=nbsd)
    op.status()
    if form == "epilogue":
        assert op.info.tile_n % call.d_head == 0
    return check_outputs(call, inp, out, ss, inv, rows=rows, name=name or f"{call.name}_{form}")


@pytest.mark.parametrize("form", ["stats", "epilogue"])
@pytest.mark.parametrize("norm", [RMS, LAYER])
@pytest.mark.parametrize("gemm", ["auto", "single", "pair"])
def test_head_norm_tiny(norm, gemm, form):
    flags = {"auto": 0, "single": QKV_CTE_FLAG_GEMM_SINGLE_CTA, "pair": QKV_CTE_FLAG_GEMM_CTA_PAIR}[gemm]
    call = wl.custom_call(name=f"head{norm}_{gemm}", tokens=256, hidden=512, n_q_heads=4, n_kv_heads=4, d_head=128,
                          norm=norm, rope=1, seed=norm * 10 + len(gemm), has_w_col_scale=True)
    _case(call, flags=flags, form=form)


@pytest.mark.parametrize("form", ["stats", "epilogue"])
@pytest.mark.parametrize("T", [1, 129, 300])
@pytest.mark.parametrize("norm,rope", [(RMS, 1), (LAYER, 1), (RMS, 0), (LAYER, 0)])
def test_head_norm_ragged(T, norm, rope, form):
    call = wl.custom_call(name=f"headT{T}", tokens=T, hidden=256, n_q_heads=3, n_kv_heads=1, d_head=128,
                          norm=norm, rope=rope, seed=T + norm, has_w_col_scale=True)
    _case(call, name=f"head_T{T}_n{norm}_r{rope}_{form}", form=form)


@pytest.mark.parametrize("form", ["stats", "epilogue"])
@pytest.mark.parametrize("norm,rope", [(RMS, 0), (LAYER, 1)])
@pytest.mark.parametrize("T", [129, 300])
def test_head_norm_kv_call(T, norm, rope, form):
    """A K|V call (no Q heads) with a per-head norm: K normalised per head with its
    [d_head] gamma, V as projected."""
    call = wl.custom_call(name=f"head_kv{T}", tokens=T, hidden=512, n_q_heads=0, n_kv_heads=3, d_head=128,
                          norm=norm, rope=rope, seed=61 + T + norm, has_w_col_scale=True)
    _case(call, name=f"head_kv_T{T}_n{norm}_r{rope}_{form}", form=form)


@pytest.mark.parametrize("norm,tile_n,form", [(RMS, 0, "epilogue"), (LAYER, 0, "epilogue"), (RMS, 128, "epilogue"),
                                             (LAYER, 256, "epilogue"), (RMS, 0, "stats"), (LAYER, 0, "stats"),
                                             (LAYER, 192, "stats"), (RMS, 128, "stats")])
def test_head_norm_d64_tiles(norm, tile_n, form):
    # d = 64: in the epilogue the automatic tile is 192 (three heads); 128 and 256 hold two
    # and four. From statistics any tile works (240 puts heads across tile edges).
    call = wl.custom_call(name="head_d64", tokens=200, hidden=384, n_q_heads=5, n_kv_heads=2, d_head=64,
                          norm=norm, rope=1, seed=41 + norm, has_w_col_scale=True)
    _case(call, tile_n=tile_n, name=f"head_d64_n{norm}_t{tile_n}_{form}", form=form)


@pytest.mark.parametrize("tile_n", [192, 240, 256])
def test_head_layernorm_parts_and_offset(tile_n):
    """LayerNorm statistics combined across tile parts: 128-wide heads over 192/240-wide
    tiles straddle tile edges, d = 256 over 240 spans up to three parts. A common offset
    of 1000 on every column (the bias) with deviations of ~0.3 loses everything in a
    one-pass variance (sum of squares ~1e6 in fp32) and in an uncentred fp16 hand-off
    (resolution ~0.5 at 1000); the centred parts and their pairwise combination must
    not."""
    for d, nq in ((128, 5), (256, 3)):
        call = wl.custom_call(name=f"ln_parts_d{d}_t{tile_n}", tokens=300, hidden=256, n_q_heads=nq,
                              n_kv_heads=1, d_head=d, norm=LAYER, rope=1, seed=tile_n + d, has_w_col_scale=True)
        inp = dict(wl.make_inputs(call))
        inp["bias"] = torch.full_like(inp["bias"], 1000.0)   # exact in bf16
        _case(call, tile_n=tile_n, inp=inp, name=call.name)


@pytest.mark.parametrize("form", ["stats", "epilogue"])
@pytest.mark.parametrize("norm", [RMS, LAYER])
def test_head_norm_separate_and_nbsd(norm, form):
    call = wl.custom_call(name="head_sep", tokens=333, hidden=512, n_q_heads=6, n_kv_heads=0, d_head=128,
                          norm=norm, rope=0, seed=51 + norm)
    _case(call, nbsd=True, name=f"head_sep_nbsd_n{norm}_{form}", form=form)


@pytest.mark.parametrize("form", ["stats", "epilogue"])
@pytest.mark.parametrize("norm", [RMS, LAYER])
def test_head_norm_wan480p_sampled(norm, form):
    base = wl.workload("wan480p")[0]
    call = wl.custom_call(name=f"wan480p_head{norm}", tokens=base.tokens, hidden=base.hidden,
                          n_q_heads=base.n_q_heads, n_kv_heads=base.n_kv_heads, d_head=base.d_head, norm=norm,
                          rope=1, rope_grid=base.rope_grid, outlier_frac=base.outlier_frac, seed=base.seed)
    _case(call, rows=sampled_rows(call), form=form)


# --- interleaved -> rotate-half ----------------------------------------------------

@pytest.mark.parametrize("rows,row_bytes,nq,nkv,d", [(640, 256, 3, 1, 128), (640, 8, 3, 1, 128), (640, 2, 3, 1, 128),
                                                    (640, 1, 3, 1, 128), (1000 * 64, 4, 1000, 0, 64),
                                                    (448, 12, 5, 2, 64)])
def test_permutation_byte_exact(rows, row_bytes, nq, nkv, d):
    g = torch.Generator().manual_seed(rows + row_bytes)
    src = torch.randint(0, 256, (rows, row_bytes), generator=g, dtype=torch.uint8)
    dst = qkv_cte_interleaved_to_rotate_half(src.to(DEV), nq, nkv, d)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), O.permute_qk_rows(src.numpy(), nq, nkv, d))


@pytest.mark.parametrize("norm", [O.NORM_ACROSS_HEADS, RMS, LAYER])
def test_interleaved_checkpoint_through_the_path(norm):
    """Treat the generated tensors as an interleaved-RoPE checkpoint, convert them on
    the GPU, run the rotate-half path, and compare with the oracle's interleaved model
    on the original tensors (output Q/K columns in rotate-half order)."""
    call = wl.custom_call(name=f"interleaved_n{norm}", tokens=300, hidden=512, n_q_heads=3, n_kv_heads=2, d_head=128,
                          norm=norm, rope=1, seed=61 + norm, has_w_col_scale=True)
    nq, nkv, d = call.n_q_heads, call.n_kv_heads, call.d_head
    inp = wl.make_inputs(call)
    # interleaved tables: the generator's rotate-half tables put back in interleaved order
    inv_perm = np.argsort(O.interleaved_to_rotate_half(d))
    cos_il = inp["cos"][:, torch.as_tensor(inv_perm)].contiguous()
    sin_il = inp["sin"][:, torch.as_tensor(inv_perm)].contiguous()
    n = {k: wl.as_numpy_bits(v) for k, v in inp.items()}
    ref = O.qkv_cte(n["A"], n["a_scale"], n["W"], n["w_sf"], n["bias"], n["gamma_q"], n["gamma_k"], cos_il.numpy(),
                    sin_il.numpy(), n_q_heads=nq, n_kv_heads=nkv, d_head=d, norm=norm, rope=1, eps=call.eps,
                    w_col_scale=n["w_col_scale"], rope_layout="interleaved")
    expect = O.permute_qk_rows(ref["O"].T, nq, nkv, d).T

    g = to_device(inp, DEV)
    conv = dict(g)
    for k in ("W", "w_sf", "bias", "w_col_scale"):
        conv[k] = qkv_cte_interleaved_to_rotate_half(g[k], nq, nkv, d)
    per_head = norm in (RMS, LAYER)
    conv["gamma_q"] = qkv_cte_interleaved_to_rotate_half(g["gamma_q"], 1 if per_head else nq, 0, d)
    conv["gamma_k"] = qkv_cte_interleaved_to_rotate_half(g["gamma_k"], 1 if per_head else nkv, 0, d)
    T = call.tokens
    conv["cos"] = qkv_cte_interleaved_to_rotate_half(cos_il.to(DEV).reshape(T * d), T, 0, d).reshape(T, d)
    conv["sin"] = qkv_cte_interleaved_to_rotate_half(sin_il.to(DEV).reshape(T * d), T, 0, d).reshape(T, d)
    # the converted tables are the generator's rotate-half tables again
    assert torch.equal(conv["cos"].cpu(), inp["cos"]) and torch.equal(conv["sin"].cpu(), inp["sin"])
    op, out, ss, _ = run_path(call, conv, want_inv=False)
    op.status()
    got = out.float().cpu().double().numpy()
    err = np.abs(got - expect)
    assert np.all(err <= 1e-2 * np.abs(expect) + 1e-2), f"max err {err.max()}"
