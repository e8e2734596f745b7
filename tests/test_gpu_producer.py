"""GPU parity of the producer step (bf16 -> ROW_MX rows, packed [T, H + 4] rows)
and of the path fed packed or bf16 inputs, against the oracle.

Codes and scales are integers / exact fp32 values decided in fp32 on both sides,
so the comparisons are bit-exact.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import qkv_cte_oracle as O
from rope_tcgen05_mxfp8_gb300 import (QKV_CTE_INPUT_BF16, QKV_CTE_INPUT_PACKED, qkv_cte_row_quantize,
                                      qkv_cte_unpack_rows)

from gpu_harness import assert_same_to_rounding, check_outputs, run_path, sampled_rows, to_device

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _bits(x):
    return wl.bf16_bits(x.cpu())


def _special_rows(H, seed):
    """Rows that exercise every branch of the quantiser: all zeros, negative zeros,
    bf16 subnormals, values near the bf16 maximum, a one-hot row, and rows whose
    scale is a power of two so that x / s falls exactly on e4m3 midpoints (ties)."""
    g = np.random.default_rng(seed)
    grid = O.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[1:] + grid[:-1]) / 2
    rows = [np.zeros(H), -np.zeros(H), g.normal(0, 1, H) * 1e-39, g.normal(0, 1, H) * 1e37,
            np.eye(1, H, H // 3)[0] * -7.25]
    for j in (-8, 0, 9):
        r = g.choice(mids, size=H) * g.choice([-1.0, 1.0], size=H)
        r[H // 2] = 448.0
        rows.append(r * 2.0 ** j)   # every element exact in bf16 (<= 5 significant bits)
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    assert np.all(O.decode_bf16(_bits(x))[5:] == np.stack(rows)[5:])
    return x


def _activations(T, H, seed, outliers=True):
    call = wl.custom_call(name="act", tokens=T, hidden=H, n_q_heads=1, n_kv_heads=1, d_head=128, seed=seed)
    if not outliers:
        return wl.make_activations(call)
    x = wl.make_activations(call).float()
    g = torch.Generator().manual_seed(seed)
    rows = torch.randperm(T, generator=g)[: max(1, T // 50)]
    x[rows] *= 300.0
    return x.to(torch.bfloat16)


def _check_quantised(x_cpu, A, a_scale, packed=None, rows=None):
    bits = _bits(x_cpu)
    idx = np.arange(x_cpu.shape[0]) if rows is None else np.asarray(rows)
    ref_codes, ref_s = O.row_quantise(bits[idx])
    if A is not None:
        got = A.index_select(0, torch.as_tensor(idx, device=A.device)).cpu().numpy()
        bad = got != ref_codes
        assert not bad.any(), (f"{int(bad.sum())} codes differ; first at row {idx[np.nonzero(bad)[0][0]]} "
                               f"col {np.nonzero(bad)[1][0]}: got {got[bad][0]:#x} ref {ref_codes[bad][0]:#x}")
        gs = a_scale.index_select(0, torch.as_tensor(idx, device=a_scale.device)).cpu().numpy()
        assert np.array_equal(gs.view(np.uint32), ref_s.view(np.uint32)), "scales differ"
    if packed is not None:
        got = packed.index_select(0, torch.as_tensor(idx, device=packed.device)).cpu().numpy()
        assert np.array_equal(got, O.pack_rows(ref_codes, ref_s)), "packed rows differ"


@pytest.mark.parametrize("T,H", [(1, 16), (5, 128), (37, 5120), (300, 6400), (1000, 1024)])
def test_row_quantize_bit_exact(T, H):
    x = _activations(T, H, seed=T + H)
    x_dev = x.to(DEV)
    A, s, _ = qkv_cte_row_quantize(x_dev)
    packed = torch.empty(T, H + 4, dtype=torch.uint8, device=DEV)
    qkv_cte_row_quantize(x_dev, packed=packed)
    A2 = torch.empty(T, H, dtype=torch.uint8, device=DEV)
    s2 = torch.empty(T, dtype=torch.float32, device=DEV)
    packed2 = torch.empty(T, H + 4, dtype=torch.uint8, device=DEV)
    qkv_cte_row_quantize(x_dev, A2, s2, packed2)
    torch.cuda.synchronize()
    _check_quantised(x, A, s, packed)
    assert torch.equal(A, A2) and torch.equal(s, s2) and torch.equal(packed, packed2)


@pytest.mark.parametrize("H", [128, 640])
def test_row_quantize_special_rows_and_ties(H):
    x = _special_rows(H, seed=H)
    x_dev = x.to(DEV)
    packed = torch.empty(x.shape[0], H + 4, dtype=torch.uint8, device=DEV)
    A, s, _ = qkv_cte_row_quantize(x_dev)
    qkv_cte_row_quantize(x_dev, packed=packed)
    torch.cuda.synchronize()
    _check_quantised(x, A, s, packed)
    # the tie rows really hold ties: the quotients sit exactly on midpoints
    assert float(s[5].cpu()) == 2.0 ** -8


def test_row_quantize_empty():
    x = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    A, s, _ = qkv_cte_row_quantize(x)
    torch.cuda.synchronize()
    assert A.numel() == 0 and s.numel() == 0


@pytest.mark.parametrize("T,H", [(1, 16), (2, 128), (3, 128), (4, 128), (9, 48), (1000, 5120)])
def test_unpack_rows_byte_exact(T, H):
    """Random bytes, every alignment phase of the 4 mod 16 packed pitch."""
    g = torch.Generator().manual_seed(T * 7 + H)
    packed = torch.randint(0, 256, (T, H + 4), generator=g, dtype=torch.uint8)
    A, s = qkv_cte_unpack_rows(packed.to(DEV))
    torch.cuda.synchronize()
    ref_c, ref_s = O.unpack_rows(packed.numpy())
    assert np.array_equal(A.cpu().numpy(), ref_c)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def _packed_input(inp):
    return torch.from_numpy(O.pack_rows(inp["A"].numpy(), inp["a_scale"].numpy()))


def _fp8_from_bf16(x):
    codes, s = O.row_quantise(_bits(x))
    return torch.from_numpy(codes), torch.from_numpy(s)


@pytest.mark.parametrize("T", [1, 300, 1000])
def test_path_with_packed_input(T):
    call = wl.custom_call(name=f"packed_T{T}", tokens=T, hidden=1024, n_q_heads=3, n_kv_heads=2, d_head=128,
                          seed=T + 3, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    packed = _packed_input(inp).to(DEV)
    op, out, ss, inv = run_path(call, g, input_layout=QKV_CTE_INPUT_PACKED, A_in=packed)
    op.status()
    check_outputs(call, inp, out, ss, inv, name=f"packed_T{T}")
    op_r, out_r, _, _ = run_path(call, g)
    op_r.status()
    assert_same_to_rounding(call, out, out_r, name=f"packed_vs_rows_T{T}")


@pytest.mark.parametrize("T,norm,rope", [(1, 1, 1), (333, 1, 1), (333, 0, 0), (1000, 1, 0)])
def test_path_with_bf16_input(T, norm, rope):
    call = wl.custom_call(name=f"bf16_T{T}", tokens=T, hidden=1024, n_q_heads=3, n_kv_heads=2, d_head=128,
                          norm=norm, rope=rope, seed=T + 5, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    x = wl.make_activations(call)
    # the oracle's own quantisation of the same activations is what the path must use
    inp = dict(inp)
    inp["A"], inp["a_scale"] = _fp8_from_bf16(x)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, input_layout=QKV_CTE_INPUT_BF16, A_in=x.to(DEV))
    op.status()
    check_outputs(call, inp, out, ss, inv, name=f"bf16_T{T}_n{norm}_r{rope}")


def test_path_with_bf16_input_separate_nbsd():
    call = wl.custom_call(name="bf16_sep", tokens=520, hidden=512, n_q_heads=6, n_kv_heads=0, d_head=128,
                          norm=1, rope=0, seed=91)
    inp = dict(wl.make_inputs(call))
    x = wl.make_activations(call)
    inp["A"], inp["a_scale"] = _fp8_from_bf16(x)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, input_layout=QKV_CTE_INPUT_BF16, A_in=x.to(DEV), nbsd=True)
    op.status()
    check_outputs(call, inp, out, ss, inv, name="bf16_sep_nbsd")


def test_wan480p_bf16_input_sampled():
    """The full Wan 480p shape fed bf16 activations: the standalone quantiser on
    sampled rows bit-exact, and the path's outputs on sampled rows."""
    call = wl.workload("wan480p")[0]
    inp = dict(wl.make_inputs(call))
    x = wl.make_activations(call)
    rows = sampled_rows(call)
    x_dev = x.to(DEV)
    A, s, _ = qkv_cte_row_quantize(x_dev)
    torch.cuda.synchronize()
    _check_quantised(x, A, s, rows=rows)
    # the path's own producer output equals the standalone one; feed the oracle the
    # oracle's quantisation of the sampled rows (only those rows are compared)
    codes = A.cpu()
    scale = s.cpu()
    rc, rs = O.row_quantise(_bits(x[torch.as_tensor(rows)]))
    codes[torch.as_tensor(rows)] = torch.from_numpy(rc)
    scale[torch.as_tensor(rows)] = torch.from_numpy(rs)
    inp["A"], inp["a_scale"] = codes, scale
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, input_layout=QKV_CTE_INPUT_BF16, A_in=x_dev)
    op.status()
    check_outputs(call, inp, out, ss, inv, rows=rows, name="bf16_wan480p")
    op_r, out_r, _, _ = run_path(call, g)
    op_r.status()
    assert_same_to_rounding(call, out, out_r, name="bf16_vs_rows_wan480p")
