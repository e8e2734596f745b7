"""GPU parity of the host-streaming entry point (qkv_cte_run_host): activations in and
O out through pinned host memory, in row chunks with the copies overlapped."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import qkv_cte_oracle as O
from rope_tcgen05_mxfp8_gb300 import (QKV_CTE_ERR_DEVICE_TIMEOUT, QKV_CTE_ERR_UNSUPPORTED, QKV_CTE_FLAG_TEST_STALL,
                                      QKV_CTE_INPUT_BF16, QKV_CTE_INPUT_PACKED, QKV_CTE_LAYOUT_BSD,
                                      QKV_CTE_LAYOUT_NBSD, QkvCte, QkvCteError)

from gpu_harness import assert_same_to_rounding, check_outputs, run_path, sampled_rows, to_device

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _host_run(call, inp, g, chunk_rows, nbsd=False, input_layout=0, A_host=None, flags=0):
    op = QkvCte(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, norm=call.norm,
                rope=call.rope, eps=call.eps, flags=flags, device=DEV,
                output_layout=QKV_CTE_LAYOUT_NBSD if nbsd else QKV_CTE_LAYOUT_BSD, input_layout=input_layout)
    if A_host is None:
        A_host, s_host = inp["A"].pin_memory(), inp["a_scale"].pin_memory()
    else:
        s_host = None
    heads = call.width // call.d_head
    shape = (heads, call.tokens, call.d_head) if nbsd else (call.tokens, call.width)
    O_host = torch.full(shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    sumsq = torch.full((call.tokens, 2), float("nan"), dtype=torch.float32, device=DEV)
    inv = torch.full((call.tokens, 2), float("nan"), dtype=torch.float32, device=DEV) if call.norm == 1 else None
    op.run_host(A_host, s_host, g["W"], g["w_sf"], g["bias"], g["gamma_q"] if call.norm else None,
                g["gamma_k"] if call.norm else None, g["cos"], g["sin"], O_host, w_col_scale=g["w_col_scale"],
                sumsq=sumsq, inv_rms=inv, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    out = O_host.permute(1, 0, 2).reshape(call.tokens, call.width) if nbsd else O_host
    return op, out, sumsq, inv


@pytest.mark.parametrize("T,chunk", [(300, 256), (1000, 0), (1000, 512), (1300, 256), (129, 0)])
@pytest.mark.parametrize("nbsd", [False, True])
def test_run_host_matches_oracle_and_device_run(T, chunk, nbsd):
    call = wl.custom_call(name=f"host_T{T}_c{chunk}", tokens=T, hidden=512, n_q_heads=3, n_kv_heads=2, d_head=128,
                          seed=T + chunk, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = _host_run(call, inp, g, chunk, nbsd=nbsd)
    op.host_status()
    check_outputs(call, inp, out, ss, inv, name=call.name)
    op_d, out_d, _, _ = run_path(call, g, nbsd=nbsd)
    op_d.status()
    assert_same_to_rounding(call, out, out_d.cpu(), name=f"{call.name}_vs_device")


@pytest.mark.parametrize("layout", ["bf16", "packed"])
def test_run_host_producer_inputs(layout):
    call = wl.custom_call(name=f"host_{layout}", tokens=1100, hidden=512, n_q_heads=3, n_kv_heads=2, d_head=128,
                          seed=97, has_w_col_scale=True)
    inp = dict(wl.make_inputs(call))
    if layout == "bf16":
        x = wl.make_activations(call)
        codes, s = O.row_quantise(wl.bf16_bits(x))
        inp["A"], inp["a_scale"] = torch.from_numpy(codes), torch.from_numpy(s)
        A_host, il = x.pin_memory(), QKV_CTE_INPUT_BF16
    else:
        A_host = torch.from_numpy(O.pack_rows(inp["A"].numpy(), inp["a_scale"].numpy())).pin_memory()
        il = QKV_CTE_INPUT_PACKED
    g = to_device(inp, DEV)
    op, out, ss, inv = _host_run(call, inp, g, 256, input_layout=il, A_host=A_host)
    op.host_status()
    check_outputs(call, inp, out, ss, inv, name=call.name)


def test_run_host_reports_a_stalled_chunk():
    call = wl.custom_call(name="host_stall", tokens=600, hidden=512, n_q_heads=2, n_kv_heads=1, d_head=128, seed=5)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = _host_run(call, inp, g, 256, flags=QKV_CTE_FLAG_TEST_STALL)
    with pytest.raises(QkvCteError) as ei:
        op.host_status()
    assert ei.value.code == QKV_CTE_ERR_DEVICE_TIMEOUT


def test_run_host_refuses_pageable_memory():
    call = wl.custom_call(name="host_pageable", tokens=300, hidden=512, n_q_heads=2, n_kv_heads=1, d_head=128, seed=6)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op = QkvCte(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, device=DEV)
    O_host = torch.empty(call.tokens, call.width, dtype=torch.bfloat16)   # not pinned
    with pytest.raises(QkvCteError) as ei:
        op.run_host(inp["A"], inp["a_scale"], g["W"], g["w_sf"], g["bias"], g["gamma_q"], g["gamma_k"], g["cos"],
                    g["sin"], O_host)
    assert ei.value.code == QKV_CTE_ERR_UNSUPPORTED


def test_run_host_wan480p_sampled():
    call = wl.workload("wan480p")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = _host_run(call, inp, g, 0)
    op.host_status()
    check_outputs(call, inp, out, ss, inv, rows=sampled_rows(call), name="host_wan480p")
