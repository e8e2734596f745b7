"""The allocation-free entry point, qkv_cte_run_noalloc.

Some callers cannot allocate device memory at the moment they run the projection: a
server that allocates everything at start-up and forbids cudaMalloc afterwards, a
plug-in whose host framework owns all device memory, a latency-critical path where an
allocation could synchronise the device. qkv_cte_run_noalloc serves them: it runs the
same kernels with their scratch in a fixed array inside the library instead of a
caller-provided workspace.

These tests call it through the C ABI twice in a row and check each result against
qkv_cte_run (the entry point with a workspace) and the float64 oracle; check that its
first call after a warm-up run leaves the device's free memory unchanged; that a
bounded-wait timeout in it is reported by qkv_cte_noalloc_status; and that a problem
too large for the fixed array is refused before anything is launched. The file is
named so that pytest collects it after every other test file.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from rope_tcgen05_mxfp8_gb300 import qkv_cte as q

from gpu_harness import ABS, REL, SS_REL, check_outputs, run_path, to_device


def _cases():
    return {
        "tiny": wl.workload("tiny")[0],
        "cross_k": wl.workload("cross")[1],
        "edge": wl.custom_call(name="edge_noalloc", tokens=300, hidden=1024, n_q_heads=3, n_kv_heads=2,
                               d_head=128, seed=99, has_w_col_scale=True),
    }


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "cross_k", "edge"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name):
    call = _cases()[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(call)
    g = to_device(inp, dev)
    op, ref_out, ref_ss, ref_inv = run_path(call, g)  # qkv_cte_run with its own workspace
    op.status()
    ref = ref_out.float()
    desc = q.make_desc(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, norm=call.norm,
                       rope=call.rope, eps=call.eps)
    plan, ws_bytes = q.qkv_cte_plan(desc)
    assert ws_bytes <= q.QKV_CTE_NOALLOC_SCRATCH_BYTES
    try:
        for call_no in range(2):
            out = torch.full((call.tokens, call.width), float("nan"), dtype=torch.bfloat16, device=dev)
            ss = torch.full((call.tokens, 2), float("nan"), dtype=torch.float32, device=dev)
            inv = torch.full((call.tokens, 2), float("nan"), dtype=torch.float32, device=dev)
            q.qkv_cte_run_noalloc(plan, g["A"], g["a_scale"], g["W"], g["w_sf"], g["w_col_scale"], g["bias"],
                                  g["gamma_q"] if call.norm else None, g["gamma_k"] if call.norm else None,
                                  g["cos"], g["sin"], out, ss, inv)
            torch.cuda.synchronize(dev)
            got = out.float()
            bad = ~((got - ref).abs() <= REL * ref.abs() + ABS)
            assert not bool(bad.any()), f"{name} call {call_no}: {int(bad.sum())} outputs differ from qkv_cte_run"
            segs = [0] + ([1] if call.n_kv_heads > 0 else [])
            for c in segs:
                rel = ((ss[:, c] - ref_ss[:, c]).abs() / ref_ss[:, c].abs().clamp_min(1e-30)).max()
                assert float(rel) <= SS_REL, f"{name} call {call_no}: sumsq[{c}] rel err {float(rel):.3e}"
                if call.norm:
                    rel = ((inv[:, c] - ref_inv[:, c]).abs() / ref_inv[:, c].abs()).max()
                    assert float(rel) <= SS_REL, f"{name} call {call_no}: inv_rms[{c}] rel err {float(rel):.3e}"
            check_outputs(call, inp, out, ss, inv, name=f"noalloc_{name}_{call_no}")
    finally:
        q.qkv_cte_destroy(plan)


@pytest.mark.gpu
def test_noalloc_first_call_after_warm_up_allocates_nothing():
    """A caller that forbids allocation warms the library up once (any run on the
    device maps its device code, the scratch array included); the first allocation-free
    call after that must not change the device's free memory."""
    call = _cases()["edge"]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(call)
    g = to_device(inp, dev)
    op, _, _, _ = run_path(call, g)  # warm-up through qkv_cte_run (its own workspace)
    op.status()
    desc = q.make_desc(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, norm=call.norm,
                       rope=call.rope, eps=call.eps)
    plan, _ = q.qkv_cte_plan(desc)
    out = torch.empty(call.tokens, call.width, dtype=torch.bfloat16, device=dev)
    ss = torch.empty(call.tokens, 2, dtype=torch.float32, device=dev)
    inv = torch.empty(call.tokens, 2, dtype=torch.float32, device=dev)
    try:
        torch.cuda.synchronize(dev)
        free_before, _ = torch.cuda.mem_get_info(dev)
        q.qkv_cte_run_noalloc(plan, g["A"], g["a_scale"], g["W"], g["w_sf"], g["w_col_scale"], g["bias"],
                              g["gamma_q"], g["gamma_k"], g["cos"], g["sin"], out, ss, inv)
        q.qkv_cte_noalloc_status()
        torch.cuda.synchronize(dev)
        free_after, _ = torch.cuda.mem_get_info(dev)
        assert free_after == free_before, f"free device memory changed by {free_before - free_after} bytes"
        check_outputs(call, inp, out, ss, inv, name="noalloc_after_warm_up")
    finally:
        q.qkv_cte_destroy(plan)


@pytest.mark.gpu
def test_noalloc_status_reports_a_stalled_call_and_the_next_call_is_correct():
    """The test hook that stalls the GEMM's load warp makes every bounded wait of an
    allocation-free call run out; qkv_cte_noalloc_status reports it (and clears the
    word), and the next allocation-free call on the same context is correct."""
    call = _cases()["edge"]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(call)
    g = to_device(inp, dev)
    out = torch.empty(call.tokens, call.width, dtype=torch.bfloat16, device=dev)
    ss = torch.empty(call.tokens, 2, dtype=torch.float32, device=dev)
    inv = torch.empty(call.tokens, 2, dtype=torch.float32, device=dev)
    for flags, expect_timeout in ((q.QKV_CTE_FLAG_TEST_STALL, True), (0, False)):
        plan, _ = q.qkv_cte_plan(q.make_desc(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head,
                                             norm=call.norm, rope=call.rope, eps=call.eps, flags=flags))
        try:
            q.qkv_cte_run_noalloc(plan, g["A"], g["a_scale"], g["W"], g["w_sf"], g["w_col_scale"], g["bias"],
                                  g["gamma_q"], g["gamma_k"], g["cos"], g["sin"], out, ss, inv)
            if expect_timeout:
                with pytest.raises(q.QkvCteError) as ei:
                    q.qkv_cte_noalloc_status()
                assert ei.value.code == q.QKV_CTE_ERR_DEVICE_TIMEOUT
                q.qkv_cte_noalloc_status()  # cleared
            else:
                q.qkv_cte_noalloc_status()
                check_outputs(call, inp, out, ss, inv, name="noalloc_after_stall")
        finally:
            q.qkv_cte_destroy(plan)


def test_noalloc_refuses_a_problem_larger_than_its_scratch():
    """4096 Wan tokens need far more scratch than the fixed array: refused on the host
    with a clear message, before any pointer is read or kernel launched."""
    plan, ws_bytes = q.qkv_cte_plan(q.make_desc(4096, 5120, 40, 40, 128))
    try:
        assert ws_bytes > q.QKV_CTE_NOALLOC_SCRATCH_BYTES
        rc = q.load().qkv_cte_run_noalloc(plan, *([None] * 13), None)
        assert rc == q.QKV_CTE_ERR_UNSUPPORTED
        msg = q.qkv_cte_last_error()
        assert "scratch" in msg and str(q.QKV_CTE_NOALLOC_SCRATCH_BYTES) in msg
    finally:
        q.qkv_cte_destroy(plan)


def test_noalloc_scratch_holds_the_documented_problems():
    """The header promises that 640 tokens of the fused Wan layout and the 512-token
    cross-attention K, V and K|V calls fit the fixed array (planning only, no GPU)."""
    cases = [(640, 40, 40, 1), (512, 40, 0, 0), (512, 0, 40, 0)]
    for tokens, nq, nkv, rope in cases:
        plan, ws_bytes = q.qkv_cte_plan(q.make_desc(tokens, 5120, nq, nkv, 128, rope=rope))
        q.qkv_cte_destroy(plan)
        assert ws_bytes <= q.QKV_CTE_NOALLOC_SCRATCH_BYTES, (tokens, nq, nkv, ws_bytes)
