"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small shapes are compared element by element on every row (several 128-row tiles
and N tiles, with ragged tails); the full Wan shapes are compared on 4096 seeded
sampled rows (rows are independent, so each sampled row is exact), in the same
launch configuration the benchmark times.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as wl
from rope_tcgen05_mxfp8_gb300 import QKV_CTE_ERR_DEVICE_TIMEOUT, QKV_CTE_FLAG_TEST_STALL, QkvCteError

from gpu_harness import assert_same_to_rounding, check_outputs, run_path, sampled_rows, to_device

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _case(call, tile_n=0, rows=None, name=None):
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, tile_n=tile_n)
    op.status()
    return check_outputs(call, inp, out, ss, inv, rows=rows, name=name or call.name)


@pytest.mark.parametrize("tile_n", [0, 128, 192, 240, 256])
def test_tiny_full(tile_n):
    _case(wl.workload("tiny")[0], tile_n=tile_n, name=f"tiny_n{tile_n}")


@pytest.mark.parametrize("T", [1, 127, 129, 300])
@pytest.mark.parametrize("norm,rope", [(1, 1), (1, 0), (0, 1), (0, 0)])
def test_ragged_rows_and_unaligned_segments(T, norm, rope):
    # n_q = 3, n_kv = 1, d = 128: I = 640, Q|K boundary at 384 (inside a 256 tile),
    # K|V boundary at 512, ragged last N tile; per-column weight scales on.
    call = wl.custom_call(name=f"edge_T{T}", tokens=T, hidden=256, n_q_heads=3, n_kv_heads=1, d_head=128,
                          norm=norm, rope=rope, seed=T, has_w_col_scale=True)
    _case(call, name=f"edge_T{T}_n{norm}_r{rope}")


@pytest.mark.parametrize("tile_n", [128, 240, 256])
def test_d_head_64_many_heads(tile_n):
    call = wl.custom_call(name="d64", tokens=200, hidden=384, n_q_heads=5, n_kv_heads=2, d_head=64,
                          seed=21, has_w_col_scale=True)
    _case(call, tile_n=tile_n, name=f"d64_n{tile_n}")


@pytest.mark.parametrize("norm,rope", [(1, 0), (0, 0), (1, 1)])
def test_separate_mode_small(norm, rope):
    call = wl.custom_call(name="sep", tokens=333, hidden=512, n_q_heads=6, n_kv_heads=0, d_head=128,
                          norm=norm, rope=rope, seed=31)
    _case(call, name=f"sep_n{norm}_r{rope}")


def test_large_hidden_small_tokens():
    call = wl.custom_call(name="deepk", tokens=64, hidden=5120, n_q_heads=2, n_kv_heads=2, d_head=128, seed=41)
    _case(call)


def test_short_full():
    _case(wl.workload("short")[0])


def test_wan480p_sampled():
    call = wl.workload("wan480p")[0]
    _case(call, rows=sampled_rows(call))


def test_wan720p_sampled():
    call = wl.workload("wan720p")[0]
    _case(call, rows=sampled_rows(call))


def test_cross_attention_calls():
    q, k, v = wl.workload("cross")
    _case(q, rows=sampled_rows(q))
    _case(k)
    _case(v)


@pytest.mark.parametrize("nbsd", [False, True])
def test_cross_kv_call(nbsd):
    """The cross-attention K and V projections of the 512 context tokens as one call (no
    Q heads): every element against the oracle, BSD and NBSd."""
    call = wl.workload("cross_kv")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, nbsd=nbsd)
    op.status()
    check_outputs(call, inp, out, ss, inv, name=f"cross_kv_{'nbsd' if nbsd else 'bsd'}")


@pytest.mark.parametrize("T,rope", [(300, 0), (129, 1), (1, 0)])
def test_kv_call_equals_separate_k_and_v_calls(T, rope):
    """A K|V call against the oracle, and against the separate K call (normalised as its
    only segment with gamma_k) and the separate plain V call on the same weights: V bit
    for bit, K to rounding (its sums of squares are accumulated in a run-dependent order)."""
    call = wl.custom_call(name=f"kv_{T}", tokens=T, hidden=1024, n_q_heads=0, n_kv_heads=3, d_head=128, norm=1,
                          rope=rope, seed=71 + T, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g)
    op.status()
    check_outputs(call, inp, out, ss, inv, name=call.name)
    k = call.n_kv_heads * call.d_head
    sep = wl.custom_call(name="sep", tokens=T, hidden=1024, n_q_heads=3, n_kv_heads=0, d_head=128, norm=1,
                         rope=rope, seed=1)
    gk = dict(g, W=g["W"][:k], w_sf=g["w_sf"][:k], bias=g["bias"][:k], w_col_scale=g["w_col_scale"][:k],
              gamma_q=g["gamma_k"], gamma_k=None)
    op_k, out_k, ss_k, _ = run_path(sep, gk)
    op_k.status()
    sep_v = dataclasses.replace(sep, norm=0, rope=0)
    gv = dict(g, W=g["W"][k:], w_sf=g["w_sf"][k:], bias=g["bias"][k:], w_col_scale=g["w_col_scale"][k:],
              gamma_q=None, gamma_k=None, cos=None, sin=None)
    op_v, out_v, _, _ = run_path(sep_v, gv)
    op_v.status()
    assert torch.equal(out[:, k:], out_v), "V columns differ from the separate V call"
    a, b = out[:, :k].float(), out_k.float()
    mag = torch.maximum(a.abs(), b.abs())
    tol = 2 ** -7 * mag + 2 ** -18 * mag.amax(dim=1, keepdim=True)
    assert int(((a - b).abs() > tol).sum()) == 0, "K columns differ from the separate K call by more than rounding"
    torch.testing.assert_close(ss[:, 1], ss_k[:, 0], rtol=1e-5, atol=0)


def test_outputs_repeatable_on_side_stream():
    """Two runs on a non-default stream: same results to rounding, both correct."""
    call = wl.workload("tiny")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        op1, out1, ss1, _ = run_path(call, g, stream=s)
        op2, out2, ss2, _ = run_path(call, g, stream=s)
    s.synchronize()
    # The per-row sums of squares are fp32 atomics whose order varies between runs:
    # repeat runs agree to rounding, and each matches the oracle.
    assert_same_to_rounding(call, out1, out2, name="side_stream")
    torch.testing.assert_close(ss1, ss2, rtol=1e-6, atol=0)
    check_outputs(call, inp, out1, ss1, None, name="side_stream_1")
    check_outputs(call, inp, out2, ss2, None, name="side_stream_2")


def test_norm_off_still_reports_sumsq():
    call = wl.custom_call(name="ss_only", tokens=150, hidden=256, n_q_heads=2, n_kv_heads=1, d_head=128,
                          norm=0, rope=0, seed=51)
    _case(call)


def test_zero_tokens():
    call = wl.custom_call(name="empty", tokens=0, hidden=256, n_q_heads=2, n_kv_heads=1, d_head=128, seed=1)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g)
    op.status()
    assert out.numel() == 0


def test_bounded_wait_reports_timeout_and_context_survives():
    """The test hook stops the GEMM's load warp; every downstream wait must run out
    (about two seconds each), the kernel must return, the status call must report
    it, and the next ordinary call on the same context must be correct."""
    call = wl.workload("tiny")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_TEST_STALL)
    with pytest.raises(QkvCteError) as ei:
        op.status()
    assert ei.value.code == QKV_CTE_ERR_DEVICE_TIMEOUT
    assert "mma-operands-ready" in str(ei.value)
    op.status()  # the status word was cleared
    op2, out2, ss2, inv2 = run_path(call, g)
    op2.status()
    check_outputs(call, inp, out2, ss2, inv2, name="after_timeout")


@pytest.mark.parametrize("name", ["tiny", "edge"])
def test_serial_and_overlapped_passes_agree(name):
    """The norm/RoPE pass launched after the GEMM (serial flag) and overlapped with it
    (the default, gated on per-panel ready counters) give the same, correct result."""
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_SERIAL_PASSES

    if name == "tiny":
        call = wl.workload("tiny")[0]
    else:
        call = wl.custom_call(name="edge", tokens=1000, hidden=1024, n_q_heads=3, n_kv_heads=2, d_head=128,
                              seed=77, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op_a, out_a, ss_a, inv_a = run_path(call, g)
    op_b, out_b, ss_b, inv_b = run_path(call, g, flags=QKV_CTE_FLAG_SERIAL_PASSES)
    op_a.status()
    op_b.status()
    check_outputs(call, inp, out_a, ss_a, inv_a, name=f"{name}_overlapped")
    check_outputs(call, inp, out_b, ss_b, inv_b, name=f"{name}_serial")
    diff = (out_a.float() - out_b.float()).abs()
    assert float(diff.max()) <= 2 ** -6 * float(out_a.float().abs().max())


@pytest.mark.parametrize("d_head,nq,nkv", [(64, 5, 2), (96, 3, 2), (256, 2, 1)])
def test_serial_pass_other_head_sizes(d_head, nq, nkv):
    """The stand-alone norm/RoPE pass (serial flag: a full grid, two heads' loads in
    flight per lane) with 16, 8 (and 8 idle lanes) and 4 rows per warp task."""
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_SERIAL_PASSES

    call = wl.custom_call(name=f"serial_d{d_head}", tokens=333, hidden=512, n_q_heads=nq, n_kv_heads=nkv,
                          d_head=d_head, seed=140 + d_head, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_SERIAL_PASSES)
    op.status()
    check_outputs(call, inp, out, ss, inv, name=call.name)


def test_pass_times_reported():
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_PROFILE

    call = wl.workload("short")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_PROFILE)
    prep, gemm, norm, run = op.pass_times()
    op.status()
    assert prep > 0 and gemm > 0 and norm > 0 and run > 0
    assert run >= gemm
    flops = call.flops / (gemm * 1e-3) / 1e12
    assert 10 < flops < 6000, f"implausible GEMM rate {flops} TFLOP/s"


# --- the CTA-pair GEMM (256-row tiles, M = 256 MMAs on two SMs) ------------------

def _pair_case(call, tile_n=0, rows=None, name=None):
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_GEMM_CTA_PAIR

    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, tile_n=tile_n, flags=QKV_CTE_FLAG_GEMM_CTA_PAIR)
    assert op.info.cta_pair == 1
    op.status()
    return check_outputs(call, inp, out, ss, inv, rows=rows, name=name or f"pair_{call.name}")


@pytest.mark.parametrize("tile_n", [240, 128, 256])
def test_cta_pair_tiny_full(tile_n):
    _pair_case(wl.workload("tiny")[0], tile_n=tile_n, name=f"pair_tiny_n{tile_n}")


@pytest.mark.parametrize("T", [1, 129, 257, 300, 640])
def test_cta_pair_ragged_rows(T):
    # T mod 256 in (0, 128] leaves the second CTA's half of the last tile empty.
    call = wl.custom_call(name=f"pair_T{T}", tokens=T, hidden=256, n_q_heads=3, n_kv_heads=1, d_head=128,
                          seed=T + 7, has_w_col_scale=True)
    _pair_case(call)


def test_cta_pair_d64_and_separate():
    _pair_case(wl.custom_call(name="pair_d64", tokens=200, hidden=384, n_q_heads=5, n_kv_heads=2, d_head=64,
                              seed=23, has_w_col_scale=True))
    _pair_case(wl.custom_call(name="pair_sep", tokens=333, hidden=512, n_q_heads=6, n_kv_heads=0, d_head=128,
                              norm=1, rope=0, seed=33))


def test_cta_pair_short_full():
    _pair_case(wl.workload("short")[0])


def test_cta_pair_wan480p_sampled():
    call = wl.workload("wan480p")[0]
    _pair_case(call, rows=sampled_rows(call))


def test_cta_pair_bounded_wait_reports_timeout():
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_GEMM_CTA_PAIR

    call = wl.workload("tiny")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_TEST_STALL | QKV_CTE_FLAG_GEMM_CTA_PAIR)
    with pytest.raises(QkvCteError) as ei:
        op.status()
    assert ei.value.code == QKV_CTE_ERR_DEVICE_TIMEOUT
    _pair_case(call, name="pair_after_timeout")


# --- the single-CTA GEMM (128-row tiles), forced ---------------------------------

def _single_case(call, tile_n=0, rows=None, name=None):
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_GEMM_SINGLE_CTA

    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, tile_n=tile_n, flags=QKV_CTE_FLAG_GEMM_SINGLE_CTA)
    assert op.info.cta_pair == 0
    op.status()
    return check_outputs(call, inp, out, ss, inv, rows=rows, name=name or f"single_{call.name}")


@pytest.mark.parametrize("tile_n", [240, 128, 192, 256])
def test_single_cta_tiny_full(tile_n):
    _single_case(wl.workload("tiny")[0], tile_n=tile_n, name=f"single_tiny_n{tile_n}")


@pytest.mark.parametrize("T", [129, 300])
def test_single_cta_ragged_rows(T):
    call = wl.custom_call(name=f"single_T{T}", tokens=T, hidden=256, n_q_heads=3, n_kv_heads=1, d_head=128,
                          seed=T + 11, has_w_col_scale=True)
    _single_case(call)


def test_single_cta_wan480p_sampled():
    call = wl.workload("wan480p")[0]
    _single_case(call, rows=sampled_rows(call))


# --- NBSd output layout [heads, T, d_head] ----------------------------------------

def _nbsd_case(call, flags=0, tile_n=0, rows=None, name=None):
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, tile_n=tile_n, flags=flags, nbsd=True)
    op.status()
    # run_path hands back the NBSd buffer viewed as BSD; every element was written
    # (the buffer starts as NaN, which the tolerance check rejects)
    return check_outputs(call, inp, out, ss, inv, rows=rows, name=name or f"nbsd_{call.name}")


@pytest.mark.parametrize("form", ["auto", "single", "pair"])
def test_nbsd_tiny_full(form):
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_GEMM_CTA_PAIR, QKV_CTE_FLAG_GEMM_SINGLE_CTA

    flags = {"auto": 0, "single": QKV_CTE_FLAG_GEMM_SINGLE_CTA, "pair": QKV_CTE_FLAG_GEMM_CTA_PAIR}[form]
    _nbsd_case(wl.workload("tiny")[0], flags=flags, name=f"nbsd_tiny_{form}")


@pytest.mark.parametrize("T", [1, 129, 300])
def test_nbsd_ragged_rows_d64(T):
    call = wl.custom_call(name=f"nbsd_T{T}", tokens=T, hidden=384, n_q_heads=5, n_kv_heads=2, d_head=64,
                          seed=T + 101, has_w_col_scale=True)
    _nbsd_case(call)


def test_nbsd_serial_passes_and_separate_mode():
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_SERIAL_PASSES

    call = wl.custom_call(name="nbsd_edge", tokens=1000, hidden=1024, n_q_heads=3, n_kv_heads=2, d_head=128,
                          seed=78, has_w_col_scale=True)
    _nbsd_case(call, flags=QKV_CTE_FLAG_SERIAL_PASSES, name="nbsd_edge_serial")
    _nbsd_case(call, name="nbsd_edge_overlapped")
    sep = wl.custom_call(name="nbsd_sep", tokens=333, hidden=512, n_q_heads=6, n_kv_heads=0, d_head=128,
                         norm=1, rope=1, seed=34)
    _nbsd_case(sep)


def test_nbsd_cross_attention_calls():
    q, k, v = wl.workload("cross")
    _nbsd_case(q, rows=sampled_rows(q))
    _nbsd_case(k)
    _nbsd_case(v)


def test_nbsd_wan480p_sampled_matches_bsd():
    """At the full size: NBSd on sampled rows against the oracle, and the whole NBSd
    result against the BSD run permuted (same kernels, same arithmetic, different
    addresses: V bit-identical, Q/K equal to rounding, the sums of squares being
    fp32 atomics)."""
    call = wl.workload("wan480p")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op_n, out_n, ss_n, inv_n = run_path(call, g, nbsd=True)
    op_n.status()
    check_outputs(call, inp, out_n, ss_n, inv_n, rows=sampled_rows(call), name="nbsd_wan480p")
    op_b, out_b, _, _ = run_path(call, g)
    op_b.status()
    assert_same_to_rounding(call, out_n, out_b, name="nbsd_vs_bsd_wan480p")


@pytest.mark.parametrize("norm", [1, 2, 3])
def test_d_head_32(norm):
    """The smallest head the norm/RoPE pairing takes: d/2 = 16, one chunk per half."""
    call = wl.custom_call(name=f"d32_n{norm}", tokens=300, hidden=256, n_q_heads=6, n_kv_heads=3, d_head=32,
                          norm=norm, rope=1, seed=71 + norm, has_w_col_scale=True)
    _case(call)


def test_d_head_48_plain_projection():
    """d % 32 != 0 is refused with a norm or RoPE, but a plain projection takes it."""
    call = wl.custom_call(name="d48_plain", tokens=257, hidden=384, n_q_heads=3, n_kv_heads=2, d_head=48,
                          norm=0, rope=0, seed=81, has_w_col_scale=True)
    _case(call)


# --- the norm/RoPE work inside the GEMM's epilogue warps (on request) vs its own kernel

@pytest.mark.parametrize("name", ["edge", "short"])
def test_norm_in_gemm_and_separate_pass_agree(name):
    """With QKV_CTE_FLAG_NORM_IN_GEMM the pair GEMM runs the norm/RoPE tasks in its
    epilogue warps; by default the same work is a kernel of its own overlapped with
    the GEMM. Both are correct and agree to rounding."""
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_NORM_IN_GEMM

    if name == "edge":
        call = wl.custom_call(name="fuse_edge", tokens=1000, hidden=1024, n_q_heads=3, n_kv_heads=2, d_head=128,
                              seed=79, has_w_col_scale=True)
    else:
        call = wl.workload("short")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op_f, out_f, ss_f, inv_f = run_path(call, g, flags=QKV_CTE_FLAG_NORM_IN_GEMM)
    op_s, out_s, ss_s, inv_s = run_path(call, g)
    assert op_f.info.norm_in_gemm == 1 and op_s.info.norm_in_gemm == 0
    op_f.status()
    op_s.status()
    check_outputs(call, inp, out_f, ss_f, inv_f, name=f"{name}_in_gemm")
    check_outputs(call, inp, out_s, ss_s, inv_s, name=f"{name}_separate")
    assert_same_to_rounding(call, out_f, out_s, name=f"{name}_in_gemm_vs_separate")


def test_norm_in_gemm_wan480p_sampled():
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_NORM_IN_GEMM

    call = wl.workload("wan480p")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_NORM_IN_GEMM)
    op.status()
    check_outputs(call, inp, out, ss, inv, rows=sampled_rows(call), name="in_gemm_wan480p")


@pytest.mark.parametrize("norm,rope", [(1, 0), (0, 1)])
def test_norm_in_gemm_partial_work(norm, rope):
    """Norm without RoPE and RoPE without norm through the in-GEMM tasks, NBSd output."""
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_NORM_IN_GEMM

    call = wl.custom_call(name=f"fuse_n{norm}_r{rope}", tokens=700, hidden=512, n_q_heads=4, n_kv_heads=2,
                          d_head=64, norm=norm, rope=rope, seed=83 + norm, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_NORM_IN_GEMM, nbsd=True)
    assert op.info.norm_in_gemm == 1
    op.status()
    check_outputs(call, inp, out, ss, inv, name=call.name)


def test_norm_in_gemm_bounded_wait_reports_timeout():
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_GEMM_CTA_PAIR, QKV_CTE_FLAG_NORM_IN_GEMM

    call = wl.workload("tiny")[0]
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g, flags=QKV_CTE_FLAG_TEST_STALL | QKV_CTE_FLAG_GEMM_CTA_PAIR |
                                QKV_CTE_FLAG_NORM_IN_GEMM)
    assert op.info.norm_in_gemm == 1
    with pytest.raises(QkvCteError) as ei:
        op.status()
    assert ei.value.code == QKV_CTE_ERR_DEVICE_TIMEOUT
    op2, out2, ss2, inv2 = run_path(call, g, flags=QKV_CTE_FLAG_NORM_IN_GEMM)
    op2.status()
    check_outputs(call, inp, out2, ss2, inv2, name="in_gemm_after_timeout")


# --- degenerate and extreme shapes -------------------------------------------------

@pytest.mark.parametrize("gemm", ["pair", "single"])
def test_single_k_stage(gemm):
    """H = 128: one 128-byte K stage per tile (the pipeline ring barely turns)."""
    from rope_tcgen05_mxfp8_gb300 import QKV_CTE_FLAG_GEMM_CTA_PAIR, QKV_CTE_FLAG_GEMM_SINGLE_CTA

    call = wl.custom_call(name=f"h128_{gemm}", tokens=700, hidden=128, n_q_heads=3, n_kv_heads=2, d_head=128,
                          seed=91, has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    flags = QKV_CTE_FLAG_GEMM_CTA_PAIR if gemm == "pair" else QKV_CTE_FLAG_GEMM_SINGLE_CTA
    op, out, ss, inv = run_path(call, g, flags=flags)
    op.status()
    check_outputs(call, inp, out, ss, inv, name=call.name)


@pytest.mark.parametrize("norm,rope", [(1, 1), (2, 0), (3, 1)])
def test_single_head_separate_call(norm, rope):
    """One Q head, no K/V: the smallest separate-mode call."""
    call = wl.custom_call(name=f"onehead_n{norm}", tokens=257, hidden=256, n_q_heads=1, n_kv_heads=0, d_head=128,
                          norm=norm, rope=rope, seed=93 + norm)
    _case(call)


def test_large_token_count_sampled():
    """131072 tokens at the Wan layout (4x the 480p rows; ~15 GB on the device), on
    sampled rows: index arithmetic past 2^31 bytes in every buffer."""
    base = wl.workload("wan480p")[0]
    call = wl.custom_call(name="t131072", tokens=131072, hidden=base.hidden, n_q_heads=base.n_q_heads,
                          n_kv_heads=base.n_kv_heads, d_head=base.d_head, rope_grid=(88, 30, 52),
                          outlier_frac=base.outlier_frac, seed=131)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    op, out, ss, inv = run_path(call, g)
    op.status()
    rows = np.unique(np.concatenate([sampled_rows(call, 2048), [0, call.tokens - 1]]))
    check_outputs(call, inp, out, ss, inv, rows=rows, name=call.name)


# --- streams and graphs ---------------------------------------------------------------

def test_cuda_graph_capture_and_replay():
    """The launch sequence (prep, the GEMM, the norm/RoPE pass as a programmatic
    dependent) captures into a CUDA graph; every replay recomputes O correctly."""
    call = wl.custom_call(name="graph", tokens=1000, hidden=1024, n_q_heads=3, n_kv_heads=2, d_head=128, seed=111,
                          has_w_col_scale=True)
    inp = wl.make_inputs(call)
    g = to_device(inp, DEV)
    from rope_tcgen05_mxfp8_gb300 import QkvCte

    op = QkvCte(call.tokens, call.hidden, call.n_q_heads, call.n_kv_heads, call.d_head, device=DEV)
    out = torch.empty(call.tokens, call.width, dtype=torch.bfloat16, device=DEV)
    ss = torch.empty(call.tokens, 2, dtype=torch.float32, device=DEV)
    inv = torch.empty(call.tokens, 2, dtype=torch.float32, device=DEV)
    args = (g["A"], g["a_scale"], g["W"], g["w_sf"], g["bias"], g["gamma_q"], g["gamma_k"], g["cos"], g["sin"])
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        op(*args, out=out, w_col_scale=g["w_col_scale"], sumsq=ss, inv_rms=inv)   # warm-up outside the capture
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        op(*args, out=out, w_col_scale=g["w_col_scale"], sumsq=ss, inv_rms=inv)
    for i in range(3):
        out.fill_(float("nan"))
        ss.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        op.status()
        check_outputs(call, inp, out, ss, inv, name=f"graph_replay_{i}")


def test_independent_calls_on_two_streams():
    """Two plans, each with its own workspace, run at the same time on two streams."""
    from rope_tcgen05_mxfp8_gb300 import QkvCte

    calls = [wl.custom_call(name="stream_a", tokens=1500, hidden=1024, n_q_heads=4, n_kv_heads=2, d_head=128, seed=121),
             wl.custom_call(name="stream_b", tokens=900, hidden=512, n_q_heads=6, n_kv_heads=0, d_head=64, norm=1,
                            rope=0, seed=122)]
    inps = [wl.make_inputs(c) for c in calls]
    gs = [to_device(i, DEV) for i in inps]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ops, outs, sss = [], [], []
    for c, g in zip(calls, gs):
        ops.append(QkvCte(c.tokens, c.hidden, c.n_q_heads, c.n_kv_heads, c.d_head, norm=c.norm, rope=c.rope,
                          device=DEV))
        outs.append(torch.full((c.tokens, c.width), float("nan"), dtype=torch.bfloat16, device=DEV))
        sss.append(torch.empty(c.tokens, 2, dtype=torch.float32, device=DEV))
    for _ in range(3):
        for c, g, op, out, ss, s in zip(calls, gs, ops, outs, sss, streams):
            with torch.cuda.stream(s):
                op(g["A"], g["a_scale"], g["W"], g["w_sf"], g["bias"], g["gamma_q"], g["gamma_k"], g["cos"], g["sin"],
                   out=out, sumsq=ss, stream=s)
    torch.cuda.synchronize()
    for c, inp, op, out, ss, s in zip(calls, inps, ops, outs, sss, streams):
        op.status(s)
        check_outputs(c, inp, out, ss, None, name=c.name)
