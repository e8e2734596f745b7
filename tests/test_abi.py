"""CPU checks of the C ABI: the library loads, exports every declared entry point,
and its host-side plan validation returns the documented codes. No compute call
is made here (there may be no GPU)."""
import ctypes
import os
import re

import pytest

import rope_tcgen05_mxfp8_gb300 as pkg
from rope_tcgen05_mxfp8_gb300 import build as b
from rope_tcgen05_mxfp8_gb300 import qkv_cte as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    b.build()


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(inc, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(qkv_cte_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    declared = _declared_functions()
    assert set(q.EXPORTED) <= set(declared)
    lib = ctypes.CDLL(pkg.library_path())
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_version():
    assert pkg.qkv_cte_version() == 4


def _plan_code(**kw):
    base = dict(tokens=256, hidden=512, n_q_heads=4, n_kv_heads=4, d_head=128)
    base.update(kw)
    desc = q.make_desc(**{k: v for k, v in base.items() if k in
                          ("tokens", "hidden", "n_q_heads", "n_kv_heads", "d_head", "norm", "rope", "eps",
                           "mode", "output_layout", "flags", "tile_n", "input_layout")})
    try:
        plan, ws = q.qkv_cte_plan(desc)
    except q.QkvCteError as e:
        return e.code
    q.qkv_cte_destroy(plan)
    return 0


@pytest.mark.parametrize("kw,code", [
    (dict(), 0),
    (dict(tokens=0), 0),
    (dict(tokens=1), 0),
    (dict(tokens=-1), -1),
    (dict(tokens=2 ** 31), -2),
    (dict(hidden=0), -1),
    (dict(hidden=100), -2),
    (dict(hidden=192), -2),
    (dict(d_head=0), -1),
    (dict(d_head=24), -2),
    (dict(n_q_heads=0), 0),                      # fused mode with no Q heads: a K|V call
    (dict(n_q_heads=-1), -1),
    (dict(n_q_heads=0, n_kv_heads=0, mode=1), -1),  # separate mode needs a Q segment
    (dict(n_q_heads=0, n_kv_heads=0, mode=0), -1),
    (dict(n_kv_heads=-1), -1),
    (dict(n_kv_heads=0, mode=0), -1),
    (dict(n_kv_heads=2, mode=1), -1),
    (dict(mode=7), -1),
    (dict(norm=4), -1),
    (dict(d_head=48), -2),                       # norm + RoPE pair chunks d/2 apart: d % 32
    (dict(d_head=16, norm=0, rope=1), -2),
    (dict(d_head=80, norm=2, rope=0), -2),
    (dict(d_head=48, norm=0, rope=0), 0),        # plain projection: d % 16 is enough
    (dict(norm=2), 0),
    (dict(norm=3), 0),
    (dict(norm=2, tile_n=240), 0),      # per-head norm from statistics: any tile
    (dict(norm=2, tile_n=240, flags=0x40), -2),  # ... in the epilogue: 128-wide heads do not divide 240
    (dict(norm=3, tile_n=256), 0),
    (dict(rope=-1), -1),
    (dict(eps=-1.0), -1),
    (dict(eps=float("nan")), -1),
    (dict(output_layout=1), 0),
    (dict(output_layout=5), -1),
    (dict(flags=0x100), -1),
    (dict(tile_n=100), -2),
    (dict(tile_n=240), 0),
    (dict(input_layout=3), -1),
    (dict(input_layout=-1), -1),
    (dict(input_layout=1), 0),
    (dict(input_layout=2), 0),
    (dict(n_kv_heads=0, mode=1, norm=1, rope=0), 0),
])
def test_plan_validation(kw, code):
    assert _plan_code(**kw) == code


def test_per_head_norm_chooses_a_tile_of_whole_heads():
    for d, tile in ((128, 128), (64, 192), (256, 256), (32, 192), (96, 192)):
        plan, ws = q.qkv_cte_plan(q.make_desc(300, 512, 4, 4, d, norm=2,
                                        flags=q.QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE))
        try:
            info = q.qkv_cte_get_plan_info(plan)
            assert info.tile_n == tile and info.tile_n % d == 0
        finally:
            q.qkv_cte_destroy(plan)


def test_per_head_norm_rejects_heads_no_tile_holds():
    with pytest.raises(q.QkvCteError) as ei:
        q.qkv_cte_plan(q.make_desc(300, 512, 4, 4, 160, norm=2, flags=q.QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE))
    assert ei.value.code == q.QKV_CTE_ERR_UNSUPPORTED and "whole heads" in str(ei.value)


def test_norm_runs_in_the_gemm_only_on_request():
    F = q.QKV_CTE_FLAG_NORM_IN_GEMM
    cases = (
        (dict(tokens=1000), 0),                                   # default: its own kernel
        (dict(tokens=1000, flags=F), 1),
        (dict(tokens=1000, flags=F | q.QKV_CTE_FLAG_SERIAL_PASSES), 0),
        (dict(tokens=1000, flags=F | q.QKV_CTE_FLAG_GEMM_SINGLE_CTA), 0),
        (dict(tokens=100, flags=F), 0),                           # one 128-row block: single-CTA form
        (dict(tokens=1000, norm=0, rope=0, flags=F), 0),          # nothing to run
        (dict(tokens=1000, norm=2, flags=F), 0),                  # per head: finished in the epilogue itself
        (dict(tokens=1000, norm=0, rope=1, flags=F), 1),
    )
    for kw, expect in cases:
        args = dict(hidden=512, n_q_heads=4, n_kv_heads=4, d_head=128)
        args.update(kw)
        plan, ws = q.qkv_cte_plan(q.make_desc(**args))
        try:
            assert q.qkv_cte_get_plan_info(plan).norm_in_gemm == expect, kw
        finally:
            q.qkv_cte_destroy(plan)


def test_per_head_norm_workspace():
    """In the epilogue the per-head kinds need no Q/K hand-off; from statistics they need
    the hand-off plus per-(row, head) statistics: one float (RMS) or, per tile part of a
    head, a (mean, M2) pair (LayerNorm)."""
    T = 1000
    align = lambda x: -(-x // 256) * 256
    rows = -(-T // 128) * 128
    kq = 8 * 128
    hand_off = align(rows * kq * 2) + align(rows * kq // 16)
    F = q.QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE
    sizes = {}
    for key, norm, flags in (("across", 1, 0), ("epi", 2, F), ("rms", 2, 0), ("ln", 3, 0)):
        plan, ws = q.qkv_cte_plan(q.make_desc(T, 512, 4, 4, 128, norm=norm, tile_n=128, flags=flags))
        q.qkv_cte_destroy(plan)
        sizes[key] = ws
    assert sizes["across"] - sizes["epi"] == hand_off
    assert sizes["rms"] - sizes["across"] == align(rows * 8 * 4)
    parts = (128 + 128 - 2) // 128 + 1          # tiles a 128-column head can touch at tile 128
    assert sizes["ln"] - sizes["across"] == align(rows * 8 * parts * 16)


def test_plan_info_reports_the_choices():
    plan, ws = q.qkv_cte_plan(q.make_desc(32760, 5120, 40, 40, 128))
    try:
        info = q.qkv_cte_get_plan_info(plan)
        assert info.tile_n == 240 and info.m_tiles == 128 and info.n_tiles == 64 and info.cta_pair == 1
        assert info.workspace_bytes == ws and 1 <= info.n_bands <= 16
    finally:
        q.qkv_cte_destroy(plan)
    plan, ws = q.qkv_cte_plan(q.make_desc(512, 512, 4, 4, 128, tile_n=128))
    try:
        assert q.qkv_cte_get_plan_info(plan).tile_n == 128
    finally:
        q.qkv_cte_destroy(plan)
    for T, flags, pair, m_tiles in ((100, 0, 0, 1), (300, 0, 1, 2), (300, q.QKV_CTE_FLAG_GEMM_SINGLE_CTA, 0, 3),
                                    (100, q.QKV_CTE_FLAG_GEMM_CTA_PAIR, 1, 1)):
        plan, ws = q.qkv_cte_plan(q.make_desc(T, 512, 4, 4, 128, flags=flags))
        try:
            info = q.qkv_cte_get_plan_info(plan)
            assert (info.cta_pair, info.m_tiles) == (pair, m_tiles), (T, flags)
        finally:
            q.qkv_cte_destroy(plan)
    with pytest.raises(q.QkvCteError):
        q.qkv_cte_plan(q.make_desc(300, 512, 4, 4, 128,
                                   flags=q.QKV_CTE_FLAG_GEMM_CTA_PAIR | q.QKV_CTE_FLAG_GEMM_SINGLE_CTA))


def test_error_message_is_recorded():
    with pytest.raises(q.QkvCteError) as ei:
        q.qkv_cte_plan(q.make_desc(256, 100, 4, 4, 128))
    assert "multiple of 128" in str(ei.value)
    assert "multiple of 128" in q.qkv_cte_last_error()


@pytest.mark.parametrize("input_layout", [0, 1, 2])
def test_workspace_size_formula(input_layout):
    for T, I_heads, tile in ((32760, (40, 40), 256), (1, (1, 1), 128), (4096, (40, 0), 240)):
        nq, nkv = I_heads
        desc = q.make_desc(T, 5120, nq, nkv, 128, rope=0 if nkv == 0 else 1, tile_n=tile,
                           input_layout=input_layout)
        plan, ws = q.qkv_cte_plan(desc)
        q.qkv_cte_destroy(plan)
        I = (nq + 2 * nkv) * 128
        n_tiles = -(-I // tile)
        sf = n_tiles * (5120 // 128) * (-(-tile // 128)) * 2048  # 4 lane-quarter copies of 512 B
        ss = -(-(T * 8) // 256) * 256
        rows = -(-T // 128) * 128
        kq = (nq + nkv) * 128
        qk = -(-(rows * kq * 2) // 256) * 256 + -(-(rows * kq // 16) // 256) * 256  # hand-off
        ready = -(-(-(-T // 128) * 4) // 256) * 256        # per-panel counters
        ready += 1024 * 4                                   # per-SM sub-partition table
        # a packed or bf16 input: the producer's codes [T, H] and row scales [T]
        act = (-(-(T * 5120) // 256) * 256 + -(-(T * 4) // 256) * 256) if input_layout else 0
        assert ws == 256 + ss + -(-sf // 256) * 256 + ready + qk + act


def test_run_rejects_null_plan_without_launch():
    lib = pkg.load()
    rc = lib.qkv_cte_run(None, *([None] * 14), ctypes.c_size_t(0), None)
    assert rc == q.QKV_CTE_ERR_INVALID
    assert "null plan" in q.qkv_cte_last_error()


def test_destroy_null_is_noop():
    pkg.load().qkv_cte_destroy(None)


def test_run_argument_checks_precede_any_cuda_call():
    """Missing required pointers are rejected on the host (no device touched)."""
    lib = pkg.load()
    plan, ws = q.qkv_cte_plan(q.make_desc(256, 512, 4, 4, 128))
    try:
        fake = ctypes.c_void_p(4096)
        args = [fake] * 14
        args[0] = None  # A missing
        rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws), None)
        assert rc == q.QKV_CTE_ERR_INVALID
        args = [fake] * 14
        args[7] = None  # gamma_k missing while norm and n_kv > 0
        rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws), None)
        assert rc == q.QKV_CTE_ERR_INVALID and "gamma_k" in q.qkv_cte_last_error()
        args = [fake] * 14
        args[8] = None  # cos missing while rope
        rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws), None)
        assert rc == q.QKV_CTE_ERR_INVALID and "cos" in q.qkv_cte_last_error()
        args = [fake] * 14
        args[0] = ctypes.c_void_p(4097)  # misaligned A
        rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws), None)
        assert rc == q.QKV_CTE_ERR_UNSUPPORTED
        args = [fake] * 14
        rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws - 1), None)
        assert rc == q.QKV_CTE_ERR_INVALID and "workspace" in q.qkv_cte_last_error()
    finally:
        q.qkv_cte_destroy(plan)


def test_run_input_layout_checks():
    """a_scale goes with separate FP8 rows only; packed rows need only 4-byte alignment."""
    lib = pkg.load()
    fake = ctypes.c_void_p(4096)
    for layout in (1, 2):
        plan, ws = q.qkv_cte_plan(q.make_desc(256, 512, 4, 4, 128, input_layout=layout))
        try:
            args = [fake] * 14
            rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws), None)    # a_scale given
            assert rc == q.QKV_CTE_ERR_INVALID and "a_scale must be NULL" in q.qkv_cte_last_error()
            args[0] = ctypes.c_void_p(4100)                                    # A 4-byte aligned only
            args[1] = None
            rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws - 1), None)
            if layout == 1:   # passes the alignment check, stops at the workspace size
                assert rc == q.QKV_CTE_ERR_INVALID and "workspace" in q.qkv_cte_last_error()
            else:
                assert rc == q.QKV_CTE_ERR_UNSUPPORTED and "aligned" in q.qkv_cte_last_error()
        finally:
            q.qkv_cte_destroy(plan)
    plan, ws = q.qkv_cte_plan(q.make_desc(256, 512, 4, 4, 128))
    try:
        args = [fake] * 14
        args[1] = None
        rc = lib.qkv_cte_run(plan, *args, ctypes.c_size_t(ws), None)
        assert rc == q.QKV_CTE_ERR_INVALID and "a_scale is required" in q.qkv_cte_last_error()
    finally:
        q.qkv_cte_destroy(plan)


def test_producer_entry_points_check_arguments_on_the_host():
    lib = pkg.load()
    f = ctypes.c_void_p(4096)
    g = ctypes.c_void_p(1 << 40)
    assert lib.qkv_cte_row_quantize(f, 4, 100, g, g, None, None) == q.QKV_CTE_ERR_UNSUPPORTED   # H % 16
    assert lib.qkv_cte_row_quantize(f, -1, 128, g, g, None, None) == q.QKV_CTE_ERR_INVALID
    assert lib.qkv_cte_row_quantize(f, 4, 128, None, None, None, None) == q.QKV_CTE_ERR_INVALID  # no output
    assert lib.qkv_cte_row_quantize(f, 4, 128, g, None, None, None) == q.QKV_CTE_ERR_INVALID     # A without scale
    assert lib.qkv_cte_row_quantize(ctypes.c_void_p(4098), 4, 128, g, g, None, None) == q.QKV_CTE_ERR_UNSUPPORTED
    # X [4, 128] bf16 spans 1 KB from 4096; codes written into it overlap
    assert lib.qkv_cte_row_quantize(f, 4, 128, ctypes.c_void_p(4096 + 512), g, None, None) == q.QKV_CTE_ERR_INVALID
    assert "overlap" in q.qkv_cte_last_error()
    assert lib.qkv_cte_row_quantize(None, 0, 128, g, g, None, None) == 0      # empty: nothing launched
    assert lib.qkv_cte_unpack_rows(f, 4, 128, None, g, None) == q.QKV_CTE_ERR_INVALID
    assert lib.qkv_cte_unpack_rows(f, 4, 120, g, g, None) == q.QKV_CTE_ERR_UNSUPPORTED
    assert lib.qkv_cte_unpack_rows(ctypes.c_void_p(4098), 4, 128, g, ctypes.c_void_p(1 << 41), None) == \
        q.QKV_CTE_ERR_UNSUPPORTED
    assert lib.qkv_cte_unpack_rows(None, 0, 128, None, None, None) == 0


def test_zero_tokens_launches_nothing():
    """An empty problem returns before any pointer check or CUDA call (no workspace
    given, so not even the status word is touched)."""
    lib = pkg.load()
    plan, ws = q.qkv_cte_plan(q.make_desc(0, 512, 4, 4, 128))
    try:
        rc = lib.qkv_cte_run(plan, *([None] * 14), ctypes.c_size_t(0), None)
        assert rc == 0
    finally:
        q.qkv_cte_destroy(plan)


def test_host_scratch_bytes_formula():
    """Two staging slots (input rows, row scales, output rows) plus one chunk's workspace."""
    T, H, nq, nkv, d = 10000, 512, 4, 4, 128
    I = (nq + 2 * nkv) * d
    align = lambda x: -(-x // 256) * 256
    for layout, in_row in ((0, H), (1, H + 4), (2, 2 * H)):
        plan, ws = q.qkv_cte_plan(q.make_desc(T, H, nq, nkv, d, input_layout=layout))
        cplan, cws = q.qkv_cte_plan(q.make_desc(1024, H, nq, nkv, d, input_layout=layout))
        try:
            n = q.qkv_cte_host_scratch_bytes(plan, 1000)   # rounded up to 1024 rows
            slot = align(1024 * in_row) + align(1024 * 4) + align(1024 * I * 2)
            assert n == 256 + 2 * slot + align(cws)
            assert q.qkv_cte_host_scratch_bytes(plan, 10 ** 6) > n     # capped at T rows
        finally:
            q.qkv_cte_destroy(plan)
            q.qkv_cte_destroy(cplan)


def test_run_host_argument_checks_precede_any_copy():
    lib = pkg.load()
    plan, ws = q.qkv_cte_plan(q.make_desc(300, 512, 4, 4, 128))
    try:
        P = ctypes.c_void_p
        f = P(4096)
        args = [f] * 14
        args[0] = None
        rc = lib.qkv_cte_run_host(plan, *args, ctypes.c_size_t(1 << 30), 0, None)
        assert rc == q.QKV_CTE_ERR_INVALID and "required" in q.qkv_cte_last_error()
        args = [f] * 14
        args[1] = None      # separate FP8 rows need their scales
        rc = lib.qkv_cte_run_host(plan, *args, ctypes.c_size_t(1 << 30), 0, None)
        assert rc == q.QKV_CTE_ERR_INVALID and "a_scale_host" in q.qkv_cte_last_error()
        args = [f] * 14     # not pinned host memory (here: no device at all)
        rc = lib.qkv_cte_run_host(plan, *args, ctypes.c_size_t(1 << 30), 0, None)
        assert rc == q.QKV_CTE_ERR_UNSUPPORTED and "pinned" in q.qkv_cte_last_error()
    finally:
        q.qkv_cte_destroy(plan)
