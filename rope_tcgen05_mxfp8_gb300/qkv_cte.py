"""Thin ctypes binding over libqkvcte.so (argument marshalling only).

Each function has the name of the C entry point it calls (see include/qkv_cte.h).
Tensors are torch CUDA tensors used as device memory; every step of the
computation runs in the library's CUDA kernels. If the library has not been built
the first call raises: there is no other implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libqkvcte.so")

QKV_CTE_OK = 0
QKV_CTE_ERR_INVALID = -1
QKV_CTE_ERR_UNSUPPORTED = -2
QKV_CTE_ERR_CUDA = -3
QKV_CTE_ERR_ARCH = -4
QKV_CTE_ERR_DEVICE_TIMEOUT = -5
QKV_CTE_MODE_FUSED = 0
QKV_CTE_MODE_SEPARATE = 1
QKV_CTE_LAYOUT_BSD = 0
QKV_CTE_LAYOUT_NBSD = 1
QKV_CTE_NORM_NONE = 0
QKV_CTE_NORM_ACROSS_HEADS = 1
QKV_CTE_NORM_HEAD_RMS = 2
QKV_CTE_NORM_HEAD_LAYER = 3
QKV_CTE_INPUT_ROW_FP8 = 0
QKV_CTE_INPUT_PACKED = 1
QKV_CTE_INPUT_BF16 = 2
QKV_CTE_FLAG_TEST_STALL = 0x1
QKV_CTE_FLAG_PROFILE = 0x2
QKV_CTE_FLAG_SERIAL_PASSES = 0x4
QKV_CTE_FLAG_GEMM_CTA_PAIR = 0x8
QKV_CTE_FLAG_GEMM_SINGLE_CTA = 0x10
QKV_CTE_FLAG_NORM_IN_GEMM = 0x20
QKV_CTE_FLAG_HEAD_NORM_IN_EPILOGUE = 0x40

EXPORTED = ("qkv_cte_plan", "qkv_cte_run", "qkv_cte_status", "qkv_cte_pass_times", "qkv_cte_destroy",
            "qkv_cte_last_error", "qkv_cte_version", "qkv_cte_run_noalloc", "qkv_cte_get_plan_info",
            "qkv_cte_row_quantize", "qkv_cte_unpack_rows", "qkv_cte_interleaved_to_rotate_half",
            "qkv_cte_run_host", "qkv_cte_host_scratch_bytes", "qkv_cte_noalloc_status")
QKV_CTE_NOALLOC_SCRATCH_BYTES = 24 << 20


class qkv_cte_desc(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int64),
        ("hidden", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("d_head", ctypes.c_int32),
        ("mode", ctypes.c_int32),
        ("norm", ctypes.c_int32),
        ("rope", ctypes.c_int32),
        ("output_layout", ctypes.c_int32),
        ("eps", ctypes.c_float),
        ("flags", ctypes.c_uint32),
        ("tile_n", ctypes.c_int32),
        ("input_layout", ctypes.c_int32),
    ]


class qkv_cte_plan_info(ctypes.Structure):
    _fields_ = [
        ("tile_n", ctypes.c_int32),
        ("m_tiles", ctypes.c_int32),
        ("n_tiles", ctypes.c_int32),
        ("n_bands", ctypes.c_int32),
        ("cta_pair", ctypes.c_int32),
        ("norm_in_gemm", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
    ]


class QkvCteError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qkv_cte error {code}: {msg}")
        self.code = code


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libqkvcte.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    lib.qkv_cte_plan.argtypes = [ctypes.POINTER(P), ctypes.POINTER(qkv_cte_desc), ctypes.POINTER(ctypes.c_size_t)]
    lib.qkv_cte_plan.restype = ctypes.c_int
    lib.qkv_cte_run.argtypes = [P] * 15 + [ctypes.c_size_t, P]
    lib.qkv_cte_run.restype = ctypes.c_int
    lib.qkv_cte_get_plan_info.argtypes = [P, ctypes.POINTER(qkv_cte_plan_info)]
    lib.qkv_cte_get_plan_info.restype = ctypes.c_int
    lib.qkv_cte_run_noalloc.argtypes = [P] * 15
    lib.qkv_cte_run_noalloc.restype = ctypes.c_int
    lib.qkv_cte_noalloc_status.argtypes = [P]
    lib.qkv_cte_noalloc_status.restype = ctypes.c_int
    lib.qkv_cte_row_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, P, P]
    lib.qkv_cte_row_quantize.restype = ctypes.c_int
    lib.qkv_cte_unpack_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, P]
    lib.qkv_cte_unpack_rows.restype = ctypes.c_int
    lib.qkv_cte_interleaved_to_rotate_half.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                       ctypes.c_int32, ctypes.c_int32, P]
    lib.qkv_cte_interleaved_to_rotate_half.restype = ctypes.c_int
    lib.qkv_cte_run_host.argtypes = [P] * 15 + [ctypes.c_size_t, ctypes.c_int32, P]
    lib.qkv_cte_run_host.restype = ctypes.c_int
    lib.qkv_cte_host_scratch_bytes.argtypes = [P, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
    lib.qkv_cte_host_scratch_bytes.restype = ctypes.c_int
    lib.qkv_cte_status.argtypes = [P, P]
    lib.qkv_cte_status.restype = ctypes.c_int
    lib.qkv_cte_pass_times.argtypes = [P, ctypes.POINTER(ctypes.c_float)]
    lib.qkv_cte_pass_times.restype = ctypes.c_int
    lib.qkv_cte_destroy.argtypes = [P]
    lib.qkv_cte_destroy.restype = None
    lib.qkv_cte_last_error.argtypes = []
    lib.qkv_cte_last_error.restype = ctypes.c_char_p
    lib.qkv_cte_version.argtypes = []
    lib.qkv_cte_version.restype = ctypes.c_int
    _lib = lib
    return lib


def qkv_cte_last_error() -> str:
    return load().qkv_cte_last_error().decode()


def qkv_cte_version() -> int:
    return load().qkv_cte_version()


def _check(rc: int) -> int:
    if rc != QKV_CTE_OK:
        raise QkvCteError(rc, qkv_cte_last_error())
    return rc


def make_desc(tokens, hidden, n_q_heads, n_kv_heads, d_head, norm=1, rope=1, eps=1e-6,
              mode=None, output_layout=QKV_CTE_LAYOUT_BSD, flags=0, tile_n=0,
              input_layout=QKV_CTE_INPUT_ROW_FP8) -> qkv_cte_desc:
    if mode is None:
        mode = QKV_CTE_MODE_FUSED if n_kv_heads > 0 else QKV_CTE_MODE_SEPARATE
    return qkv_cte_desc(tokens, hidden, n_q_heads, n_kv_heads, d_head, mode, norm, rope, output_layout,
                        eps, flags, tile_n, input_layout)


def qkv_cte_plan(desc: qkv_cte_desc):
    """Returns (plan handle, workspace bytes); raises QkvCteError on a rejected desc."""
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(load().qkv_cte_plan(ctypes.byref(plan), ctypes.byref(desc), ctypes.byref(ws)))
    return plan, ws.value


def qkv_cte_get_plan_info(plan) -> qkv_cte_plan_info:
    info = qkv_cte_plan_info()
    _check(load().qkv_cte_get_plan_info(plan, ctypes.byref(info)))
    return info


def qkv_cte_destroy(plan) -> None:
    load().qkv_cte_destroy(plan)


_DTYPES = {
    "A": (torch.uint8, torch.bfloat16, torch.int16, torch.uint16), "W": (torch.uint8,), "w_sf": (torch.uint8,),
    "X": (torch.bfloat16, torch.int16, torch.uint16), "packed": (torch.uint8,),
    "a_scale": (torch.float32,), "w_col_scale": (torch.float32,),
    "bias": (torch.bfloat16, torch.int16, torch.uint16),
    "gamma_q": (torch.bfloat16, torch.int16, torch.uint16),
    "gamma_k": (torch.bfloat16, torch.int16, torch.uint16),
    "cos": (torch.float32,), "sin": (torch.float32,),
    "O": (torch.bfloat16, torch.int16, torch.uint16),
    "sumsq": (torch.float32,), "inv_rms": (torch.float32,), "workspace": (torch.uint8,),
}


def _ptr(name: str, t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor or None")
    if t.dtype not in _DTYPES[name]:
        raise TypeError(f"{name}: dtype {t.dtype} not in {_DTYPES[name]}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def qkv_cte_run(plan, A, a_scale, W, w_sf, w_col_scale, bias, gamma_q, gamma_k, cos, sin, O,
                sumsq, inv_rms, workspace, stream=None) -> int:
    """Launch the path on `stream` (torch.cuda.Stream, raw handle, or None = current stream)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = [_ptr("A", A), _ptr("a_scale", a_scale), _ptr("W", W), _ptr("w_sf", w_sf),
            _ptr("w_col_scale", w_col_scale), _ptr("bias", bias), _ptr("gamma_q", gamma_q),
            _ptr("gamma_k", gamma_k), _ptr("cos", cos), _ptr("sin", sin), _ptr("O", O),
            _ptr("sumsq", sumsq), _ptr("inv_rms", inv_rms), _ptr("workspace", workspace)]
    return _check(load().qkv_cte_run(plan, *args, ctypes.c_size_t(ws_bytes), ctypes.c_void_p(handle)))


def qkv_cte_run_noalloc(plan, A, a_scale, W, w_sf, w_col_scale, bias, gamma_q, gamma_k, cos, sin, O,
                        sumsq, inv_rms, stream=None) -> int:
    """qkv_cte_run with the library's fixed scratch array instead of a workspace: for
    callers that cannot allocate device memory when they run (see qkv_cte.h)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    args = [_ptr("A", A), _ptr("a_scale", a_scale), _ptr("W", W), _ptr("w_sf", w_sf),
            _ptr("w_col_scale", w_col_scale), _ptr("bias", bias), _ptr("gamma_q", gamma_q),
            _ptr("gamma_k", gamma_k), _ptr("cos", cos), _ptr("sin", sin), _ptr("O", O),
            _ptr("sumsq", sumsq), _ptr("inv_rms", inv_rms)]
    return _check(load().qkv_cte_run_noalloc(plan, *args, ctypes.c_void_p(handle)))


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def qkv_cte_row_quantize(X, A=None, a_scale=None, packed=None, stream=None):
    """bf16 X [T, H] -> e4m3 codes A [T, H] + fp32 a_scale [T] and/or packed [T, H + 4]
    rows (the outputs given, or, with none given, A and a_scale allocated here).
    Returns (A, a_scale, packed)."""
    T, H = X.shape
    if A is None and a_scale is None and packed is None:
        A = torch.empty(T, H, dtype=torch.uint8, device=X.device)
        a_scale = torch.empty(T, dtype=torch.float32, device=X.device)
    _check(load().qkv_cte_row_quantize(_ptr("X", X), T, H, _ptr("A", A), _ptr("a_scale", a_scale),
                                       _ptr("packed", packed), _stream_handle(stream)))
    return A, a_scale, packed


def qkv_cte_unpack_rows(packed, A=None, a_scale=None, stream=None):
    """Packed [T, H + 4] rows -> (A uint8 [T, H], a_scale fp32 [T])."""
    T, H = packed.shape[0], packed.shape[1] - 4
    if A is None:
        A = torch.empty(T, H, dtype=torch.uint8, device=packed.device)
    if a_scale is None:
        a_scale = torch.empty(T, dtype=torch.float32, device=packed.device)
    _check(load().qkv_cte_unpack_rows(_ptr("packed", packed), T, H, _ptr("A", A), _ptr("a_scale", a_scale),
                                      _stream_handle(stream)))
    return A, a_scale


def qkv_cte_interleaved_to_rotate_half(src, n_q_heads, n_kv_heads, d_head, dst=None, stream=None):
    """Permute the Q/K rows of a per-output-channel tensor (first dimension = rows)
    from the interleaved to the rotate-half lane order; returns dst (allocated here
    when not given). See qkv_cte.h for how to lay out each tensor as rows."""
    if not (src.is_cuda and src.is_contiguous()):
        raise ValueError("src: must be a contiguous CUDA tensor")
    if dst is None:
        dst = torch.empty_like(src)
    if not (dst.is_cuda and dst.is_contiguous()) or dst.numel() * dst.element_size() != src.numel() * src.element_size():
        raise ValueError("dst: must be a contiguous CUDA tensor of src's size")
    rows = src.shape[0] if src.dim() > 0 else 0
    row_bytes = (src.numel() * src.element_size()) // rows if rows else 1
    _check(load().qkv_cte_interleaved_to_rotate_half(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()),
                                                     rows, row_bytes, n_q_heads, n_kv_heads, d_head,
                                                     _stream_handle(stream)))
    return dst


def _host_ptr(name: str, t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name}: expected a pinned CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def qkv_cte_host_scratch_bytes(plan, chunk_rows=0) -> int:
    n = ctypes.c_size_t()
    _check(load().qkv_cte_host_scratch_bytes(plan, chunk_rows, ctypes.byref(n)))
    return n.value


def qkv_cte_run_host(plan, A_host, a_scale_host, W, w_sf, w_col_scale, bias, gamma_q, gamma_k, cos, sin, O_host,
                     sumsq, inv_rms, scratch, chunk_rows=0, stream=None) -> int:
    """The path on pinned host activations, writing O to pinned host memory, with the
    copies overlapped with the computation (see qkv_cte.h)."""
    ws_bytes = scratch.numel() * scratch.element_size() if scratch is not None else 0
    args = [_host_ptr("A_host", A_host), _host_ptr("a_scale_host", a_scale_host), _ptr("W", W), _ptr("w_sf", w_sf),
            _ptr("w_col_scale", w_col_scale), _ptr("bias", bias), _ptr("gamma_q", gamma_q),
            _ptr("gamma_k", gamma_k), _ptr("cos", cos), _ptr("sin", sin), _host_ptr("O_host", O_host),
            _ptr("sumsq", sumsq), _ptr("inv_rms", inv_rms), _ptr("workspace", scratch)]
    return _check(load().qkv_cte_run_host(plan, *args, ctypes.c_size_t(ws_bytes), chunk_rows,
                                          _stream_handle(stream)))


def qkv_cte_status(workspace, stream=None) -> int:
    """Synchronise the stream and raise QkvCteError if a bounded device wait ran out."""
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return _check(load().qkv_cte_status(_ptr("workspace", workspace), ctypes.c_void_p(handle)))


def qkv_cte_noalloc_status(stream=None) -> int:
    """qkv_cte_status for the scratch array of qkv_cte_run_noalloc on the current device."""
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return _check(load().qkv_cte_noalloc_status(ctypes.c_void_p(handle)))


def qkv_cte_pass_times(plan):
    """(prep, GEMM, norm+RoPE, whole run) device milliseconds of the plan's latest run."""
    ms = (ctypes.c_float * 4)()
    _check(load().qkv_cte_pass_times(plan, ms))
    return tuple(float(x) for x in ms)


class QkvCte:
    """A plan plus its workspace on one device: the usual way to call the library.

    >>> op = QkvCte(tokens=T, hidden=H, n_q_heads=40, n_kv_heads=40, d_head=128)
    >>> op(A, a_scale, W, w_sf, bias, gamma_q, gamma_k, cos, sin, out=O)
    """

    def __init__(self, tokens, hidden, n_q_heads, n_kv_heads, d_head, norm=1, rope=1, eps=1e-6,
                 tile_n=0, flags=0, device=None, output_layout=QKV_CTE_LAYOUT_BSD,
                 input_layout=QKV_CTE_INPUT_ROW_FP8):
        self.desc = make_desc(tokens, hidden, n_q_heads, n_kv_heads, d_head, norm=norm, rope=rope,
                              eps=eps, tile_n=tile_n, flags=flags, output_layout=output_layout,
                              input_layout=input_layout)
        self.plan, self.workspace_bytes = qkv_cte_plan(self.desc)
        self.info = qkv_cte_get_plan_info(self.plan)
        self.width = (n_q_heads + 2 * n_kv_heads) * d_head
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.workspace = torch.zeros(max(self.workspace_bytes, 256), dtype=torch.uint8, device=dev)

    def plan_info(self) -> qkv_cte_plan_info:
        """The plan's choices."""
        return qkv_cte_get_plan_info(self.plan)

    def __call__(self, A, a_scale, W, w_sf, bias, gamma_q, gamma_k, cos, sin, out=None,
                 w_col_scale=None, sumsq=None, inv_rms=None, stream=None):
        if out is None:
            if self.desc.output_layout == QKV_CTE_LAYOUT_NBSD:
                d = self.desc.d_head
                out = torch.empty(self.width // d, self.desc.tokens, d, dtype=torch.bfloat16, device=A.device)
            else:
                out = torch.empty(self.desc.tokens, self.width, dtype=torch.bfloat16, device=A.device)
        qkv_cte_run(self.plan, A, a_scale, W, w_sf, w_col_scale, bias, gamma_q, gamma_k, cos, sin, out,
                    sumsq, inv_rms, self.workspace, stream)
        return out

    def run_host(self, A_host, a_scale_host, W, w_sf, bias, gamma_q, gamma_k, cos, sin, O_host, w_col_scale=None,
                 sumsq=None, inv_rms=None, chunk_rows=0, stream=None):
        """qkv_cte_run_host with a scratch buffer kept per chunk size."""
        n = qkv_cte_host_scratch_bytes(self.plan, chunk_rows)
        if getattr(self, "_host_scratch", None) is None or self._host_scratch.numel() < max(n, 256):
            dev = self.workspace.device
            self._host_scratch = torch.zeros(max(n, 256), dtype=torch.uint8, device=dev)
        qkv_cte_run_host(self.plan, A_host, a_scale_host, W, w_sf, w_col_scale, bias, gamma_q, gamma_k, cos, sin,
                         O_host, sumsq, inv_rms, self._host_scratch, chunk_rows, stream)
        return O_host

    def host_status(self, stream=None):
        return qkv_cte_status(self._host_scratch, stream)

    def status(self, stream=None):
        return qkv_cte_status(self.workspace, stream)

    def pass_times(self):
        return qkv_cte_pass_times(self.plan)

    def close(self):
        if self.plan is not None:
            qkv_cte_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
