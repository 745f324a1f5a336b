"""ctypes binding of libnvfp4.so (include/nvfp4.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but turn PyTorch tensors into pointers, sizes and the current CUDA
stream.  All arithmetic runs in the library's CUDA kernels.  If the library is
missing or fails to load, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass

import torch

from . import build as _build

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_UNSUPPORTED_SHAPE = 2
NVFP4_ERR_WORKSPACE = 3
NVFP4_ERR_CUDA = 4
NVFP4_ERR_DEVICE_TIMEOUT = 5

NVFP4_STATUS_WORD_OFFSET = 128

NVFP4_OP_QUANTIZE = 0
NVFP4_OP_GEMV_SKINNY = 1
NVFP4_OP_GATEUP_SWIGLU = 2
NVFP4_OP_GEMM_PREFILL = 3
NVFP4_OP_FP6_GEMM = 4
NVFP4_OP_FP6_GATEUP_SWIGLU = 5

NVFP4_OUT_F32 = 0
NVFP4_OUT_BF16 = 1

_lock = threading.Lock()
_lib = None


class SkinnyJobC(ctypes.Structure):
    """nvfp4_skinny_job of include/nvfp4.h."""
    _fields_ = [("x", ctypes.c_void_p), ("x_ld", ctypes.c_int64), ("input", ctypes.c_int32),
                ("n_weights", ctypes.c_int32), ("codes", ctypes.c_void_p * 2), ("scales", ctypes.c_void_p * 2),
                ("tensor_scale", ctypes.c_void_p * 2), ("M", ctypes.c_int64), ("K", ctypes.c_int64),
                ("y", ctypes.c_void_p), ("out_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {nvfp4_status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libnvfp4.so (built by gemm_nvfp4_gb300.build / __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libnvfp4.so not found at {path}: build it with `python -m gemm_nvfp4_gb300.build` "
                "(the NVFP4 path has no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, i64, sz, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        lib.nvfp4_status_string.restype = ctypes.c_char_p
        lib.nvfp4_status_string.argtypes = [i32]
        lib.nvfp4_version.restype = i32
        lib.nvfp4_version.argtypes = []
        lib.nvfp4_workspace_bytes.restype = sz
        lib.nvfp4_workspace_bytes.argtypes = [i32, i64, i64, i64]
        lib.nvfp4_quantize.restype = i32
        lib.nvfp4_quantize.argtypes = [P, i64, i64, P, P, P, P, sz, P]
        lib.nvfp4_quantize_bf16.restype = i32
        lib.nvfp4_quantize_bf16.argtypes = [P, i64, i64, P, P, P, P, sz, P]
        lib.nvfp4_blocked_scale_bytes.restype = sz
        lib.nvfp4_blocked_scale_bytes.argtypes = [i64, i64]
        lib.nvfp4_import_blocked_scales.restype = i32
        lib.nvfp4_import_blocked_scales.argtypes = [P, i64, i64, P, P]
        lib.nvfp4_fp6_quantize.restype = i32
        lib.nvfp4_fp6_quantize.argtypes = [P, i64, i64, P, P, P]
        lib.nvfp4_fp6_quantize_bf16.restype = i32
        lib.nvfp4_fp6_quantize_bf16.argtypes = [P, i64, i64, P, P, P]
        lib.nvfp4_fp6_gemm.restype = i32
        lib.nvfp4_fp6_gemm.argtypes = [P, i64, P, P, i64, i64, P, i32, P, sz, P]
        lib.nvfp4_fp6_gateup_swiglu.restype = i32
        lib.nvfp4_fp6_gateup_swiglu.argtypes = [P, i64, P, P, P, P, i64, i64, P, i32, P, sz, P]
        lib.nvfp4_gemv_skinny.restype = i32
        lib.nvfp4_gemv_skinny.argtypes = [P, i64, P, P, P, i64, i64, P, i32, P, sz, P]
        lib.nvfp4_gateup_swiglu.restype = i32
        lib.nvfp4_gateup_swiglu.argtypes = [P, i64, P, P, P, P, P, P, i64, i64, P, i32, P, sz, P]
        lib.nvfp4_gemm_prefill.restype = i32
        lib.nvfp4_gemm_prefill.argtypes = [P, i64, P, P, P, i64, i64, P, i32, P, sz, P]
        lib.nvfp4_gemv_skinny_noalloc.restype = i32
        lib.nvfp4_gemv_skinny_noalloc.argtypes = [P, i64, P, P, P, i64, i64, P, i32, P]
        lib.nvfp4_stream_plan_bytes.restype = sz
        lib.nvfp4_stream_plan_bytes.argtypes = [ctypes.POINTER(SkinnyJobC), i32, i64]
        lib.nvfp4_stream_plan.restype = i32
        lib.nvfp4_stream_plan.argtypes = [ctypes.POINTER(SkinnyJobC), i32, i64, P, sz, P]
        lib.nvfp4_stream_run.restype = i32
        lib.nvfp4_stream_run.argtypes = [P, sz, P]
        lib.nvfp4_noalloc_status.restype = i32
        lib.nvfp4_noalloc_status.argtypes = [i32, ctypes.POINTER(ctypes.c_uint32), P]
        lib.nvfp4_noalloc_selftest_wait_timeout.restype = i32
        lib.nvfp4_noalloc_selftest_wait_timeout.argtypes = [P]
        lib.nvfp4_device_status.restype = i32
        lib.nvfp4_device_status.argtypes = [P, sz, i32, ctypes.POINTER(ctypes.c_uint32), P]
        lib.nvfp4_selftest_wait_timeout.restype = i32
        lib.nvfp4_selftest_wait_timeout.argtypes = [P, sz, P]
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/nvfp4.h."""
    text = open(_build.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


# ---------------------------------------------------------------------------
# Thin wrappers with the C names
# ---------------------------------------------------------------------------

def nvfp4_status_string(status: int) -> str:
    return load_library().nvfp4_status_string(int(status)).decode()


def nvfp4_version() -> int:
    return load_library().nvfp4_version()


def nvfp4_workspace_bytes(op: int, N: int, M: int, K: int) -> int:
    return load_library().nvfp4_workspace_bytes(int(op), int(N), int(M), int(K))


@dataclass
class NVFP4Weight:
    """One NVFP4 tensor W[M][K] in device memory (see include/nvfp4.h)."""
    codes: torch.Tensor         # uint8 [M, K/2]
    scales: torch.Tensor        # uint8 [M, K/16]
    tensor_scale: torch.Tensor  # float32 [1]

    @property
    def M(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1] * 2

    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != NVFP4_OK:
        raise NVFP4Error(status, where)


def _workspace(op, N, M, K, device, workspace):
    need = nvfp4_workspace_bytes(op, N, M, K)
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    if need == 0:
        return None, 0
    # zero-filled: the skinny calls keep split-K counters in it
    return torch.zeros(need, dtype=torch.uint8, device=device), need


def _out_code(dtype) -> int:
    if dtype == torch.float32:
        return NVFP4_OUT_F32
    if dtype == torch.bfloat16:
        return NVFP4_OUT_BF16
    raise ValueError(f"unsupported output dtype {dtype}")


def nvfp4_quantize(w: torch.Tensor, workspace: torch.Tensor | None = None,
                   out: NVFP4Weight | None = None, stream=None) -> NVFP4Weight:
    """fp32 [M, K] CUDA tensor -> NVFP4Weight (codes, scales, tensor scale)."""
    M, K = w.shape
    if out is None:
        out = NVFP4Weight(torch.empty(M, K // 2, dtype=torch.uint8, device=w.device),
                          torch.empty(M, K // 16, dtype=torch.uint8, device=w.device),
                          torch.empty(1, dtype=torch.float32, device=w.device))
    ws, ws_bytes = _workspace(NVFP4_OP_QUANTIZE, 0, M, K, w.device, workspace)
    st = load_library().nvfp4_quantize(_ptr(w), M, K, _ptr(out.codes), _ptr(out.scales),
                                       _ptr(out.tensor_scale), _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "nvfp4_quantize")
    return out


def nvfp4_quantize_bf16(w: torch.Tensor, workspace: torch.Tensor | None = None,
                        out: NVFP4Weight | None = None, stream=None) -> NVFP4Weight:
    """bf16 [M, K] CUDA tensor -> NVFP4Weight, identical to quantising w.float()."""
    if w.dtype != torch.bfloat16:
        raise ValueError(f"nvfp4_quantize_bf16 takes bf16 weights, got {w.dtype}")
    M, K = w.shape
    if out is None:
        out = NVFP4Weight(torch.empty(M, K // 2, dtype=torch.uint8, device=w.device),
                          torch.empty(M, K // 16, dtype=torch.uint8, device=w.device),
                          torch.empty(1, dtype=torch.float32, device=w.device))
    ws, ws_bytes = _workspace(NVFP4_OP_QUANTIZE, 0, M, K, w.device, workspace)
    st = load_library().nvfp4_quantize_bf16(_ptr(w), M, K, _ptr(out.codes), _ptr(out.scales),
                                            _ptr(out.tensor_scale), _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "nvfp4_quantize_bf16")
    return out


def nvfp4_blocked_scale_bytes(M: int, K: int) -> int:
    return load_library().nvfp4_blocked_scale_bytes(M, K)


def nvfp4_import_blocked_scales(blocked: torch.Tensor, M: int, K: int,
                                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Blocked (128 x 4) E4M3 scale bytes -> row-major uint8 [M, K/16] scales."""
    if blocked.dtype != torch.uint8:
        raise ValueError(f"blocked scales are uint8 bytes, got {blocked.dtype}")
    if blocked.numel() < nvfp4_blocked_scale_bytes(M, K):
        raise ValueError("blocked scale buffer smaller than nvfp4_blocked_scale_bytes(M, K)")
    if out is None:
        out = torch.empty(M, K // 16, dtype=torch.uint8, device=blocked.device)
    st = load_library().nvfp4_import_blocked_scales(_ptr(blocked), M, K, _ptr(out), _stream(stream))
    _check(st, "nvfp4_import_blocked_scales")
    return out


def _new_out(N, M, dtype, device, out):
    return out if out is not None else torch.empty(N, M, dtype=dtype, device=device)


def nvfp4_gemv_skinny(x: torch.Tensor, W: NVFP4Weight, out_dtype=torch.float32,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """y[N, M] = x[N, K] (bf16) . dequant(W)^T for N = 1..16."""
    N, K = x.shape
    y = _new_out(N, W.M, out_dtype, x.device, out)
    ws, ws_bytes = _workspace(NVFP4_OP_GEMV_SKINNY, N, W.M, K, x.device, workspace)
    st = load_library().nvfp4_gemv_skinny(_ptr(x), N, _ptr(W.codes), _ptr(W.scales), _ptr(W.tensor_scale),
                                          W.M, K, _ptr(y), _out_code(y.dtype), _ptr(ws), ws_bytes,
                                          _stream(stream))
    _check(st, "nvfp4_gemv_skinny")
    return y


def nvfp4_gateup_swiglu(x: torch.Tensor, Wg: NVFP4Weight, Wu: NVFP4Weight, out_dtype=torch.float32,
                        out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """h[N, M] = silu(x . Wg^T) * (x . Wu^T), any N >= 1."""
    N, K = x.shape
    h = _new_out(N, Wg.M, out_dtype, x.device, out)
    ws, ws_bytes = _workspace(NVFP4_OP_GATEUP_SWIGLU, N, Wg.M, K, x.device, workspace)
    st = load_library().nvfp4_gateup_swiglu(_ptr(x), N, _ptr(Wg.codes), _ptr(Wg.scales),
                                            _ptr(Wg.tensor_scale), _ptr(Wu.codes), _ptr(Wu.scales),
                                            _ptr(Wu.tensor_scale), Wg.M, K, _ptr(h), _out_code(h.dtype),
                                            _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "nvfp4_gateup_swiglu")
    return h


def nvfp4_gemm_prefill(x: torch.Tensor, W: NVFP4Weight, out_dtype=torch.float32,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """y[N, M] = x[N, K] (bf16) . dequant(W)^T, any N >= 1 (tensor cores for N > 16)."""
    N, K = x.shape
    y = _new_out(N, W.M, out_dtype, x.device, out)
    ws, ws_bytes = _workspace(NVFP4_OP_GEMM_PREFILL, N, W.M, K, x.device, workspace)
    st = load_library().nvfp4_gemm_prefill(_ptr(x), N, _ptr(W.codes), _ptr(W.scales), _ptr(W.tensor_scale),
                                           W.M, K, _ptr(y), _out_code(y.dtype), _ptr(ws), ws_bytes,
                                           _stream(stream))
    _check(st, "nvfp4_gemm_prefill")
    return y


def nvfp4_device_status(workspace: torch.Tensor, clear: bool = True, stream=None) -> tuple[int, int]:
    """(status, code) of the device status word in a product call's workspace:
    (NVFP4_OK, 0), or (NVFP4_ERR_DEVICE_TIMEOUT, code) when a kernel's bounded
    wait gave up since the word was last cleared.  Synchronises the stream;
    with clear=True a nonzero word is reset."""
    code = ctypes.c_uint32(0)
    st = load_library().nvfp4_device_status(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                            int(bool(clear)), ctypes.byref(code), _stream(stream))
    if st not in (NVFP4_OK, NVFP4_ERR_DEVICE_TIMEOUT):
        raise NVFP4Error(st, "nvfp4_device_status")
    return st, code.value


def nvfp4_selftest_wait_timeout(workspace: torch.Tensor, stream=None) -> None:
    """Enqueue the failure-path self-test: a bounded wait that runs out after
    2 s and records code 127 in the workspace's status word."""
    st = load_library().nvfp4_selftest_wait_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                                    _stream(stream))
    _check(st, "nvfp4_selftest_wait_timeout")


@dataclass
class FP6Weight:
    """One FP6 E2M3 block-scaled tensor W[M][K] in device memory (include/nvfp4.h)."""
    codes: torch.Tensor   # uint8 [M, 3K/4]
    scales: torch.Tensor  # uint8 [M, K/128] (UE8M0)

    @property
    def M(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1] // 6 * 8

    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel()


def _fp6_out(M, K, device, out):
    if out is not None:
        return out
    return FP6Weight(torch.empty(M, K // 8 * 6, dtype=torch.uint8, device=device),
                     torch.empty(M, K // 128, dtype=torch.uint8, device=device))


def nvfp4_fp6_quantize(w: torch.Tensor, out: FP6Weight | None = None, stream=None) -> FP6Weight:
    """fp32 [M, K] CUDA tensor (K % 128 == 0) -> FP6Weight."""
    if w.dtype != torch.float32:
        raise ValueError(f"nvfp4_fp6_quantize takes fp32 weights, got {w.dtype}")
    M, K = w.shape
    out = _fp6_out(M, K, w.device, out)
    st = load_library().nvfp4_fp6_quantize(_ptr(w), M, K, _ptr(out.codes), _ptr(out.scales), _stream(stream))
    _check(st, "nvfp4_fp6_quantize")
    return out


def nvfp4_fp6_quantize_bf16(w: torch.Tensor, out: FP6Weight | None = None, stream=None) -> FP6Weight:
    """bf16 [M, K] CUDA tensor -> FP6Weight, identical to quantising w.float()."""
    if w.dtype != torch.bfloat16:
        raise ValueError(f"nvfp4_fp6_quantize_bf16 takes bf16 weights, got {w.dtype}")
    M, K = w.shape
    out = _fp6_out(M, K, w.device, out)
    st = load_library().nvfp4_fp6_quantize_bf16(_ptr(w), M, K, _ptr(out.codes), _ptr(out.scales),
                                                _stream(stream))
    _check(st, "nvfp4_fp6_quantize_bf16")
    return out


def nvfp4_fp6_gemm(x: torch.Tensor, W: FP6Weight, out_dtype=torch.float32, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[N, M] = x[N, K] (bf16) . dequant(W)^T for FP6 weights, any N >= 1."""
    N, K = x.shape
    y = _new_out(N, W.M, out_dtype, x.device, out)
    ws, ws_bytes = _workspace(NVFP4_OP_FP6_GEMM, N, W.M, K, x.device, workspace)
    st = load_library().nvfp4_fp6_gemm(_ptr(x), N, _ptr(W.codes), _ptr(W.scales), W.M, K, _ptr(y),
                                       _out_code(y.dtype), _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "nvfp4_fp6_gemm")
    return y


def nvfp4_fp6_gateup_swiglu(x: torch.Tensor, Wg: FP6Weight, Wu: FP6Weight, out_dtype=torch.float32,
                            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """h[N, M] = silu(x . Wg^T) * (x . Wu^T) for FP6 weights, any N >= 1."""
    N, K = x.shape
    h = _new_out(N, Wg.M, out_dtype, x.device, out)
    ws, ws_bytes = _workspace(NVFP4_OP_FP6_GATEUP_SWIGLU, N, Wg.M, K, x.device, workspace)
    st = load_library().nvfp4_fp6_gateup_swiglu(_ptr(x), N, _ptr(Wg.codes), _ptr(Wg.scales), _ptr(Wu.codes),
                                                _ptr(Wu.scales), Wg.M, K, _ptr(h), _out_code(h.dtype),
                                                _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "nvfp4_fp6_gateup_swiglu")
    return h


def nvfp4_gemv_skinny_noalloc(x: torch.Tensor, W: NVFP4Weight, out_dtype=torch.float32,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Skinny product whose scratch is the library's fixed device array (for
    callers that cannot allocate device memory; see include/nvfp4.h).  The
    output tensor is the only buffer created here, and only when `out` is None."""
    N, K = x.shape
    y = _new_out(N, W.M, out_dtype, x.device, out)
    st = load_library().nvfp4_gemv_skinny_noalloc(_ptr(x), N, _ptr(W.codes), _ptr(W.scales),
                                                  _ptr(W.tensor_scale), W.M, K, _ptr(y),
                                                  _out_code(y.dtype), _stream(stream))
    _check(st, "nvfp4_gemv_skinny_noalloc")
    return y


def nvfp4_noalloc_status(clear: bool = True, stream=None) -> tuple[int, int]:
    """(status, code) of the status word in the no-allocation array of the
    current device; with clear=True a nonzero word zero-fills the array."""
    code = ctypes.c_uint32(0)
    st = load_library().nvfp4_noalloc_status(int(bool(clear)), ctypes.byref(code), _stream(stream))
    if st not in (NVFP4_OK, NVFP4_ERR_DEVICE_TIMEOUT):
        raise NVFP4Error(st, "nvfp4_noalloc_status")
    return st, code.value


def nvfp4_noalloc_selftest_wait_timeout(stream=None) -> None:
    """Enqueue the bounded-wait self-test against the no-allocation array."""
    _check(load_library().nvfp4_noalloc_selftest_wait_timeout(_stream(stream)),
           "nvfp4_noalloc_selftest_wait_timeout")


# ---------------------------------------------------------------------------
# Product lists in one launch (nvfp4_stream_plan / nvfp4_stream_run)
# ---------------------------------------------------------------------------

@dataclass
class SkinnyJob:
    """One product of a list: y = x . W^T, or silu(x . Wg^T) * (x . Wu^T) when
    W is a (gate, up) pair.  x is a bf16 [N, K] tensor (rows may be strided),
    or None with `input` the index of an earlier job whose bf16 output is x."""
    W: object                       # NVFP4Weight, or (gate, up) NVFP4Weights
    y: torch.Tensor                 # [N, M] float32 or bfloat16
    x: torch.Tensor | None = None
    input: int = -1

    def weights(self):
        return list(self.W) if isinstance(self.W, (tuple, list)) else [self.W]


def _job_structs(jobs):
    arr = (SkinnyJobC * len(jobs))()
    for i, j in enumerate(jobs):
        ws = j.weights()
        c = arr[i]
        if j.x is not None:
            if j.x.dtype != torch.bfloat16 or j.x.stride(1) != 1:
                raise ValueError("job activations must be bf16 with unit stride along K")
            c.x = j.x.data_ptr()
            c.x_ld = j.x.stride(0)
        c.input = int(j.input)
        c.n_weights = len(ws)
        for k, W in enumerate(ws):
            c.codes[k] = W.codes.data_ptr()
            c.scales[k] = W.scales.data_ptr()
            c.tensor_scale[k] = W.tensor_scale.data_ptr()
        c.M = ws[0].M
        c.K = ws[0].K
        c.y = j.y.data_ptr()
        c.out_dtype = _out_code(j.y.dtype)
    return arr


class StreamPlan:
    """A plan buffer (device) and the tensors its jobs point to (kept alive)."""

    def __init__(self, buffer: torch.Tensor, jobs, N: int):
        self.buffer = buffer
        self.jobs = list(jobs)
        self.N = N

    def nbytes(self) -> int:
        return self.buffer.numel()


def nvfp4_stream_plan_bytes(jobs, N: int) -> int:
    arr = _job_structs(jobs)
    return load_library().nvfp4_stream_plan_bytes(arr, len(jobs), int(N))


def nvfp4_stream_plan(jobs, N: int, device=None, stream=None) -> StreamPlan:
    """Build the device plan of a job list (synchronises the stream)."""
    arr = _job_structs(jobs)
    lib = load_library()
    need = lib.nvfp4_stream_plan_bytes(arr, len(jobs), int(N))
    if need == 0:
        raise NVFP4Error(NVFP4_ERR_INVALID_ARG, "nvfp4_stream_plan_bytes")
    dev = device or jobs[0].y.device
    buf = torch.empty(need, dtype=torch.uint8, device=dev)
    st = lib.nvfp4_stream_plan(arr, len(jobs), int(N), _ptr(buf), need, _stream(stream))
    _check(st, "nvfp4_stream_plan")
    return StreamPlan(buf, jobs, int(N))


def nvfp4_stream_run(plan: StreamPlan, stream=None) -> None:
    """Run every job of a plan (one launch, asynchronous)."""
    st = load_library().nvfp4_stream_run(_ptr(plan.buffer), plan.nbytes(), _stream(stream))
    _check(st, "nvfp4_stream_run")

