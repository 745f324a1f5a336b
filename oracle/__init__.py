"""CPU oracle for the NVFP4 weight x bf16 activation path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never imports, links or calls it, and it shares no
code with the CUDA library: the only thing both sides consume is the seeded
synthetic inputs.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C11, single-threaded, fp32
quantiser steps in the order the recipe writes them, fp64 dot products in k
order).  This module compiles it with gcc on first use and wraps it with
ctypes for numpy arrays.

It also covers the ingest helpers (bf16-input quantiser, the blocked 128 x 4
scale layout), the FP6 E2M3 block-scaled variant of the weights, and the W4A4
product (activations quantised to NVFP4 as well).

Pins (tests/test_oracle_pins.py) tie every function here to something other
than itself: brute-force nearest-value searches, PyTorch's float8_e4m3fn
conversions, hand-worked blocks, exact rational arithmetic and closed forms.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

# Strict IEEE fp32/fp64: no contraction into FMA, no fast-math.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libnvfp4_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-shared", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    i64, f32, f64 = ctypes.c_int64, ctypes.c_float, ctypes.c_double
    P = ctypes.c_void_p
    lib.nvfp4_oracle_e2m1_value.restype = f64
    lib.nvfp4_oracle_e2m1_value.argtypes = [ctypes.c_int]
    lib.nvfp4_oracle_e4m3_value.restype = f64
    lib.nvfp4_oracle_e4m3_value.argtypes = [ctypes.c_int]
    lib.nvfp4_oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.nvfp4_oracle_e4m3_encode.argtypes = [f32]
    lib.nvfp4_oracle_e2m1_encode.restype = ctypes.c_uint8
    lib.nvfp4_oracle_e2m1_encode.argtypes = [f32]
    lib.nvfp4_oracle_quantize.restype = ctypes.c_int
    lib.nvfp4_oracle_quantize.argtypes = [P, i64, i64, P, P, P]
    lib.nvfp4_oracle_gemv.restype = None
    lib.nvfp4_oracle_gemv.argtypes = [P, i64, i64, P, i64, P, P, f32,
                                      i64, P, i64, P, P]
    lib.nvfp4_oracle_swiglu.restype = None
    lib.nvfp4_oracle_swiglu.argtypes = [P, i64, i64, P, i64,
                                        P, P, f32, P, P, f32,
                                        i64, P, i64, P, P, P, P, P]
    lib.nvfp4_oracle_e2m3_value.restype = f64
    lib.nvfp4_oracle_e2m3_value.argtypes = [ctypes.c_int]
    lib.nvfp4_oracle_e2m3_encode.restype = ctypes.c_uint8
    lib.nvfp4_oracle_e2m3_encode.argtypes = [f32]
    lib.nvfp4_oracle_fp6_quantize.restype = ctypes.c_int
    lib.nvfp4_oracle_fp6_quantize.argtypes = [P, i64, i64, P, P]
    lib.nvfp4_oracle_fp6_gemv.restype = None
    lib.nvfp4_oracle_fp6_gemv.argtypes = [P, i64, i64, P, i64, P, P, i64, P, i64, P, P]
    lib.nvfp4_oracle_w4a4_gemm.restype = None
    lib.nvfp4_oracle_w4a4_gemm.argtypes = [P, P, f32, i64, i64, P, i64, P, P, f32, i64, P, i64, P, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# --------------------------------------------------------------------------
# Element formats
# --------------------------------------------------------------------------

def e2m1_value(code: int, lib=None) -> float:
    return (lib or _load()).nvfp4_oracle_e2m1_value(int(code))


def e4m3_value(byte: int, lib=None) -> float:
    return (lib or _load()).nvfp4_oracle_e4m3_value(int(byte))


def e4m3_encode(q, lib=None) -> int:
    """fp32 -> E4M3 byte (RNE, saturating at 448)."""
    return int((lib or _load()).nvfp4_oracle_e4m3_encode(float(np.float32(q))))


def e2m1_encode(v, lib=None) -> int:
    """fp32 -> E2M1 code (nearest, ties to even code, clamp 6, sign kept)."""
    return int((lib or _load()).nvfp4_oracle_e2m1_encode(float(np.float32(v))))


# --------------------------------------------------------------------------
# Quantiser and products
# --------------------------------------------------------------------------

def quantize(w, lib=None):
    """fp32 [M, K] -> (codes uint8 [M, K/2], scales uint8 [M, K/16], ts float32)."""
    w = _c(w, np.float32)
    M, K = w.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    rc = (lib or _load()).nvfp4_oracle_quantize(_ptr(w), M, K, _ptr(codes), _ptr(scales), _ptr(ts))
    if rc != 0:
        raise ValueError(f"oracle quantize failed ({rc}): K % 16 != 0 or non-finite weight")
    return codes, scales, np.float32(ts[0])


def quantize_bf16(w_bits, lib=None):
    """bf16 weights (uint16 bit patterns [M, K]) -> NVFP4 with the same recipe.

    The plain definition: every bf16 value is exactly an fp32 value (its bits
    followed by 16 zero bits), and the quantiser recipe then runs on those
    fp32 values unchanged (the ingest step before the path; bw24 README,
    safetensors loader re-encoding weights to NVFP4 at load time).
    """
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    w = (w_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return quantize(w, lib)


# --------------------------------------------------------------------------
# External scale layout (ingest repack)
# --------------------------------------------------------------------------
#
# The pages re-encode NVFP4 checkpoints into each engine's own layout at load
# time (bw24 README, safetensors loader; bw24 wiki Home) without printing the
# source layout.  This library defines one external layout to import: the codes
# as in the canonical layout ([M][K/2], even k in the low nibble) and the
# E4M3 block scales in 128 x 4 blocks, the block arrangement block-scaled
# tensor-core GEMMs read:
#   blocks in row-major order over (M/128 rounded up) x (K/64 rounded up);
#   inside a block, scale (row r, scale column c) at byte
#       (r % 32) * 16 + (r / 32) * 4 + c;
#   padding entries (rows >= M, columns >= K/16) are zero.

def blocked_scale_bytes(M: int, K: int) -> int:
    """Bytes of the external blocked scale buffer."""
    return ((M + 127) // 128) * ((K // 16 + 3) // 4) * 512


def interleave_scales(scales):
    """Canonical scales uint8 [M, K/16] -> external blocked layout (1-D)."""
    scales = np.asarray(scales, dtype=np.uint8)
    M, S = scales.shape
    nb = (S + 3) // 4
    out = np.zeros(((M + 127) // 128) * nb * 512, np.uint8)
    for m in range(M):
        for c in range(S):
            blk = (m // 128) * nb + c // 4
            r, cc = m % 128, c % 4
            out[blk * 512 + (r % 32) * 16 + (r // 32) * 4 + cc] = scales[m, c]
    return out


def deinterleave_scales(blocked, M: int, K: int):
    """External blocked layout -> canonical scales uint8 [M, K/16]."""
    blocked = np.asarray(blocked, dtype=np.uint8).reshape(-1)
    S = K // 16
    nb = (S + 3) // 4
    out = np.zeros((M, S), np.uint8)
    for m in range(M):
        for c in range(S):
            blk = (m // 128) * nb + c // 4
            r, cc = m % 128, c % 4
            out[m, c] = blocked[blk * 512 + (r % 32) * 16 + (r // 32) * 4 + cc]
    return out


def _index(idx, total):
    if idx is None:
        return None, total
    idx = _c(idx, np.int64)
    return idx, len(idx)


def gemv(x_bf16_bits, codes, scales, ts, rows=None, tokens=None, lib=None):
    """y_ref, A (fp64) of shape [n_tokens, n_rows]; x given as uint16 bf16 bits [N, K].

    Pass criterion for a device result y: |y - y_ref| <= 1e-5 * A + 1e-7.
    """
    x = _c(x_bf16_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N, K = x.shape
    M = codes.shape[0]
    assert codes.shape == (M, K // 2) and scales.shape == (M, K // 16)
    r, nr = _index(rows, M)
    t, nt = _index(tokens, N)
    y = np.zeros((nt, nr), np.float64)
    A = np.zeros((nt, nr), np.float64)
    (lib or _load()).nvfp4_oracle_gemv(_ptr(x), N, K, _ptr(t), nt, _ptr(codes), _ptr(scales),
                              float(np.float32(ts)), M, _ptr(r), nr, _ptr(y), _ptr(A))
    return y, A


def swiglu(x_bf16_bits, gate, up, rows=None, tokens=None, lib=None):
    """h_ref, g_ref, u_ref, Ag, Au (fp64) for gate=(codes, scales, ts), up=(...)."""
    x = _c(x_bf16_bits, np.uint16)
    gc, gs, gts = _c(gate[0], np.uint8), _c(gate[1], np.uint8), gate[2]
    uc, us, uts = _c(up[0], np.uint8), _c(up[1], np.uint8), up[2]
    N, K = x.shape
    M = gc.shape[0]
    assert gc.shape == uc.shape == (M, K // 2)
    r, nr = _index(rows, M)
    t, nt = _index(tokens, N)
    outs = [np.zeros((nt, nr), np.float64) for _ in range(5)]
    (lib or _load()).nvfp4_oracle_swiglu(_ptr(x), N, K, _ptr(t), nt,
                                _ptr(gc), _ptr(gs), float(np.float32(gts)),
                                _ptr(uc), _ptr(us), float(np.float32(uts)),
                                M, _ptr(r), nr, *[_ptr(o) for o in outs])
    return tuple(outs)


def dequantize(codes, scales, ts, lib=None):
    """Exact fp64 weights [M, K] (for small pins only)."""
    lib = lib or _load()
    e2 = np.array([lib.nvfp4_oracle_e2m1_value(c) for c in range(16)])
    e4 = np.array([lib.nvfp4_oracle_e4m3_value(b) for b in range(256)])
    codes = np.asarray(codes, np.uint8)
    M, K2 = codes.shape
    K = 2 * K2
    c = np.empty((M, K), np.uint8)
    c[:, 0::2] = codes & 0xF
    c[:, 1::2] = codes >> 4
    s = np.repeat(np.asarray(scales, np.uint8), 16, axis=1)
    return e2[c] * e4[s] * float(np.float32(ts))


# --------------------------------------------------------------------------
# FP6 E2M3 block-scaled variant (128-wide UE8M0 block scales, no tensor scale)
# --------------------------------------------------------------------------

def e2m3_value(code: int, lib=None) -> float:
    return (lib or _load()).nvfp4_oracle_e2m3_value(int(code))


def e2m3_encode(v, lib=None) -> int:
    """fp32 -> E2M3 code (nearest, ties to even code, saturating at 7.5, sign kept)."""
    return int((lib or _load()).nvfp4_oracle_e2m3_encode(float(np.float32(v))))


def fp6_quantize(w, lib=None):
    """fp32 [M, K], K % 128 == 0 -> (codes uint8 [M, 3K/4], scales uint8 [M, K/128])."""
    w = _c(w, np.float32)
    M, K = w.shape
    codes = np.zeros((M, K // 8 * 6), np.uint8)
    scales = np.zeros((M, K // 128), np.uint8)
    rc = (lib or _load()).nvfp4_oracle_fp6_quantize(_ptr(w), M, K, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError(f"oracle fp6_quantize failed ({rc}): K % 128 != 0 or non-finite weight")
    return codes, scales


def fp6_quantize_bf16(w_bits, lib=None):
    """bf16 bits [M, K] -> FP6, quantising the exact fp32 values of the inputs."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    return fp6_quantize((w_bits.astype(np.uint32) << np.uint32(16)).view(np.float32), lib)


def fp6_gemv(x_bf16_bits, codes, scales, rows=None, tokens=None, lib=None):
    """y_ref, A (fp64) [n_tokens, n_rows] for FP6 weights; |y - y_ref| <= 1e-5 A + 1e-7."""
    x = _c(x_bf16_bits, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N, K = x.shape
    M = codes.shape[0]
    assert codes.shape == (M, K // 8 * 6) and scales.shape == (M, K // 128)
    r, nr = _index(rows, M)
    t, nt = _index(tokens, N)
    y = np.zeros((nt, nr), np.float64)
    A = np.zeros((nt, nr), np.float64)
    (lib or _load()).nvfp4_oracle_fp6_gemv(_ptr(x), N, K, _ptr(t), nt, _ptr(codes), _ptr(scales),
                                           M, _ptr(r), nr, _ptr(y), _ptr(A))
    return y, A


def fp6_swiglu(x_bf16_bits, gate, up, rows=None, tokens=None, lib=None):
    """h_ref, g_ref, u_ref, Ag, Au for gate = (codes, scales), up = (codes, scales):
    h = silu(g) * u with silu(g) = g / (1 + exp(-g)), in fp64."""
    g, Ag = fp6_gemv(x_bf16_bits, gate[0], gate[1], rows, tokens, lib)
    u, Au = fp6_gemv(x_bf16_bits, up[0], up[1], rows, tokens, lib)
    return g / (1.0 + np.exp(-g)) * u, g, u, Ag, Au


def fp6_dequantize(codes, scales, lib=None):
    """Exact fp64 FP6 weights [M, K] (for small pins only)."""
    lib = lib or _load()
    e = np.array([lib.nvfp4_oracle_e2m3_value(c) for c in range(64)])
    codes = np.asarray(codes, np.uint8)
    M, nb = codes.shape
    K = nb // 6 * 8
    bits = np.unpackbits(codes, axis=1, bitorder="little").reshape(M, K, 6)
    c = (bits.astype(np.int64) << np.arange(6)).sum(axis=2)
    s = np.repeat(np.asarray(scales, np.int64), 128, axis=1)
    return e[c] * np.exp2(s - 127.0)


def load_variant(path: str):
    """Bind a separately compiled copy of the oracle (used only by the tests
    that plant a mistake in a copy of the oracle source and check that the pins
    catch it)."""
    return _bind(ctypes.CDLL(path))


# --------------------------------------------------------------------------
# W4A4: activations quantised to NVFP4 as well
# --------------------------------------------------------------------------

def quantize_activations(x_bf16_bits, lib=None):
    """bf16 activations [N, K] -> one NVFP4 tensor (codes, scales, ts) by the
    weights' recipe: the matrix is quantised exactly as a bf16 weight matrix."""
    return quantize_bf16(x_bf16_bits, lib)


def w4a4_gemm(xq, wq, rows=None, tokens=None, lib=None):
    """y_ref, A (fp64) [n_tokens, n_rows] of ts_x * ts_w * sum_k dec(x) dec(w)
    for xq = (codes, scales, ts) of the activations [N, K] and wq = (codes,
    scales, ts) of the weights [M, K]; |y - y_ref| <= 1e-5 A + 1e-7."""
    xc, xs = _c(xq[0], np.uint8), _c(xq[1], np.uint8)
    wc, ws = _c(wq[0], np.uint8), _c(wq[1], np.uint8)
    N, K = xc.shape[0], 2 * xc.shape[1]
    M = wc.shape[0]
    assert xs.shape == (N, K // 16) and wc.shape == (M, K // 2) and ws.shape == (M, K // 16)
    r, nr = _index(rows, M)
    t, nt = _index(tokens, N)
    y = np.zeros((nt, nr), np.float64)
    A = np.zeros((nt, nr), np.float64)
    (lib or _load()).nvfp4_oracle_w4a4_gemm(_ptr(xc), _ptr(xs), float(np.float32(xq[2])), N, K, _ptr(t), nt,
                                            _ptr(wc), _ptr(ws), float(np.float32(wq[2])), M, _ptr(r), nr,
                                            _ptr(y), _ptr(A))
    return y, A
