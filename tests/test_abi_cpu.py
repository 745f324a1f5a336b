"""C-ABI library checks that need no GPU: it builds, loads, exports every
symbol include/nvfp4.h declares, and rejects bad arguments on the host before
any CUDA call (every case below returns before the library touches the device).
"""
from __future__ import annotations

import ctypes

import pytest

import gemm_nvfp4_gb300 as g
from gemm_nvfp4_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return g.load_library()


def test_exports_every_declared_function(lib):
    names = g.header_functions()
    assert set(names) >= {"nvfp4_quantize", "nvfp4_gemv_skinny", "nvfp4_gateup_swiglu",
                          "nvfp4_gemm_prefill", "nvfp4_workspace_bytes", "nvfp4_status_string"}
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/nvfp4.h but not exported"


def test_exports_nothing_undeclared(lib):
    """Every nvfp4_* function the library exports is declared in the header."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("no nm on this host")
    out = subprocess.run([nm, "-D", "--defined-only", g.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {f[2] for f in (line.split() for line in out.splitlines())
                if len(f) == 3 and f[1] == "T" and f[2].startswith("nvfp4_")}
    assert exported == set(g.header_functions())


def test_python_binding_has_the_c_names():
    for name in g.header_functions():
        assert callable(getattr(g, name)), name


def test_version_and_status_strings(lib):
    assert g.nvfp4_version() >= 100
    for st in range(6):
        assert g.nvfp4_status_string(st).startswith("NVFP4_")
    assert "TIMEOUT" in g.nvfp4_status_string(g.NVFP4_ERR_DEVICE_TIMEOUT)
    assert "unknown" in g.nvfp4_status_string(99)


def test_workspace_bytes(lib):
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_QUANTIZE, 0, 4096, 4096) > 0
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 1, 4096, 4096) > 0
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 17, 4096, 4096) == 0  # rejected N
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 1, 4096, 4100) == 0   # K % 16
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_GATEUP_SWIGLU, 16, 17408, 5120) >= \
        g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 16, 17408, 5120)
    assert g.nvfp4_workspace_bytes(99, 1, 16, 16) == 0
    # independent of the device: same answer twice, no CUDA needed
    a = g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMM_PREFILL, 8192, 17408, 5120)
    assert a == g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMM_PREFILL, 8192, 17408, 5120)


FAKE = 1 << 20  # an aligned address that is never dereferenced (the call fails first)


def _P(v):
    return ctypes.c_void_p(v)


def test_gemv_rejects_bad_arguments(lib):
    ws = g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMV_SKINNY, 4, 64, 64)
    call = lambda **kw: lib.nvfp4_gemv_skinny(
        _P(kw.get("x", FAKE)), kw.get("N", 4), _P(kw.get("codes", FAKE)), _P(kw.get("scales", FAKE)),
        _P(kw.get("ts", FAKE)), kw.get("M", 64), kw.get("K", 64), _P(kw.get("y", FAKE)),
        kw.get("dt", 0), _P(kw.get("ws", FAKE)), kw.get("wsb", ws), None)
    assert call(K=72) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert call(N=17) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert call(N=-1) == binding.NVFP4_ERR_INVALID_ARG
    assert call(M=-5) == binding.NVFP4_ERR_INVALID_ARG
    assert call(x=0) == binding.NVFP4_ERR_INVALID_ARG
    assert call(codes=0) == binding.NVFP4_ERR_INVALID_ARG
    assert call(scales=0) == binding.NVFP4_ERR_INVALID_ARG
    assert call(ts=0) == binding.NVFP4_ERR_INVALID_ARG
    assert call(y=0) == binding.NVFP4_ERR_INVALID_ARG
    assert call(x=FAKE + 2) == binding.NVFP4_ERR_INVALID_ARG      # x not 16-byte aligned
    assert call(codes=FAKE + 8) == binding.NVFP4_ERR_INVALID_ARG  # codes not 16-byte aligned
    assert call(dt=7) == binding.NVFP4_ERR_INVALID_ARG
    assert call(wsb=ws - 1) == binding.NVFP4_ERR_WORKSPACE
    assert call(ws=0) == binding.NVFP4_ERR_INVALID_ARG
    # empty problems are no-ops that touch nothing
    assert call(N=0, x=0, y=0) == binding.NVFP4_OK
    assert call(M=0, codes=0, scales=0, ts=0, y=0) == binding.NVFP4_OK


def test_gateup_and_prefill_reject_bad_arguments(lib):
    ws = g.nvfp4_workspace_bytes(g.NVFP4_OP_GATEUP_SWIGLU, 4, 64, 64)
    st = lib.nvfp4_gateup_swiglu(_P(FAKE), 4, _P(FAKE), _P(FAKE), _P(FAKE), _P(0), _P(FAKE), _P(FAKE),
                                 64, 64, _P(FAKE), 0, _P(FAKE), ws, None)
    assert st == binding.NVFP4_ERR_INVALID_ARG  # null up codes
    st = lib.nvfp4_gateup_swiglu(_P(FAKE), 4, _P(FAKE), _P(FAKE), _P(FAKE), _P(FAKE), _P(FAKE), _P(FAKE),
                                 64, 64, _P(FAKE), 0, _P(FAKE), ws - 1, None)
    assert st == binding.NVFP4_ERR_WORKSPACE
    ws = g.nvfp4_workspace_bytes(g.NVFP4_OP_GEMM_PREFILL, 600, 64, 64)
    st = lib.nvfp4_gemm_prefill(_P(FAKE), 600, _P(FAKE), _P(FAKE), _P(FAKE), 64, 40, _P(FAKE), 0,
                                _P(FAKE), ws, None)
    assert st == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    if ws > 0:
        st = lib.nvfp4_gemm_prefill(_P(FAKE), 600, _P(FAKE), _P(FAKE), _P(FAKE), 64, 64, _P(FAKE), 1,
                                    _P(FAKE), ws - 1, None)
        assert st == binding.NVFP4_ERR_WORKSPACE


def test_quantize_rejects_bad_arguments(lib):
    ws = g.nvfp4_workspace_bytes(g.NVFP4_OP_QUANTIZE, 0, 64, 64)
    q = lambda **kw: lib.nvfp4_quantize(_P(kw.get("w", FAKE)), kw.get("M", 64), kw.get("K", 64),
                                        _P(kw.get("c", FAKE)), _P(kw.get("s", FAKE)), _P(kw.get("ts", FAKE)),
                                        _P(kw.get("ws", FAKE)), kw.get("wsb", ws), None)
    assert q(K=40) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert q(M=-1) == binding.NVFP4_ERR_INVALID_ARG
    assert q(w=0) == binding.NVFP4_ERR_INVALID_ARG
    assert q(w=FAKE + 4) == binding.NVFP4_ERR_INVALID_ARG
    assert q(ts=0) == binding.NVFP4_ERR_INVALID_ARG
    assert q(wsb=ws - 4) == binding.NVFP4_ERR_WORKSPACE


def test_quantize_bf16_rejects_bad_arguments(lib):
    ws = g.nvfp4_workspace_bytes(g.NVFP4_OP_QUANTIZE, 0, 64, 64)
    q = lambda **kw: lib.nvfp4_quantize_bf16(_P(kw.get("w", FAKE)), kw.get("M", 64), kw.get("K", 64),
                                             _P(kw.get("c", FAKE)), _P(kw.get("s", FAKE)), _P(kw.get("ts", FAKE)),
                                             _P(kw.get("ws", FAKE)), kw.get("wsb", ws), None)
    assert q(K=40) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert q(M=-1) == binding.NVFP4_ERR_INVALID_ARG
    assert q(w=0) == binding.NVFP4_ERR_INVALID_ARG
    assert q(w=FAKE + 2) == binding.NVFP4_ERR_INVALID_ARG
    assert q(c=FAKE + 8) == binding.NVFP4_ERR_INVALID_ARG
    assert q(ts=0) == binding.NVFP4_ERR_INVALID_ARG
    assert q(wsb=ws - 4) == binding.NVFP4_ERR_WORKSPACE


def test_blocked_scale_import_arguments(lib):
    assert g.nvfp4_blocked_scale_bytes(130, 128) == 2048
    assert g.nvfp4_blocked_scale_bytes(128, 64) == 512
    assert g.nvfp4_blocked_scale_bytes(1, 16) == 512
    assert g.nvfp4_blocked_scale_bytes(17408, 5120) == 136 * 80 * 512
    assert g.nvfp4_blocked_scale_bytes(16, 24) == 0   # K % 16
    assert g.nvfp4_blocked_scale_bytes(-1, 16) == 0
    imp = lambda **kw: lib.nvfp4_import_blocked_scales(_P(kw.get("b", FAKE)), kw.get("M", 64), kw.get("K", 64),
                                                       _P(kw.get("s", FAKE)), None)
    assert imp(K=40) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert imp(M=-1) == binding.NVFP4_ERR_INVALID_ARG
    assert imp(b=0) == binding.NVFP4_ERR_INVALID_ARG
    assert imp(s=0) == binding.NVFP4_ERR_INVALID_ARG
    assert imp(b=FAKE + 4) == binding.NVFP4_ERR_INVALID_ARG
    assert imp(M=0, b=0, s=0) == binding.NVFP4_OK
    assert imp(K=0, b=0, s=0) == binding.NVFP4_OK


def test_fp6_calls_reject_bad_arguments(lib):
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GEMM, 4, 1024, 1024) > 0
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GEMM, 4, 1024, 1040) == 0   # K % 128
    assert g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GATEUP_SWIGLU, 600, 1024, 1024) > 0
    q = lambda **kw: lib.nvfp4_fp6_quantize(_P(kw.get("w", FAKE)), kw.get("M", 64), kw.get("K", 128),
                                            _P(kw.get("c", FAKE)), _P(kw.get("s", FAKE)), None)
    assert q(K=144) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert q(M=-1) == binding.NVFP4_ERR_INVALID_ARG
    assert q(w=0) == binding.NVFP4_ERR_INVALID_ARG
    assert q(c=FAKE + 4) == binding.NVFP4_ERR_INVALID_ARG
    assert q(M=0, w=0, c=0, s=0) == binding.NVFP4_OK
    assert lib.nvfp4_fp6_quantize_bf16(_P(FAKE), 64, 96, _P(FAKE), _P(FAKE), None) == \
        binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    ws = g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GEMM, 4, 64, 128)
    mm = lambda **kw: lib.nvfp4_fp6_gemm(_P(kw.get("x", FAKE)), kw.get("N", 4), _P(kw.get("c", FAKE)),
                                         _P(kw.get("s", FAKE)), kw.get("M", 64), kw.get("K", 128),
                                         _P(kw.get("y", FAKE)), kw.get("dt", 0), _P(kw.get("ws", FAKE)),
                                         kw.get("wsb", ws), None)
    assert mm(K=144) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert mm(x=0) == binding.NVFP4_ERR_INVALID_ARG
    assert mm(s=FAKE + 1) == binding.NVFP4_ERR_INVALID_ARG
    assert mm(dt=5) == binding.NVFP4_ERR_INVALID_ARG
    assert mm(wsb=ws - 1) == binding.NVFP4_ERR_WORKSPACE
    assert mm(N=0, x=0, y=0) == binding.NVFP4_OK
    st = lib.nvfp4_fp6_gateup_swiglu(_P(FAKE), 4, _P(FAKE), _P(FAKE), _P(0), _P(FAKE), 64, 128, _P(FAKE), 0,
                                     _P(FAKE), g.nvfp4_workspace_bytes(g.NVFP4_OP_FP6_GATEUP_SWIGLU, 4, 64, 128),
                                     None)
    assert st == binding.NVFP4_ERR_INVALID_ARG  # null up codes


def test_status_calls_reject_bad_workspaces(lib):
    """Argument checks of the device-status calls, all before any CUDA call."""
    code = ctypes.c_uint32(7)
    need = binding.NVFP4_STATUS_WORD_OFFSET + 4
    rd = lambda ws, n: lib.nvfp4_device_status(_P(ws), n, 1, ctypes.byref(code), None)
    assert rd(0, 256) == binding.NVFP4_ERR_INVALID_ARG
    assert rd(FAKE + 4, 256) == binding.NVFP4_ERR_INVALID_ARG
    assert rd(FAKE, need - 1) == binding.NVFP4_ERR_INVALID_ARG
    assert code.value == 7  # untouched on a rejected call
    st = lambda ws, n: lib.nvfp4_selftest_wait_timeout(_P(ws), n, None)
    assert st(0, 256) == binding.NVFP4_ERR_INVALID_ARG
    assert st(FAKE + 8, 256) == binding.NVFP4_ERR_INVALID_ARG
    assert st(FAKE, need - 1) == binding.NVFP4_ERR_INVALID_ARG
    # every product workspace holds the status word (the header promises 256 bytes at least)
    for op, N in ((g.NVFP4_OP_GEMV_SKINNY, 1), (g.NVFP4_OP_GATEUP_SWIGLU, 4), (g.NVFP4_OP_GEMM_PREFILL, 600),
                  (g.NVFP4_OP_GATEUP_SWIGLU, 600), (g.NVFP4_OP_FP6_GEMM, 4), (g.NVFP4_OP_FP6_GEMM, 600),
                  (g.NVFP4_OP_FP6_GATEUP_SWIGLU, 1)):
        for M, K in ((64, 128), (4096, 4096), (333, 4112)):
            if op in (g.NVFP4_OP_FP6_GEMM, g.NVFP4_OP_FP6_GATEUP_SWIGLU) and K % 128:
                continue
            assert g.nvfp4_workspace_bytes(op, N, M, K) >= 256 >= need, (op, N, M, K)


def _job(x=FAKE, inp=-1, nw=1, M=256, K=512, out=1, codes=FAKE, y=FAKE, x_ld=0):
    j = binding.SkinnyJobC()
    j.x = x
    j.x_ld = x_ld
    j.input = inp
    j.n_weights = nw
    for k in range(min(nw, 2)):
        j.codes[k] = codes
        j.scales[k] = FAKE
        j.tensor_scale[k] = FAKE
    j.M, j.K, j.y, j.out_dtype = M, K, y, out
    return j


def _arr(*jobs):
    a = (binding.SkinnyJobC * len(jobs))()
    for i, j in enumerate(jobs):
        a[i] = j
    return a


def test_stream_plan_size_and_checks_on_the_host(lib):
    """nvfp4_stream_plan_bytes is host arithmetic; bad lists are refused by it
    and by nvfp4_stream_plan before any CUDA call."""
    size = lambda a, N=4: lib.nvfp4_stream_plan_bytes(a, len(a), N)
    ok = _arr(_job(), _job(inp=0, K=256), _job(nw=2, M=512, K=256, inp=1, out=1), _job(inp=2, M=128, K=512))
    n_ok = size(ok)
    assert n_ok >= 256 and n_ok % 256 == 0
    assert size(ok, N=16) >= n_ok            # more tokens, more statistics items
    assert size(ok, N=0) == 0 and size(ok, N=17) == 0
    bad = [
        _arr(_job(inp=0)),                            # job 0 cannot read an output
        _arr(_job(out=0), _job(inp=0, K=256)),        # input is not bf16
        _arr(_job(M=128), _job(inp=0, K=256)),        # input narrower than K
        _arr(_job(M=260), _job(inp=0, K=256)),        # input row stride not a multiple of 8 elements
        _arr(_job(K=272)),                            # K % 256 != 0
        _arr(_job(nw=3)),
        _arr(_job(out=2)),
        _arr(_job(x=0)),                              # null activations
        _arr(_job(x=FAKE + 8)),                       # misaligned activations
        _arr(_job(codes=FAKE + 4)),                   # misaligned codes
        _arr(_job(y=0)),
        _arr(_job(x_ld=520)),                         # a valid row stride (>= K, multiple of 8)
    ]
    for a in bad[:-1]:
        assert size(a) == 0
    assert size(bad[-1]) > 0                      # 520 is a valid row stride
    assert size(_arr(_job(x_ld=500))) == 0        # a row stride below K
    plan = lambda a, p, n: lib.nvfp4_stream_plan(a, len(a), 4, _P(p), n, None)
    assert plan(ok, FAKE, n_ok - 1) == binding.NVFP4_ERR_WORKSPACE
    assert plan(ok, 0, n_ok) == binding.NVFP4_ERR_INVALID_ARG
    assert plan(ok, FAKE + 16, n_ok) == binding.NVFP4_ERR_INVALID_ARG  # the plan must be 256-byte aligned
    assert plan(bad[0], FAKE, n_ok) == binding.NVFP4_ERR_INVALID_ARG
    assert lib.nvfp4_stream_plan(ok, len(ok), 17, _P(FAKE), n_ok, None) == binding.NVFP4_ERR_UNSUPPORTED_SHAPE
    run = lambda p, n: lib.nvfp4_stream_run(_P(p), n, None)
    assert run(0, n_ok) == binding.NVFP4_ERR_INVALID_ARG
    assert run(FAKE + 16, n_ok) == binding.NVFP4_ERR_INVALID_ARG
    assert run(FAKE, 255) == binding.NVFP4_ERR_INVALID_ARG
