"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol the headers declare, and rejects bad arguments before any CUDA call.
No GPU is needed."""

import ctypes
import os
import re

import pytest

from top_kl_loss_tcgen05_b300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in ("kd.h", "kd_testing.h", "kd_profile.h"):
        with open(os.path.join(ROOT, "include", h)) as f:
            src = f.read()
        names.update(re.findall(r"KD_API[^;(]*?\b(kd_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    return _native.load()


def test_headers_declare_the_three_calls():
    names = _declared_symbols()
    for n in ("kd_topk_cache", "kd_fused_kl_fwd", "kd_fused_kl_bwd", "kd_fused_kl_workspace_size",
              "kd_topk_workspace_size", "kd_read_device_status", "kd_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), n
        assert n in _native.SIGNATURES, n
    # and nothing else is bound by the Python side
    assert set(_native.SIGNATURES) == names


def test_built_for_sm103a():
    assert "arch=compute_103a,code=sm_103a" in build.ARCH
    assert os.path.exists(build.LIB)


def test_status_strings(lib):
    for code, name in [(0, "KD_OK"), (1, "KD_ERR_INVALID_ARG"), (2, "KD_ERR_UNSUPPORTED"), (3, "KD_ERR_WORKSPACE"),
                       (4, "KD_ERR_CUDA"), (5, "KD_ERR_DEVICE_TIMEOUT"), (6, "KD_ERR_BAD_ID"),
                       (7, "KD_ERR_IO"), (8, "KD_ERR_FORMAT")]:
        assert lib.kd_status_string(code).decode() == name
    assert lib.kd_status_string(99).decode() == "KD_ERR_UNKNOWN"
    assert lib.kd_version() >= 100


def test_fused_workspace_is_independent_of_T_and_follows_the_group_rule(lib):
    f = lib.kd_fused_kl_workspace_size
    V = 201088
    # dominated by the bf16 dz of one backward group of G = clamp(4096 / chunk, 1, 4)
    # chunks: G * chunk * V * 2 bytes
    for chunk, G in ((64, 4), (1024, 4), (1500, 2), (2048, 2), (3000, 1), (4096, 1), (8192, 1)):
        n = f(2880, V, 100, chunk)
        dz = G * chunk * V * 2
        assert dz < n < 1.05 * dz + 64 * 2**20, (chunk, n, dz)
        assert n <= 8 * chunk * V + 64 * 2**20
    assert 1.9 < f(2880, V, 100, 128) / f(2880, V, 100, 64) < 2.1
    assert f(0, 10, 1, 1) == 0 and f(8, 0, 1, 1) == 0 and f(8, 10, 0, 1) == 0 and f(8, 10, 1, 0) == 0


# Fake but non-null "device" pointers: every call below must fail in argument
# validation, before anything touches CUDA.
P = ctypes.c_void_p(0x1000)
P16 = ctypes.c_void_p(0x10000)


def test_topk_argument_errors(lib):
    ws = ctypes.c_void_p(0x100000)
    call = lib.kd_topk_cache
    assert call(None, 0, 4, 8, 8, 2, P16, P16, ws, 256, None) == _native.KD_ERR_INVALID_ARG
    assert call(P16, 0, 0, 8, 8, 2, P16, P16, ws, 256, None) == _native.KD_ERR_INVALID_ARG
    assert call(P16, 0, 4, 8, 8, 9, P16, P16, ws, 256, None) == _native.KD_ERR_INVALID_ARG  # K > V
    assert call(P16, 0, 4, 8, 7, 2, P16, P16, ws, 256, None) == _native.KD_ERR_INVALID_ARG  # ld < V
    assert call(P16, 7, 4, 8, 8, 2, P16, P16, ws, 256, None) == _native.KD_ERR_INVALID_ARG  # dtype
    assert call(ctypes.c_void_p(0x1001), 0, 4, 8, 8, 2, P16, P16, ws, 256, None) == _native.KD_ERR_UNSUPPORTED
    assert call(ctypes.c_void_p(0x1002), 1, 4, 8, 8, 2, P16, P16, ws, 256, None) == _native.KD_ERR_UNSUPPORTED
    assert call(P16, 0, 4, 8, 8, 2, P16, P16, None, 256, None) == _native.KD_ERR_WORKSPACE
    assert call(P16, 0, 4, 8, 8, 2, P16, P16, ws, 16, None) == _native.KD_ERR_WORKSPACE
    assert call(P16, 0, 4, 8, 8, 2, P16, P16, ctypes.c_void_p(0x100010), 256, None) == _native.KD_ERR_WORKSPACE


def test_fused_argument_errors(lib):
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 40
    fwd = lib.kd_fused_kl_fwd
    args = dict(H=P16, W=P16, ids=P16, logp=P16, T=64, d=64, V=128, K=4, chunk=32, loss=P16, lse=P16, rows=None,
                ws=ws, wsb=big, s=None)

    def f(**kw):
        a = dict(args)
        a.update(kw)
        return fwd(*a.values())

    assert f(H=None) == _native.KD_ERR_INVALID_ARG
    assert f(T=0) == _native.KD_ERR_INVALID_ARG
    assert f(K=129) == _native.KD_ERR_INVALID_ARG
    assert f(loss=None) == _native.KD_ERR_INVALID_ARG
    assert f(d=60) == _native.KD_ERR_UNSUPPORTED  # d % 8
    assert f(K=4097, V=5000) == _native.KD_ERR_UNSUPPORTED
    assert f(W=ctypes.c_void_p(0x10008)) == _native.KD_ERR_UNSUPPORTED
    assert f(wsb=10) == _native.KD_ERR_WORKSPACE
    assert f(ws=None) == _native.KD_ERR_WORKSPACE
    bwd = lib.kd_fused_kl_bwd
    assert bwd(P16, P16, P16, P16, None, 64, 64, 128, 4, 32, 1.0, None, P16, P16, 0, ws, big, None) == \
        _native.KD_ERR_INVALID_ARG
    # dH or dW may be NULL (that gradient is skipped), not both
    assert bwd(P16, P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, None, None, 0, ws, big, None) == \
        _native.KD_ERR_INVALID_ARG
    assert bwd(P16, P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, ctypes.c_void_p(0x10004), P16, 0, ws,
               big, None) == _native.KD_ERR_UNSUPPORTED
    assert bwd(P16, P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, P16, ctypes.c_void_p(0x10004), 0, ws,
               big, None) == _native.KD_ERR_UNSUPPORTED
    fb = lib.kd_fused_kl_fwdbwd
    assert fb(P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, P16, P16, None, None, None, 0, ws, big, None) == \
        _native.KD_ERR_INVALID_ARG


@pytest.mark.parametrize("tau,over,bf", [(0.0, 0, 0), (-1.0, 0, 0), (float("inf"), 0, 0), (float("nan"), 0, 0),
                                         (1e-45, 0, 0), (1.0, 2, 0), (1.0, 0, -1)])
def test_invalid_loss_options_are_rejected_on_every_call(lib, tau, over, bf):
    """Bad kd_kl_options (tau <= 0, not finite or so small that 1/tau
    overflows; flags outside {0, 1}) come back as KD_ERR_INVALID_ARG from
    all three _ex calls, before anything touches CUDA."""
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 40
    o = ctypes.byref(_native.KLOptions(tau, None, over, bf))
    assert lib.kd_fused_kl_fwd_ex(P16, P16, P16, P16, 64, 64, 128, 4, 32, P16, P16, None, o, ws, big, None) == \
        _native.KD_ERR_INVALID_ARG
    assert lib.kd_fused_kl_bwd_ex(P16, P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, P16, P16, 0, o, ws, big,
                                  None) == _native.KD_ERR_INVALID_ARG
    assert lib.kd_fused_kl_fwdbwd_ex(P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, P16, P16, None, P16, P16, 0,
                                     o, ws, big, None) == _native.KD_ERR_INVALID_ARG


def test_single_call_and_teacher_argument_errors(lib):
    ws = ctypes.c_void_p(0x100000)
    big = 1 << 40
    one = lib.kd_fused_kl_fwdbwd
    assert one(P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, None, P16, None, P16, P16, 0, ws, big, None) == \
        _native.KD_ERR_INVALID_ARG  # no loss output
    assert one(P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, P16, P16, None, ctypes.c_void_p(0x10004), P16, 0,
               ws, big, None) == _native.KD_ERR_UNSUPPORTED  # dH not 16-byte aligned
    t = lib.kd_teacher_topk_cache
    assert t(P16, P16, 0, 64, 128, 4, 32, P16, P16, ws, big, None) == _native.KD_ERR_INVALID_ARG  # T = 0
    assert t(P16, P16, 8, 64, 128, 129, 32, P16, P16, ws, big, None) == _native.KD_ERR_INVALID_ARG  # K > V
    assert t(P16, P16, 8, 60, 128, 4, 32, P16, P16, ws, big, None) == _native.KD_ERR_UNSUPPORTED  # d % 8
    assert t(ctypes.c_void_p(0x10008), P16, 8, 64, 128, 4, 32, P16, P16, ws, big, None) == _native.KD_ERR_UNSUPPORTED
    assert t(P16, P16, 8, 64, 128, 4, 32, P16, P16, None, big, None) == _native.KD_ERR_WORKSPACE
    need = lib.kd_teacher_topk_workspace_size(64, 128, 4, 32)
    assert need > 0
    assert t(P16, P16, 8, 64, 128, 4, 32, P16, P16, ws, need - 1, None) == _native.KD_ERR_WORKSPACE


def test_group_option_sets_the_workspace(lib):
    """kd_fused_kl_workspace_size_ex grows with chunk * group; group = 1 makes
    chunk alone the unit (one chunk's dz), and group = 0 is the default rule."""
    f = lib.kd_fused_kl_workspace_size_ex
    d, V, K = 2880, 201088, 100
    for chunk in (256, 1024, 2048):
        n1 = f(d, V, K, chunk, 1)
        dz1 = chunk * V * 2
        assert dz1 < n1 < 1.05 * dz1 + 64 * 2**20
        for G in (2, 3, 4, 8):
            nG = f(d, V, K, chunk, G)
            assert G * dz1 < nG < 1.05 * G * dz1 + 64 * 2**20, (chunk, G)
        assert f(d, V, K, chunk, 0) == lib.kd_fused_kl_workspace_size(d, V, K, chunk)
    assert 1.9 < f(d, V, K, 2048, 1) / f(d, V, K, 1024, 1) < 2.1
    assert f(d, V, K, 1024, -1) == 0


def test_invalid_group_is_rejected_and_workspace_follows_the_group(lib):
    ws = ctypes.c_void_p(0x100000)
    o_neg = ctypes.byref(_native.KLOptions(1.0, None, 0, 0, -1))
    assert lib.kd_fused_kl_fwd_ex(P16, P16, P16, P16, 64, 64, 128, 4, 32, P16, P16, None, o_neg, ws, 1 << 40,
                                  None) == _native.KD_ERR_INVALID_ARG
    # a workspace sized for group 1 is too small for group 4
    need1 = lib.kd_fused_kl_workspace_size_ex(64, 4096, 4, 256, 1)
    o4 = ctypes.byref(_native.KLOptions(1.0, None, 0, 0, 4))
    assert lib.kd_fused_kl_fwd_ex(P16, P16, P16, P16, 64, 64, 4096, 4, 256, P16, P16, None, o4, ws, need1,
                                  None) == _native.KD_ERR_WORKSPACE
    # group * chunk beyond 2^24 rows per launch
    o_big = ctypes.byref(_native.KLOptions(1.0, None, 0, 0, 1 << 20))
    assert lib.kd_fused_kl_bwd_ex(P16, P16, P16, P16, P16, 64, 64, 128, 4, 32, 1.0, None, P16, P16, 0, o_big, ws,
                                  1 << 40, None) == _native.KD_ERR_UNSUPPORTED


def test_test_switches_are_setters_not_environment(lib, monkeypatch):
    """The tile-shape and exact-selection switches live behind kd_testing.h
    setters; the environment does not change them."""
    a, b = ctypes.c_int32(7), ctypes.c_int32(7)
    monkeypatch.setenv("KD_GEMM_CTA2", "0")
    monkeypatch.setenv("KD_GEMM_WIDE", "1")
    assert lib.kd_test_get_gemm_tiles(ctypes.byref(a), ctypes.byref(b)) == 0
    assert (a.value, b.value) == (-1, -1)
    assert lib.kd_test_set_gemm_tiles(2, 0) == _native.KD_ERR_INVALID_ARG
    assert lib.kd_test_set_gemm_tiles(0, -2) == _native.KD_ERR_INVALID_ARG
    try:
        assert lib.kd_test_set_gemm_tiles(0, 1) == 0
        assert lib.kd_test_get_gemm_tiles(ctypes.byref(a), ctypes.byref(b)) == 0
        assert (a.value, b.value) == (0, 1)
    finally:
        assert lib.kd_test_set_gemm_tiles(-1, -1) == 0
    assert lib.kd_test_set_topk_force_exact(2) == _native.KD_ERR_INVALID_ARG
    assert lib.kd_test_set_topk_force_exact(1) == 0 and lib.kd_test_set_topk_force_exact(0) == 0
    with open(os.path.join(ROOT, "top_kl_loss_tcgen05_b300", "csrc", "kd_api.cu")) as f:
        src = f.read()
    assert re.findall(r'getenv\("([A-Z_]+)"\)', src) == ["KD_DEBUG"]


def test_noalloc_refuses_before_touching_the_stream(lib):
    """kd_topk_cache_noalloc runs kd_topk_cache's checks before anything is
    enqueued: these refusals return without a CUDA call (no GPU here)."""
    call = lib.kd_topk_cache_noalloc
    assert call(ctypes.c_void_p(0x1001), 0, 4, 8, 8, 2, P16, P16, None) == _native.KD_ERR_UNSUPPORTED  # alignment
    assert call(P16, 0, 4, 1 << 31, 1 << 31, 2, P16, P16, None) == _native.KD_ERR_UNSUPPORTED  # V
    assert call(P16, 0, 4, 70000, 70000, 65537, P16, P16, None) == _native.KD_ERR_UNSUPPORTED  # K
    assert call(P16, 0, 4, 8, 8, 9, P16, P16, None) == _native.KD_ERR_INVALID_ARG


def test_workspace_queries_refuse_what_the_calls_refuse(lib):
    """Size queries return 0, not a wrapped-around size, for shapes the calls
    would refuse."""
    f = lib.kd_fused_kl_workspace_size_ex
    assert f(2880, 201088, 100, 4096, 0) > 0
    assert f(2880, 201088, 100, 1 << 25, 0) == 0            # chunk above 2^24
    assert f(2880, 201088, 100, 1 << 20, 64) == 0           # group * chunk above 2^24
    assert f(2880, 201088, 100, 4096, (1 << 31) - 1) == 0   # absurd group
    assert f(2880, 201088, 5000, 4096, 0) == 0              # K > 4096
    assert f(2880, 100, 101, 64, 0) == 0                    # K > V
    assert f(1 << 25, 1000, 10, 64, 0) == 0                 # d above 2^24
    assert lib.kd_fused_kl_workspace_size(2880, 1 << 31, 100, 4096) == 0
    t = lib.kd_teacher_topk_workspace_size
    assert t(4096, 128256, 100, 1024) > 0
    assert t(4096, 128256, 100, 1 << 25) == 0 and t(4096, 100, 101, 64) == 0 and t(4096, 1 << 31, 10, 64) == 0
