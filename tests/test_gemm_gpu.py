"""The tcgen05 GEMM building block (TMA -> smem -> tcgen05.mma -> TMEM -> TMA
store / reduce-add) against a plain PyTorch fp64 product of the same bf16
operands, for every operand layout the backward pass uses and ragged edges in
M, N and K, with one CTA per 128 x 256 tile and with CTA-pair 256 x 256 tiles
(tcgen05 cta_group::2) both 256 x 256 and 256 x 512 wide."""

import pytest
import torch

from top_kl_loss_tcgen05_b300 import _native, workspace

pytestmark = pytest.mark.gpu


def _run(M, N, K, a_mn, b_mn, reduce_add=False, seed=0, c_trans=False, pair=False, wide=False, n240=False):
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(seed)
    A = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g, device=dev).to(torch.bfloat16)
    Ain = A.t().contiguous() if a_mn else A.contiguous()
    Bin = B.t().contiguous() if b_mn else B.contiguous()
    shape = (N, M) if c_trans else (M, N)
    C0 = torch.randn(*shape, generator=g, device=dev) if reduce_add else torch.full(shape, float("nan"), device=dev)
    C = C0.clone()
    ws = workspace(256, dev)
    flags = (1 if reduce_add else 0) | (2 if c_trans else 0) | (4 if pair else 0) | (8 if wide else 0) | \
        (16 if n240 else 0)
    rc = _native.lib().kd_test_gemm(Ain.data_ptr(), Bin.data_ptr(), C.data_ptr(), M, N, K, a_mn, b_mn,
                                    flags, ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _native.status_string(rc)
    assert _native.lib().kd_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    ref = A.double() @ B.double().t()
    if c_trans:
        ref = ref.t()
    if reduce_add:
        ref = ref + C0.double()
    err = (C.double() - ref).norm() / ref.norm()
    assert torch.isfinite(C).all()
    assert err < 1e-5, err.item()


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_gemm_layouts_exact_tiles(cuda_dev, a_mn, b_mn):
    _run(256, 384, 256, a_mn, b_mn)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
def test_gemm_layouts_ragged(cuda_dev, a_mn, b_mn):
    _run(136, 200, 72, a_mn, b_mn, seed=1)
    _run(1000, 584, 1032, a_mn, b_mn, seed=2)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 1), (1, 1)])
def test_gemm_reduce_add(cuda_dev, a_mn, b_mn):
    _run(520, 392, 200, a_mn, b_mn, reduce_add=True, seed=3)


def test_gemm_many_tiles_persistent(cuda_dev):
    # more tiles than SMs: every CTA loops over several tiles and both TMEM
    # accumulators
    _run(128 * 40, 192 * 9, 128, 0, 1, seed=4)


@pytest.mark.parametrize("a_mn,b_mn", [(1, 0), (0, 0), (1, 1)])
def test_gemm_transposed_store(cuda_dev, a_mn, b_mn):
    _run(264, 1000, 520, a_mn, b_mn, seed=5, c_trans=True)
    _run(3072, 1024, 4096, a_mn, b_mn, seed=6, c_trans=True)


def test_gemm_transposed_reduce_add(cuda_dev):
    _run(136, 520, 64, 1, 0, reduce_add=True, seed=7, c_trans=True)


# CTA-pair tiles (256 x 256, and wide 256 x 512): B is K-major.
@pytest.mark.parametrize("wide", [False, True], ids=["pair", "wide"])
@pytest.mark.parametrize("a_mn", [0, 1])
def test_pair_tiles_layouts(cuda_dev, a_mn, wide):
    _run(256, 512, 256, a_mn, 0, pair=True, wide=wide)
    _run(136, 200, 72, a_mn, 0, seed=1, pair=True, wide=wide)       # one tile, every part ragged
    _run(1000, 584, 1032, a_mn, 0, seed=2, pair=True, wide=wide)    # second N half partly past N
    _run(64, 1000, 128, a_mn, 0, seed=8, pair=True, wide=wide)      # odd CTA's rows all out of range
    _run(296, 248, 64, a_mn, 0, seed=10, pair=True, wide=wide)      # wide: second half entirely past N


@pytest.mark.parametrize("wide", [False, True], ids=["pair", "wide"])
def test_pair_tiles_many_tiles_and_reduce_add(cuda_dev, wide):
    _run(256 * 30, 256 * 11, 192, 0, 0, seed=9, pair=True, wide=wide)   # several tiles per CTA pair
    _run(520, 392, 200, 1, 0, reduce_add=True, seed=3, pair=True, wide=wide)


@pytest.mark.parametrize("wide", [False, True], ids=["pair", "wide"])
@pytest.mark.parametrize("a_mn", [0, 1])
def test_pair_tiles_transposed_store(cuda_dev, a_mn, wide):
    _run(264, 1000, 520, a_mn, 0, seed=5, c_trans=True, pair=True, wide=wide)
    _run(3072, 1024, 4096, a_mn, 0, seed=6, c_trans=True, pair=True, wide=wide)
    _run(136, 520, 64, 1, 0, reduce_add=True, seed=7, c_trans=True, pair=True, wide=wide)


@pytest.mark.parametrize("a_mn", [0, 1])
def test_480_wide_tiles(cuda_dev, a_mn):
    """256 x 480 pair tiles (two N = 240 MMAs, the dW tile at d = 2880): exact
    and ragged N, the 16-column tail box of each half, stores and reduce-adds
    that must not touch the neighbouring tile's columns."""
    _run(256, 480, 128, a_mn, 0, pair=True, wide=True, n240=True)
    _run(512, 2880, 256, a_mn, 0, seed=11, pair=True, wide=True, n240=True)              # the dW width
    _run(1000, 2880, 200, a_mn, 0, seed=12, reduce_add=True, pair=True, wide=True, n240=True)
    _run(296, 1000, 72, a_mn, 0, seed=13, pair=True, wide=True, n240=True)               # ragged N: 480 + 480 + 40
    _run(136, 232, 64, a_mn, 0, seed=14, pair=True, wide=True, n240=True)                # one half, ends mid-tail
    _run(256 * 20, 480 * 6, 320, a_mn, 0, seed=15, reduce_add=True, pair=True, wide=True, n240=True)


def test_480_wide_tiles_refused_outside_wide_pairs(cuda_dev):
    dev = torch.device("cuda:0")
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(64, 64, device=dev)
    ws = workspace(256, dev)
    for flags in (16, 16 | 4, 16 | 4 | 8 | 2):
        rc = _native.lib().kd_test_gemm(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64, 0, 0, flags,
                                        ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 2  # KD_ERR_UNSUPPORTED, nothing launched


def test_pair_tiles_reject_n_major_b(cuda_dev):
    dev = torch.device("cuda:0")
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(64, 64, device=dev)
    ws = workspace(256, dev)
    for flags in (4, 12):
        rc = _native.lib().kd_test_gemm(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64, 0, 1, flags,
                                        ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 2  # KD_ERR_UNSUPPORTED, nothing launched
