"""kd_topk_cache against the fp64 oracle: ids bit-exact (value descending,
ties to the lowest id), log-softmax within 1e-4 absolute."""

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import _native, synth
from topk_props import check_topk_rows

pytestmark = pytest.mark.gpu

LOGP_TOL = 1e-4


def _check(logits_dev, K, rows=None, force_exact=False):
    _native.set_topk_force_exact(force_exact)
    try:
        ids, logp = kd.topk_cache(logits_dev, K)
        torch.cuda.synchronize()
    finally:
        _native.set_topk_force_exact(False)
    sel = slice(None) if rows is None else rows
    x = logits_dev[sel].float().cpu().numpy()
    oi, ol = O.topk_cache(x, K)
    gi = ids[sel].cpu().numpy()
    gl = logp[sel].cpu().numpy()
    assert np.array_equal(gi, oi), np.argwhere(gi != oi)[:5]
    assert np.max(np.abs(gl.astype(np.float64) - ol)) <= LOGP_TOL
    return ids, logp


def test_topk_tiny_teacher_fp32(cuda_dev):
    c = synth.CONFIGS["tiny"]
    H, W = synth.student(c["T"], c["d"], c["V"], c["seed"])
    tl = synth.teacher_logits(H, W, c["seed"]).to(cuda_dev)
    _check(tl, c["K"])
    _check(tl, c["K"], force_exact=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topk_heavy_ties_small_ints(cuda_dev, dtype):
    g = torch.Generator().manual_seed(5)
    x = torch.randint(-4, 5, (64, 3001), generator=g).to(dtype)
    x[x == 0] = torch.where(torch.rand(int((x == 0).sum()), generator=g) < 0.5, -0.0, 0.0).to(dtype)
    xd = x.to(cuda_dev)
    for K in (1, 7, 100, 513):
        _check(xd, K)
        _check(xd, K, force_exact=True)


@pytest.mark.parametrize("dtype,V", [(torch.float32, 20011), (torch.bfloat16, 40009)])
def test_topk_rows_with_full_batches(cuda_dev, dtype, V):
    """Rows long enough for full load batches (6 x 256 vectors of 16 bytes:
    6144 fp32 or 12288 bf16 elements), the common case at real vocabulary
    sizes, with a ragged tail; the whole result against the oracle. The
    values are heavy-tailed and rounded to a coarse grid, so the top-K
    boundary has ties."""
    g = torch.Generator().manual_seed(V)
    x = (torch.randn(24, V, generator=g) * 3).round() / 4
    x[3] = 0.0  # one row all ties
    x[5, ::7] = 9.0  # many equal maxima
    _check(x.to(dtype).to(cuda_dev), 100)
    _check(x.to(dtype).to(cuda_dev), 1)


def test_topk_degenerate_rows(cuda_dev):
    V = 1000
    rows = [torch.zeros(V), torch.full((V,), -3.5), torch.arange(V, dtype=torch.float32),
            -torch.arange(V, dtype=torch.float32), torch.where(torch.arange(V) % 2 == 0, -0.0, 0.0)]
    x = torch.stack(rows).to(torch.bfloat16).to(cuda_dev)
    for K in (1, 10, 257, V):
        _check(x, K)


def test_topk_K_equals_V_and_tiny_rows(cuda_dev):
    g = torch.Generator().manual_seed(9)
    for V in (1, 3, 8, 37):
        x = torch.randn(5, V, generator=g).to(cuda_dev)
        _check(x, V)
        _check(x, 1)


def test_topk_unaligned_stride_and_ragged_V(cuda_dev):
    g = torch.Generator().manual_seed(3)
    base = torch.randn(33, 5003, generator=g).to(torch.bfloat16).to(cuda_dev)
    view = base[:, :4999]  # ld = 5003 (rows start at odd 16-byte offsets), V = 4999
    _check(view, 64)
    basef = torch.randn(17, 2051, generator=g).to(cuda_dev)
    _check(basef[:, 3:2050], 20)  # rows start 12 bytes past a 16-byte boundary


def test_topk_large_K_exact_path(cuda_dev):
    g = torch.Generator().manual_seed(4)
    x = torch.randn(6, 9000, generator=g).to(torch.bfloat16).to(cuda_dev)
    _check(x, 1024)  # the largest K of the candidate-buffer path
    _check(x, 1500)  # K > 1024 goes to the radix selection directly
    _check(x, 2500)


def test_topk_full_size_workload_sampled(cuda_dev):
    """The extraction workload at its full size ([8192, 201088] bf16, N(0,2)
    plus a Zipf-like per-row bias). All rows run in one launch, as in the
    bench. The oracle checks 256 rows spread over the matrix, and every row
    passes the exact property check of tests/topk_props.py."""
    c = synth.CONFIGS["topk"]
    x = synth.topk_logits(c["T"], c["V"], c["seed"], device=cuda_dev)
    ws = kd.workspace(256, cuda_dev)
    ids, logp = kd.topk_cache(x, c["K"], ws=ws)
    torch.cuda.synchronize()
    rs = np.random.default_rng(0).choice(c["T"], 256, replace=False)
    xs = x[torch.as_tensor(rs, device=cuda_dev)].float().cpu().numpy()
    oi, ol = O.topk_cache(xs, c["K"])
    assert np.array_equal(ids[torch.as_tensor(rs, device=cuda_dev)].cpu().numpy(), oi)
    assert np.max(np.abs(logp[torch.as_tensor(rs, device=cuda_dev)].cpu().numpy().astype(np.float64) - ol)) <= LOGP_TOL
    # every row: ids distinct and in range, values non-increasing
    ic = ids.long()
    assert int(ic.min()) >= 0 and int(ic.max()) < c["V"]
    vals = torch.gather(x, 1, ic).float()
    assert bool((vals[:, 1:] <= vals[:, :-1]).all())
    srt = torch.sort(ic, dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all())
    fallback_rows = int(ws[4:8].view(torch.int32).item())
    assert fallback_rows < c["T"] // 20  # the radix path is the exception
    check_topk_rows(x, ids, logp, LOGP_TOL)  # all 8192 rows
