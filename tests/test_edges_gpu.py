"""Edge cases of the fused loss and the teacher-side cache against the fp64
oracle: one position, K = 1, chunk = 1 and chunk > T, the smallest d, the
largest supported K, and argument errors returned before any launch."""


import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import _native, synth

pytestmark = pytest.mark.gpu

KD_ERR_INVALID_ARG, KD_ERR_UNSUPPORTED, KD_ERR_WORKSPACE = 1, 2, 3


def frob(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def run_all(H, W, ids, logp, chunk):
    """Separate calls and the single call, both against the oracle."""
    T = H.shape[0]
    Hn, Wn = H.float().cpu().numpy(), W.float().cpu().numpy()
    i, lp = ids.cpu().numpy(), logp.cpu().numpy()
    lo, lse_o, L_o = O.fused_kl_forward(Hn, Wn, i, lp)
    dH_o, dW_o = O.fused_kl_backward(Hn, Wn, i, lp, 1.0 / T)
    loss, lse, rows = kd.fused_kl_fwd(H, W, ids, logp, chunk, want_rows=True)
    dH, dW = kd.fused_kl_bwd(H, W, ids, logp, lse, chunk, 1.0 / T)
    l1, lse1, r1, dH1, dW1 = kd.fused_kl_fwdbwd(H, W, ids, logp, chunk, want_rows=True)
    torch.cuda.synchronize()
    for lv, lsev, rv, dHv, dWv in ((loss, lse, rows, dH, dW), (l1, lse1, r1, dH1, dW1)):
        assert abs(lv.item() - lo) <= 1e-3 * abs(lo) + 1e-6
        np.testing.assert_allclose(lsev.cpu().numpy(), lse_o, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(rv.cpu().numpy(), L_o, rtol=1e-3, atol=2e-4)
        assert frob(dHv.cpu().numpy(), dH_o) <= 1e-2
        assert frob(dWv.cpu().numpy(), dW_o) <= 1e-2


def case(T, d, V, K, seed):
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    dev = torch.device("cuda:0")
    return H.to(dev), W.to(dev), ids.to(dev), logp.to(dev)


@pytest.mark.parametrize("T,d,V,K,chunk", [
    (1, 8, 17, 1, 1),          # one position, K = 1, the smallest d
    (5, 64, 300, 3, 1),        # chunk = 1: groups of four positions, the last ragged
    (10, 128, 5000, 1, 4096),  # chunk > T, K = 1
    (64, 256, 8192, 4096, 64), # the largest supported K (block-wide teacher prep)
    (5000, 64, 700, 5, 1365),  # groups of three chunks (4095 positions), the second ragged
    (5000, 64, 700, 5, 4097),  # chunk above 4096: groups of one chunk
])
def test_loss_edges_match_oracle(cuda_dev, T, d, V, K, chunk):
    run_all(*case(T, d, V, K, T * 31 + K), chunk)


def test_teacher_cache_edges(cuda_dev):
    g = torch.Generator().manual_seed(5)
    for T, d, V, K, chunk in ((1, 8, 1, 1, 1), (3, 8, 7, 7, 2), (9, 16, 513, 1, 4)):
        H = torch.randint(-2, 3, (T, d), generator=g).to(torch.bfloat16)
        W = torch.randint(-2, 3, (V, d), generator=g).to(torch.bfloat16)
        ids, logp = kd.teacher_topk_cache(H.to(cuda_dev), W.to(cuda_dev), K, chunk=chunk)
        torch.cuda.synchronize()
        ids_o, logp_o = O.teacher_topk_cache(H.float().numpy(), W.float().numpy(), K)
        assert np.array_equal(ids.cpu().numpy(), ids_o)
        np.testing.assert_allclose(logp.cpu().numpy(), logp_o, rtol=0, atol=1e-4)


def test_argument_errors_return_before_launch(cuda_dev):
    H, W, ids, logp = case(16, 64, 500, 4, 3)
    L = _native.lib()
    st = torch.cuda.current_stream().cuda_stream
    ws = kd.fused_kl_workspace(64, 500, 4, 8, cuda_dev)
    out = torch.empty(16, device=cuda_dev)

    def fwd(T=16, d=64, V=500, K=4, chunk=8, ws_bytes=None, Hp=None):
        return L.kd_fused_kl_fwd(Hp if Hp is not None else H.data_ptr(), W.data_ptr(), ids.data_ptr(),
                                 logp.data_ptr(), T, d, V, K, chunk, out.data_ptr(), out.data_ptr(), None,
                                 ws.data_ptr(), ws.numel() if ws_bytes is None else ws_bytes, st)

    assert fwd(T=0) == KD_ERR_INVALID_ARG            # empty input
    assert fwd(K=501) == KD_ERR_INVALID_ARG          # K > V
    assert fwd(chunk=0) == KD_ERR_INVALID_ARG
    assert fwd(d=60) == KD_ERR_UNSUPPORTED           # rows not 16-byte multiples
    assert fwd(K=4097, V=5000) == KD_ERR_UNSUPPORTED
    assert fwd(Hp=H.data_ptr() + 2) == KD_ERR_UNSUPPORTED  # misaligned H
    assert fwd(ws_bytes=1024) == KD_ERR_WORKSPACE
    assert kd.read_device_status(ws) == 0  # nothing ran
    tws = kd.workspace(256, cuda_dev)
    assert L.kd_teacher_topk_cache(H.data_ptr(), W.data_ptr(), 16, 64, 500, 4, 8, ids.data_ptr(), logp.data_ptr(),
                                   tws.data_ptr(), 256, st) == KD_ERR_WORKSPACE
    assert L.kd_topk_cache(out.data_ptr(), 1, 0, 16, 16, 1, ids.data_ptr(), logp.data_ptr(), tws.data_ptr(), 256,
                           st) == KD_ERR_INVALID_ARG
