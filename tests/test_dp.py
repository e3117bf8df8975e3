"""Position-sharded data parallelism (top_kl_loss_tcgen05_b300/dp.py) on CPU:
two gloo ranks, each with its shard of the positions and the full W. The
per-shard call is the fp64 oracle, injected here (in the test only), so
what is checked is the reduction: the 1 / T_global gradient scale, the sum of
the loss, and the all-reduce of dW. The sharded loss, dH rows and dW must
equal the oracle's on the full T. No GPU is used."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from top_kl_loss_tcgen05_b300 import dp, synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(T, d, V, K, seed):
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    return H.float().numpy().astype(np.float64), W.float().numpy().astype(np.float64), ids.numpy(), logp.numpy()


def oracle_shard_call(H, W, ids, logp, chunk, s):
    """The loss on one shard from the oracle (fp64, CPU tensors in and out).
    Like libkd, it refuses a shard without positions (libkd returns
    KD_ERR_INVALID_ARG for T = 0), so the helper must not make that call."""
    from oracle import kd_oracle as O

    if H.shape[0] == 0:
        raise ValueError("the loss refuses T = 0")

    Hn, Wn = H.numpy(), W.numpy()
    _, _, L = O.fused_kl_forward(Hn, Wn, ids.numpy(), logp.numpy())
    dH, dW = O.fused_kl_backward(Hn, Wn, ids.numpy(), logp.numpy(), s)
    return dp.ShardResult(torch.tensor(float(np.sum(L)), dtype=torch.float64), torch.from_numpy(dH),
                          torch.from_numpy(np.ascontiguousarray(dW)))


def _rank_main(rank, world, port, T, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H, W, ids, logp = _inputs(T, 32, 300, 8, 77)
        t0, t1 = dp.shard_range(T, world, rank)
        loss, dH, dW = dp.dp_fused_kl_step(torch.from_numpy(H[t0:t1]), torch.from_numpy(W),
                                           torch.from_numpy(ids[t0:t1]), torch.from_numpy(logp[t0:t1]), 64, T,
                                           shard_call=oracle_shard_call, grad_scale=2.0)
        q.put((rank, t0, t1, float(loss), dH.numpy(), dW.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T", [200, 201, 1])  # T = 1: rank 1 holds no positions
def test_two_gloo_ranks_reproduce_the_full_batch_loss_and_gradients(T):
    from oracle import kd_oracle as O

    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, T, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    H, W, ids, logp = _inputs(T, 32, 300, 8, 77)
    loss_o, _, _ = O.fused_kl_forward(H, W, ids, logp)
    dH_o, dW_o = O.fused_kl_backward(H, W, ids, logp, 2.0 / T)  # grad_scale 2 on the mean loss
    assert out[0][1] == 0 and out[0][2] == out[1][1] and out[1][2] == T
    for rank, t0, t1, loss, dH, dW in out:
        assert abs(loss - loss_o) <= 1e-6 * abs(loss_o)  # fp32 result of an fp64 sum
        np.testing.assert_allclose(dW, dW_o, rtol=1e-12, atol=1e-15)  # same dW on every rank
        np.testing.assert_allclose(dH, dH_o[t0:t1], rtol=1e-12, atol=1e-15)


def test_shard_ranges_cover_the_positions_once():
    for T in (0, 1, 7, 200, 201, 262144):
        for world in (1, 2, 3, 8):
            spans = [dp.shard_range(T, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        dp.shard_range(10, 2, 2)


def test_single_rank_without_a_process_group_is_the_plain_loss():
    """With no process group the helper is the loss of the one shard."""
    from oracle import kd_oracle as O

    H, W, ids, logp = _inputs(50, 16, 40, 4, 5)
    loss, dH, dW = dp.dp_fused_kl_step(torch.from_numpy(H), torch.from_numpy(W), torch.from_numpy(ids),
                                       torch.from_numpy(logp), 16, 50, shard_call=oracle_shard_call)
    loss_o, _, _ = O.fused_kl_forward(H, W, ids, logp)
    dH_o, dW_o = O.fused_kl_backward(H, W, ids, logp, 1.0 / 50)
    assert abs(float(loss) - loss_o) <= 1e-6 * abs(loss_o)
    np.testing.assert_allclose(dH.numpy(), dH_o, rtol=1e-12)
    np.testing.assert_allclose(dW.numpy(), dW_o, rtol=1e-12)


hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402


@settings(max_examples=25, deadline=None, derandomize=True)
@given(st.integers(1, 12), st.integers(1, 6), st.floats(0.25, 4.0), st.integers(0, 1000))
def test_shards_of_any_split_sum_to_the_full_batch(T, world, gscale, seed):
    """Without a process group each rank's result is its share; summed over
    the ranks (as the all-reduce sums them) the loss and dW are the
    full-batch ones and the dH rows tile the full dH. world > T leaves ranks
    without positions: they contribute zeros."""
    from oracle import kd_oracle as O

    H, W, ids, logp = _inputs(T, 8, 24, 3, seed)
    loss, dW, dH_rows = 0.0, 0.0, []
    for r in range(world):
        t0, t1 = dp.shard_range(T, world, r)
        l, dH, dWr = dp.dp_fused_kl_step(torch.from_numpy(H[t0:t1]), torch.from_numpy(W), torch.from_numpy(ids[t0:t1]),
                                         torch.from_numpy(logp[t0:t1]), 4, T, shard_call=oracle_shard_call,
                                         grad_scale=gscale)
        assert dH.shape == (t1 - t0, 8) and dWr.shape == W.shape
        loss += float(l)
        dW = dW + dWr.numpy()
        dH_rows.append(dH.numpy())
    loss_o, _, _ = O.fused_kl_forward(H, W, ids, logp)
    dH_o, dW_o = O.fused_kl_backward(H, W, ids, logp, gscale / T)
    assert abs(loss - loss_o) <= 1e-6 * abs(loss_o) + 1e-12
    np.testing.assert_allclose(np.concatenate(dH_rows), dH_o, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dW, dW_o, rtol=1e-12, atol=1e-15)


def test_empty_shard_gives_zeros_in_the_loss_precision_without_calling_the_loss():
    """bf16 weights (as libkd takes them): the empty shard's dW is fp32, the
    precision libkd returns dW in, so every rank all-reduces the same dtype."""
    def must_not_run(*a, **k):
        raise AssertionError("the loss was called on an empty shard")

    H = torch.zeros(0, 16, dtype=torch.bfloat16)
    W = torch.randn(40, 16).to(torch.bfloat16)
    ids, logp = torch.zeros(0, 4, dtype=torch.int32), torch.zeros(0, 4)
    loss, dH, dW = dp.dp_fused_kl_step(H, W, ids, logp, 8, 100, shard_call=must_not_run)
    assert float(loss) == 0.0 and dH.shape == (0, 16)
    assert dW.dtype == torch.float32 and dW.shape == (40, 16) and not dW.any()
    with pytest.raises(ValueError):
        dp.dp_fused_kl_step(H, W, ids, logp, 8, 0, shard_call=must_not_run)
