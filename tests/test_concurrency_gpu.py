"""Calls on distinct workspaces may run at the same time (include/kd.h):
two host threads, each on its own stream and workspace, run the loss
(forward, backward and the single call) and the top-K cache on different
inputs at once. Every result must equal, bit for bit, the same call run
alone."""

import threading

import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from top_kl_loss_tcgen05_b300 import synth

pytestmark = pytest.mark.gpu


def _case(dev, seed, T=700, d=264, V=3000, K=24, chunk=128):
    H, W = synth.student(T, d, V, seed)
    ids, logp = synth.synthetic_cache(T, V, K, seed + 1)
    logits = synth.topk_logits(T // 4, V, seed + 2)
    return dict(H=H.to(dev), W=W.to(dev), ids=ids.to(dev), logp=logp.to(dev), logits=logits.to(dev), chunk=chunk,
                ws=kd.fused_kl_workspace(d, V, K, chunk, dev))


def _run(c, reps=1):
    T = c["H"].shape[0]
    out = None
    for _ in range(reps):
        loss, lse, rows = kd.fused_kl_fwd(c["H"], c["W"], c["ids"], c["logp"], c["chunk"], ws=c["ws"], want_rows=True)
        dH, dW = kd.fused_kl_bwd(c["H"], c["W"], c["ids"], c["logp"], lse, c["chunk"], 1.0 / T, ws=c["ws"])
        l1, lse1, r1, dH1, dW1 = kd.fused_kl_fwdbwd(c["H"], c["W"], c["ids"], c["logp"], c["chunk"], ws=c["ws"],
                                                   want_rows=True)
        tid, tlp = kd.topk_cache(c["logits"], 50)
        out = [loss, lse, rows, dH, dW, l1, lse1, r1, dH1, dW1, tid, tlp]
    return out


def test_two_threads_two_streams_match_sequential(cuda_dev):
    cases = [_case(cuda_dev, 100), _case(cuda_dev, 200)]
    ref = []
    for c in cases:
        r = _run(c)
        torch.cuda.synchronize()
        ref.append([t.clone() for t in r])
        assert kd.read_device_status(c["ws"]) == 0

    results = [None, None]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream(device=cuda_dev)
            with torch.cuda.stream(s):
                r = _run(cases[i], reps=3)  # repeated so that the two streams overlap
                s.synchronize()
                results[i] = [t.clone() for t in r]
        except BaseException as e:  # re-raised in the test thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert kd.read_device_status(cases[i]["ws"]) == 0
        for a, b in zip(results[i], ref[i]):
            assert torch.equal(a, b)
