"""Failure detection without a GPU fault: a device-side wait that runs out.

Every pipeline wait in libkd (TMA stages, TMEM accumulators, tile queue,
top-K) is bounded by wall-clock time; on expiry the kernel records
KD_ERR_DEVICE_TIMEOUT in the workspace status word, unwinds and returns. Here
a kernel waits on an mbarrier that nothing arrives at; the test checks the
status the host reads and that the context is still usable afterwards."""

import time

import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from top_kl_loss_tcgen05_b300 import _native

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_reports_timeout(cuda_dev):
    ws = kd.workspace(256, cuda_dev)
    s = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    assert _native.lib().kd_test_wait_timeout(50_000_000, ws.data_ptr(), s) == 0
    assert kd.read_device_status(ws) == _native.KD_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert kd.read_device_status(ws) == 0  # cleared by the read
    # the context still runs work normally (continuous values: no ties)
    x = torch.randn(4, 1000, device=cuda_dev)
    ids, _ = kd.topk_cache(x, 5)
    torch.cuda.synchronize()
    assert torch.equal(ids.long(), torch.topk(x, 5, dim=1).indices)


def test_timeout_hook_rejects_bad_limits(cuda_dev):
    ws = kd.workspace(256, cuda_dev)
    L = _native.lib()
    assert L.kd_test_wait_timeout(0, ws.data_ptr(), None) == _native.KD_ERR_INVALID_ARG
    assert L.kd_test_wait_timeout(20_000_000_000, ws.data_ptr(), None) == _native.KD_ERR_INVALID_ARG
    assert L.kd_test_wait_timeout(1000, None, None) == _native.KD_ERR_INVALID_ARG
