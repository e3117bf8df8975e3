"""kd_topk_cache_noalloc: top-K cache extraction for callers that cannot
allocate device memory (no workspace argument; the scratch is a fixed array
inside libkd). It must give what kd_topk_cache gives with a caller-provided
workspace, on two calls in a row (the second call reuses the array the first
one left behind). Runs through the C ABI."""

import numpy as np
import pytest
import torch

import top_kl_loss_tcgen05_b300 as kd
from top_kl_loss_tcgen05_b300 import _native, synth

pytestmark = pytest.mark.gpu


def _noalloc(x, K):
    T, V = x.shape
    ids = torch.empty(T, K, dtype=torch.int32, device=x.device)
    logp = torch.empty(T, K, dtype=torch.float32, device=x.device)
    dt = _native.KD_BF16 if x.dtype == torch.bfloat16 else _native.KD_F32
    rc = _native.lib().kd_topk_cache_noalloc(x.data_ptr(), dt, T, V, x.stride(0), K, ids.data_ptr(),
                                             logp.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _native.status_string(rc)
    torch.cuda.synchronize()
    return ids, logp


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_dev):
    c = synth.CONFIGS["topk"]
    # two different inputs, back to back: Zipf-biased bf16 rows, then fp32 rows with ties
    a = synth.topk_logits(c["T"], c["V"], c["seed"], device=cuda_dev, rows=512)
    g = torch.Generator().manual_seed(21)
    b = torch.randint(-6, 7, (300, 7001), generator=g).to(torch.float32).to(cuda_dev)
    for x, K in ((a, c["K"]), (b, 37)):
        ids_n, logp_n = _noalloc(x, K)
        ids_w, logp_w = kd.topk_cache(x, K)
        torch.cuda.synchronize()
        assert torch.equal(ids_n, ids_w)
        assert float((logp_n - logp_w).abs().max()) <= 1e-4


def test_noalloc_allocates_no_device_memory(cuda_dev):
    """After the first call on the device (which looks up the array's
    address), further calls leave the device's free memory unchanged: the
    entry point allocates nothing, and neither does anything it calls."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(256, 5000, generator=g).to(torch.bfloat16).to(cuda_dev)
    ids = torch.empty(256, 20, dtype=torch.int32, device=cuda_dev)
    logp = torch.empty(256, 20, dtype=torch.float32, device=cuda_dev)
    L = _native.lib()
    s = torch.cuda.current_stream().cuda_stream

    def call():
        rc = L.kd_topk_cache_noalloc(x.data_ptr(), _native.KD_BF16, 256, 5000, 5000, 20, ids.data_ptr(),
                                     logp.data_ptr(), s)
        assert rc == 0, _native.status_string(rc)

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    ids_w, _ = kd.topk_cache(x, 20)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_w)


def test_noalloc_rejects_bad_arguments(cuda_dev):
    L = _native.lib()
    assert L.kd_topk_cache_noalloc(None, 0, 4, 8, 8, 2, None, None, None) == _native.KD_ERR_INVALID_ARG
    x = torch.zeros(4, 8, device=cuda_dev)
    out = torch.empty(4, 9, dtype=torch.int32, device=cuda_dev)
    assert L.kd_topk_cache_noalloc(x.data_ptr(), 1, 4, 8, 8, 9, out.data_ptr(), out.data_ptr(), None) == \
        _native.KD_ERR_INVALID_ARG
