"""The on-disk teacher cache (kd_cache_* in libkd, host only): round trips are
bit-exact, ranges read back what was written, and damaged or unfinished
files are refused. The records written are the oracle's top-K of synthetic
teacher logits, the content a real cache holds."""

import os
import struct

import numpy as np
import pytest
import torch

from oracle import kd_oracle as O
from top_kl_loss_tcgen05_b300 import _native, synth
from top_kl_loss_tcgen05_b300.cache_file import CacheReader, CacheWriter

KD_ERR_INVALID_ARG, KD_ERR_BAD_ID, KD_ERR_IO, KD_ERR_FORMAT = 1, 6, 7, 8


def _cache(T=300, V=1000, K=12, seed=5):
    H, W = synth.student(T, 64, V, seed)
    tl = synth.teacher_logits(H, W, seed)
    ids, logp = O.topk_cache(tl.numpy(), K)
    return torch.from_numpy(ids), torch.from_numpy(logp)


def test_round_trip_is_bit_exact(tmp_path):
    ids, logp = _cache()
    p = tmp_path / "c.kdtopk"
    with CacheWriter(p, 1000, 12) as w:
        w.append(ids[:1], logp[:1])       # appends of several sizes
        w.append(ids[1:200], logp[1:200])
        w.append(ids[200:200], logp[200:200])
        w.append(ids[200:], logp[200:])
    assert os.path.getsize(p) == 64 + 300 * 12 * 8
    with CacheReader(p) as r:
        assert (r.T, r.V, r.K) == (300, 1000, 12)
        i2, l2 = r.read(0, 300)
        assert torch.equal(i2, ids)
        assert torch.equal(l2.view(torch.int32), logp.view(torch.int32))  # bitwise, not just close
        i3, l3 = r.read(137, 41)
        assert torch.equal(i3, ids[137:178]) and torch.equal(l3, logp[137:178])


def test_header_layout(tmp_path):
    ids, logp = _cache(T=3, V=50, K=4)
    p = tmp_path / "h.kdtopk"
    with CacheWriter(p, 50, 4) as w:
        w.append(ids, logp)
    raw = open(p, "rb").read()
    magic, ver, hdr, T, V, K, flags = struct.unpack_from("<8sIIqqiI", raw, 0)
    assert (magic, ver, hdr, T, V, K, flags) == (b"KDTOPK01", 1, 64, 3, 50, 4, 0)
    assert raw[40:64] == bytes(24)
    rec = np.frombuffer(raw[64:64 + 32], dtype="<i4")
    assert np.array_equal(rec[:4], ids[0].numpy())
    assert np.array_equal(rec[4:].view("<f4"), logp[0].numpy())


def test_batches_cover_every_row_in_order(tmp_path):
    ids, logp = _cache(T=257)
    p = tmp_path / "b.kdtopk"
    with CacheWriter(p, 1000, 12) as w:
        w.append(ids, logp)
    with CacheReader(p) as r:
        got = list(r.batches(64))
        assert [g[0] for g in got] == [0, 64, 128, 192, 256]
        assert torch.equal(torch.cat([g[1] for g in got]), ids)
        assert torch.equal(torch.cat([g[2] for g in got]), logp)
        sub = list(r.batches(100, start=50, stop=180))
        assert [(g[0], g[1].shape[0]) for g in sub] == [(50, 100), (150, 30)]
        it = r.batches(16)
        next(it)
        it.close()  # stopping early joins the read in flight


def test_refuses_bad_ids_unfinished_truncated_and_foreign_files(tmp_path):
    ids, logp = _cache(T=20, V=1000, K=12)
    p = tmp_path / "x.kdtopk"
    w = CacheWriter(p, 1000, 12)
    bad = ids.clone()
    bad[3, 5] = 1000
    with pytest.raises(_native.KDError) as e:
        w.append(bad, logp)
    assert e.value.code == KD_ERR_BAD_ID and w.rows == 0
    w.append(ids, logp)
    with pytest.raises(_native.KDError) as e:  # the writer has not closed it yet
        CacheReader(p)
    assert e.value.code == KD_ERR_FORMAT
    w.close()
    with CacheReader(p) as r:
        with pytest.raises(_native.KDError) as e:
            r.read(15, 6)  # past the end
        assert e.value.code == KD_ERR_INVALID_ARG
    raw = open(p, "rb").read()
    t = tmp_path / "t.kdtopk"
    open(t, "wb").write(raw[:-8])
    with pytest.raises(_native.KDError) as e:
        CacheReader(t)
    assert e.value.code == KD_ERR_FORMAT
    f = tmp_path / "f.kdtopk"
    open(f, "wb").write(b"NOTACACH" + raw[8:])
    with pytest.raises(_native.KDError) as e:
        CacheReader(f)
    assert e.value.code == KD_ERR_FORMAT
    with pytest.raises(_native.KDError) as e:
        CacheReader(tmp_path / "missing.kdtopk")
    assert e.value.code == KD_ERR_IO


@pytest.mark.gpu
def test_gpu_cache_to_file_and_back_to_the_device(cuda_dev, tmp_path):
    import top_kl_loss_tcgen05_b300 as kd

    T, V, K = 512, 4096, 16
    H, W = synth.student(T, 128, V, 9)
    tl = synth.teacher_logits(H, W, 9).to(cuda_dev)
    ids, logp = kd.topk_cache(tl, K)
    p = tmp_path / "g.kdtopk"
    with CacheWriter(p, V, K) as w:
        for t0 in range(0, T, 200):
            w.append(ids[t0:t0 + 200], logp[t0:t0 + 200])
    with CacheReader(p) as r:
        parts = list(r.batches(96, device=cuda_dev))
        torch.cuda.synchronize()
    assert all(g[1].device.type == "cuda" for g in parts)
    assert torch.equal(torch.cat([g[1] for g in parts]), ids)
    assert torch.equal(torch.cat([g[2] for g in parts]), logp)


def test_concurrent_reads_on_one_reader(tmp_path):
    """kd_cache_read may run from several threads on one reader (pread, no
    shared file offset): every thread gets exactly its own ranges."""
    import threading

    ids, logp = _cache(T=2000, V=5000, K=24)
    p = tmp_path / "c.kdtopk"
    with CacheWriter(p, 5000, 24) as w:
        w.append(ids, logp)
    errors = []
    with CacheReader(p) as r:
        def worker(seed):
            try:
                g = torch.Generator().manual_seed(seed)
                for _ in range(200):
                    r0 = int(torch.randint(0, 2000, (1,), generator=g))
                    n = int(torch.randint(0, 2000 - r0 + 1, (1,), generator=g))
                    i2, l2 = r.read(r0, n)
                    if not (torch.equal(i2, ids[r0:r0 + n]) and torch.equal(l2, logp[r0:r0 + n])):
                        errors.append((seed, r0, n))
            except BaseException as e:  # reported in the test thread
                errors.append(e)

        threads = [threading.Thread(target=worker, args=(s,)) for s in range(8)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
    assert not errors, errors[:3]
