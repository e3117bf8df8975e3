"""Property checks of the on-disk teacher cache (kd_cache_* in libkd, host
only) on generated files (hypothesis). The fixed cases in test_cache_file.py
check the header layout and the refusals one by one; these check, for any
shape, any split of the appends and any record contents:

* a file reads back bit for bit, whatever float bit patterns the log-probs
  hold (NaNs with payloads, infinities, signed zeros, subnormals): the
  format stores them, it does not interpret them;
* every in-range read [row0, row0 + rows) returns exactly those records, and
  a read that reaches past the end is refused with KD_ERR_INVALID_ARG;
* `batches` covers [start, stop) once, in order, in ranges of the requested
  size (the last one shorter);
* the file size is the 64-byte header plus 8·K bytes per record.
"""

import os

import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from top_kl_loss_tcgen05_b300 import _native  # noqa: E402
from top_kl_loss_tcgen05_b300.cache_file import CacheReader, CacheWriter  # noqa: E402

KD_ERR_INVALID_ARG = 1
SETTINGS = settings(max_examples=40, deadline=None, derandomize=True,
                    suppress_health_check=[HealthCheck.function_scoped_fixture])


@st.composite
def caches(draw):
    """(V, K, ids [T, K] int32 in [0, V), logp [T, K] float32 of arbitrary bit
    patterns, cut points of the appends)."""
    V = draw(st.integers(1, 5000))
    K = draw(st.integers(1, min(V, 64)))
    T = draw(st.integers(0, 300))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, V, size=(T, K), dtype=np.int64).astype(np.int32)
    bits = rng.integers(0, 2**32, size=(T, K), dtype=np.uint64).astype(np.uint32)
    special = np.array([0x7FC00001, 0xFFC12345, 0x7F800000, 0xFF800000, 0x80000000, 0x00000001, 0x3F800000],
                       dtype=np.uint32)
    pick = rng.random(size=(T, K)) < 0.1
    bits[pick] = rng.choice(special, size=int(pick.sum()))
    cuts = sorted(draw(st.lists(st.integers(0, T), max_size=5)))
    return V, K, ids, bits.view(np.float32), cuts


def _write(path, V, K, ids, logp, cuts):
    with CacheWriter(path, V, K) as w:
        prev = 0
        for c in cuts + [ids.shape[0]]:
            w.append(torch.from_numpy(ids[prev:c]), torch.from_numpy(logp[prev:c]))
            prev = c
    return ids.shape[0]


@SETTINGS
@given(caches(), st.data())
def test_any_cache_reads_back_bit_for_bit(tmp_path, c, data):
    V, K, ids, logp, cuts = c
    p = tmp_path / "p.kdtopk"
    T = _write(p, V, K, ids, logp, cuts)
    assert os.path.getsize(p) == 64 + T * K * 8
    with CacheReader(p) as r:
        assert (r.T, r.V, r.K) == (T, V, K)
        i_all, l_all = r.read(0, T)
        assert np.array_equal(i_all.numpy(), ids)
        assert np.array_equal(l_all.numpy().view(np.uint32), logp.view(np.uint32))
        for _ in range(4):
            row0 = data.draw(st.integers(0, T))
            rows = data.draw(st.integers(0, T - row0))
            i2, l2 = r.read(row0, rows)
            assert np.array_equal(i2.numpy(), ids[row0:row0 + rows])
            assert np.array_equal(l2.numpy().view(np.uint32), logp[row0:row0 + rows].view(np.uint32))
        row0 = data.draw(st.integers(0, T))
        with pytest.raises(_native.KDError) as e:
            r.read(row0, T - row0 + 1)
        assert e.value.code == KD_ERR_INVALID_ARG


@SETTINGS
@given(caches(), st.data())
def test_batches_cover_any_range_once_in_order(tmp_path, c, data):
    V, K, ids, logp, cuts = c
    p = tmp_path / "b.kdtopk"
    T = _write(p, V, K, ids, logp, cuts)
    start = data.draw(st.integers(0, T))
    stop = data.draw(st.integers(start, T))
    n = data.draw(st.integers(1, 97))
    with CacheReader(p) as r:
        got = list(r.batches(n, start=start, stop=stop))
    assert [g[0] for g in got] == list(range(start, stop, n))
    assert all(g[1].shape[0] == min(n, stop - g[0]) for g in got)
    if got:
        assert np.array_equal(torch.cat([g[1] for g in got]).numpy(), ids[start:stop])
        assert np.array_equal(torch.cat([g[2] for g in got]).numpy().view(np.uint32),
                              logp[start:stop].view(np.uint32))
    else:
        assert start == stop
