"""The teacher top-K cache on disk: a thin binding of libkd's kd_cache_* calls.

The method computes the teacher's top-K once, offline, and reuses it in every
training run ("ทำให้ Knowledge Distillation มีประสิทธิภาพ..." (ai-thai.com),
section "การทำ Distillation แบบ Offline"). The file holds one fixed-size
record per position (K int32 ids, then K float32 log-probs); the format is
specified next to the C declarations in include/kd.h.

    with CacheWriter(path, V, K) as w:
        w.append(ids, logp)              # [rows, K] each, any device
    r = CacheReader(path)
    for row0, ids, logp in r.batches(4096, device="cuda:0"):
        ...                              # ids/logp on the device

The reads run in libkd (pread). ctypes releases the GIL during the call, so
the background read in `batches` overlaps the caller's GPU work.
"""

from __future__ import annotations

import ctypes
import threading

import torch

from . import _native


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise _native.KDError(fn, rc)


def _host(t, dtype) -> torch.Tensor:
    t = torch.as_tensor(t)
    if t.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, t.dtype))
    return t.detach().to("cpu").contiguous()


class CacheWriter:
    """Creates (or truncates) a cache file and appends records to it. The
    row count is written when the writer is closed; a file that was never
    closed is rejected by readers."""

    def __init__(self, path: str, V: int, K: int):
        self._h = ctypes.c_void_p()
        _check("kd_cache_create", _native.lib().kd_cache_create(str(path).encode(), V, K, ctypes.byref(self._h)))
        self.V, self.K, self.rows = V, K, 0

    def append(self, ids, logp) -> None:
        ids = _host(ids, torch.int32)
        logp = _host(logp, torch.float32)
        if ids.dim() != 2 or ids.shape != logp.shape or ids.shape[1] != self.K:
            raise ValueError("ids and logp must both be [rows, %d]" % self.K)
        _check("kd_cache_append",
               _native.lib().kd_cache_append(self._h, ids.data_ptr(), logp.data_ptr(), ids.shape[0]))
        self.rows += ids.shape[0]

    def close(self) -> None:
        if self._h:
            h, self._h = self._h, ctypes.c_void_p()
            _check("kd_cache_close", _native.lib().kd_cache_close(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class CacheReader:
    """Opens a finished cache file; `read` returns any range of positions and
    `batches` streams consecutive ranges with one read ahead."""

    def __init__(self, path: str):
        self._h = ctypes.c_void_p()
        T, V, K = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _check("kd_cache_open", _native.lib().kd_cache_open(str(path).encode(), ctypes.byref(self._h),
                                                            ctypes.byref(T), ctypes.byref(V), ctypes.byref(K)))
        self.T, self.V, self.K = T.value, V.value, K.value

    def read(self, row0: int, rows: int, out=None, pin: bool = False):
        """(ids [rows, K] int32, logp [rows, K] float32) in host memory
        (pinned if `pin`), or into `out` = (ids, logp) host tensors."""
        if out is None:
            ids = torch.empty(rows, self.K, dtype=torch.int32, pin_memory=pin)
            logp = torch.empty(rows, self.K, dtype=torch.float32, pin_memory=pin)
        else:
            ids, logp = out
            if ids.shape[0] < rows or logp.shape[0] < rows or not (ids.is_contiguous() and logp.is_contiguous()):
                raise ValueError("output buffers too small or not contiguous")
        _check("kd_cache_read", _native.lib().kd_cache_read(self._h, row0, rows, ids.data_ptr(), logp.data_ptr()))
        return ids[:rows], logp[:rows]

    def batches(self, rows_per_batch: int, device=None, start: int = 0, stop: int | None = None):
        """Yields (row0, ids, logp) for consecutive ranges of positions in
        [start, stop). The next range is read into pinned memory by a
        background thread while the caller works on the current one. With a
        CUDA `device`, each batch is copied there on the current stream
        (the copy is ordered before any later work on that stream)."""
        stop = self.T if stop is None else min(stop, self.T)
        if rows_per_batch <= 0 or start < 0 or start > stop:
            raise ValueError("bad range")
        dev = torch.device(device) if device is not None else None
        cuda = dev is not None and dev.type == "cuda"
        bufs = [(torch.empty(rows_per_batch, self.K, dtype=torch.int32, pin_memory=cuda),
                 torch.empty(rows_per_batch, self.K, dtype=torch.float32, pin_memory=cuda)) for _ in range(2)]
        done = [None, None]  # CUDA event: the last copy out of buffer b has finished
        ranges = [(r0, min(rows_per_batch, stop - r0)) for r0 in range(start, stop, rows_per_batch)]

        def start_fill(i, b):
            box = []

            def run():
                try:
                    r0, n = ranges[i]
                    self.read(r0, n, out=bufs[b])
                except BaseException as e:  # re-raised in the caller's thread
                    box.append(e)

            th = threading.Thread(target=run, daemon=True)
            th.start()
            return th, box

        pending = start_fill(0, 0) if ranges else None
        try:
            for i, (r0, n) in enumerate(ranges):
                b = i & 1
                th, box = pending
                th.join()
                pending = None
                if box:
                    raise box[0]
                if i + 1 < len(ranges):
                    if done[b ^ 1] is not None:
                        done[b ^ 1].synchronize()  # its last device copy has read the buffer
                    pending = start_fill(i + 1, b ^ 1)
                ids, logp = bufs[b][0][:n], bufs[b][1][:n]
                if cuda:
                    ids = ids.to(dev, non_blocking=True)
                    logp = logp.to(dev, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record()
                    done[b] = ev
                else:
                    ids, logp = ids.clone(), logp.clone()  # the buffer is refilled while the caller holds these
                yield r0, ids, logp
        finally:
            if pending is not None:
                pending[0].join()  # no read may outlive the generator (the handle may be closed next)

    def close(self) -> None:
        if self._h:
            h, self._h = self._h, ctypes.c_void_p()
            _check("kd_cache_close", _native.lib().kd_cache_close(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
