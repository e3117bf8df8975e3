"""The oracle's pins must catch plausible mistakes in the oracle.

Each mutant below is one oracle function with one planted mistake of the
kind that is easy to make when writing the definition down (a dropped term,
a wrong sign or index, a transposed operand, the wrong tie order, a variant
option ignored). The mutant is patched into the oracle module on the CPU,
every pin of tests/test_oracle.py runs against it, and at least one pin must
fail. Nothing here touches the CUDA path.
"""

import functools

import numpy as np
import pytest

import test_oracle as pins
from oracle import kd_oracle as O

_f64 = O._f64


def _all_pins():
    out = []
    for name in sorted(dir(pins)):
        if not name.startswith("test_"):
            continue
        f = getattr(pins, name)
        par = [m for m in getattr(f, "pytestmark", []) if m.name == "parametrize"]
        if par:
            arg, values = par[0].args[0], par[0].args[1]
            out.extend(("%s[%s]" % (name, v), functools.partial(f, **{arg: v})) for v in values)
        else:
            out.append((name, f))
    return out


def _first_failing_pin():
    """Name of the first pin whose check fails. Only a failed check counts:
    any other error means the mutant itself is broken, and it propagates."""
    for name, pin in _all_pins():
        try:
            pin()
        except (AssertionError, pytest.fail.Exception):
            return name
    return None


# ------------------------------------------------------------------ mutants
# Each returns {oracle attribute: replacement}.


def m_lse_counts_the_shift_twice():
    def logsumexp_rows(x):
        x = _f64(x)
        m = x.max(axis=1, keepdims=True)
        return (m + np.log(np.exp(x).sum(axis=1, keepdims=True)))[:, 0]
    return {"logsumexp_rows": logsumexp_rows}


def m_topk_ties_to_highest_id():
    def topk_cache(logits, K):
        x = _f64(logits)
        T, V = x.shape
        if not 1 <= K <= V:
            raise ValueError("need 1 <= K <= V")
        lse = O.logsumexp_rows(x)
        ids = np.empty((T, K), np.int32)
        logp = np.empty((T, K), np.float32)
        for t in range(T):
            order = (V - 1 - np.argsort(-x[t][::-1], kind="stable"))[:K]
            ids[t] = order
            logp[t] = (x[t][order] - lse[t]).astype(np.float32)
        return ids, logp
    return {"topk_cache": topk_cache}


def m_topk_stores_raw_logits():
    orig = O.topk_cache

    def topk_cache(logits, K):
        ids, _ = orig(logits, K)
        x = _f64(logits)
        return ids, np.take_along_axis(x, ids.astype(np.int64), 1).astype(np.float32)
    return {"topk_cache": topk_cache}


def m_teacher_cache_from_permuted_head():
    def teacher_topk_cache(H, W, K):
        return O.topk_cache(_f64(H) @ _f64(W)[::-1].T, K)  # LM-head rows in the wrong order
    return {"teacher_topk_cache": teacher_topk_cache}


def m_teacher_not_renormalised():
    def teacher_probs(logp, temperature=1.0):
        l = _f64(logp) / float(temperature)
        return np.exp(l), l
    return {"teacher_probs": teacher_probs}


def m_teacher_ignores_temperature():
    def teacher_probs(logp, temperature=1.0):
        l = _f64(logp)
        lp = l - O.logsumexp_rows(l)[:, None]
        return np.exp(lp), lp
    return {"teacher_probs": teacher_probs}


def _kl_rows(mistake):
    def kl_rows_from_logits(z, ids, logp, temperature=1.0):
        z = _f64(z) / float(temperature)
        ids = np.asarray(ids, dtype=np.int64)
        rows = np.arange(z.shape[0])[:, None]
        lse = O.logsumexp_rows(z)
        p, logp_n = O.teacher_probs(logp, temperature)
        if mistake == "student_over_K":
            lse_k = O.logsumexp_rows(z[rows, ids])
            return (p * (logp_n - (z[rows, ids] - lse_k[:, None]))).sum(1), lse
        logq = z[rows, ids] - lse[:, None]
        if mistake == "reverse_direction":
            q = np.exp(logq)
            return (q * (logq - logp_n)).sum(1), lse
        if mistake == "entropy_dropped":
            return (-p * logq).sum(1), lse
        if mistake == "wrong_sign_on_q":
            return (p * (logp_n + logq)).sum(1), lse
        raise AssertionError(mistake)
    return {"kl_rows_from_logits": kl_rows_from_logits}


def _dlogits(mistake):
    def dlogits(z, ids, logp, scale, temperature=1.0):
        tau = float(temperature)
        z = _f64(z) / tau
        ids = np.asarray(ids, dtype=np.int64)
        T, V = z.shape
        g = np.exp(z - O.logsumexp_rows(z)[:, None])
        p, _ = O.teacher_probs(logp, tau)
        rows = np.broadcast_to(np.arange(T)[:, None], ids.shape)
        if mistake == "sign":
            np.add.at(g, (rows, ids), p)
        elif mistake == "index":
            np.add.at(g, (rows, (ids + 1) % V), -p)
        elif mistake == "assign_not_add":
            g[rows, ids] -= p  # duplicates overwrite instead of adding
        else:
            np.add.at(g, (rows, ids), -p)
        factor = scale if mistake == "no_chain_factor" else scale / tau
        return factor * g
    return {"dlogits": dlogits}


def _forward(mistake):
    def fused_kl_forward(H, W, ids, logp, temperature=1.0, mask=None, mean_over_mask=False):
        z = O.student_logits(H, W)
        L, lse = O.kl_rows_from_logits(z, ids, logp, temperature)
        w = O._mask_weights(mask, L.shape[0])
        if mistake != "mask_ignored":
            L = L * w
        n = w.sum() if (mean_over_mask and mistake != "mean_always_over_T") else float(L.shape[0])
        if mistake == "sum_not_mean":
            n = 1.0
        return (float(L.sum() / n) if n > 0 else 0.0), lse, L
    return {"fused_kl_forward": fused_kl_forward}


def _backward(mistake):
    def fused_kl_backward(H, W, ids, logp, scale, rows_per_block=None, temperature=1.0, mask=None):
        H64, W64 = _f64(H), _f64(W)
        ids = np.asarray(ids)
        T = H64.shape[0]
        w = O._mask_weights(mask, T)
        step = T if rows_per_block is None else max(1, int(rows_per_block))
        dH = np.empty_like(H64)
        dW = np.zeros_like(W64)
        for t0 in range(0, T, step):
            t1 = min(T, t0 + step)
            z = H64[t0:t1] @ W64.T
            g = O.dlogits(z, ids[t0:t1], np.asarray(logp)[t0:t1], scale, temperature)
            if mistake != "mask_ignored":
                g = g * w[t0:t1, None]
            dH[t0:t1] = g @ (W64[::-1] if mistake == "dH_wrong_rows_of_W" else W64)
            Hb = H64[0:t1 - t0] if mistake == "dW_block_offset" else H64[t0:t1]
            if mistake == "dW_transposed":
                dW += (Hb.T @ g).T[:, ::-1]
            else:
                dW += g.T @ Hb
        return dH, dW
    return {"fused_kl_backward": fused_kl_backward}


MUTANTS = {
    "lse counts the max shift twice": m_lse_counts_the_shift_twice,
    "top-K ties go to the highest id": m_topk_ties_to_highest_id,
    "top-K stores raw logits, not log-softmax": m_topk_stores_raw_logits,
    "teacher cache from a permuted LM head": m_teacher_cache_from_permuted_head,
    "teacher not renormalised over K": m_teacher_not_renormalised,
    "temperature not applied to the teacher": m_teacher_ignores_temperature,
    "student softmax renormalised over K": lambda: _kl_rows("student_over_K"),
    "KL in the reverse direction": lambda: _kl_rows("reverse_direction"),
    "teacher entropy term dropped": lambda: _kl_rows("entropy_dropped"),
    "wrong sign on log q": lambda: _kl_rows("wrong_sign_on_q"),
    "gradient sign of the teacher term": lambda: _dlogits("sign"),
    "gradient scattered one id off": lambda: _dlogits("index"),
    "duplicate ids overwrite instead of adding": lambda: _dlogits("assign_not_add"),
    "1/tau chain factor dropped": lambda: _dlogits("no_chain_factor"),
    "sum over positions instead of the mean": lambda: _forward("sum_not_mean"),
    "mask ignored in the forward": lambda: _forward("mask_ignored"),
    "mean over T despite mean_over_mask": lambda: _forward("mean_always_over_T"),
    "mask ignored in the backward": lambda: _backward("mask_ignored"),
    "dH from the wrong rows of W": lambda: _backward("dH_wrong_rows_of_W"),
    "dW from the wrong block of H": lambda: _backward("dW_block_offset"),
    "dW with a transposed operand": lambda: _backward("dW_transposed"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(monkeypatch, name):
    for attr, fn in MUTANTS[name]().items():
        assert hasattr(O, attr)
        monkeypatch.setattr(O, attr, fn)
    caught = _first_failing_pin()
    assert caught is not None, "no pin fails when the oracle has: %s" % name


def test_pins_pass_on_the_unmodified_oracle():
    assert _first_failing_pin() is None
