"""fp64 CPU oracle for offline top-K KL distillation.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (the CUDA library and its Python binding) never
calls it, and this module imports nothing from the product package.

It is the plain definition of what the method computes, written out in
float64 with numpy. It applies no chunking, fusion or recompute. The fused
chunked loss only has to reach the same numbers faster. Sources, by page title
and section:

* [KD-TH] "ทำให้ Knowledge Distillation มีประสิทธิภาพ คุ้มค่า และใช้งานได้จริงในระดับ
  Scale ใหญ่" (ai-thai.com):
  - section "การทำ Distillation แบบ Offline" (offline distillation): the
    teacher runs once and the K=100 most probable tokens per position are
    cached.
  - section "กลไก Fused Chunked KL Loss" (the fused chunked KL mechanism):
    the Dense, Forward-chunked and Fused-chunked KL variants compute the same
    loss. Dense KL expands the cached top-100 into a full teacher table and
    compares it with the student's logits over the full vocabulary.
  - section "โมเดลนักเรียนที่ได้" (the resulting student): a closed-form
    gradient of the fused loss exists. The page does not print it; it is
    derived below.
* [KD-RU] "Multiverse Computing сократила видеопамять для дистилляции
  нейросетей до 15,6 раза" (iitog.ru), fourth paragraph: top-100 cache,
  KL loss fused with the final projection, chunk recompute in backward.
* [KD-PT] "Um Novo Método Reduz Drasticamente o Custo de Compressão de
  Grandes Modelos de IA" (ai2day.live), section "O que os investigadores
  alteraram?": KL divergence measures how far the student's predictions are
  from the teacher's.

Readings where the pages are silent:

* KL direction is KL(p_teacher || q_student). It is the only direction that
  stays finite when the teacher has no mass outside its K cached ids.
* The teacher distribution is the K cached log-probs renormalised over K,
  with zero mass elsewhere. The student distribution is its softmax over the
  full vocabulary, not renormalised over K.
* The loss is reduced by the mean over positions. The core has no
  temperature and no padding mask. Two optional variants, which the pages
  leave open, follow the usual distillation conventions:
  - temperature tau: the student distribution is softmax(z / tau) and the
    teacher's is its cached log-probs divided by tau, renormalised over K.
    No tau^2 factor is applied; a caller who wants Hinton's scaling
    multiplies the loss and the gradient scale by tau^2.
  - a position mask: excluded positions add nothing to the loss and get a
    zero gradient; the mean runs over all T positions or over the included
    ones only (mean_over_mask).
* Top-K order is value descending, then id ascending, so ties at the K-th
  place go to the lowest ids. -0.0 and +0.0 tie.
* Duplicate ids in a cache row are separate entries. Their gradient is the
  scatter-add of their probabilities.

Parity pins are in tests/test_oracle.py. Every function here is pinned.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "topk_cache",
    "logsumexp_rows",
    "teacher_probs",
    "student_logits",
    "kl_rows_from_logits",
    "dlogits",
    "fused_kl_forward",
    "fused_kl_backward",
]


def _f64(a) -> np.ndarray:
    """Widen a float array (bf16 already widened to fp32 by the caller) to fp64."""
    return np.asarray(a, dtype=np.float64)


def logsumexp_rows(x: np.ndarray) -> np.ndarray:
    """log(sum_j exp(x[t, j])) per row t, in fp64, shifted by the row max."""
    x = _f64(x)
    m = x.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(x - m).sum(axis=1, keepdims=True)))[:, 0]


def topk_cache(logits, K: int):
    """Teacher logits [T, V] -> (ids int32 [T, K], logp float32 [T, K]).

    The offline cache of [KD-TH] section "การทำ Distillation แบบ Offline" and of
    [KD-RU] fourth paragraph: per position the K most probable token ids and
    their full-vocabulary log-softmax values. Softmax is monotone, so the K
    largest logits are the K most probable tokens.

    Order: value descending, then id ascending. A stable sort of the negated
    row keeps equal values in id order, and -0.0 == +0.0 under comparison.
    logp[t, k] = x[t, id] - logsumexp(x[t, :]) is rounded to float32 once.
    """
    x = _f64(logits)
    if x.ndim != 2:
        raise ValueError("logits must be [T, V]")
    T, V = x.shape
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    ids = np.empty((T, K), dtype=np.int32)
    logp = np.empty((T, K), dtype=np.float32)
    lse = logsumexp_rows(x)
    for t in range(T):
        row = x[t]
        order = np.argsort(-row, kind="stable")[:K]
        ids[t] = order
        logp[t] = (row[order] - lse[t]).astype(np.float32)
    return ids, logp


def teacher_topk_cache(H, W, K: int):
    """The offline cache straight from the teacher's final hidden states H
    [T, d] and LM head W [V, d]: topk_cache of the logits x = H W^T, taken in
    fp64. This is the teacher-side path of [KD-TH] section "การทำ Distillation
    แบบ Offline" (the teacher's projection, then its top-K)."""
    return topk_cache(_f64(H) @ _f64(W).T, K)


def teacher_probs(logp, temperature: float = 1.0):
    """Cached log-probs [T, K] -> (p, log p) renormalised over the K entries.

    p_tk = exp(l_tk - log sum_k' exp(l_tk')). The teacher has zero mass outside
    its K ids: the Dense KL variant builds its full teacher table from the
    cached top-100 alone ([KD-TH] section "กลไก Fused Chunked KL Loss").
    With a temperature, l is replaced by l / tau before the renormalisation.
    """
    l = _f64(logp) / float(temperature)
    lse_k = logsumexp_rows(l)[:, None]
    logp_n = l - lse_k
    return np.exp(logp_n), logp_n


def student_logits(H, W) -> np.ndarray:
    """Student logits z = H W^T in fp64. This is the final projection that the
    fused loss folds into its chunks ([KD-TH] "กลไก Fused Chunked KL Loss":
    hidden states -> logits per chunk). H is [T, d] and W is [V, d]."""
    return _f64(H) @ _f64(W).T


def kl_rows_from_logits(z, ids, logp, temperature: float = 1.0):
    """Per-position loss from student logits z [T, V] and the cache.

    L_t = sum_k p_tk (log p_tk - log q_t,id_tk), where
    log q_tj = z_tj - lse_t and lse_t = log sum_j exp z_tj over the full
    vocabulary. With a temperature, z is replaced by z / tau and p by the
    tempered teacher (teacher_probs). Returns (L [T], lse [T]); lse is that
    of z / tau.
    """
    z = _f64(z) / float(temperature)
    ids = np.asarray(ids, dtype=np.int64)
    T = z.shape[0]
    lse = logsumexp_rows(z)
    p, logp_n = teacher_probs(logp, temperature)
    rows = np.arange(T)[:, None]
    logq_ids = z[rows, ids] - lse[:, None]
    L = (p * (logp_n - logq_ids)).sum(axis=1)
    return L, lse


def dlogits(z, ids, logp, scale: float, temperature: float = 1.0) -> np.ndarray:
    """Closed-form logit gradient, times `scale`.

    d L_t / d z_tj = q_tj - sum_k p_tk [id_tk == j]. Since
    d lse_t / d z_t = q_t and sum_k p_tk = 1, the entropy term drops out.
    With a temperature the chain rule through z / tau adds a factor 1/tau,
    and q, p are the tempered distributions.
    `scale` carries the reduction, e.g. 1/T for the mean over positions.
    Duplicate ids add their probabilities (np.add.at is a scatter-add).
    """
    tau = float(temperature)
    z = _f64(z) / tau
    ids = np.asarray(ids, dtype=np.int64)
    T = z.shape[0]
    lse = logsumexp_rows(z)
    g = np.exp(z - lse[:, None])
    p, _ = teacher_probs(logp, tau)
    rows = np.broadcast_to(np.arange(T)[:, None], ids.shape)
    np.add.at(g, (rows, ids), -p)
    return (scale / tau) * g


def _mask_weights(mask, T):
    if mask is None:
        return np.ones(T)
    m = np.asarray(mask).reshape(-1)
    if m.shape[0] != T:
        raise ValueError("mask must have T entries")
    return (m != 0).astype(np.float64)


def fused_kl_forward(H, W, ids, logp, temperature: float = 1.0, mask=None, mean_over_mask: bool = False):
    """(loss, lse [T], L [T]): the mean over positions of the top-K KL, with the
    student logits taken from the final projection z = H W^T.

    With a mask, excluded positions have L_t = 0 and the mean runs over T
    positions, or over the N included ones if mean_over_mask (loss 0 when
    N = 0). lse is reported for every position."""
    z = student_logits(H, W)
    L, lse = kl_rows_from_logits(z, ids, logp, temperature)
    w = _mask_weights(mask, L.shape[0])
    L = L * w
    n = w.sum() if mean_over_mask else float(L.shape[0])
    return (float(L.sum() / n) if n > 0 else 0.0), lse, L


def fused_kl_backward(H, W, ids, logp, scale: float, rows_per_block: int | None = None, temperature: float = 1.0,
                      mask=None):
    """(dH [T, d], dW [V, d]) for the loss scaled by `scale`.

    With g_t = scale * (q_t - sum_k p_tk e_id_tk):
    dH_t = sum_j g_tj W_j (that is, g W) and dW = sum_t g_t h_t^T (that is,
    g^T H). `rows_per_block` only bounds host memory. Positions are summed
    block by block, and blocking over positions is the sum over t in the
    definition of dW. With a temperature, g is that of dlogits; with a mask,
    g_t = 0 at excluded positions. `scale` is the full per-position factor
    (1/T, or 1/N for the mean over the included positions).
    """
    H64 = _f64(H)
    W64 = _f64(W)
    ids = np.asarray(ids)
    T = H64.shape[0]
    w = _mask_weights(mask, T)
    step = T if rows_per_block is None else max(1, int(rows_per_block))
    dH = np.empty_like(H64)
    dW = np.zeros_like(W64)
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        z = H64[t0:t1] @ W64.T
        g = dlogits(z, ids[t0:t1], np.asarray(logp)[t0:t1], scale, temperature) * w[t0:t1, None]
        dH[t0:t1] = g @ W64
        dW += g.T @ H64[t0:t1]
    return dH, dW
