"""Seeded synthetic workloads shared by the tests, the bench and the smoke run.

This module only draws random numbers and builds input tensors. It holds no
step of the method: no softmax, no top-K selection and no KL. Both the CUDA
path and the oracle take their inputs from here.

Workloads (sizes from the pages' settings):

* Student: H ~ N(0, 1) [T, d] and W ~ N(0, 1/d) [V, d], both bf16. The
  second argument of N is the variance, so each logit H W^T has unit variance.
* Teacher logits (perturbed-W teacher): 1.5 * H (W + E)^T with
  E ~ N(0, 0.5/d), in fp32.
* Top-K extraction logits: N(0, 2) plus a Zipf-like per-row bias
  b_t[v] = -log(1 + ((v + o_t) mod V)), where o_t is uniform per row. Stored
  as bf16.
* Teacher head (teacher-side cache): H ~ N(0, 1) [T, d] and W ~ N(0, 3.375/d)
  [V, d], both bf16, so each logit has variance 3.375 = 1.5^2 * (1 + 0.5), the
  variance of the perturbed-W teacher logits above.
* Synthetic cache: K distinct ids per row, (a_t + k * b_t) mod V with
  gcd(b_t, V) = 1, and log-probs that are a descending N(0, 2) sample shifted
  down by log V. The loss renormalises them over K.
"""

from __future__ import annotations

import math

import torch

__all__ = [
    "CONFIGS",
    "student",
    "teacher_weight",
    "teacher_logits_from",
    "teacher_logits",
    "topk_logits",
    "teacher_head",
    "synthetic_cache",
]

# (T, d, V, K, chunk) per workload, by name. "tiny" is small enough for the
# full oracle; "llama3b", "gptoss20b" and "long" are the projection shapes of
# Llama-3.2-3B (d=3072, V=128256) and GPT-OSS-20B (d=2880, V=201088); "topk" is
# the cache-extraction workload (T=8192 rows of V=201088 teacher logits).
CONFIGS = {
    "tiny": dict(T=256, d=256, V=4096, K=16, chunk=64, seed=1000),
    "llama3b": dict(T=8192, d=3072, V=128256, K=100, chunk=1024, seed=1001),
    "gptoss20b": dict(T=32768, d=2880, V=201088, K=100, chunk=2048, seed=1002),
    "long": dict(T=262144, d=2880, V=201088, K=100, chunk=4096, seed=1003),
    "topk": dict(T=8192, V=201088, K=100, seed=1004),
    # teacher-side cache straight from a Llama-3.1-8B-shaped LM head
    "teacher": dict(T=8192, d=4096, V=128256, K=100, chunk=1024, seed=1005),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def student(T: int, d: int, V: int, seed: int, device="cpu"):
    """H [T, d] ~ N(0, 1) and W [V, d] ~ N(0, 1/d), drawn in fp32 then rounded to bf16."""
    g = _gen(seed, device)
    H = torch.randn(T, d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=device, dtype=torch.float32) * (1.0 / math.sqrt(d))).to(
        torch.bfloat16
    )
    return H, W


def teacher_head(T: int, d: int, V: int, seed: int, device="cpu"):
    """Teacher final hidden states H [T, d] ~ N(0, 1) and LM head W [V, d] ~
    N(0, 3.375/d), drawn in fp32 then rounded to bf16."""
    g = _gen(seed, device)
    H = torch.randn(T, d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=device, dtype=torch.float32) * math.sqrt(3.375 / d)).to(
        torch.bfloat16
    )
    return H, W


def teacher_weight(W: torch.Tensor, seed: int) -> torch.Tensor:
    """fp32 perturbed teacher projection W + E with E ~ N(0, 0.5/d)."""
    V, d = W.shape
    g = _gen(seed + 7919, W.device)
    E = torch.randn(V, d, generator=g, device=W.device, dtype=torch.float32) * math.sqrt(0.5 / d)
    return W.float() + E


def teacher_logits_from(Hs: torch.Tensor, Wt: torch.Tensor) -> torch.Tensor:
    """fp32 teacher logits 1.5 * Hs Wt^T for a block of positions."""
    with _no_tf32():
        return 1.5 * (Hs.float() @ Wt.T)


def teacher_logits(H: torch.Tensor, W: torch.Tensor, seed: int, rows: slice | None = None):
    """fp32 teacher logits 1.5 * H (W + E)^T with E ~ N(0, 0.5/d).

    E is drawn for the whole of W from `seed`, so the same teacher serves
    every row. `rows` restricts the output to those positions.
    """
    Hs = H if rows is None else H[rows]
    return teacher_logits_from(Hs, teacher_weight(W, seed))


class _no_tf32:
    """Keep fp32 matmuls in full fp32 while generating teacher logits."""

    def __enter__(self):
        self.prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False

    def __exit__(self, *exc):
        torch.backends.cuda.matmul.allow_tf32 = self.prev
        return False


def topk_logits(T: int, V: int, seed: int, device="cpu", row0: int = 0, rows: int | None = None):
    """bf16 [rows, V] teacher logits: N(0, 2) plus a per-row Zipf-like bias.

    The bias is -log(1 + ((v + o_t) mod V)), with o_t drawn uniformly per row.
    `row0`/`rows` give a slice of the full [T, V] matrix. Rows are drawn in
    blocks of 256, each from a generator seeded by (seed, first row of the
    block), so a slice that starts on a block boundary and ends on one (or at
    T) holds the same values as that part of the full draw. Within a block
    the per-row offsets are drawn after the noise, so a slice that ends
    inside a block gets other offsets for its last rows.
    """
    if row0 % 256:
        raise ValueError("row0 must be a multiple of 256")
    rows = T - row0 if rows is None else rows
    out = torch.empty(rows, V, dtype=torch.bfloat16, device=device)
    v = torch.arange(V, device=device, dtype=torch.float64)
    blk = 256
    for r0 in range(0, rows, blk):
        r1 = min(rows, r0 + blk)
        g = _gen(seed * 1000003 + row0 + r0, device)
        noise = torch.randn(r1 - r0, V, generator=g, device=device, dtype=torch.float32) * math.sqrt(2.0)
        off = torch.randint(0, V, (r1 - r0, 1), generator=g, device=device).to(torch.float64)
        bias = -torch.log1p(torch.remainder(v[None, :] + off, V))
        out[r0:r1] = (noise.double() + bias).to(torch.bfloat16)
    return out


def synthetic_cache(T: int, V: int, K: int, seed: int, device="cpu"):
    """(ids int32 [T, K], logp float32 [T, K]) with K distinct ids per row.

    ids_tk = (a_t + k * b_t) mod V, where b_t is coprime with V, so the K ids
    of a row are distinct. logp is a descending N(0, 2) sample minus log V.
    """
    if K > V:
        raise ValueError("K > V")
    g = _gen(seed + 104729, "cpu")
    a = torch.randint(0, V, (T,), generator=g, dtype=torch.int64)
    b = torch.randint(1, max(2, V), (T,), generator=g, dtype=torch.int64)
    bl = b.tolist()
    for i, x in enumerate(bl):
        while math.gcd(int(x), V) != 1:
            x = (x + 1) % V or 1
        bl[i] = x
    b = torch.tensor(bl, dtype=torch.int64)
    k = torch.arange(K, dtype=torch.int64)
    ids = torch.remainder(a[:, None] + k[None, :] * b[:, None], V).to(torch.int32)
    vals = torch.randn(T, K, generator=g, dtype=torch.float32) * math.sqrt(2.0)
    logp = torch.sort(vals, dim=1, descending=True).values - math.log(V)
    return ids.to(device), logp.to(device)
