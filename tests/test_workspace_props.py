"""Property checks of libkd's workspace queries (host-only C calls, no GPU)
on generated sizes (hypothesis). For every size the calls accept:

* the fused-loss workspace holds at least what its contents need: one
  group's bf16 dz (G·chunk rows of V rounded up to 64) and the transposed
  hidden-state group (d rows of G·chunk rounded up to 64), where G is the
  group (the default rule: 4096 / chunk, clamped to [1, 4]);
* it grows with each of d, V, K, chunk and group and never with T (T is not
  an argument), and group = 0 is the default rule;
* the teacher-cache workspace is the one chunk of fp32 logits plus 8 bytes
  per position and 256-column vocabulary tile that kd.h states, up to the
  header and alignment;
* every size is a multiple of 256 bytes (so a workspace can be carved from
  a larger 256-aligned buffer).
"""

import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from top_kl_loss_tcgen05_b300 import _native  # noqa: E402

SETTINGS = settings(max_examples=200, deadline=None, derandomize=True)


def _up(x, a):
    return (x + a - 1) // a * a


def _group(chunk, group):
    return group if group > 0 else min(4, max(1, 4096 // chunk))


sizes = st.tuples(
    st.integers(1, 2048).map(lambda x: 8 * x),   # d (a multiple of 8)
    st.integers(1, 300000),                     # V
    st.integers(1, 4096),                       # K
    st.integers(1, 8192),                       # chunk
    st.integers(0, 8),                          # group (0 = default)
).filter(lambda s: s[2] <= s[1])


@SETTINGS
@given(sizes)
def test_fused_workspace_holds_its_contents(s):
    d, V, K, chunk, group = s
    f = _native.lib().kd_fused_kl_workspace_size_ex
    n = f(d, V, K, chunk, group)
    G = _group(chunk, group)
    assert n > 0 and n % 256 == 0
    dz = G * chunk * _up(V, 64) * 2
    hct = d * _up(G * chunk, 64) * 2
    parts = 2 * 4 * G * chunk * ((V + 255) // 256)
    assert n >= dz + hct + parts
    if group == 0:
        assert n == _native.lib().kd_fused_kl_workspace_size(d, V, K, chunk)
        assert n == f(d, V, K, chunk, G)


@SETTINGS
@given(sizes, st.sampled_from(["d", "V", "K", "chunk", "group"]), st.integers(1, 5000))
def test_fused_workspace_grows_with_every_size(s, which, step):
    d, V, K, chunk, group = s
    group = max(group, 1)  # an explicit group, so chunk alone moves
    f = _native.lib().kd_fused_kl_workspace_size_ex
    base = f(d, V, K, chunk, group)
    args = dict(d=d, V=V, K=K, chunk=chunk, group=group)
    args[which] += 8 * step if which == "d" else (step % 8 + 1 if which == "group" else step)
    if args["K"] > min(args["V"], 4096) or args["chunk"] * args["group"] > (1 << 24):
        return
    assert f(args["d"], args["V"], args["K"], args["chunk"], args["group"]) >= base


@SETTINGS
@given(st.integers(1, 2048).map(lambda x: 8 * x), st.integers(1, 300000), st.integers(1, 100), st.integers(1, 4096))
def test_teacher_workspace_is_one_chunk_of_logits_and_its_partials(d, V, K, chunk):
    if K > V:
        return
    n = _native.lib().kd_teacher_topk_workspace_size(d, V, K, chunk)
    need = 4 * chunk * _up(V, 64) + 8 * chunk * ((V + 255) // 256)
    assert n % 256 == 0
    assert need <= n <= need + 1024 + 3 * 256
