"""The online-softmax rescale rule with a lazily moved reference (CPU).

The decode kernel's 16-bit stages and the tcgen05 kernel keep, per query row,
a reference m that moves to the running maximum only when a stage's scores
exceed it by more than 2^8 ([vllm-06] 2.2.2, the m / l rescale of the online
softmax, applied lazily).  These tests run that rule in fp64 on score
sequences built to cross the threshold in known ways and compare the result
with the oracle's attention on the same inputs: the output and the
log-sum-exp do not depend on which reference was kept, and every exponential
stays at most 2^8.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import bits

LAZY_LOG2 = 8.0
STAGE = 16


def lazy_online_softmax(s2: np.ndarray, v: np.ndarray):
    """One query row: base-2 scores s2 [n], values v [n, d], streamed in stages
    of 16 tokens.  Returns (O / l, lse in natural log, largest e^(s - m) seen,
    number of reference moves)."""
    m, l = -math.inf, 0.0
    o = np.zeros(v.shape[1])
    top, moves = 0.0, 0
    for t0 in range(0, len(s2), STAGE):
        s = s2[t0:t0 + STAGE]
        mx = float(s.max())
        if not mx <= m + LAZY_LOG2:  # the stage does not fit under the reference
            m_new = max(m, mx)
            alpha = 0.0 if m == -math.inf else 2.0 ** (m - m_new)
            o *= alpha
            l *= alpha
            m = m_new
            moves += 1
        p = np.exp2(s - m)
        top = max(top, float(p.max()))
        l += float(p.sum())
        o += p @ v[t0:t0 + STAGE]
    return o / l, (m + math.log2(l)) * math.log(2.0), top, moves


def _scores_and_values(n, rise, seed):
    """q = e_0 and k_t = c_t e_0, so the base-2 score of token t is exactly
    rise * (t - n / 2) with the scale below; values N(0, 1)."""
    d = 8
    scale = 1.0 / math.sqrt(d)
    k = np.zeros((n, d))
    k[:, 0] = rise * (np.arange(n) - n / 2) / (scale * math.log2(math.e))
    v = np.random.default_rng(seed).normal(size=(n, d))
    q = np.zeros(d)
    q[0] = 1.0
    return q, k, v, scale


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _oracle_row(qt, kt, vt, scale):
    """The oracle's decode attention of one sequence and head over bf16 K/V in
    pages of 16 tokens, in order."""
    n, d = kt.shape
    bs = 16
    pages = (n + bs - 1) // bs
    kc = torch.zeros(pages * bs, 1, d, dtype=torch.bfloat16)
    vc = torch.zeros(pages * bs, 1, d, dtype=torch.bfloat16)
    kc[:n, 0] = kt
    vc[:n, 0] = vt
    out = oracle.decode_attention(bits(qt.view(1, 1, d)), bits(kc.view(pages, bs, 1, d)),
                                  bits(vc.view(pages, bs, 1, d)),
                                  np.arange(pages, dtype=np.int32)[None, :],
                                  np.array([n], dtype=np.int32), scale, "bf16")
    return out[0, 0]


# 400 tokens = 25 stages; each stage's maximum lies 16 * rise above the last.
# The reference stays where it last moved until a stage exceeds it by more
# than 8: a rise of 2.5 a stage moves it at stages 0, 4, 8, ..., 24 (7 moves),
# 4.8 and 7.5 at every second stage (13), 14.4 at every stage (25); falling
# scores set it once.
@pytest.mark.parametrize("rise,expect_moves", [
    (2.5 / STAGE, 7),
    (4.8 / STAGE, 13),
    (7.5 / STAGE, 13),
    (14.4 / STAGE, 25),
    (-4.8 / STAGE, 1),
])
def test_lazy_reference_gives_the_plain_softmax(rise, expect_moves):
    n = 400
    q, k, v, scale = _scores_and_values(n, rise, seed=3)
    s2 = (k @ q) * scale * math.log2(math.e)
    got, lse, top, moves = lazy_online_softmax(s2, v)
    # the plain definition, written out
    w = np.exp(s2 * math.log(2.0) - (s2 * math.log(2.0)).max())
    exact = (w @ v) / w.sum()
    exact_lse = float((s2 * math.log(2.0)).max() + math.log(w.sum()))
    assert np.allclose(got, exact, rtol=1e-12, atol=1e-13)
    assert abs(lse - exact_lse) <= 1e-12 * max(1.0, abs(exact_lse))
    assert top <= 2.0 ** LAZY_LOG2
    assert moves == expect_moves


def test_lazy_reference_agrees_with_the_oracle():
    """The same rule against the oracle's decode attention of the same bf16 inputs."""
    n = 333
    q, k, v, scale = _scores_and_values(n, 0.47, seed=5)
    qt, kt, vt = _bf16(q), _bf16(k), _bf16(v)
    s2 = (kt.double().numpy() @ qt.double().numpy()) * scale * math.log2(math.e)
    got, _, top, moves = lazy_online_softmax(s2, vt.double().numpy())
    ref = _oracle_row(qt, kt, vt, scale)
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-10)
    assert top <= 2.0 ** LAZY_LOG2 and moves > 1


def test_a_rise_past_the_threshold_inside_one_stage_moves_the_reference():
    """A single token 2^8.5 above the reference forces the move (else e^(s - m)
    would exceed 2^8); one just under it does not."""
    s2 = np.zeros(32)
    v = np.eye(32)[:, :4]
    s2[20] = 8.5
    _, _, top, moves = lazy_online_softmax(s2, v)
    assert moves == 2 and top <= 1.0 + 1e-15
    s2[20] = 7.9
    _, _, top, moves = lazy_online_softmax(s2, v)
    assert moves == 1 and abs(top - 2.0 ** 7.9) < 1e-9
