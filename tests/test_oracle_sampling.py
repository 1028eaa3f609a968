"""Pins of the oracle's sampling-mode verification (speculative sampling at
temperature T, Philox4x32-10 random numbers): the generator's published
known-answer vectors, Gumbel-max draws against the softmax they sample, and
the invariant the method exists for -- the emitted token follows the
target's distribution whatever the draft (lossless in distribution)."""
import json
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def softmax(x, T):
    z = np.asarray(x, dtype=np.float64) / T
    z = np.exp(z - z.max())
    return z / z.sum()


def test_philox_known_answers():
    with open(os.path.join(GOLD, "philox4x32_10_kat.json")) as f:
        kat = json.load(f)
    for vec in kat["vectors"]:
        got = O.philox4x32_10([int(x, 16) for x in vec["ctr"]], [int(x, 16) for x in vec["key"]])
        assert got == [int(x, 16) for x in vec["out"]]


def test_uniform_is_the_top_24_bits_of_the_first_word():
    seed = 0x1234_5678_9ABC_DEF0
    for v, pos, seq, purpose, cycle in [(0, 0, 0, 1, 0), (151935, 4111, 31, 3, 7), (5, 9, 2, 2, 123456)]:
        x0 = O.philox4x32_10([v, pos, (seq << 8) | purpose, cycle], [seed & 0xFFFFFFFF, seed >> 32])[0]
        u = O.uniform(seed, v, pos, seq, purpose, cycle)
        assert u == ((x0 >> 8) + 0.5) / 2 ** 24
        assert 0.0 < u < 1.0


def test_gumbel_max_draws_follow_the_softmax():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal(6).astype(np.float32)
    T, n = 0.7, 20000
    counts = np.zeros(6)
    for c in range(n):
        tok, lse, _ = O.sample_row(logits, T, seed=99, pos=3, seq=0, purpose=O.RNG_DRAFT, cycle=c)
        counts[tok] += 1
    p = softmax(logits, T)
    assert lse == pytest.approx(np.log(np.exp(logits.astype(np.float64) / T).sum()), rel=1e-12)
    # every frequency within 4.5 standard errors of its probability
    se = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(counts / n - p) < 4.5 * se), (counts / n, p)


def test_speculative_sampling_is_lossless_in_distribution():
    """Block of 3 rows, vocabulary 6: drafts sampled from a deliberately
    different draft distribution; the first emitted token (accepted draft or
    residual draw) must be distributed as softmax(target row 0 / T), and the
    acceptance rate must equal sum_v min(p_v, q_v)."""
    rng = np.random.default_rng(2)
    B, V, T, n = 3, 6, 0.9, 20000
    tl = rng.standard_normal((B, V)).astype(np.float32)
    dl = (tl[:B - 1] * 0.3 + rng.standard_normal((B - 1, V))).astype(np.float32)
    first = np.zeros(V)
    accepted0 = 0
    for c in range(n):
        drafts = [O.sample_row(dl[j], T, seed=7, pos=11 + j, seq=1, purpose=O.RNG_DRAFT, cycle=c)[0]
                  for j in range(B - 1)]
        k, out, _ = O.spec_sample_accept(tl, dl, drafts, T, seed=7, seq=1, P=10, cycle=c)
        assert 0 <= k <= B - 1 and len(out) == k + 1
        assert list(out[:k]) == drafts[:k]
        first[out[0]] += 1
        accepted0 += k > 0
    p, q = softmax(tl[0], T), softmax(dl[0], T)
    se = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(first / n - p) < 4.5 * se), (first / n, p, q)
    alpha = np.minimum(p, q).sum()
    assert abs(accepted0 / n - alpha) < 4.5 * np.sqrt(alpha * (1 - alpha) / n)


def test_identical_distributions_accept_everything():
    rng = np.random.default_rng(3)
    B, V, T = 5, 40, 1.3
    tl = rng.standard_normal((B, V)).astype(np.float32)
    for c in range(50):
        drafts = [O.sample_row(tl[j], T, seed=5, pos=j + 1, seq=0, purpose=O.RNG_DRAFT, cycle=c)[0]
                  for j in range(B - 1)]
        k, out, _ = O.spec_sample_accept(tl, tl[:B - 1], drafts, T, seed=5, seq=0, P=0, cycle=c)
        assert k == B - 1 and list(out[:B - 1]) == drafts


def test_low_temperature_is_greedy():
    rng = np.random.default_rng(4)
    B, V = 4, 50
    tl = rng.standard_normal((B, V)).astype(np.float32)
    g = tl.argmax(1)
    for c in range(20):
        tok, _, _ = O.sample_row(tl[0], 1e-4, seed=3, pos=1, seq=0, purpose=O.RNG_DRAFT, cycle=c)
        assert tok == g[0]
        # drafts = the target's greedy tokens: all accepted, bonus = greedy of the last row
        k, out, _ = O.spec_sample_accept(tl, tl[:B - 1], list(g[:B - 1]), 1e-4, seed=3, seq=0, P=0, cycle=c)
        assert k == B - 1 and list(out) == list(g)
