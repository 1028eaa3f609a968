"""Pins of the oracle's sampled DFlash 2 path walk and of speculative
sampling against its sparse proposal: the proposal against a numpy
log-softmax of the pair scores, draw frequencies against it, zero factors
give the uniform proposal, a tiny temperature reduces to the greedy walk,
and the first emitted token follows the target distribution whatever the
walk proposes."""
import numpy as np
import pytest

from block_diffusion_speculative_step_gb300 import synth
from oracle import oracle as O
from tests import helpers as Hh


def _model(seed=0, V=60, K=5, R=6, B=4):
    w = Hh.small_workload(dtype="f32", V=V, topk=K, rank=R, block=B)
    m = synth.make_model(w, seed=seed, jitter=0.1, with_target=True)
    om = Hh.omodel(w, m)
    rng = np.random.default_rng(seed)
    U = rng.standard_normal((R, w.draft.hidden)).astype(np.float32) * 0.3
    Vm = rng.standard_normal((R, w.draft.hidden)).astype(np.float32) * 0.3
    logits = rng.standard_normal((B - 1, V)).astype(np.float32)
    _, cand, _ = O.path_select(om.draft.cfg, logits, om.E, U, Vm, anchor=3, topk=K)
    return w, om, U, Vm, logits, cand


def _scores(om, U, Vm, a, cands):
    E = om.E.astype(np.float64)
    return np.array([(U.astype(np.float64) @ E[a]) @ (Vm.astype(np.float64) @ E[b]) for b in cands])


def test_proposal_is_the_log_softmax_of_the_pair_scores():
    w, om, U, Vm, logits, cand = _model()
    T = 0.7
    path, lq, mg = O.path_walk_sample(om.draft.cfg, cand, om.E, U, Vm, 3, T, seed=1, seq=0, P=10, cycle=0)
    prev = 3
    for j in range(len(path)):
        z = _scores(om, U, Vm, prev, cand[j]) / T
        ref = z - (z.max() + np.log(np.exp(z - z.max()).sum()))
        np.testing.assert_allclose(lq[j], ref, rtol=0, atol=1e-10)
        assert path[j] in cand[j]
        prev = path[j]


def test_step_frequencies_follow_the_proposal():
    w, om, U, Vm, logits, cand = _model(seed=1)
    T, n = 0.8, 6000
    counts = np.zeros(cand.shape[1])
    for c in range(n):
        path, lq, _ = O.path_walk_sample(om.draft.cfg, cand, om.E, U, Vm, 3, T, seed=9, seq=2, P=5, cycle=c)
        counts[list(cand[0]).index(path[0])] += 1
    q = np.exp(lq[0])
    se = np.sqrt(q * (1 - q) / n)
    assert np.all(np.abs(counts / n - q) < 4.5 * se), (counts / n, q)


def test_zero_factors_give_the_uniform_proposal():
    w, om, U, Vm, logits, cand = _model(seed=2)
    z = np.zeros_like(U)
    K = cand.shape[1]
    path, lq, _ = O.path_walk_sample(om.draft.cfg, cand, om.E, z, z, 3, 1.0, seed=4, seq=0, P=0, cycle=0)
    np.testing.assert_allclose(lq, np.full_like(lq, -np.log(K)), rtol=0, atol=1e-12)


def test_tiny_temperature_is_the_greedy_walk():
    for seed in range(4):
        w, om, U, Vm, logits, cand = _model(seed=10 + seed)
        greedy, cg, gm = O.path_select(om.draft.cfg, logits, om.E, U, Vm, anchor=3, topk=cand.shape[1])
        if gm.min() < 1e-6:
            continue
        for c in range(5):
            path, _, _ = O.path_walk_sample(om.draft.cfg, cg, om.E, U, Vm, 3, 1e-9, seed=2, seq=0, P=0, cycle=c)
            np.testing.assert_array_equal(path, greedy)


def test_sparse_proposal_sampling_is_lossless_in_distribution():
    """Block of 3 rows over 12 tokens, candidate lists of 4: drafts from the
    sampled walk; the first emitted token follows softmax(target row 0 / T)
    -- tokens outside the candidates included -- and the first draft is
    accepted at rate sum_v min(p_v, q_v)."""
    V, K, B, T, n = 12, 4, 3, 0.9, 20000
    w, om, U, Vm, logits, cand = _model(seed=5, V=V, K=K, B=B)
    rng = np.random.default_rng(6)
    tl = rng.standard_normal((B, V)).astype(np.float32)
    first = np.zeros(V)
    acc0 = 0
    lq0 = None
    for c in range(n):
        path, lq, _ = O.path_walk_sample(om.draft.cfg, cand, om.E, U, Vm, 3, T, seed=8, seq=1, P=20, cycle=c)
        lq0 = lq[0]
        k, out, _ = O.spec_sample_accept_sparse(tl, cand, lq, path, T, seed=8, seq=1, P=20, cycle=c)
        assert list(out[:k]) == list(path[:k])
        first[out[0]] += 1
        acc0 += k > 0
    z = tl[0].astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    se = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(first / n - p) < 4.5 * se), (first / n, p)
    q = np.zeros(V)
    q[cand[0]] = np.exp(lq0)
    alpha = np.minimum(p, q).sum()
    assert abs(acc0 / n - alpha) < 4.5 * np.sqrt(alpha * (1 - alpha) / n)
