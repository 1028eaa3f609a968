"""Pins of the oracle's top-k / top-p filter for sampling mode: the kept set
against a numpy restatement (np.lexsort order, cumulative softmax), the
special cases (top-k 1 is greedy, no filter changes nothing, a tiny top-p
keeps the top entry), and speculative sampling with filtered target and
draft rows following the filtered target distribution."""
import numpy as np
import pytest

from oracle import oracle as O


def _ref_keep(l, T, k, p):
    V = len(l)
    order = np.lexsort((np.arange(V), -l.astype(np.float64)))  # logit desc, index asc
    n = k if 0 < k < V else V
    if p < 1.0:
        x = l[order[:n]].astype(np.float64) / T
        w = np.exp(x - x.max())
        cum = np.cumsum(w) / w.sum()
        n = int(np.argmax(cum >= p)) + 1
    keep = np.zeros(V, dtype=np.uint8)
    keep[order[:n]] = 1
    return keep


@pytest.mark.parametrize("k,p", [(0, 1.0), (1, 1.0), (5, 1.0), (50, 1.0), (0, 0.9), (0, 0.5), (7, 0.8), (0, 1e-9)])
def test_filter_matches_numpy_restatement(k, p):
    rng = np.random.default_rng(k * 100 + int(p * 1000))
    for trial in range(20):
        l = (rng.standard_normal(50) * 2).astype(np.float32)
        l[rng.integers(0, 50, 6)] = l[3]  # planted ties
        T = float(rng.uniform(0.5, 1.5))
        keep, n, mg = O.filter_row(l, T, k, p)
        ref = _ref_keep(l, T, k, p)
        if mg < 1e-9:  # the cumulative mass meets top_p exactly: either side is a valid reading
            continue
        np.testing.assert_array_equal(keep, ref)
        assert n == int(ref.sum())


def test_top_k_one_is_greedy():
    rng = np.random.default_rng(5)
    l = rng.standard_normal(200).astype(np.float32)
    l[[17, 90]] = l.max() + 1.0  # a tie at the top: the lower index wins
    keep, n, _ = O.filter_row(l, 1.0, 1, 1.0)
    assert n == 1 and keep[17] == 1
    for c in range(30):
        tok, lse, _ = O.sample_row(l, 1.0, seed=2, pos=4, seq=0, purpose=O.RNG_DRAFT, cycle=c, keep=keep)
        assert tok == 17 and lse == pytest.approx(float(l[17]), abs=1e-12)


def test_no_filter_changes_nothing():
    rng = np.random.default_rng(6)
    B, V, T = 4, 64, 0.8
    tl = rng.standard_normal((B, V)).astype(np.float32)
    dl = rng.standard_normal((B - 1, V)).astype(np.float32)
    kt = np.stack([O.filter_row(tl[j], T, 0, 1.0)[0] for j in range(B)])
    kd = np.stack([O.filter_row(dl[j], T, V, 1.0)[0] for j in range(B - 1)])
    assert kt.all() and kd.all()
    for c in range(20):
        drafts = [O.sample_row(dl[j], T, 4, j + 1, 0, O.RNG_DRAFT, c)[0] for j in range(B - 1)]
        a = O.spec_sample_accept(tl, dl, drafts, T, 4, 0, 0, c)
        b = O.spec_sample_accept(tl, dl, drafts, T, 4, 0, 0, c, keep_t=kt, keep_d=kd)
        assert a[0] == b[0] and list(a[1]) == list(b[1])


def test_tiny_top_p_keeps_the_top_entry():
    rng = np.random.default_rng(7)
    l = rng.standard_normal(300).astype(np.float32)
    keep, n, _ = O.filter_row(l, 1.0, 0, 1e-12)
    assert n == 1 and keep[int(np.argmax(l))] == 1


def test_filtered_speculative_sampling_follows_the_filtered_target():
    """Block of 3 rows, vocabulary 8, top-k 5 and top-p 0.85 on both sides:
    the first emitted token is distributed as the filtered, renormalised
    softmax of target row 0 (tokens outside its kept set never appear), and
    the acceptance rate equals sum_v min(p_v, q_v) of the filtered rows."""
    rng = np.random.default_rng(8)
    B, V, T, n, k, p = 3, 8, 0.9, 20000, 5, 0.85
    tl = rng.standard_normal((B, V)).astype(np.float32)
    dl = (tl[:B - 1] * 0.3 + rng.standard_normal((B - 1, V))).astype(np.float32)
    kt = np.stack([O.filter_row(tl[j], T, k, p)[0] for j in range(B)])
    kd = np.stack([O.filter_row(dl[j], T, k, p)[0] for j in range(B - 1)])
    first = np.zeros(V)
    accepted0 = 0
    for c in range(n):
        drafts = [O.sample_row(dl[j], T, 7, 11 + j, 1, O.RNG_DRAFT, c, keep=kd[j])[0] for j in range(B - 1)]
        assert all(kd[j][drafts[j]] for j in range(B - 1))
        kk, out, _ = O.spec_sample_accept(tl, dl, drafts, T, 7, 1, 10, c, keep_t=kt, keep_d=kd)
        first[out[0]] += 1
        accepted0 += kk > 0

    def fsoft(x, keep):
        z = np.where(keep > 0, x.astype(np.float64) / T, -np.inf)
        z = np.exp(z - z.max())
        return z / z.sum()

    pt, qd = fsoft(tl[0], kt[0]), fsoft(dl[0], kd[0])
    assert np.all(first[kt[0] == 0] == 0)
    se = np.sqrt(pt * (1 - pt) / n) + 1e-12
    assert np.all(np.abs(first / n - pt) < 4.5 * se), (first / n, pt)
    alpha = np.minimum(pt, qd).sum()
    assert abs(accepted0 / n - alpha) < 4.5 * np.sqrt(alpha * (1 - alpha) / n)
