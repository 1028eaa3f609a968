"""Pins of the CPU oracle to things other than itself: library routines
(torch float64 SDPA / rms_norm / bf16 conversion, numpy argmax), closed forms,
invariants, brute force on tiny inputs, and the worked examples the pages
print (tests/golden/).  CPU only."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import synth
from tests import helpers as Hh

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ bf16 rounding


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -3.4e38, 1e-40,
                         np.inf, -np.inf]])
    # exact ties: bf16 mantissa boundary halfway points, both parities
    base = np.array([1.0, 1.0078125, 2.0, 3.0], dtype=np.float32)
    ties = base.view(np.uint32) + 0x8000
    x = np.concatenate([x, ties.view(np.float32).astype(np.float64)])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_round_array(x)
    np.testing.assert_array_equal(got, ref)
    got_c = np.array([orc.lib().or_bf16_round(float(v)) for v in x])
    np.testing.assert_array_equal(got_c, ref)
    assert np.isnan(orc.lib().or_bf16_round(float("nan")))


# ------------------------------------------------------------------------- RoPE


def test_rope_closed_forms(orc):
    rng = np.random.default_rng(1)
    d, theta = 64, 1e4
    v = rng.standard_normal(d)
    np.testing.assert_allclose(orc.rope(v, 0, theta), v, rtol=0, atol=0)
    for pos in (1, 7, 1000, 131071):
        r = orc.rope(v, pos, theta)
        assert abs(np.linalg.norm(r) - np.linalg.norm(v)) < 1e-12
        ref = Hh.trope(torch.from_numpy(v)[None, :], torch.tensor([pos]), theta)[0].numpy()
        np.testing.assert_allclose(r, ref, rtol=0, atol=1e-11)
    # relative-position property: <R(q,m), R(k,n)> depends on m - n only
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    a = orc.rope(q, 10, theta) @ orc.rope(k, 3, theta)
    b = orc.rope(q, 510, theta) @ orc.rope(k, 503, theta)
    assert abs(a - b) < 1e-10
    # first pair at pos 1 rotates by exactly 1 radian (w_0 = 1)
    e = np.zeros(d); e[0] = 1.0
    r = orc.rope(e, 1, theta)
    assert abs(r[0] - np.cos(1.0)) < 1e-15 and abs(r[d // 2] - np.sin(1.0)) < 1e-15


# ------------------------------------------------------------- RMSNorm, linear


def test_rmsnorm_and_linear_match_library(orc):
    rng = np.random.default_rng(2)
    c = orc.Cfg(96, 4, 2, 16, 64, False, 1e4, 1e-5)
    x = rng.standard_normal((5, 96))
    g = (1 + 0.1 * rng.standard_normal(96)).astype(np.float32)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g.astype(np.float64)),
                                       1e-5).numpy()
    np.testing.assert_allclose(orc.rmsnorm(c, x, g), ref, rtol=1e-13, atol=1e-13)
    W = rng.standard_normal((33, 96)).astype(np.float32)
    np.testing.assert_allclose(orc.linear(c, W, x), x @ W.astype(np.float64).T, rtol=1e-12, atol=1e-12)
    Wb = synth.to_numpy(torch.from_numpy(W).to(torch.bfloat16))
    cb = orc.Cfg(96, 4, 2, 16, 64, True, 1e4, 1e-5)
    np.testing.assert_allclose(orc.linear(cb, Wb, x), x @ Hh.t64(Wb).numpy().T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- decoder layer


def _layer_setup(dtype, seed=0, **kw):
    w = Hh.small_workload(dtype=dtype, **kw)
    m = synth.make_model(w, seed=seed, jitter=0.1, with_target=True)
    om = Hh.omodel(w, m)
    return w, om


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_causal_layer_matches_torch_sdpa(orc, dtype):
    w, om = _layer_setup(dtype)
    c, L = om.target.cfg, om.target.layers[0]
    rng = np.random.default_rng(3)
    cap = 32
    kc = np.zeros((c.nkv, cap, c.d)); vc = np.zeros((c.nkv, cap, c.d))
    h0 = rng.standard_normal((9, c.H))
    # prefix of 5 rows, then 4 more rows against the cache
    h_pre = h0[:5].copy(); orc.decoder_layer(c, L, h_pre, 0, orc.CAUSAL, kc, vc)
    h_suf = h0[5:].copy(); orc.decoder_layer(c, L, h_suf, 5, orc.CAUSAL, kc, vc)
    ref, _, _ = Hh.torch_layer(c, L, torch.from_numpy(h0), torch.arange(9), causal=True)
    tol = 1e-10 if dtype == "f32" else 2e-2
    np.testing.assert_allclose(np.concatenate([h_pre, h_suf]), ref.numpy(), rtol=0, atol=tol)
    if dtype == "f32":
        # incremental (cached) == one pass over all rows, bit for bit
        kc2 = np.zeros_like(kc); vc2 = np.zeros_like(vc)
        h_all = h0.copy(); orc.decoder_layer(c, L, h_all, 0, orc.CAUSAL, kc2, vc2)
        np.testing.assert_array_equal(np.concatenate([h_pre, h_suf]), h_all)
        np.testing.assert_array_equal(kc, kc2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("window", [0, 6])
def test_bidir_layer_matches_torch_sdpa(orc, dtype, window):
    w, om = _layer_setup(dtype)
    c, L = om.draft.cfg, om.draft.layers[1]
    rng = np.random.default_rng(4)
    P, M = 11, 4
    cap = window if window else 16
    kc = np.zeros((c.nkv, cap, c.d)); vc = np.zeros((c.nkv, cap, c.d))
    ctx_k = orc.rnd(c, rng.standard_normal((P, c.nkv, c.d)))
    ctx_v = orc.rnd(c, rng.standard_normal((P, c.nkv, c.d)))
    for t in range(P):
        s = t % window if window else t
        kc[:, s] = ctx_k[t]; vc[:, s] = ctx_v[t]
    h0 = rng.standard_normal((M, c.H))
    h = h0.copy()
    orc.decoder_layer(c, L, h, P, orc.BIDIR, kc, vc, window)
    lo = max(0, P - window) if window else 0
    ref, _, _ = Hh.torch_layer(c, L, torch.from_numpy(h0), torch.arange(P, P + M),
                               ctx_k=torch.from_numpy(ctx_k[lo:]), ctx_v=torch.from_numpy(ctx_v[lo:]),
                               causal=False)
    tol = 1e-10 if dtype == "f32" else 2e-2
    np.testing.assert_allclose(h, ref.numpy(), rtol=0, atol=tol)


def test_window_at_least_context_equals_no_window(orc):
    w, om = _layer_setup("f32")
    c, L = om.draft.cfg, om.draft.layers[0]
    rng = np.random.default_rng(5)
    P, M, W = 9, 4, 12
    ck = rng.standard_normal((c.nkv, W, c.d)); cv = rng.standard_normal((c.nkv, W, c.d))
    h0 = rng.standard_normal((M, c.H))
    a = h0.copy(); orc.decoder_layer(c, L, a, P, orc.BIDIR, ck, cv, W)
    b = h0.copy(); orc.decoder_layer(c, L, b, P, orc.BIDIR, ck.copy(), cv.copy(), 0)
    np.testing.assert_array_equal(a, b)


def test_attention_special_cases(orc):
    """Identity projections: a single key returns its value; identical keys
    return the mean of the values; the bidirectional block with no context is
    plain non-causal self-attention; causal == bidirectional at one row."""
    H = d = 8
    c = orc.Cfg(H, 1, 1, d, 4, False, 1e4, 1e-6)
    eye = np.eye(H, dtype=np.float32)
    z = np.zeros((4, H), dtype=np.float32)
    one = np.ones(H, dtype=np.float32)
    L = orc.Layer(eye, eye, eye, eye, z, z, np.zeros((H, 4), dtype=np.float32), one, one)
    rng = np.random.default_rng(6)
    # causal at p0 = 0, one row: attends only itself -> out = own v (= normed x, rotated at pos 0)
    h = rng.standard_normal((1, H))
    x = orc.rmsnorm(c, h, one)
    kc = np.zeros((1, 4, d)); vc = np.zeros((1, 4, d))
    hc = h.copy(); orc.decoder_layer(c, L, hc, 0, orc.CAUSAL, kc, vc)
    np.testing.assert_allclose(hc, h + x, rtol=0, atol=1e-13)
    # bidirectional, one row, zero context == the causal result
    hb = h.copy(); orc.decoder_layer(c, L, hb, 0, orc.BIDIR, np.zeros((1, 4, d)), np.zeros((1, 4, d)))
    np.testing.assert_array_equal(hb, hc)
    # identical keys (all-zero context keys, block row whose rotated key is 0 is impossible, so use
    # zero queries): with q = 0 every score is 0 and the output is the mean of all values.
    Lz = orc.Layer(np.zeros_like(eye), eye, eye, eye, z, z, np.zeros((H, 4), dtype=np.float32), one, one)
    P = 3
    ck = rng.standard_normal((1, 4, d)); cv = rng.standard_normal((1, 4, d))
    h = rng.standard_normal((1, H))
    x = orc.rmsnorm(c, h, one)[0]
    hz = h.copy(); orc.decoder_layer(c, Lz, hz, P, orc.BIDIR, ck, cv)
    mean_v = (cv[0, :P].sum(0) + x) / (P + 1)
    np.testing.assert_allclose(hz[0], h[0] + mean_v, rtol=0, atol=1e-13)


# --------------------------------------------------------------- LM head argmax


def test_lm_head_argmax_bruteforce_and_ties(orc):
    rng = np.random.default_rng(7)
    c = orc.Cfg(32, 2, 1, 16, 8, False, 1e4, 1e-6)
    W = rng.standard_normal((50, 32)).astype(np.float32)
    W[17] = W[5]  # exact duplicate rows -> exact ties
    x = rng.standard_normal((6, 32))
    x[2] = W[5].astype(np.float64) * 10  # row 2's max is the tie between 5 and 17
    am, mg, lg = orc.lm_head_argmax(c, W, x, True)
    ref = (x @ W.astype(np.float64).T).astype(np.float32)
    np.testing.assert_array_equal(lg, ref)
    np.testing.assert_array_equal(am, np.argmax(ref, axis=1))  # numpy: first (lowest) index on ties
    assert am[2] == 5 and mg[2] == 0.0
    srt = np.sort(ref.astype(np.float64), axis=1)
    np.testing.assert_allclose(mg, srt[:, -1] - srt[:, -2])


# ------------------------------------------------------------------- acceptance


def test_accept_worked_example(orc):
    g = gold("prefix_accept_example.json")
    n, agree = g["drafted"], g["agree_prefix"]
    B = n + 1
    target = np.arange(100, 100 + B, dtype=np.int32)          # target greedy after rows 0..B-1
    drafts = target[:n].copy()
    drafts[agree] += 1000                                       # the 7th draft differs
    drafts[agree + 1:] = target[agree + 1:n]                    # later agreement must not count
    k, out = orc.accept(drafts, target)
    assert k == g["expected_accept"]
    assert len(out) == g["expected_emitted"]
    np.testing.assert_array_equal(out[:agree], drafts[:agree])
    assert out[agree] == target[agree]                          # 7th comes from the target


def test_accept_exhaustive_small():
    """Every draft/target pattern with B = 4 and 3 token values: accepted
    drafts agree with the target, the first rejected one does not, the bonus
    is the target's token there, 1 <= emitted <= B."""
    from oracle import oracle as O
    B, V = 4, 3
    for drafts in itertools.product(range(V), repeat=B - 1):
        for g in itertools.product(range(V), repeat=B):
            k, out = O.accept(np.array(drafts), np.array(g))
            assert 0 <= k <= B - 1 and len(out) == k + 1
            assert all(drafts[j] == g[j] for j in range(k))
            assert k == B - 1 or drafts[k] != g[k]
            assert out[k] == g[k] and list(out[:k]) == list(drafts[:k])


# ------------------------------------------------------------ fusion + injection


def test_fusion_closed_form(orc):
    H, F = 16, 3
    c = orc.Cfg(H, 2, 1, 8, 8, False, 1e4, 1e-6)
    Wfc = np.zeros((H, F * H), dtype=np.float32); Wfc[:, :H] = np.eye(H)
    g = np.ones(H, dtype=np.float32)
    rng = np.random.default_rng(8)
    wk = rng.standard_normal((8, H)).astype(np.float32)
    wv = rng.standard_normal((8, H)).astype(np.float32)
    hot = 5
    feats = np.zeros((2, F * H)); feats[:, hot] = 1.0; feats[:, H + 2] = 7.0  # 2nd tap ignored by W_fc
    kc = [np.zeros((1, 4, 8))]; vc = [np.zeros((1, 4, 8))]
    cvec = orc.fuse_context(c, F, Wfc, g, feats, [0, 3], [wk], [wv], kc, vc)
    scale = 1.0 / np.sqrt(1.0 / H + 1e-6)                       # RMSNorm of a one-hot
    expect_c = np.zeros(H); expect_c[hot] = scale
    np.testing.assert_allclose(cvec[0], expect_c, rtol=1e-14)
    np.testing.assert_allclose(kc[0][0, 0], wk[:, hot] * scale, rtol=1e-12)   # pos 0: no rotation
    np.testing.assert_allclose(vc[0][0, 3], wv[:, hot] * scale, rtol=1e-12)   # V never rotated
    k3 = orc.rope(wk[:, hot].astype(np.float64) * scale, 3, 1e4)
    np.testing.assert_allclose(kc[0][0, 3], k3, rtol=1e-12)
    # linearity in W_v
    vc2 = [np.zeros((1, 4, 8))]
    orc.fuse_context(c, F, Wfc, g, feats, [0, 3], [wk], [2 * wv], [np.zeros((1, 4, 8))], vc2)
    np.testing.assert_allclose(vc2[0], 2 * vc[0], rtol=1e-14)


def test_fusion_window_ring_slots(orc):
    H, F, W = 16, 2, 4
    c = orc.Cfg(H, 2, 1, 8, 8, False, 1e4, 1e-6)
    rng = np.random.default_rng(9)
    Wfc = rng.standard_normal((H, F * H)).astype(np.float32)
    g = np.ones(H, dtype=np.float32)
    wk = rng.standard_normal((8, H)).astype(np.float32)
    wv = rng.standard_normal((8, H)).astype(np.float32)
    feats = rng.standard_normal((6, F * H))
    kc = [np.zeros((1, W, 8))]; vc = [np.zeros((1, W, 8))]
    orc.fuse_context(c, F, Wfc, g, feats, list(range(6)), [wk], [wv], kc, vc, W)
    kf = [np.zeros((1, 8, 8))]; vf = [np.zeros((1, 8, 8))]
    orc.fuse_context(c, F, Wfc, g, feats, list(range(6)), [wk], [wv], kf, vf, 0)
    for t in range(2, 6):  # the last W positions live at slot t % W
        np.testing.assert_array_equal(kc[0][0, t % W], kf[0][0, t])


# -------------------------------------------------------------- whole-model pins


def _tiny_model(dtype="f32", seed=0, **kw):
    w = Hh.small_workload(dtype=dtype, **kw)
    m = synth.make_model(w, seed=seed, jitter=0.1, with_target=True)
    return w, Hh.omodel(w, m)


def test_target_forward_matches_torch_restatement(orc):
    w, om = _tiny_model()
    prompt = synth.make_tokens(1, 12, w.vocab).numpy()
    st = orc.new_state(om, 32)
    am, mg, feats, lg = orc.target_forward(om, st, prompt, 0, want_logits=True)
    c = om.target.cfg
    h = Hh.t64(om.E[prompt])
    taps = {}
    for li, L in enumerate(om.target.layers):
        h, _, _ = Hh.torch_layer(c, L, h, torch.arange(12), causal=True)
        taps[li] = h.clone()
    x = torch.nn.functional.rms_norm(h, (c.H,), Hh.t64(om.target.g_final), c.eps)
    logits = x @ Hh.t64(om.Wlm).T
    np.testing.assert_allclose(lg, logits.numpy(), rtol=0, atol=1e-5)
    np.testing.assert_allclose(feats, torch.cat([taps[l] for l in w.taps], 1).numpy(), atol=1e-10)
    ok = mg > 1e-4
    np.testing.assert_array_equal(am[ok], logits.argmax(1).numpy()[ok])


def test_cached_decode_equals_full_recompute(orc):
    """Brute force: every greedy token equals the argmax of a fresh, cache-free
    forward over the whole prefix."""
    w, om = _tiny_model()
    prompt = synth.make_tokens(2, 10, w.vocab).numpy()
    toks, margins = orc.greedy_generate(om, prompt, 8, cap=32)
    seq = list(prompt)
    for i in range(8):
        st = orc.new_state(om, 32)
        am, mg, _, _ = orc.target_forward(om, st, seq, 0)
        assert am[-1] == toks[i]
        assert abs(mg[-1] - margins[i]) < 1e-12
        seq.append(int(toks[i]))


@pytest.mark.parametrize("dtype,block", [("f32", 4), ("bf16", 5)])
def test_speculative_equals_greedy(orc, dtype, block):
    """Lossless: the speculative loop emits exactly the plain greedy tokens."""
    w, om = _tiny_model(dtype=dtype, block=block)
    prompt = synth.make_tokens(3, 12, w.vocab).numpy()
    n = 30
    ref, _ = orc.greedy_generate(om, prompt, n, cap=64)
    got, acc = orc.speculative_generate(om, prompt, n, cap=64)
    np.testing.assert_array_equal(got, ref)
    assert all(0 <= k <= block - 1 for k in acc)


def test_perfect_and_wrong_drafters(orc):
    w, om = _tiny_model(block=4)
    prompt = synth.make_tokens(4, 12, w.vocab).numpy()
    n = 25
    ref, _ = orc.greedy_generate(om, prompt, n + 8, cap=80)
    pos_of = {}

    def perfect(m, st, anchor, P):
        i = P - len(prompt)                 # anchor is greedy token i
        return ref[i + 1:i + m.block]

    def wrong(m, st, anchor, P):
        i = P - len(prompt)
        return (ref[i + 1:i + m.block] + 1) % (w.vocab - 1)

    got, acc = orc.speculative_generate(om, prompt, n, cap=80, drafter=perfect)
    np.testing.assert_array_equal(got, ref[:n])
    assert all(k == w.block - 1 for k in acc)
    got, acc = orc.speculative_generate(om, prompt, n, cap=80, drafter=wrong)
    np.testing.assert_array_equal(got, ref[:n])
    assert all(k == 0 for k in acc)


def test_tiny_lossless_workload(orc):
    """The 4-layer / 2-draft-layer fp32 workload: 64 generated tokens after a
    64-token prompt, speculative == greedy."""
    w = synth.WORKLOADS["tiny-lossless"]
    m = synth.make_model(w, seed=0)
    om = Hh.omodel(w, m)
    prompt = synth.make_tokens(0, w.prompt, w.vocab).numpy()
    cap = w.prompt + w.generate + w.block
    ref, margins = orc.greedy_generate(om, prompt, w.generate, cap)
    got, acc = orc.speculative_generate(om, prompt, w.generate, cap)
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------- path selector


def test_path_selector_zero_factors_is_top1(orc):
    w, om = _tiny_model(dtype="bf16", topk=4, rank=8, block=5)
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((4, w.vocab)).astype(np.float32)
    z = np.zeros((8, w.draft.hidden), dtype=np.uint16)
    path, cand, mg = orc.path_select(om.draft.cfg, logits, om.E, z, z, anchor=3, topk=4)
    np.testing.assert_array_equal(path, np.argmax(logits, axis=1))
    np.testing.assert_array_equal(cand, np.argsort(-logits, axis=1, kind="stable")[:, :4])
    assert np.all(mg == 0.0)


def test_path_selector_bruteforce(orc):
    w, om = _tiny_model(dtype="f32", V=40, topk=5, rank=6, block=4)
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((3, w.vocab)).astype(np.float32)
    U = rng.standard_normal((6, w.draft.hidden)).astype(np.float32)
    Vm = rng.standard_normal((6, w.draft.hidden)).astype(np.float32)
    path, cand, mg = orc.path_select(om.draft.cfg, logits, om.E, U, Vm, anchor=7, topk=5)
    E = om.E.astype(np.float64)
    prev = 7
    for j in range(3):
        top = np.argsort(-logits[j], kind="stable")[:5]
        sc = np.array([(U @ E[prev]) @ (Vm @ E[b]) for b in top]).astype(np.float32)
        assert path[j] == top[int(np.argmax(sc))]
        prev = path[j]


# --------------------------------------------------------- taps and cost model


def test_tap_layer_rule(orc):
    for case in gold("tap_layers.json")["cases"]:
        ids = orc.tap_layers(case["n_layers"], case["n_taps"])
        assert ids[0] == case["first"] and ids[-1] == case["last"]
        assert len(ids) == case["n_taps"] and all(a < b for a, b in zip(ids, ids[1:]))
        gaps = np.diff(ids)
        assert gaps.max() - gaps.min() <= 1          # uniform up to rounding
    for wname, w in synth.WORKLOADS.items():
        if len(w.taps) == 5:
            assert tuple(orc.tap_layers(w.target.layers)) == w.taps


def test_cost_model_example(orc):
    g = gold("cost_model_example.json")
    for case in g["cases"]:
        v = orc.per_token_cost_ms(g["t_draft_ms"], g["t_verify_ms"], case["accepted"])
        assert abs(v - case["ms_per_token"]) <= case["abs_tol"]
    sp = g["baseline_ms_per_token"] / orc.per_token_cost_ms(g["t_draft_ms"], g["t_verify_ms"], 6)
    assert abs(sp - g["speedup_at_6"]) <= g["speedup_tol"]


# ------------------------------------------------------ teacher-forced stages


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["causal", "bidir"])
def test_layer_stages_open_for_teacher_forcing(orc, dtype, mode):
    """decoder_layer_tf is decoder_layer with its stages open: with nothing
    given it is the plain layer bit for bit, its stage outputs are the torch
    restatement's intermediates (each named stage is the tensor its name
    says), and feeding every stage its own value back changes nothing; a
    given stage replaces the oracle's value (a perturbed attention output
    moves the output by exactly the O projection of the perturbation)."""
    w, om = _layer_setup(dtype)
    causal = mode == "causal"
    c = om.target.cfg if causal else om.draft.cfg
    L = om.target.layers[0] if causal else om.draft.layers[0]
    rng = np.random.default_rng(12)
    P, M, cap = 7, 4, 16
    kc = np.zeros((c.nkv, cap, c.d)); vc = np.zeros((c.nkv, cap, c.d))
    ctx_k = orc.rnd(c, rng.standard_normal((P, c.nkv, c.d)))
    ctx_v = orc.rnd(c, rng.standard_normal((P, c.nkv, c.d)))
    for t in range(P):
        kc[:, t] = ctx_k[t]; vc[:, t] = ctx_v[t]
    h0 = rng.standard_normal((M, c.H))
    mo = orc.CAUSAL if causal else orc.BIDIR
    h_plain = h0.copy(); kp, vp = kc.copy(), vc.copy()
    orc.decoder_layer(c, L, h_plain, P, mo, kp, vp)
    h_tf = h0.copy(); kt, vt = kc.copy(), vc.copy()
    st = orc.decoder_layer_tf(c, L, h_tf, P, mo, kt, vt)
    np.testing.assert_array_equal(h_tf, h_plain)
    np.testing.assert_array_equal(kt, kp)
    ref = {}
    if causal:
        Hh.torch_layer(c, L, torch.from_numpy(h0), torch.arange(P, P + M), causal=True,
                       past_k=torch.from_numpy(ctx_k), past_v=torch.from_numpy(ctx_v), stages=ref)
    else:
        Hh.torch_layer(c, L, torch.from_numpy(h0), torch.arange(P, P + M), ctx_k=torch.from_numpy(ctx_k),
                       ctx_v=torch.from_numpy(ctx_v), causal=False, stages=ref)
    tol = 1e-10 if dtype == "f32" else 2e-2
    for n in orc.STAGES:
        np.testing.assert_allclose(st[n], ref[n].numpy(), rtol=0, atol=tol, err_msg=n)
    h_again = h0.copy()
    st2 = orc.decoder_layer_tf(c, L, h_again, P, mo, kc.copy(), vc.copy(), given=st)
    np.testing.assert_array_equal(h_again, h_plain)
    for n in orc.STAGES:
        np.testing.assert_array_equal(st2[n], st[n], err_msg=n)
    # a given attention output replaces the oracle's: the output moves by the
    # O projection of the change, and the stages before it do not move
    delta = np.zeros_like(st["o"]); delta[1, 3] = 0.5
    h_pert = h0.copy()
    st3 = orc.decoder_layer_tf(c, L, h_pert, P, mo, kc.copy(), vc.copy(),
                               given={"o": st["o"] + delta, "x2": st["x2"], "act": st["act"]})
    np.testing.assert_array_equal(st3["q"], st["q"])
    wo = orc.wfloat(c, L.wo)
    np.testing.assert_allclose(h_pert - h_plain, delta @ wo.T, rtol=0, atol=1e-12)
