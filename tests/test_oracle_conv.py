"""Pins of the oracle's DFlash 2 two-tap dynamic depthwise convolution
(dyn_conv, and the draft layer that carries four of them): a library
reduction (identical rows make the taps static, so the convolution is a
depthwise F.conv1d with causal padding), locality, the zero generator, and
the draft layer against a float64 torch restatement.  CPU only."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from block_diffusion_speculative_step_gb300 import synth
from tests import helpers as Hh


def _conv_model(dtype="f32", seed=7, **kw):
    w = Hh.small_workload(dtype=dtype, conv_rank=8, **kw)
    m = synth.make_model(w, seed=seed, jitter=0.1, with_target=True, std=0.2)
    return w, m, Hh.omodel(w, m)


def test_dyn_conv_identical_rows_is_depthwise_conv1d(orc):
    """All rows equal: every row gets the same taps (a, b), so the layer is a
    static two-tap depthwise convolution, which F.conv1d computes with
    groups = H, kernel [b, 1 + a] and one zero of left padding."""
    w, _, om = _conv_model()
    c, cv = om.draft.cfg, om.draft.layers[0].conv
    rng = np.random.default_rng(1)
    u = np.repeat(rng.standard_normal((1, c.H)), 5, axis=0)
    got = orc.dyn_conv(c, cv.w1[2], cv.w2[2], u)
    ab = F.silu(Hh.t64(cv.w1[2]) @ torch.from_numpy(u[0])) @ Hh.t64(cv.w2[2]).T
    a, b = ab[:c.H], ab[c.H:]
    weight = torch.stack([b, 1.0 + a], dim=1).unsqueeze(1)          # [H][1][2]
    seq = torch.from_numpy(u).T.unsqueeze(0)                        # [1][H][M]
    ref = F.conv1d(F.pad(seq, (1, 0)), weight, groups=c.H)[0].T
    np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)
    assert not np.allclose(got[0], got[1])  # row 0 has no predecessor


def test_dyn_conv_locality(orc):
    """Changing row t changes rows t (its taps and value) and t + 1 (its
    previous-position input) and nothing else: the two taps are the current
    and the previous position, not the next one."""
    w, _, om = _conv_model()
    c, cv = om.draft.cfg, om.draft.layers[1].conv
    rng = np.random.default_rng(2)
    u = rng.standard_normal((6, c.H))
    y0 = orc.dyn_conv(c, cv.w1[0], cv.w2[0], u)
    for t in range(6):
        u2 = u.copy()
        u2[t] += rng.standard_normal(c.H)
        y1 = orc.dyn_conv(c, cv.w1[0], cv.w2[0], u2)
        changed = np.where(np.abs(y1 - y0).max(axis=1) > 0)[0].tolist()
        assert changed == [r for r in (t, t + 1) if r < 6], (t, changed)


def test_dyn_conv_zero_generator_is_identity(orc):
    w, _, om = _conv_model()
    c, cv = om.draft.cfg, om.draft.layers[0].conv
    u = np.random.default_rng(3).standard_normal((4, c.H))
    np.testing.assert_array_equal(orc.dyn_conv(c, cv.w1[1], np.zeros_like(cv.w2[1]), u), u)
    np.testing.assert_array_equal(orc.dyn_conv(c, np.zeros_like(cv.w1[1]), cv.w2[1], u), u)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_draft_layer_with_conv_matches_torch(orc, dtype):
    """The draft layer with its four convolutions (attention input / output,
    MLP input / output), bidirectional over injected context, against the
    float64 torch restatement with F.scaled_dot_product_attention."""
    w, _, om = _conv_model(dtype)
    c, L = om.draft.cfg, om.draft.layers[1]
    rng = np.random.default_rng(4)
    P, M = 11, 5
    kc = np.zeros((c.nkv, 16, c.d)); vc = np.zeros((c.nkv, 16, c.d))
    ctx_k = orc.rnd(c, rng.standard_normal((P, c.nkv, c.d)))
    ctx_v = orc.rnd(c, rng.standard_normal((P, c.nkv, c.d)))
    kc[:, :P] = ctx_k.transpose(1, 0, 2); vc[:, :P] = ctx_v.transpose(1, 0, 2)
    h0 = rng.standard_normal((M, c.H))
    h = h0.copy()
    orc.decoder_layer(c, L, h, P, orc.BIDIR, kc, vc)
    ref, _, _ = Hh.torch_layer(c, L, torch.from_numpy(h0), torch.arange(P, P + M),
                               ctx_k=torch.from_numpy(ctx_k), ctx_v=torch.from_numpy(ctx_v), causal=False)
    tol = 1e-10 if dtype == "f32" else 2e-2
    np.testing.assert_allclose(h, ref.numpy(), rtol=0, atol=tol)
    plain = h0.copy()
    L0 = orc.Layer(**{k: getattr(L, k) for k in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g1", "g2")})
    orc.decoder_layer(c, L0, plain, P, orc.BIDIR, kc, vc)
    assert np.abs(plain - h).max() > 1e-3  # the convolutions do change the layer


def test_draft_layer_zero_conv_equals_plain_layer(orc):
    """Zero tap generators: every convolution returns its input exactly, so
    the layer equals the layer without them, bit for bit."""
    w, _, om = _conv_model("bf16")
    c, L = om.draft.cfg, om.draft.layers[0]
    z = orc.Conv([a.copy() for a in L.conv.w1], [np.zeros_like(a) for a in L.conv.w2])
    Lz = orc.Layer(L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd, L.g1, L.g2, z)
    L0 = orc.Layer(L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd, L.g1, L.g2)
    rng = np.random.default_rng(5)
    kc = rng.standard_normal((c.nkv, 16, c.d)); vc = rng.standard_normal((c.nkv, 16, c.d))
    h0 = rng.standard_normal((4, c.H))
    a = h0.copy(); orc.decoder_layer(c, Lz, a, 9, orc.BIDIR, kc, vc)
    b = h0.copy(); orc.decoder_layer(c, L0, b, 9, orc.BIDIR, kc, vc)
    np.testing.assert_array_equal(a, b)
