"""Pins of the oracle's multi-round block denoising (draft_denoise): a
closed form built from an identity draft and a shifted LM head, the
one-round reduction, and the path-selector special case.  CPU only."""
import numpy as np
import torch

from block_diffusion_speculative_step_gb300 import synth
from tests import helpers as Hh


def _successor_model(dtype="f32", **kw):
    """A draft whose layers leave the residual unchanged (every projection
    zero: attention and MLP outputs are exactly 0) and whose LM head row v is
    the embedding of token v-1.  Then row j's logits are RMSNorm(e_x) . e_{v-1}
    for its input token x, which peak at v = x + 1 (mod V): a Gaussian
    embedding's self product dominates its cross products."""
    w = Hh.small_workload(dtype=dtype, **kw)
    m = synth.make_model(w, seed=3, jitter=0.1, with_target=True)
    for L in m["draft"]["layers"]:
        for k in ("w_qkv", "w_o", "w_gu", "w_down"):
            L[k].zero_()
    m["lm_head"] = torch.roll(m["embed"], 1, dims=0).contiguous()
    return w, Hh.omodel(w, m)


def test_denoise_rounds_closed_form(orc):
    """After R rounds every draft is (mask + R) mod V: round 1 reads the mask
    tokens, each later round reads row j's own previous draft.  A feedback
    that shifted rows (row j reading draft j-1, row 1 the anchor) would give
    anchor + R at row 1."""
    w, om = _successor_model(V=128, block=6)
    st = orc.new_state(om, 32)
    anchor = 5
    for R in range(1, 5):
        d, mg, _ = orc.draft_denoise(om, st, anchor, 7, R)
        np.testing.assert_array_equal(d, np.full(w.block - 1, (w.mask_id + R) % w.vocab))
        assert np.all(mg > 0)


def test_denoise_one_round_is_single_step(orc):
    w, om = Hh.small_workload(), None
    m = synth.make_model(w, seed=4, jitter=0.1, with_target=True)
    om = Hh.omodel(w, m)
    st = orc.new_state(om, 48)
    rng = np.random.default_rng(2)
    for li in range(len(om.draft.layers)):
        st.dk[li][:, :20] = rng.standard_normal(st.dk[li][:, :20].shape)
        st.dv[li][:, :20] = rng.standard_normal(st.dv[li][:, :20].shape)
    a1, m1, l1 = orc.draft_forward(om, st, 9, 20, want_logits=True)
    a2, m2, l2 = orc.draft_denoise(om, st, 9, 20, 1, want_logits=True)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(m1, m2)
    np.testing.assert_array_equal(l1, l2)


def test_denoise_zero_selector_is_plain_rounds(orc):
    """With U = V = 0 every pair score ties, the walk keeps rank 0 (the top-1
    draft) at every row, so the selector changes no round's drafts."""
    w = Hh.small_workload(dtype="bf16", V=128, block=5, topk=4, rank=8)
    m = synth.make_model(w, seed=5, jitter=0.1, with_target=True)
    om = Hh.omodel(w, m)
    st = orc.new_state(om, 48)
    rng = np.random.default_rng(3)
    for li in range(len(om.draft.layers)):
        st.dk[li][:, :16] = rng.standard_normal(st.dk[li][:, :16].shape)
        st.dv[li][:, :16] = rng.standard_normal(st.dv[li][:, :16].shape)
    z = np.zeros((8, w.draft.hidden), dtype=np.uint16)
    for R in (2, 3):
        plain, _, _ = orc.draft_denoise(om, st, 11, 16, R)
        walked, mg, _ = orc.draft_denoise(om, st, 11, 16, R, selector=(z, z, 4))
        np.testing.assert_array_equal(walked, plain)
        assert np.all(mg == 0.0)


def test_denoise_init_continues_rounds(orc):
    """Rounds compose: R rounds from the masks == R - r rounds started from
    the drafts of the first r rounds."""
    w = Hh.small_workload(V=128, block=5)
    m = synth.make_model(w, seed=6, jitter=0.1, with_target=True)
    om = Hh.omodel(w, m)
    st = orc.new_state(om, 48)
    rng = np.random.default_rng(4)
    for li in range(len(om.draft.layers)):
        st.dk[li][:, :16] = rng.standard_normal(st.dk[li][:, :16].shape)
        st.dv[li][:, :16] = rng.standard_normal(st.dv[li][:, :16].shape)
    d3, m3, l3 = orc.draft_denoise(om, st, 2, 16, 3, want_logits=True)
    d1, _, _ = orc.draft_denoise(om, st, 2, 16, 1)
    e2, n2, k2 = orc.draft_denoise(om, st, 2, 16, 2, want_logits=True, init=d1)
    np.testing.assert_array_equal(d3, e2)
    np.testing.assert_array_equal(m3, n2)
    np.testing.assert_array_equal(l3, k2)
