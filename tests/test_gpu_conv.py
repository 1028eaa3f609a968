"""DFlash 2 two-tap dynamic depthwise convolutions in the draft layers on the
GPU (dflash_draft_block with conv_rank > 0) against the oracle's draft with
the same convolutions; logits within the tolerance, drafts bit-exact up to
reported near-ties.  Zero tap generators must reproduce the draft without
convolutions bit for bit, and a sequence's drafts must not depend on the
batch."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from oracle import oracle as O
from tests import gpu_common as G
from tests.test_gpu_parity import rand_cache, small

pytestmark = pytest.mark.gpu


def _setup(dtype, S, r=16, window=0):
    w = small(dtype, window=window, conv_rank=r)
    eng, om, _ = G.setup(w, S=S, cap=96)
    base = [9, 40, 23][:S]
    eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
    eng.anchor.copy_(torch.tensor([17, 400, 5][:S], dtype=torch.int32))
    dk, dv = [], []
    for j in range(w.draft.layers):
        k, v = rand_cache(eng, eng.caches.dk[j], eng.caches.dv[j], S, eng.dcap, 50 + j, om.draft.cfg)
        dk.append(k)
        dv.append(v)
    return w, eng, om, base, dk, dv


def _run(eng, w, S, **kw):
    logits = torch.zeros(S * (w.block - 1), w.vocab, device="cuda")
    eng.draft(logits, **kw)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    return eng.drafts.cpu().numpy().copy(), logits.cpu().numpy().reshape(S, w.block - 1, w.vocab)


@pytest.mark.parametrize("dtype,window", [("f32", 0), ("bf16", 0), ("bf16", 24)])
def test_draft_block_with_conv(dtype, window):
    S = 2
    w, eng, om, base, dk, dv = _setup(dtype, S, window=window)
    gd, gl = _run(eng, w, S)
    _, gl0 = _run(eng, w, S, conv_rank=0)
    for s in range(S):
        st = O.new_state(om, 96)
        st.dk = [k[s].copy() for k in dk]
        st.dv = [v[s].copy() for v in dv]
        am, mg, lg = O.draft_forward(om, st, int(eng.anchor[s]), base[s], want_logits=True)
        err = np.abs(gl[s] - lg).max()
        assert err <= G.LOGIT_TOL[dtype], f"draft logits with convolutions differ by {err}"
        G.check_argmax(gd[s], am, mg, tol=max(G.NEAR_TIE, 2 * err))
        np.testing.assert_array_equal(gd[s], gl[s].argmax(-1))
        # the convolutions move the logits by more than the GPU / oracle disagreement
        assert np.abs(gl0[s] - lg).max() > 2 * err + 1e-6


def test_zero_conv_generators_reproduce_plain_draft():
    S = 2
    w, eng, om, base, dk, dv = _setup("bf16", S)
    for L in eng.m["draft"]["layers"]:
        L["conv_w2"].zero_()
    gd, gl = _run(eng, w, S)
    pd, pl = _run(eng, w, S, conv_rank=0)
    np.testing.assert_array_equal(gl, pl)
    np.testing.assert_array_equal(gd, pd)


def test_conv_rows_independent_of_batch():
    """Each sequence of a 3-sequence draft equals the same sequence drafted
    alone (same seed, so the same weights), bit for bit."""
    S = 3
    w, eng, om, base, dk, dv = _setup("bf16", S)
    gd, gl = _run(eng, w, S)
    for s in range(S):
        e1, _, _ = G.setup(w, S=1, cap=96)
        e1.base_pos.copy_(eng.base_pos[s:s + 1])
        e1.anchor.copy_(eng.anchor[s:s + 1])
        for j in range(w.draft.layers):
            e1.caches.dk[j].copy_(eng.caches.dk[j][s:s + 1])
            e1.caches.dv[j].copy_(eng.caches.dv[j][s:s + 1])
        d1, l1 = _run(e1, w, 1)
        np.testing.assert_array_equal(l1[0], gl[s])
        np.testing.assert_array_equal(d1[0], gd[s])
