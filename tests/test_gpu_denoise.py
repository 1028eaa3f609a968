"""Multi-round block denoising on the GPU (dflash_draft_block with
denoise_rounds = R) against the oracle's draft_denoise.  Each round is
checked on its own: the oracle runs one round from the GPU's drafts of the
round before (its `init`), so a near-tie in an earlier round cannot make a
later comparison fail; logits within the tolerance, drafts bit-exact up to
reported near-ties."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from oracle import oracle as O
from tests import gpu_common as G
from tests.test_gpu_parity import _path_factors, rand_cache, small

pytestmark = pytest.mark.gpu


def _gpu_rounds(eng, S, B, V, R):
    """Drafts and logits of the GPU's runs with 1..R rounds."""
    out = []
    for r in range(1, R + 1):
        logits = torch.zeros(S * (B - 1), V, device="cuda")
        eng.draft(logits, rounds=r)
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        out.append((eng.drafts.cpu().numpy().copy(), logits.cpu().numpy().reshape(S, B - 1, V)))
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_denoise_rounds(dtype):
    w = small(dtype, window=0)
    S, B, R = 2, w.block, 3
    eng, om, _ = G.setup(w, S=S, cap=96)
    base = [9, 40]
    eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
    eng.anchor.copy_(torch.tensor([17, 400], dtype=torch.int32))
    dk, dv = [], []
    for j in range(w.draft.layers):
        k, v = rand_cache(eng, eng.caches.dk[j], eng.caches.dv[j], S, eng.dcap, 30 + j, om.draft.cfg)
        dk.append(k)
        dv.append(v)
    runs = _gpu_rounds(eng, S, B, w.vocab, R)
    for s in range(S):
        st = O.new_state(om, 96)
        st.dk = [k[s].copy() for k in dk]
        st.dv = [v[s].copy() for v in dv]
        prev = None
        for r, (gd, gl) in enumerate(runs):
            am, mg, lg = O.draft_denoise(om, st, int(eng.anchor[s]), base[s], 1, want_logits=True, init=prev)
            err = np.abs(gl[s] - lg).max()
            assert err <= G.LOGIT_TOL[dtype], f"seq {s} round {r + 1}: logits differ by {err}"
            G.check_argmax(gd[s], am, mg, tol=max(G.NEAR_TIE, 2 * err))
            np.testing.assert_array_equal(gd[s], gl[s].argmax(-1))
            prev = gd[s]  # the next round starts from the GPU's drafts
        # the rounds really feed back: round 2 reads drafts, not masks
        assert not np.array_equal(runs[0][1][s], runs[1][1][s])


def test_denoise_rounds_path_selector():
    """Every round ends with the DFlash 2 path walk; the next round reads the
    walked path.  Round r's logits are checked against the oracle started
    from the GPU's path of round r - 1, and the GPU's path of round r against
    the oracle's walk over the GPU's own logits (up to a score near-tie)."""
    w = small("bf16", V=1000, block=10, topk=16, rank=64)
    S, B, R = 2, w.block, 2
    eng, om, _ = G.setup(w, S=S, cap=96)
    Un, Vn = _path_factors(eng, w, 9, "bf16")
    base = [9, 40]
    eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
    eng.anchor.copy_(torch.tensor([17, 400], dtype=torch.int32))
    dk, dv = [], []
    for j in range(w.draft.layers):
        k, v = rand_cache(eng, eng.caches.dk[j], eng.caches.dv[j], S, eng.dcap, 40 + j, om.draft.cfg)
        dk.append(k)
        dv.append(v)
    runs = _gpu_rounds(eng, S, B, w.vocab, R)
    compared = 0
    for s in range(S):
        st = O.new_state(om, 96)
        st.dk = [k[s].copy() for k in dk]
        st.dv = [v[s].copy() for v in dv]
        prev = None
        for r, (gp, gl) in enumerate(runs):
            _, _, lg = O.draft_denoise(om, st, int(eng.anchor[s]), base[s], 1, want_logits=True, init=prev)
            err = np.abs(gl[s] - lg).max()
            assert err <= G.LOGIT_TOL["bf16"], f"seq {s} round {r + 1}: logits differ by {err}"
            path, _, mg = O.path_select(om.draft.cfg, gl[s], om.E, Un, Vn, int(eng.anchor[s]), topk=16)
            for j in range(B - 1):
                if mg[j] < 1e-4:
                    break
                assert gp[s, j] == path[j], f"seq {s} round {r + 1} step {j}"
                compared += 1
            prev = gp[s]
    assert compared >= S * R * (B - 1) // 2
