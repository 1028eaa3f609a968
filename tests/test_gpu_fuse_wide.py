"""Context-feature fusion and KV injection over many token rows: 20
sequences x 8 rows = 160 rows, so the FC and the K/V projections run with
160-column tiles, the shared-memory row table and the separate split-K
fixup kernel, with ragged valid-row counts (0 to 8).  Two sequences are
compared with the oracle; every sequence is also injected alone (8 rows:
the 16-column path whose last piece finishes the tile) and must give the
same fused rows and the same draft K/V bit for bit."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from oracle import oracle as O
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu


def _small(window):
    return Hh.small_workload(dtype="bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=3, d_layers=2,
                             taps=(0, 1), block=8, window=window)


@pytest.mark.parametrize("window", [0, 16])
def test_fuse_many_rows_matches_alone_and_oracle(window):
    w = _small(window)
    S, rows, cap = 20, 8, 64
    eng, om, m = G.setup(w, S=S, cap=cap)
    g = torch.Generator().manual_seed(21)
    base = torch.randint(0, 40, (S,), generator=g).to(torch.int32)
    valid = torch.randint(0, rows + 1, (S,), generator=g).to(torch.int32)
    valid[0], valid[1], valid[2] = rows, 0, 3
    eng.base_pos.copy_(base)
    vld = valid.cuda()
    F, H = len(w.taps), w.draft.hidden
    feats = synth.make_features(7, S * rows, F, H, synth.torch_dtype(w))
    eng.feats[:S * rows].copy_(feats.cuda())
    nl = w.draft.layers

    def clear():
        for t in eng.caches.dk + eng.caches.dv:
            t.zero_()

    # all sequences in one call
    clear()
    cout = torch.zeros(S * rows, H, device="cuda")
    a = eng.fuse_args(rows, eng.feats, eng.base_pos, vld)
    a.c_out = cout.data_ptr()
    D.dflash_fuse_context(a, eng.ws_ptr, eng.ws_bytes)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    batched = (cout.clone(), [t.clone() for t in eng.caches.dk], [t.clone() for t in eng.caches.dv])

    # every sequence alone (pointers into the same buffers)
    clear()
    cout1 = torch.zeros(S * rows, H, device="cuda")
    for s in range(S):
        b = eng.fuse_args(rows, eng.feats[s * rows:(s + 1) * rows], eng.base_pos[s:], vld[s:])
        b.n_seqs = 1
        for j in range(nl):
            b.kv_layers[j] = D.dflash_kv(eng.caches.dk[j][s].data_ptr(), eng.caches.dv[j][s].data_ptr(),
                                         eng.dcap, w.window)
        b.c_out = cout1[s * rows:].data_ptr()
        D.dflash_fuse_context(b, eng.ws_ptr, eng.ws_bytes)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    for s in range(S):
        n = int(valid[s])
        assert torch.equal(batched[0][s * rows:s * rows + n], cout1[s * rows:s * rows + n]), s
    for j in range(nl):
        assert torch.equal(batched[1][j], eng.caches.dk[j]), j
        assert torch.equal(batched[2][j], eng.caches.dv[j]), j

    # the oracle, for a full and a partial sequence
    for s in (0, 2):
        n = int(valid[s])
        st = O.new_state(om, cap)
        f = G.f64(feats[s * rows:s * rows + n].reshape(n, F * H))
        pos = list(range(int(base[s]), int(base[s]) + n))
        cref = O.fuse(om, st, f, pos)
        np.testing.assert_allclose(G.f64(batched[0][s * rows:s * rows + n]), cref, rtol=0, atol=3e-2)
        for j in range(nl):
            for t in pos:
                slot = t % window if window else t
                np.testing.assert_allclose(G.f64(batched[1][j][s, :, slot]), st.dk[j][:, slot], rtol=0, atol=3e-2)
                np.testing.assert_allclose(G.f64(batched[2][j][s, :, slot]), st.dv[j][:, slot], rtol=0, atol=3e-2)
