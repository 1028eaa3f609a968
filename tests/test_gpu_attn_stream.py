"""The streaming tcgen05 attention (one CTA per SM, the logical ranks of the
cluster kernel as work units, partials merged by the CTA that completes an
item) against the cluster kernel it stands in for: the same layer, draft
block and paged calls with DFLASH_ATTN_STREAM=1 and =0 must agree bit for
bit -- ragged and very short contexts (fewer chunks than logical ranks),
the bidirectional block chunk, sliding windows, page tables -- and match the
oracle; a stalled streaming launch reports the timeout and leaves the item
counters ready for the next call."""
import os

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from oracle import oracle as O
from tests import gpu_common as G
from tests.test_gpu_parity import rand_cache, small

pytestmark = pytest.mark.gpu


class _Attn:
    """Selects the attention kernel for the calls inside the block."""

    def __init__(self, stream: bool):
        self.v = "1" if stream else "0"

    def __enter__(self):
        self.old = os.environ.get("DFLASH_ATTN_STREAM")
        os.environ["DFLASH_ATTN_STREAM"] = self.v

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop("DFLASH_ATTN_STREAM", None)
        else:
            os.environ["DFLASH_ATTN_STREAM"] = self.old


def _wl(**kw):
    # head dim 128 and a GQA group of 4: the tcgen05 kernels
    return small("bf16", d=128, nq=8, nkv=2, **kw)


def _layer(eng, rows, h0, base, layer=1):
    eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
    eng.h[:len(base) * rows].copy_(h0.cuda())
    D.dflash_decoder_layer_forward(eng.target_layer_args(layer, rows, eng.h), eng.ws_ptr, eng.ws_bytes)
    torch.cuda.synchronize()
    return eng.status(), G.f64(eng.h[:len(base) * rows])


@pytest.mark.parametrize("rows,base", [(8, [0, 5, 129, 700, 1000]), (16, [3, 1007, 250])])
def test_stream_causal_layer_matches_cluster(rows, base):
    w = _wl(block=rows)
    S, cap = len(base), 1024
    eng, om, _ = G.setup(w, S=S, cap=cap)
    kc, vc = rand_cache(eng, eng.caches.tk[1], eng.caches.tv[1], S, cap, 1, None)
    h0 = torch.randn(S * rows, w.target.hidden, generator=torch.Generator().manual_seed(2))
    out = {}
    for stream in (False, True):
        with _Attn(stream):
            st, out[stream] = _layer(eng, rows, h0, base)
        assert st == D.DFLASH_OK
    np.testing.assert_array_equal(out[True], out[False])
    c, L = om.target.cfg, om.target.layers[1]
    for s in range(S):
        hs = h0[s * rows:(s + 1) * rows].double().numpy().copy()
        O.decoder_layer(c, L, hs, base[s], O.CAUSAL, kc[s].copy(), vc[s].copy())
        np.testing.assert_allclose(out[True][s * rows:(s + 1) * rows], hs, rtol=0, atol=G.LOGIT_TOL["bf16"])


@pytest.mark.parametrize("window", [0, 256])
def test_stream_draft_block_matches_cluster(window):
    w = _wl(window=window)
    S = 4
    eng, _, _ = G.setup(w, S=S, cap=1024)
    base = [40, 1000, 300, 129]
    eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
    for j in range(w.draft.layers):
        rand_cache(eng, eng.caches.dk[j], eng.caches.dv[j], S, eng.dcap, 10 + j, None)
    out = {}
    for stream in (False, True):
        eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
        eng.anchor.copy_(torch.tensor([17, 400, 3, 999], dtype=torch.int32))
        logits = torch.zeros(S * (w.block - 1), w.vocab, device="cuda")
        with _Attn(stream):
            eng.draft(logits)
            torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        out[stream] = (eng.drafts.cpu().numpy().copy(), logits.cpu().numpy())
    np.testing.assert_array_equal(out[True][1], out[False][1])
    np.testing.assert_array_equal(out[True][0], out[False][0])


def test_stream_paged_layer_matches_contiguous_cluster():
    w = _wl()
    S, rows, cap = 3, 8, 1024
    a, _, _ = G.setup(w, S=S, cap=cap)
    b, _, _ = G.setup(w, S=S, cap=cap)
    base = [5, 900, 130]
    for e in (a, b):
        e.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
        rand_cache(e, e.caches.tk[1], e.caches.tv[1], S, cap, 1, None)
    b.page_caches(256, seed=7, spare_pages=3)
    h0 = torch.randn(S * rows, w.target.hidden, generator=torch.Generator().manual_seed(3))
    with _Attn(False):
        sa, ha = _layer(a, rows, h0, base)
    with _Attn(True):
        sb, hb = _layer(b, rows, h0, base)
    assert sa == D.DFLASH_OK and sb == D.DFLASH_OK
    np.testing.assert_array_equal(hb, ha)


def test_stream_timeout_then_recovers():
    """A stalled streaming launch gives up within its wait limit and reports
    DFLASH_ERR_TIMEOUT; every unit still arrives, so the item counters are
    back at zero and the next call on the same workspace is exact."""
    w = _wl()
    S, rows, cap = 3, 8, 1024
    eng, _, _ = G.setup(w, S=S, cap=cap)
    base = [5, 900, 130]
    rand_cache(eng, eng.caches.tk[1], eng.caches.tv[1], S, cap, 1, None)
    kc0, vc0 = eng.caches.tk[1].clone(), eng.caches.tv[1].clone()
    h0 = torch.randn(S * rows, w.target.hidden, generator=torch.Generator().manual_seed(4))
    with _Attn(True):
        st, ref = _layer(eng, rows, h0, base)
        assert st == D.DFLASH_OK
        D.dflash_workspace_control(eng.ws_ptr, eng.ws_bytes, wait_limit_ns=2_000_000, stall_kv_loads=True)
        eng.caches.tk[1].copy_(kc0)
        eng.caches.tv[1].copy_(vc0)
        st, _ = _layer(eng, rows, h0, base)
        assert st == D.DFLASH_ERR_TIMEOUT, st
        D.dflash_workspace_control(eng.ws_ptr, eng.ws_bytes)
        eng.caches.tk[1].copy_(kc0)
        eng.caches.tv[1].copy_(vc0)
        st, again = _layer(eng, rows, h0, base)
    assert st == D.DFLASH_OK
    np.testing.assert_array_equal(again, ref)
