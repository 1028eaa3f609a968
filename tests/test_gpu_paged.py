"""Paged KV caches (page pools + per-sequence page tables, pages handed out
in a shuffled order) on the GPU: every call returns what the contiguous call
returns, bit for bit -- the layer (causal, ragged positions crossing pages),
the windowed draft block, the context fusion writes, whole speculative
generation -- and matches the oracle; an unmapped page id raises the range
status instead of touching memory outside the pool."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from oracle import oracle as O
from tests import gpu_common as G
from tests.test_gpu_parity import rand_cache, small

pytestmark = pytest.mark.gpu


def _pair(w, S, cap, seed=0):
    """Two engines with the same weights: one stays contiguous, one is paged later."""
    a, om, _ = G.setup(w, seed=seed, S=S, cap=cap)
    b, _, _ = G.setup(w, seed=seed, S=S, cap=cap)
    return a, b, om


def _same_caches(a, b):
    ub = b.unpaged_caches()
    for kind, ks, vs in (("t", a.caches.tk, a.caches.tv), ("d", a.caches.dk, a.caches.dv)):
        for x, y in zip(ks + vs, ub[kind][0] + ub[kind][1]):
            assert torch.equal(x, y), kind


@pytest.mark.parametrize("dtype,d,ps", [("f32", 64, 128), ("bf16", 64, 128), ("bf16", 128, 256)])
def test_paged_causal_layer(dtype, d, ps):
    w = small(dtype, d=d)
    S, rows, cap = 3, 8, 512
    a, b, om = _pair(w, S, cap)
    base = [5, 300, 124]  # ragged; the last block straddles a 128-slot page boundary
    kc = vc = None
    for e in (a, b):
        e.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
        kc, vc = rand_cache(e, e.caches.tk[1], e.caches.tv[1], S, 300, 1, None)
    b.page_caches(ps, seed=7, spare_pages=3)
    h0 = torch.randn(S * rows, w.target.hidden, generator=torch.Generator().manual_seed(2))
    for e in (a, b):
        e.h[:S * rows].copy_(h0.cuda())
        D.dflash_decoder_layer_forward(e.target_layer_args(1, rows, e.h), e.ws_ptr, e.ws_bytes)
    torch.cuda.synchronize()
    assert b.status() == D.DFLASH_OK
    np.testing.assert_array_equal(G.f64(b.h[:S * rows]), G.f64(a.h[:S * rows]))
    _same_caches(a, b)
    c, L = om.target.cfg, om.target.layers[1]
    got = G.f64(b.h[:S * rows])
    for s in range(S):
        hs = h0[s * rows:(s + 1) * rows].double().numpy().copy()
        O.decoder_layer(c, L, hs, base[s], O.CAUSAL, kc[s].copy(), vc[s].copy())
        np.testing.assert_allclose(got[s * rows:(s + 1) * rows], hs, rtol=0, atol=1e-4 if dtype == "f32" else 2e-2)


@pytest.mark.parametrize("dtype,window", [("f32", 0), ("bf16", 0), ("bf16", 256)])
def test_paged_draft_block(dtype, window):
    w = small(dtype, window=window)
    S = 2
    a, b, om = _pair(w, S, 512)
    base = [200, 400]
    for e in (a, b):
        e.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
        e.anchor.copy_(torch.tensor([17, 400], dtype=torch.int32))
        for j in range(w.draft.layers):
            rand_cache(e, e.caches.dk[j], e.caches.dv[j], S, e.dcap, 10 + j, None)
    b.page_caches(128, seed=9, spare_pages=2)
    out = []
    for e in (a, b):
        logits = torch.zeros(S * (w.block - 1), w.vocab, device="cuda")
        e.draft(logits)
        torch.cuda.synchronize()
        assert e.status() == D.DFLASH_OK
        out.append((e.drafts.cpu().numpy().copy(), logits.cpu().numpy()))
    np.testing.assert_array_equal(out[1][0], out[0][0])
    np.testing.assert_array_equal(out[1][1], out[0][1])


@pytest.mark.parametrize("window", [0, 256])
def test_paged_fuse_context(window):
    w = small("bf16", window=window)
    S, rows = 2, 6
    a, b, om = _pair(w, S, 512)
    b.page_caches(128, seed=11)
    feats = synth.make_features(5, S * rows, len(w.taps), w.draft.hidden, synth.torch_dtype(w))
    vld = torch.tensor([6, 3], dtype=torch.int32, device="cuda")
    for e in (a, b):
        e.base_pos.copy_(torch.tensor([0, 379], dtype=torch.int32))  # 379..384 crosses a page
        e.feats[:S * rows].copy_(feats.cuda())
        D.dflash_fuse_context(e.fuse_args(rows, e.feats, e.base_pos, vld), e.ws_ptr, e.ws_bytes)
    torch.cuda.synchronize()
    assert b.status() == D.DFLASH_OK
    _same_caches(a, b)


@pytest.mark.parametrize("ps", [128, 256])
def test_paged_speculative_generation(ps):
    """Whole cycles on paged caches (target and draft; the 3 x 99-row prefill
    also takes the per-sequence launch split) reproduce the plain greedy
    continuation computed on contiguous caches."""
    w = small("bf16", V=512, block=6)
    S, n, cap = 3, 40, 256
    m_cpu = synth.make_model(w, seed=3, jitter=0.1, with_target=True)
    prompts = torch.stack([synth.make_tokens(10 + s, 100, w.vocab) for s in range(S)]).cuda()
    from block_diffusion_speculative_step_gb300.engine import Engine
    greedy = Engine(w, G.to_dev(m_cpu), S, cap).greedy_generate(prompts, n)
    paged = Engine(w, G.to_dev(m_cpu), S, cap)
    paged.page_caches(ps, seed=5, spare_pages=1)
    spec, acc = paged.speculative_generate(prompts, n)
    assert paged.status() == D.DFLASH_OK
    np.testing.assert_array_equal(spec.numpy(), greedy.numpy())
    assert int(acc.max()) <= w.block - 1


def test_unmapped_page_raises_range_status():
    """A page id outside the pool: the kernels' own checks skip its writes,
    read page 0 in its place and raise the range status (reported as an
    invalid argument); nothing outside the pool is touched."""
    w = small("bf16")
    S, rows = 2, 8
    e, om, _ = G.setup(w, S=S, cap=256)
    e.base_pos.copy_(torch.tensor([5, 130], dtype=torch.int32))
    e.page_caches(128, seed=1)
    table, ps, mp, pool = e.paging["t"]
    table[1, 1] = pool + 5  # sequence 1's second page: unmapped
    e.h[:S * rows].normal_()
    D.dflash_decoder_layer_forward(e.target_layer_args(0, rows, e.h), e.ws_ptr, e.ws_bytes)
    torch.cuda.synchronize()
    assert e.status() == D.DFLASH_ERR_INVALID_ARG
