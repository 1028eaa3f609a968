"""Parity at the 32-sequence ragged verification shapes (Qwen3-8B dims,
contexts U[1024, 8192], 16-row blocks: 512 token rows per launch, split by
the library into launches of whole sequences): one causal target layer and
verification over the full 151936-entry vocabulary.  Sampled sequences are
compared with the oracle; every sampled sequence is also re-run alone and
must reproduce its rows of the 32-sequence launch bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from block_diffusion_speculative_step_gb300.engine import Engine
from oracle import oracle as O
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

S = 32
SAMPLED = (0, 19, 31)


@pytest.fixture(scope="module")
def b32():
    w = synth.WORKLOADS["qwen3-8b-b32"]
    w = dataclasses.replace(w, target=dataclasses.replace(w.target, layers=1),
                            draft=dataclasses.replace(w.draft, layers=1), taps=(0, 0, 0, 0, 0))
    m = synth.make_model(w, seed=6, device="cuda", jitter=0.1)
    ctx = synth.make_ctx_lengths(0, w)
    eng = Engine(w, m, S, w.ctx + 64, prefill_chunk=16)
    g = torch.Generator(device="cuda").manual_seed(11)
    for t in eng.caches.tk + eng.caches.tv:
        t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(t.dtype))
    torch.cuda.synchronize()
    return w, m, eng, ctx


def ocfg(w, s):
    return O.Cfg(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, True, w.rope_theta, w.rms_eps)


def _elem(t):
    return t.element_size()


def test_b32_causal_layer(b32):
    w, m, eng, ctx = b32
    B, H = w.block, w.target.hidden
    eng.base_pos.copy_(torch.tensor(ctx, dtype=torch.int32))
    h0 = torch.randn(S * B, H, generator=torch.Generator().manual_seed(1))
    eng.h[:S * B].copy_(h0.cuda())
    kc = {s: G.f64(eng.caches.tk[0][s]) for s in SAMPLED}
    vc = {s: G.f64(eng.caches.tv[0][s]) for s in SAMPLED}
    bufs = G.stage_buffers(w.target, S, B, bidir=False)
    D.dflash_decoder_layer_forward(G.attach_stages(eng.target_layer_args(0, B, eng.h), bufs), eng.ws_ptr,
                                   eng.ws_bytes)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    got = eng.h[:S * B].clone()
    n = synth.to_numpy
    L = m["target"]["layers"][0]
    ol = O.Layer.from_stacked(ocfg(w, w.target), n(L["w_qkv"]), n(L["w_o"]), n(L["w_gu"]), n(L["w_down"]),
                              n(L["ln1"]), n(L["ln2"]))
    kt, vt = eng.caches.tk[0], eng.caches.tv[0]
    for s in SAMPLED:
        # every stage against the oracle fed the GPU's inputs to it
        kr = G.f64(kt[s, :, ctx[s]:ctx[s] + B])
        vr = G.f64(vt[s, :, ctx[s]:ctx[s] + B])
        rep = G.check_layer_tf(O, ocfg(w, w.target), ol, h0[s * B:(s + 1) * B].double().numpy(), ctx[s], O.CAUSAL,
                               kc[s], vc[s], G.gpu_stages(bufs, s, B, kr, vr), G.f64(got[s * B:(s + 1) * B]))
        print(f"PARITY b32 causal layer, sequence {s} (context {ctx[s]}):", rep)
        # alone: the same rows from a one-sequence launch
        eng.h[:B].copy_(h0[s * B:(s + 1) * B].cuda())
        a = eng.target_layer_args(0, B, eng.h)
        a.n_seqs = 1
        a.base_pos = eng.base_pos.data_ptr() + 4 * s
        a.kv = D.dflash_kv(kt.data_ptr() + s * kt.stride(0) * _elem(kt), vt.data_ptr() + s * vt.stride(0) * _elem(vt),
                           eng.cap, 0)
        D.dflash_decoder_layer_forward(a, eng.ws_ptr, eng.ws_bytes)
        torch.cuda.synchronize()
        assert torch.equal(eng.h[:B], got[s * B:(s + 1) * B])


def test_b32_verify_accept(b32):
    w, m, eng, ctx = b32
    B, H = w.block, w.target.hidden
    h0 = torch.randn(S * B, H, generator=torch.Generator().manual_seed(4))
    drafts = torch.randint(0, w.vocab, (S, B - 1), generator=torch.Generator().manual_seed(5), dtype=torch.int32)
    eng.h[:S * B].copy_(h0.cuda())
    dd = drafts.cuda()
    eng.verify(B, dd)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    am_all, mg_all = eng.argmax.clone(), eng.margin.clone()
    acc_all = eng.accept_len.clone()
    # oracle on one sampled sequence
    s = SAMPLED[1]
    tc = ocfg(w, w.target)
    x = O.final_norm(tc, h0[s * B:(s + 1) * B].double().numpy(), synth.to_numpy(m["target"]["final_norm"]))
    am, mg, _ = O.lm_head_argmax(tc, synth.to_numpy(m["lm_head"]), x)
    G.check_argmax(am_all[s].cpu().numpy(), am, mg)
    np.testing.assert_allclose(mg_all[s].cpu().numpy(), mg, rtol=0, atol=1e-3)
    k, _ = O.accept(drafts[s].numpy(), am_all[s].cpu().numpy())
    assert int(acc_all[s]) == k
    # every sampled sequence alone reproduces its rows bit for bit
    for s in SAMPLED:
        eng.h[:B].copy_(h0[s * B:(s + 1) * B].cuda())
        a = eng.verify_args(B, eng.h, dd[s:s + 1], update=False)
        a.n_seqs = 1
        D.dflash_verify_accept(a, eng.ws_ptr, eng.ws_bytes)
        torch.cuda.synchronize()
        assert torch.equal(eng.argmax[0], am_all[s])
        assert torch.equal(eng.margin[0], mg_all[s])
        assert int(eng.accept_len[0]) == int(acc_all[s])
