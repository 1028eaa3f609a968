"""Parity at the full Qwen3-8B-shaped sizes of the benchmark workload, in the
launch configuration the benchmark times (batch 1, 16-row block, context
4096, the tcgen05 stream-K GEMMs, the cluster attention, the fused LM-head
argmax): one causal target layer, the five-layer draft block with its LM
head, the context fusion into five draft layers, and verification over the
full 151936-entry vocabulary.  The oracle (OpenMP over output rows) computes
every output at these sizes in seconds, so all of them are compared; layers
are compared stage by stage against the oracle fed the GPU's own inputs."""
import dataclasses

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from block_diffusion_speculative_step_gb300.engine import Engine
from oracle import oracle as O
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu

CTX = 4096


@pytest.fixture(scope="module")
def big():
    w = synth.WORKLOADS["qwen3-8b-b1"]
    w = dataclasses.replace(w, target=dataclasses.replace(w.target, layers=1),
                            draft=dataclasses.replace(w.draft, layers=5), taps=(0, 0, 0, 0, 0))
    m = synth.make_model(w, seed=5, device="cuda", jitter=0.1)
    eng = Engine(w, m, 1, CTX + 64, prefill_chunk=16)
    g = torch.Generator(device="cuda").manual_seed(9)
    for t in eng.caches.tk + eng.caches.tv + eng.caches.dk + eng.caches.dv:
        t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(t.dtype))
    torch.cuda.synchronize()
    return w, m, eng


def ocfg(w, s):
    return O.Cfg(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, True, w.rope_theta, w.rms_eps)


def olayer(w, s, L):
    n = synth.to_numpy
    return O.Layer.from_stacked(ocfg(w, s), n(L["w_qkv"]), n(L["w_o"]), n(L["w_gu"]), n(L["w_down"]), n(L["ln1"]),
                                n(L["ln2"]))


def test_fullsize_causal_layer(big):
    """One Qwen3-8B-shaped target layer over a 16-row block at position 4096,
    every stage checked against the oracle fed the GPU's inputs to it."""
    w, m, eng = big
    B = w.block
    eng.base_pos.fill_(CTX)
    h0 = torch.randn(B, w.target.hidden, generator=torch.Generator().manual_seed(1))
    eng.h[:B].copy_(h0.cuda())
    kc = G.f64(eng.caches.tk[0][0])
    vc = G.f64(eng.caches.tv[0][0])
    bufs = G.stage_buffers(w.target, 1, B, bidir=False)
    a = G.attach_stages(eng.target_layer_args(0, B, eng.h), bufs)
    D.dflash_decoder_layer_forward(a, eng.ws_ptr, eng.ws_bytes)
    assert eng.status() == D.DFLASH_OK
    got = G.f64(eng.h[:B])
    # the block's K/V went into the cache at positions CTX .. CTX+B-1
    kr = G.f64(eng.caches.tk[0][0, :, CTX:CTX + B])
    vr = G.f64(eng.caches.tv[0][0, :, CTX:CTX + B])
    rep = G.check_layer_tf(O, ocfg(w, w.target), olayer(w, w.target, m["target"]["layers"][0]),
                           h0.double().numpy(), CTX, O.CAUSAL, kc, vc, G.gpu_stages(bufs, 0, B, kr, vr), got)
    print("PARITY causal layer (teacher-forced):", rep)


def test_fullsize_draft_block(big):
    """The benchmark's draft block at full size: five Qwen3-8B-shaped draft
    layers over a 4096-position injected context, block 16, the 151936-entry
    LM head with its fused argmax.  Every layer teacher-forced, the LM head
    at the stated logit bound, drafts bit for bit up to reported near-ties;
    the end-to-end logit difference against the oracle's whole draft
    forward is reported."""
    w, m, eng = big
    B = w.block
    eng.base_pos.fill_(CTX)
    eng.anchor.fill_(4321)
    logits = torch.zeros(B - 1, w.vocab, device="cuda")
    eng.draft(logits)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    gd = eng.drafts[0].cpu().numpy()
    gl = logits.cpu().numpy()
    np.testing.assert_array_equal(gd, gl.argmax(-1))  # the fused argmax is the argmax of the logits
    om = Hh.omodel(w, m)
    rep = G.draft_parity(O, om, eng, 0, gl, gd)
    print("PARITY qwen3-8b draft block:", {k: v for k, v in rep.items() if k != "layers"},
          "layer h err", [round(L["h"], 7) for L in rep["layers"]])


def test_fullsize_fusion(big):
    w, m, eng = big
    F, H, B = len(w.taps), w.draft.hidden, w.block
    feats = synth.make_features(3, B, F, H, torch.bfloat16).cuda()
    eng.feats[:B].copy_(feats)
    base = torch.full((1,), CTX, dtype=torch.int32, device="cuda")
    valid = torch.full((1,), 11, dtype=torch.int32, device="cuda")
    cout = torch.zeros(B, H, device="cuda")
    a = eng.fuse_args(B, eng.feats, base, valid)
    a.c_out = cout.data_ptr()
    D.dflash_fuse_context(a, eng.ws_ptr, eng.ws_bytes)
    torch.cuda.synchronize()
    n = synth.to_numpy
    dc = ocfg(w, w.draft)
    wk = [olayer(w, w.draft, L).wk for L in m["draft"]["layers"]]
    wv = [olayer(w, w.draft, L).wv for L in m["draft"]["layers"]]
    kcs = [np.zeros((w.draft.n_kv, eng.dcap, w.draft.head_dim)) for _ in wk]
    vcs = [np.zeros((w.draft.n_kv, eng.dcap, w.draft.head_dim)) for _ in wk]
    pos = list(range(CTX, CTX + 11))
    cref = O.fuse_context(dc, F, n(m["fc"]), n(m["fc_norm"]), G.f64(feats[:11].reshape(11, F * H)), pos, wk, wv,
                          kcs, vcs)
    G.assert_bf16_close(G.f64(cout[:11]), cref)
    for j in range(w.draft.layers):
        G.assert_bf16_close(G.f64(eng.caches.dk[j][0, :, CTX:CTX + 11]), kcs[j][:, CTX:CTX + 11])
        G.assert_bf16_close(G.f64(eng.caches.dv[j][0, :, CTX:CTX + 11]), vcs[j][:, CTX:CTX + 11])


def test_fullsize_verify_accept(big):
    w, m, eng = big
    B, H = w.block, w.target.hidden
    h0 = torch.randn(B, H, generator=torch.Generator().manual_seed(4))
    eng.h[:B].copy_(h0.cuda())
    tc = ocfg(w, w.target)
    x = O.final_norm(tc, h0.double().numpy(), synth.to_numpy(m["target"]["final_norm"]))
    am, mg, _ = O.lm_head_argmax(tc, synth.to_numpy(m["lm_head"]), x)
    drafts = am[:B - 1].copy()
    drafts[9] = (drafts[9] + 1) % w.vocab  # accept exactly 9 unless a near-tie intervenes
    eng.drafts.copy_(torch.from_numpy(drafts.astype(np.int32))[None])
    eng.base_pos.fill_(CTX)
    eng.verify(B, eng.drafts)
    torch.cuda.synchronize()
    gam = eng.argmax[0].cpu().numpy()
    excluded = G.check_argmax(gam, am, mg)
    k, out = O.accept(drafts, gam)
    assert int(eng.accept_len[0]) == k
    np.testing.assert_array_equal(eng.out_tokens[0, :k + 1].cpu().numpy(), out)
    if excluded == 0:
        assert k == 9
    np.testing.assert_allclose(eng.margin[0].cpu().numpy(), mg, rtol=0, atol=1e-3)
    # the verification logits themselves, at the stated bound
    logits = torch.zeros(B, w.vocab, device="cuda")
    eng.base_pos.fill_(CTX)
    eng.verify(B, eng.drafts, logits)
    torch.cuda.synchronize()
    _, _, lg = O.lm_head_argmax(tc, synth.to_numpy(m["lm_head"]), x, want_logits=True)
    err = float(np.abs(logits.cpu().numpy() - lg).max())
    assert err <= G.LOGIT_TOL["bf16"], f"verification logits differ by {err}"
    print("PARITY qwen3-8b verify logits max err", err)
