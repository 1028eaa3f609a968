"""Failure detection on the GPU, made to fire without a GPU fault.

- A bounded wait that cannot complete: the workspace's stall switch makes
  the attention kernels issue none of their K/V copies (nothing is in
  flight), and a short wait limit lets their waits give up.  The call must
  come back with DFLASH_ERR_TIMEOUT through dflash_read_status, and the same
  GPU context must then run the same layer correctly.
- A NaN that reaches the argmax: a hidden state poisoned on the host must
  come back as DFLASH_ERR_NUMERIC, and a clean call after it as DFLASH_OK.
"""
import time

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from oracle import oracle as O
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu


def _layer_setup():
    # head dim 128: the tcgen05 attention kernel
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=128, I=384, V=1000, t_layers=1, d_layers=1,
                          taps=(0, 0), block=8)
    S, rows = 2, w.block
    eng, om, _ = G.setup(w, S=S, cap=512)
    g = torch.Generator().manual_seed(5)
    for t in (eng.caches.tk[0], eng.caches.tv[0]):
        t[:, :, :300] = torch.randn(t[:, :, :300].shape, generator=g).to(t.dtype).cuda()
    base = [300, 137]
    h0 = torch.randn(S * rows, w.target.hidden, generator=torch.Generator().manual_seed(6))
    return w, eng, om, S, rows, base, h0


def _run_layer(eng, S, rows, base, h0):
    eng.base_pos.copy_(torch.tensor(base, dtype=torch.int32))
    eng.h[:S * rows].copy_(h0.cuda())
    D.dflash_decoder_layer_forward(eng.target_layer_args(0, rows, eng.h), eng.ws_ptr, eng.ws_bytes)
    return eng.status()


def test_wait_timeout_is_reported_and_the_gpu_stays_usable():
    w, eng, om, S, rows, base, h0 = _layer_setup()
    kc0, vc0 = G.f64(eng.caches.tk[0]), G.f64(eng.caches.tv[0])
    limit_ns = 2_000_000  # 2 ms
    D.dflash_workspace_control(eng.ws_ptr, eng.ws_bytes, wait_limit_ns=limit_ns, stall_kv_loads=True)
    t0 = time.perf_counter()
    st = _run_layer(eng, S, rows, base, h0)
    dt = time.perf_counter() - t0
    assert st == D.DFLASH_ERR_TIMEOUT, st
    assert "status word" in D.dflash_last_error()
    assert dt < 5.0, f"the stalled call took {dt:.2f} s with a {limit_ns / 1e6} ms wait limit"
    # the status word was cleared by the read; the controls are restored to
    # their defaults (1 s limit, copies issued), and the same context runs the
    # same layer correctly from fresh inputs
    D.dflash_workspace_control(eng.ws_ptr, eng.ws_bytes)
    eng.caches.tk[0].copy_(torch.from_numpy(kc0).to(eng.caches.tk[0].dtype).cuda())
    eng.caches.tv[0].copy_(torch.from_numpy(vc0).to(eng.caches.tv[0].dtype).cuda())
    assert _run_layer(eng, S, rows, base, h0) == D.DFLASH_OK
    got = G.f64(eng.h[:S * rows])
    c, L = om.target.cfg, om.target.layers[0]
    for s in range(S):
        hs = h0[s * rows:(s + 1) * rows].double().numpy().copy()
        O.decoder_layer(c, L, hs, base[s], O.CAUSAL, kc0[s].copy(), vc0[s].copy())
        np.testing.assert_allclose(got[s * rows:(s + 1) * rows], hs, rtol=0, atol=G.LOGIT_TOL["bf16"])


def test_nan_hidden_state_raises_numeric():
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=1, d_layers=1,
                          taps=(0, 0), block=8)
    S, B = 2, w.block
    eng, om, _ = G.setup(w, S=S, cap=64)
    g = torch.Generator().manual_seed(7)
    h = torch.randn(S * B, w.target.hidden, generator=g)
    drafts = torch.randint(0, w.vocab - 1, (S, B - 1), generator=g, dtype=torch.int32).cuda()
    bad = h.clone()
    bad[B + 3, 17] = float("nan")  # one element of one row of sequence 1
    eng.h[:S * B].copy_(bad.cuda())
    eng.base_pos.fill_(10)
    eng.verify(B, drafts)
    assert eng.status() == D.DFLASH_ERR_NUMERIC
    assert "status word" in D.dflash_last_error()
    # the next call on clean inputs reports OK and the right argmax
    eng.h[:S * B].copy_(h.cuda())
    eng.base_pos.fill_(10)
    eng.verify(B, drafts)
    assert eng.status() == D.DFLASH_OK
    x = O.final_norm(om.target.cfg, h.double().numpy(), om.target.g_final)
    am, mg, _ = O.lm_head_argmax(om.target.cfg, om.Wlm, x)
    G.check_argmax(eng.argmax.cpu().numpy().ravel(), am, mg)


def test_paired_gemm_weight_stall_times_out_and_recovers():
    """512 token rows run each projection as one paired launch; with its
    weight copies switched off (stall bit 2) the MMAs' waits expire, the call
    reports DFLASH_ERR_TIMEOUT, and the same workspace then gives the bits of
    a clean run."""
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=1, d_layers=1,
                          taps=(0, 0), block=16)
    S, rows = 32, 16
    eng, _, _ = G.setup(w, S=S, cap=128)
    g = torch.Generator().manual_seed(9)
    kc = torch.randn(eng.caches.tk[0].shape, generator=g).to(eng.caches.tk[0].dtype)
    vc = torch.randn(eng.caches.tv[0].shape, generator=g).to(eng.caches.tv[0].dtype)
    base = [(13 * s + 7) % 100 for s in range(S)]
    h0 = torch.randn(S * rows, w.target.hidden, generator=g)

    def run():
        eng.caches.tk[0].copy_(kc.cuda())
        eng.caches.tv[0].copy_(vc.cuda())
        st = _run_layer(eng, S, rows, base, h0)
        return st, eng.h[:S * rows].clone().cpu()

    st, ref = run()
    assert st == D.DFLASH_OK
    D.dflash_workspace_control(eng.ws_ptr, eng.ws_bytes, wait_limit_ns=2_000_000, stall_kv_loads=2)
    t0 = time.perf_counter()
    st, _ = run()
    assert st == D.DFLASH_ERR_TIMEOUT, st
    assert time.perf_counter() - t0 < 5.0
    D.dflash_workspace_control(eng.ws_ptr, eng.ws_bytes)
    st, again = run()
    assert st == D.DFLASH_OK
    assert torch.equal(again, ref)
