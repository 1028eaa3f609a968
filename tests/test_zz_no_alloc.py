"""The allocation-free verification entry point.

Some callers cannot allocate device memory when they call into this
library -- runtimes whose memory is a pre-sized arena, plugins that are
handed only their input and output buffers, hot paths that must not
allocate.  dflash_verify_accept_noalloc serves them with a fixed scratch
array inside the library.  Here it is called through the C ABI twice in a
row with different inputs, and each result must equal what the
workspace-based dflash_verify_accept returns for the same inputs: argmax,
accept lengths and tokens exactly, margins within the tests' logit tolerance.

Kept in a file pytest collects last, so a failure here comes after every
other test has run; it also runs alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu


def _args(eng, h, drafts, argmax, margin, accept, out):
    a = eng.verify_args(eng.B, h, drafts, update=False)
    a.argmax, a.margin = argmax.data_ptr(), margin.data_ptr()
    a.accept_len, a.out_tokens = accept.data_ptr(), out.data_ptr()
    return a


def test_noalloc_matches_workspace_entry_point():
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=2, d_layers=1,
                          taps=(0, 1), block=8)
    S, B = 3, w.block
    eng, om, _ = G.setup(w, S=S, cap=64)
    dev = "cuda"
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for call, seed in enumerate((21, 22)):
        g = torch.Generator().manual_seed(seed)
        h = torch.randn(S * B, w.target.hidden, generator=g).to(dev)
        drafts = torch.randint(0, w.vocab, (S, B - 1), generator=g, dtype=torch.int32).to(dev)
        drafts[call % S] = 0  # at least one sequence whose drafts mostly disagree
        ref = [torch.zeros(S, B, dtype=torch.int32, device=dev), torch.zeros(S, B, device=dev),
               torch.zeros(S, dtype=torch.int32, device=dev), torch.zeros(S, B, dtype=torch.int32, device=dev)]
        got = [torch.full_like(ref[0], -7), torch.full_like(ref[1], -7.0), torch.full_like(ref[2], -7),
               torch.full_like(ref[3], -7)]
        D.dflash_verify_accept(_args(eng, h, drafts, *ref), eng.ws_ptr, eng.ws_bytes)
        D.dflash_verify_accept_noalloc(_args(eng, h, drafts, *got), status.data_ptr())
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0].cpu().numpy())
        np.testing.assert_allclose(got[1].cpu().numpy(), ref[1].cpu().numpy(), rtol=0, atol=G.LOGIT_TOL["bf16"])
        np.testing.assert_array_equal(got[2].cpu().numpy(), ref[2].cpu().numpy())
        np.testing.assert_array_equal(got[3].cpu().numpy(), ref[3].cpu().numpy())


def test_noalloc_rejects_oversized_request():
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=1, d_layers=1,
                          taps=(0, 0), block=8)
    eng, _, _ = G.setup(w, S=1, cap=32)
    a = eng.verify_args(eng.B, eng.h, eng.drafts, update=False)
    a.dims.hidden = 8192
    a.dims.vocab = 1 << 20          # scratch far beyond 8 MiB
    a.n_seqs, a.block = 64, 16
    rc = D.lib().dflash_verify_accept_noalloc(C.byref(a), None, None)
    assert rc == D.DFLASH_ERR_WORKSPACE
    assert "8 MiB" in D.dflash_last_error()
