"""Checkpoint / resume of the speculative decoding state.

The state a cycle carries to the next is the target and draft-context KV
caches, the committed lengths (base_pos) and the next anchor token.  Here it
is saved with torch.save in the middle of a generation, restored into a new
engine over the same weights, and the generation continues: the tokens,
accept lengths and final caches must equal those of the uninterrupted run
bit for bit.
"""
import io

import torch
import pytest

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from block_diffusion_speculative_step_gb300.engine import Engine
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu


def _state(eng):
    return {"tk": [t.clone() for t in eng.caches.tk], "tv": [t.clone() for t in eng.caches.tv],
            "dk": [t.clone() for t in eng.caches.dk], "dv": [t.clone() for t in eng.caches.dv],
            "base_pos": eng.base_pos.clone(), "anchor": eng.anchor.clone()}


def _restore(eng, st):
    for name in ("tk", "tv", "dk", "dv"):
        for dst, src in zip(getattr(eng.caches, name), st[name]):
            dst.copy_(src)
    eng.base_pos.copy_(st["base_pos"])
    eng.anchor.copy_(st["anchor"])


def _cycles(eng, n):
    toks, acc = [], []
    for _ in range(n):
        eng.cycle()
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        k = eng.accept_len.cpu()
        t = eng.out_tokens.cpu()
        acc.append(k)
        toks.append([t[s, :int(k[s]) + 1].tolist() for s in range(eng.S)])
    return toks, acc


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_resume_from_checkpoint_is_bit_exact(dtype):
    w = Hh.small_workload(dtype, H=256, nq=4, nkv=2, d=64, I=384, V=512, t_layers=3, d_layers=2, taps=(0, 2),
                          block=6)
    S = 2
    m_cpu = synth.make_model(w, seed=11, jitter=0.1, with_target=True)
    prompts = torch.stack([synth.make_tokens(30 + s, 20, w.vocab) for s in range(S)]).cuda()
    a = Engine(w, G.to_dev(m_cpu), S, 128)
    a.prefill(prompts)
    _cycles(a, 2)
    buf = io.BytesIO()
    torch.save({k: ([t.cpu() for t in v] if isinstance(v, list) else v.cpu()) for k, v in _state(a).items()}, buf)
    ref_toks, ref_acc = _cycles(a, 4)
    ref_final = _state(a)
    # a new engine over the same weights, resumed from the checkpoint
    buf.seek(0)
    st = torch.load(buf)
    b = Engine(w, G.to_dev(m_cpu), S, 128)
    _restore(b, {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in st.items()})
    toks, acc = _cycles(b, 4)
    assert toks == ref_toks
    for x, y in zip(acc, ref_acc):
        assert torch.equal(x, y)
    fin = _state(b)
    for name in ("tk", "tv", "dk", "dv"):
        for x, y in zip(fin[name], ref_final[name]):
            assert torch.equal(x, y), name
    assert torch.equal(fin["base_pos"], ref_final["base_pos"]) and torch.equal(fin["anchor"], ref_final["anchor"])
