"""Sampling-mode verification on the GPU (speculative sampling at
temperature T, Philox4x32-10 draws): the kernels' draws and decisions equal
the oracle's on the same logits and the same random-number counters (up to
reported near-ties), the emitted token is distributed as the target's
softmax whatever the draft, and a whole sampled cycle runs through the
engine."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from oracle import oracle as O
from tests import gpu_common as G
from tests import helpers as Hh

pytestmark = pytest.mark.gpu

SEED = 0x5EED_1234_ABCD_0042


def _ws(nbytes=1 << 24):
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    D.dflash_workspace_init(ws.data_ptr(), nbytes)
    return ws


def _dims(V):
    return D.dflash_dims(64, 4, 2, 16, 96, V, 1e4, 1e-6, D.DFLASH_BF16)


def _run(tl, dl, P, T, cycle, ws, top_k=0, top_p=1.0):
    """dflash_sample_drafts then dflash_sample_accept on [S][B][V] / [S][B-1][V]."""
    S, B, V = tl.shape
    tl_d, dl_d = tl.cuda().contiguous(), dl.cuda().contiguous()
    base = torch.tensor(P, dtype=torch.int32, device="cuda")
    drafts = torch.zeros(S, B - 1, dtype=torch.int32, device="cuda")
    dlse = torch.zeros(S, B - 1, device="cuda")
    a = D.dflash_sample_drafts_args()
    a.dims, a.n_seqs, a.block, a.temperature, a.cycle, a.seed = _dims(V), S, B, T, cycle, SEED
    a.base_pos, a.draft_logits, a.drafts, a.draft_lse = base.data_ptr(), dl_d.data_ptr(), drafts.data_ptr(), dlse.data_ptr()
    a.top_k, a.top_p = top_k, top_p
    assert D.dflash_workspace_bytes(D.DFLASH_OP_SAMPLE_DRAFTS, a) <= ws.numel()
    D.dflash_sample_drafts(a, ws.data_ptr(), ws.numel())
    k = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    out = torch.full((S, B), -7, dtype=torch.int32, device="cuda")
    b = D.dflash_sample_accept_args()
    b.dims, b.n_seqs, b.block, b.temperature, b.cycle, b.seed = _dims(V), S, B, T, cycle, SEED
    b.target_logits, b.draft_logits, b.draft_lse = tl_d.data_ptr(), dl_d.data_ptr(), dlse.data_ptr()
    b.drafts, b.base_pos, b.update_base_pos = drafts.data_ptr(), base.data_ptr(), 0
    b.accept_len, b.out_tokens = k.data_ptr(), out.data_ptr()
    b.top_k, b.top_p = top_k, top_p
    D.dflash_sample_accept(b, ws.data_ptr(), ws.numel())
    torch.cuda.synchronize()
    st = D.dflash_read_status(ws.data_ptr())
    assert st == D.DFLASH_OK
    return drafts.cpu().numpy(), dlse.cpu().numpy(), k.cpu().numpy(), out.cpu().numpy()


@pytest.mark.parametrize("V,T", [(1000, 0.8), (151936, 1.0)])
def test_sampling_matches_oracle(V, T):
    S, B = 3, 6
    g = torch.Generator().manual_seed(V)
    tl = torch.randn(S, B, V, generator=g) * 2.0
    dl = (tl[:, 1:] * 0.6 + torch.randn(S, B - 1, V, generator=g) * 1.2)  # a draft close to, not equal to, the target
    P = [17, 400, 4095]
    ws = _ws()
    compared = 0
    for cycle in range(3):
        dr, dlse, k, out = _run(tl, dl, P, T, cycle, ws)
        for s in range(S):
            near = False
            for j in range(B - 1):
                tok, lse, mg = O.sample_row(dl[s, j].numpy(), T, SEED, P[s] + j + 1, s, O.RNG_DRAFT, cycle)
                assert abs(dlse[s, j] - lse) <= 1e-4 * max(1.0, abs(lse))
                if mg < 1e-4:
                    near = True
                    break
                assert dr[s, j] == tok, f"cycle {cycle} seq {s} row {j}: gpu {dr[s, j]} oracle {tok}"
            if near:
                continue
            ok, oout, omg = O.spec_sample_accept(tl[s].numpy(), dl[s].numpy(), dr[s], T, SEED, s, P[s], cycle)
            if omg < 1e-4:
                continue
            assert k[s] == ok and list(out[s, :ok + 1]) == list(oout)
            assert all(out[s, ok + 1:] == -1)
            compared += 1
    assert compared >= 5


def test_emitted_token_follows_the_target_distribution():
    """300 sequences with the same block per launch, 20 cycles: 6000 draws.
    The first emitted token is distributed as softmax(target row 0 / T), the
    first draft is accepted at rate sum min(p, q)."""
    S, B, V, T = 300, 3, 6, 0.9
    g = torch.Generator().manual_seed(5)
    t1 = torch.randn(B, V, generator=g)
    d1 = t1[1:] * 0.3 + torch.randn(B - 1, V, generator=g)
    tl, dl = t1.expand(S, B, V).contiguous(), d1.expand(S, B - 1, V).contiguous()
    ws = _ws()
    first = np.zeros(V)
    acc0, n = 0, 0
    for cycle in range(20):
        _, _, k, out = _run(tl, dl, [9] * S, T, cycle, ws)
        for s in range(S):
            first[out[s, 0]] += 1
            acc0 += k[s] > 0
            n += 1
    p = torch.softmax(t1[0].double() / T, 0).numpy()
    q = torch.softmax(d1[0].double() / T, 0).numpy()
    se = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(first / n - p) < 4.5 * se), (first / n, p)
    alpha = np.minimum(p, q).sum()
    assert abs(acc0 / n - alpha) < 4.5 * np.sqrt(alpha * (1 - alpha) / n)


def test_sampled_cycle_through_the_engine():
    w = Hh.small_workload("bf16", H=256, nq=4, nkv=2, d=64, I=384, V=1000, t_layers=2, d_layers=1, taps=(0, 1),
                          block=8)
    eng, _, _ = G.setup(w, S=2, cap=128)
    prompts = torch.stack([synth.make_tokens(30 + s, 12, w.vocab) for s in range(2)]).cuda()
    eng.prefill(prompts)
    base0 = eng.base_pos.clone()
    total = torch.zeros(2, dtype=torch.int64)
    for cycle in range(4):
        eng.cycle_sampled(0.7, SEED, cycle)
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        k = eng.accept_len.cpu()
        out = eng.out_tokens.cpu()
        assert torch.all((k >= 0) & (k <= w.block - 1))
        for s in range(2):
            toks = out[s, :int(k[s]) + 1]
            assert torch.all((toks >= 0) & (toks < w.vocab))
            assert int(eng.anchor[s]) == int(toks[-1])
        total += k.long() + 1
    assert torch.equal(eng.base_pos.cpu().long(), base0.cpu().long() + total)


@pytest.mark.parametrize("V,T,top_k,top_p,q", [(1000, 0.8, 50, 1.0, 0), (1000, 0.8, 0, 0.9, 0), (1000, 1.2, 20, 0.7, 0),
                                               (1000, 1.0, 20, 0.7, 0.125), (1000, 1.0, 0, 0.8, 0.125),
                                               (151936, 1.0, 40, 1.0, 0), (151936, 1.0, 0, 0.6, 0),
                                               (151936, 1.0, 50, 0.9, 0)])
def test_filtered_sampling_matches_oracle(V, T, top_k, top_p, q):
    """Top-k / top-p: with the oracle's kept sets of the same rows, the drafts,
    the draft rows' log-normalisers over their kept entries, the accept
    lengths and the emitted tokens equal the oracle's (sequences meeting a
    near-tie -- a draw, a test or the top-p boundary -- are reported and
    skipped).  Flat logits (spread 0.5) give every kept entry a share of the
    mass, so a wrong kept set moves the normalisers far beyond the tolerance.
    At the full vocabulary the logits are peaked (spread 3) so that the kept
    sets stay small and their boundary entries carry measurable mass.  With
    q > 0 the logits are rounded to multiples of q: large groups of equal
    logits, so the top-k and top-p boundaries fall inside them and the
    index order decides (a group kept whole past the top-k index would move
    the normalisers)."""
    S, B = 3, 6
    g = torch.Generator().manual_seed(V + top_k)
    spread = 0.5 if V <= 1000 else 3.0
    tl = torch.randn(S, B, V, generator=g) * spread
    dl = tl[:, 1:] * 0.6 + torch.randn(S, B - 1, V, generator=g) * 0.8 * spread
    if q > 0:
        tl = torch.round(tl / q) * q
        dl = torch.round(dl / q) * q
    P = [17, 400, 4095]
    ws = _ws()
    compared = 0
    for cycle in range(3):
        dr, dlse, k, out = _run(tl, dl, P, T, cycle, ws, top_k, top_p)
        for s in range(S):
            kt, kd, near = [], [], False
            for j in range(B):
                keep, n, mg = O.filter_row(tl[s, j].numpy(), T, top_k, top_p)
                kt.append(keep)
                near |= mg < 1e-6  # above the float-vs-double error of the cumulative mass
            for j in range(B - 1):
                keep, n, mg = O.filter_row(dl[s, j].numpy(), T, top_k, top_p)
                kd.append(keep)
                near |= mg < 1e-6
            if near:
                continue
            for j in range(B - 1):
                tok, lse, mg = O.sample_row(dl[s, j].numpy(), T, SEED, P[s] + j + 1, s, O.RNG_DRAFT, cycle, keep=kd[j])
                assert abs(dlse[s, j] - lse) <= 1e-4 * max(1.0, abs(lse)), (s, j, dlse[s, j], lse)
                assert kd[j][dr[s, j]] == 1
                if mg < 1e-4:
                    near = True
                    break
                assert dr[s, j] == tok, f"cycle {cycle} seq {s} row {j}: gpu {dr[s, j]} oracle {tok}"
            if near:
                continue
            ok, oout, omg = O.spec_sample_accept(tl[s].numpy(), dl[s].numpy(), dr[s], T, SEED, s, P[s], cycle,
                                                 keep_t=np.stack(kt), keep_d=np.stack(kd))
            if omg < 1e-4:
                continue
            assert k[s] == ok and list(out[s, :ok + 1]) == list(oout)
            compared += 1
    assert compared >= 5


def test_filtered_emitted_token_follows_the_filtered_target():
    """Top-k 4 and top-p 0.85 on both sides, 300 sequences x 20 cycles: the
    first emitted token follows the filtered, renormalised softmax of target
    row 0 (entries outside its kept set never appear)."""
    S, B, V, T, top_k, top_p = 300, 3, 6, 0.9, 4, 0.85
    g = torch.Generator().manual_seed(6)
    t1 = torch.randn(B, V, generator=g)
    d1 = t1[1:] * 0.3 + torch.randn(B - 1, V, generator=g)
    tl, dl = t1.expand(S, B, V).contiguous(), d1.expand(S, B - 1, V).contiguous()
    ws = _ws()
    first = np.zeros(V)
    n = 0
    for cycle in range(20):
        _, _, k, out = _run(tl, dl, [9] * S, T, cycle, ws, top_k, top_p)
        for s in range(S):
            first[out[s, 0]] += 1
            n += 1
    keep, _, _ = O.filter_row(t1[0].numpy(), T, top_k, top_p)
    z = np.where(keep > 0, t1[0].double().numpy() / T, -np.inf)
    p = np.exp(z - z.max())
    p /= p.sum()
    assert np.all(first[keep == 0] == 0)
    se = np.sqrt(p * (1 - p) / n) + 1e-12
    assert np.all(np.abs(first / n - p) < 4.5 * se), (first / n, p)
