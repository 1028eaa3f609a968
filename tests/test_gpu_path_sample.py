"""The DFlash 2 path walked by sampling on the GPU (dflash_path_select /
dflash_draft_block with a path temperature) and speculative sampling against
its sparse proposal (dflash_sample_accept with draft_cand / draft_logq),
against the oracle on the same inputs and random-number counters; the
emitted token follows the target distribution; a sampled cycle with the
path selector through the engine."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_step_gb300 import dflash as D
from block_diffusion_speculative_step_gb300 import synth
from oracle import oracle as O
from tests import gpu_common as G
from tests import helpers as Hh
from tests.test_gpu_parity import _path_factors, small
from tests.test_gpu_sampling import SEED, _dims, _ws

pytestmark = pytest.mark.gpu


def _walk(eng, S, B, K, R, anchor, cand_d, base, T, cycle):
    path = torch.full((S, B - 1), -1, dtype=torch.int32, device="cuda")
    margin = torch.zeros(S, B - 1, device="cuda")
    logq = torch.zeros(S, B - 1, K, device="cuda")
    a = D.dflash_path_args()
    a.dims = eng.ddims
    a.n_seqs, a.block, a.topk, a.rank = S, B, K, R
    a.embed, a.path_u, a.path_v = eng.m["embed"].data_ptr(), eng.m["path_u"].data_ptr(), eng.m["path_v"].data_ptr()
    a.anchor, a.cand, a.path, a.margin = anchor.data_ptr(), cand_d.data_ptr(), path.data_ptr(), margin.data_ptr()
    a.temperature, a.seed, a.cycle, a.base_pos, a.logq = T, SEED, cycle, base.data_ptr(), logq.data_ptr()
    D.dflash_path_select(a, eng.ws_ptr, eng.ws_bytes)
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    return path.cpu().numpy(), logq.cpu().numpy()


def _setup(S, seed=12):
    w = small("bf16", V=600, block=6, topk=8, rank=32)
    B, K, R = w.block, 8, 32
    eng, om, _ = G.setup(w, S=S, cap=64)
    Un, Vn = _path_factors(eng, w, 8, "bf16")
    rng = np.random.default_rng(seed)
    cand = np.stack([np.stack([rng.choice(w.vocab, K, replace=False) for _ in range(B - 1)]) for _ in range(S)])
    return w, eng, om, Un, Vn, cand, B, K, R


def test_sampled_walk_matches_oracle():
    S = 3
    w, eng, om, Un, Vn, cand, B, K, R = _setup(S)
    cand_d = torch.from_numpy(cand.astype(np.int32)).cuda()
    anchor = torch.tensor([5, 77, 599], dtype=torch.int32, device="cuda")
    base = torch.tensor([10, 200, 37], dtype=torch.int32, device="cuda")
    compared = 0
    for T in (0.7, 1.5):
        for cycle in range(4):
            gp, glq = _walk(eng, S, B, K, R, anchor, cand_d, base, T, cycle)
            for s in range(S):
                op, olq, omg = O.path_walk_sample(om.draft.cfg, cand[s], om.E, Un, Vn, int(anchor[s]), T, SEED, s,
                                                  int(base[s]), cycle)
                for j in range(B - 1):
                    np.testing.assert_allclose(glq[s, j], olq[j], rtol=0, atol=2e-3)
                    assert abs(np.logaddexp.reduce(glq[s, j].astype(np.float64))) < 1e-5
                    if omg[j] < 1e-3:  # a draw near-tie: the walks may part here
                        break
                    assert gp[s, j] == op[j], f"T {T} cycle {cycle} seq {s} step {j}"
                    compared += 1
    assert compared >= 40


def test_sparse_proposal_accept_matches_oracle():
    S, B, V, K, T = 3, 6, 1000, 8, 0.9
    rng = np.random.default_rng(3)
    tl = (rng.standard_normal((S, B, V)) * 1.5).astype(np.float32)
    cand = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(B - 1)]) for _ in range(S)])
    z = rng.standard_normal((S, B - 1, K))
    lq = (z - np.log(np.exp(z).sum(-1, keepdims=True))).astype(np.float32)
    # target logits that favour the candidates, so that some drafts are accepted
    for s in range(S):
        for j in range(B - 1):
            tl[s, j, cand[s, j]] += 3.0
    ws = _ws()
    compared = 0
    for cycle in range(6):
        drafts = np.stack([np.stack([cand[s, j, rng.integers(0, K)] for j in range(B - 1)]) for s in range(S)])
        tl_d = torch.from_numpy(tl).cuda()
        base = torch.tensor([4, 90, 300], dtype=torch.int32, device="cuda")
        dr = torch.from_numpy(drafts.astype(np.int32)).cuda()
        qc = torch.from_numpy(cand.astype(np.int32)).cuda()
        ql = torch.from_numpy(lq).cuda()
        k = torch.full((S,), -1, dtype=torch.int32, device="cuda")
        out = torch.full((S, B), -7, dtype=torch.int32, device="cuda")
        b = D.dflash_sample_accept_args()
        b.dims, b.n_seqs, b.block, b.temperature, b.cycle, b.seed = _dims(V), S, B, T, cycle, SEED
        b.target_logits, b.drafts, b.base_pos, b.update_base_pos = tl_d.data_ptr(), dr.data_ptr(), base.data_ptr(), 0
        b.accept_len, b.out_tokens = k.data_ptr(), out.data_ptr()
        b.draft_topk, b.draft_cand, b.draft_logq = K, qc.data_ptr(), ql.data_ptr()
        D.dflash_sample_accept(b, ws.data_ptr(), ws.numel())
        torch.cuda.synchronize()
        assert D.dflash_read_status(ws.data_ptr()) == D.DFLASH_OK
        gk, go = k.cpu().numpy(), out.cpu().numpy()
        for s in range(S):
            ok, oout, omg = O.spec_sample_accept_sparse(tl[s], cand[s], lq[s].astype(np.float64), drafts[s], T, SEED,
                                                        s, int(base[s]), cycle)
            if omg < 1e-4:
                continue
            assert gk[s] == ok and list(go[s, :ok + 1]) == list(oout), (cycle, s)
            compared += 1
    assert compared >= 12


def test_sampled_walk_emitted_token_follows_the_target():
    """160 sequences with the same anchor, candidates and target rows, 40
    cycles: drafts walked by sampling on the GPU, accepted on the GPU
    against the walk's proposal; the first emitted token follows
    softmax(target row 0 / T) over the whole vocabulary."""
    S, T = 160, 0.9
    w, eng, om, Un, Vn, cand1, B, K, R = _setup(1, seed=13)
    e2, _, _ = G.setup(w, S=S, cap=64)
    e2.m["path_u"].copy_(eng.m["path_u"])
    e2.m["path_v"].copy_(eng.m["path_v"])
    V = w.vocab
    cand = np.repeat(cand1, S, axis=0)
    cand_d = torch.from_numpy(cand.astype(np.int32)).cuda()
    anchor = torch.full((S,), 7, dtype=torch.int32, device="cuda")
    base = torch.full((S,), 20, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(4)
    t1 = rng.standard_normal((B, V)).astype(np.float32) * 0.8
    t1[0, cand1[0, 0, :K]] += 2.0
    tl = torch.from_numpy(np.repeat(t1[None], S, axis=0)).cuda().contiguous()
    ws = _ws()
    first = np.zeros(V)
    n = 0
    for cycle in range(40):
        path, logq = _walk(e2, S, B, K, R, anchor, cand_d, base, T, cycle)
        dr = torch.from_numpy(path).cuda()
        ql = torch.from_numpy(logq).cuda()
        k = torch.full((S,), -1, dtype=torch.int32, device="cuda")
        out = torch.full((S, B), -7, dtype=torch.int32, device="cuda")
        b = D.dflash_sample_accept_args()
        b.dims, b.n_seqs, b.block, b.temperature, b.cycle, b.seed = _dims(V), S, B, T, cycle, SEED
        b.target_logits, b.drafts, b.base_pos, b.update_base_pos = tl.data_ptr(), dr.data_ptr(), base.data_ptr(), 0
        b.accept_len, b.out_tokens = k.data_ptr(), out.data_ptr()
        b.draft_topk, b.draft_cand, b.draft_logq = K, cand_d.data_ptr(), ql.data_ptr()
        D.dflash_sample_accept(b, ws.data_ptr(), ws.numel())
        torch.cuda.synchronize()
        go = out.cpu().numpy()
        for s in range(S):
            first[go[s, 0]] += 1
            n += 1
    z = t1[0].astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    se = np.sqrt(p * (1 - p) / n) + 1e-12
    big = p > 0.01  # the frequent tokens, where a wrong proposal would show
    assert big.sum() >= 5
    assert np.all(np.abs(first / n - p)[big] < 4.5 * se[big]), (first[big] / n, p[big])
    assert abs(first[~big].sum() / n - p[~big].sum()) < 4.5 * np.sqrt(p[~big].sum() / n) + 1e-3


def test_sampled_cycle_with_path_selector_through_the_engine():
    w = small("bf16", V=600, block=6, topk=8, rank=32)
    eng, _, _ = G.setup(w, S=2, cap=128)
    _path_factors(eng, w, 8, "bf16")
    prompts = torch.stack([synth.make_tokens(40 + s, 12, w.vocab) for s in range(2)]).cuda()
    eng.prefill(prompts)
    p0 = eng.base_pos.clone()
    for cycle in range(3):
        eng.cycle_sampled(0.9, 0x77, cycle, top_k=50, top_p=0.95)
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        k = eng.accept_len.cpu().numpy()
        out = eng.out_tokens.cpu().numpy()
        cand = eng.pcand.cpu().numpy()
        for s in range(2):
            assert 0 <= k[s] <= w.block - 1
            assert all(out[s, j] in cand[s, j] for j in range(k[s]))  # accepted drafts are walked candidates
            assert 0 <= out[s, k[s]] < w.vocab and all(out[s, k[s] + 1:] == -1)
    assert bool((eng.base_pos > p0).all())
