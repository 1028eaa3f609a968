"""Device buffers and the call sequence of one DFlash cycle on the C ABI.

A cycle ("DFlash ..." guide, section 4) is, all on one CUDA stream and with
no host synchronisation:

  draft_block(anchor, base_pos)            -> drafts        (draft model, block-bidirectional)
  embed([anchor, drafts]); target layers   -> h, tap feats  (causal verification forward)
  verify_accept(h, drafts)                 -> accept_len, out_tokens; anchor := bonus,
                                              commit = (base_pos, k + 1), base_pos += k + 1
  fuse_context(feats, commit)              -> draft context K/V of the committed positions

Torch here only allocates device memory and provides the stream; every step
of the cycle runs in libdflash kernels.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import dflash as D
from . import synth


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def dims_of(w: synth.Workload, s: synth.Shape) -> D.dflash_dims:
    return D.dflash_dims(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, w.vocab, w.rope_theta, w.rms_eps,
                         D.DFLASH_BF16 if w.dtype == "bf16" else D.DFLASH_F32)


def layer_weights(L: dict) -> D.dflash_layer_weights:
    return D.dflash_layer_weights(_ptr(L["w_qkv"]), _ptr(L["w_o"]), _ptr(L["w_gu"]), _ptr(L["w_down"]),
                                  _ptr(L["ln1"]), _ptr(L["ln2"]))


@dataclass
class Caches:
    tk: list  # target K per layer [S][nkv][cap][d]
    tv: list
    dk: list  # draft context K per layer [S][nkv][dcap][d]
    dv: list


class Engine:
    """One target + draft pair resident on the GPU, n_seqs sequences."""

    def __init__(self, w: synth.Workload, model: dict, n_seqs: int, cap: int, device="cuda",
                 prefill_chunk: int = 256, fuse_rows: int = 0):
        self.w = w
        self.m = model
        self.S = n_seqs
        self.B = w.block
        self.cap = cap
        self.dev = torch.device(device)
        self.dt = synth.torch_dtype(w)
        self.chunk = prefill_chunk
        self.F = len(w.taps)
        tdims = w.target
        self.ddims = dims_of(w, w.draft)
        self.tdims = dims_of(w, tdims) if "target" in model else None
        self.has_target = "target" in model
        H = w.draft.hidden
        S, B = n_seqs, self.B
        z = lambda *shape, dt=None: torch.zeros(shape, dtype=dt or self.dt, device=self.dev)
        i32 = lambda *shape: torch.zeros(shape, dtype=torch.int32, device=self.dev)
        # caches
        dcap = w.window if w.window > 0 else cap
        self.dcap = dcap
        self.caches = Caches(
            tk=[z(S, tdims.n_kv, cap, tdims.head_dim) for _ in range(tdims.layers)] if self.has_target else [],
            tv=[z(S, tdims.n_kv, cap, tdims.head_dim) for _ in range(tdims.layers)] if self.has_target else [],
            dk=[z(S, w.draft.n_kv, dcap, w.draft.head_dim) for _ in range(w.draft.layers)],
            dv=[z(S, w.draft.n_kv, dcap, w.draft.head_dim) for _ in range(w.draft.layers)])
        # RoPE tables (positions up to cap)
        self.rope_max = cap + B
        self.rope_t = z(self.rope_max, tdims.head_dim // 2, 2, dt=torch.float32) if self.has_target else None
        self.rope_d = z(self.rope_max, w.draft.head_dim // 2, 2, dt=torch.float32)
        # cycle state
        self.anchor = i32(S)
        self.base_pos = i32(S)
        self.drafts = i32(S, max(B - 1, 1))
        self.argmax = i32(S, B)
        self.margin = z(S, B, dt=torch.float32)
        self.accept_len = i32(S)
        self.out_tokens = i32(S, B)
        self.commit_base = i32(S)
        self.commit_count = i32(S)
        self.h = z(S * max(B, prefill_chunk), H, dt=torch.float32)
        self.feats = z(S * max(B, prefill_chunk), self.F, H)
        self.ones = torch.ones(S, dtype=torch.int32, device=self.dev)
        self.ws = None
        self.paging = {}  # "t" / "d" -> (page table, page size, max pages, pool pages) once paged
        # DFlash 2 draft convolutions: on when the workload has them (the
        # weights sit in the draft layers as conv_w1 / conv_w2)
        self.conv_rank = w.conv_rank
        self.ws_bytes = 0
        self._size_workspace(fuse_rows)
        st = torch.cuda.current_stream()
        if self.has_target:
            D.dflash_rope_table(w.rope_theta, tdims.head_dim, self.rope_max, self.rope_t.data_ptr(), st)
        D.dflash_rope_table(w.rope_theta, w.draft.head_dim, self.rope_max, self.rope_d.data_ptr(), st)

    # ------------------------------------------------------------ arg builders

    def target_layer_args(self, li: int, rows: int, h, tap=None, tap_offset=0, base_pos=None):
        t = self.w.target
        a = D.dflash_layer_args()
        a.dims = self.tdims
        a.w = layer_weights(self.m["target"]["layers"][li])
        a.n_seqs, a.rows = self.S, rows
        a.base_pos = _ptr(self.base_pos if base_pos is None else base_pos)
        a.h = _ptr(h)
        a.kv = self._kv("t", li)
        a.attn_mode = D.DFLASH_ATTN_CAUSAL
        a.max_pos = self.cap
        a.rope_cs = _ptr(self.rope_t)
        a.rope_max_pos = self.rope_max
        if tap is not None:
            a.tap = _ptr(tap)
            a.tap_stride = self.F * t.hidden
            a.tap_offset = tap_offset
        return a

    def fuse_args(self, rows: int, feats, base_pos, valid):
        d = self.w.draft
        a = D.dflash_fuse_args()
        a.dims = self.ddims
        a.n_taps = self.F
        a.w_fc = _ptr(self.m["fc"])
        a.fc_norm = _ptr(self.m["fc_norm"])
        a.n_layers = d.layers
        for j in range(d.layers):
            a.w_qkv_layers[j] = _ptr(self.m["draft"]["layers"][j]["w_qkv"])
            a.kv_layers[j] = self._kv("d", j)
        a.feats = _ptr(feats)
        a.n_seqs, a.rows = self.S, rows
        a.base_pos = _ptr(base_pos)
        a.valid = _ptr(valid)
        a.rope_cs = _ptr(self.rope_d)
        a.rope_max_pos = self.rope_max
        return a

    def _kv(self, kind: str, j: int):
        """The dflash_kv of target ("t") or draft-context ("d") cache layer j."""
        if kind == "t":
            k, v, cap, win = self.caches.tk[j], self.caches.tv[j], self.cap, 0
        else:
            k, v, cap, win = self.caches.dk[j], self.caches.dv[j], self.dcap, self.w.window
        kv = D.dflash_kv(_ptr(k), _ptr(v), cap, win)
        if kind in self.paging:
            table, ps, mp, pool = self.paging[kind]
            kv.pages, kv.page_size, kv.max_pages, kv.pool_pages = _ptr(table), ps, mp, pool
        return kv

    def page_caches(self, page_size: int = 128, seed: int = 0, spare_pages: int = 0):
        """Move the target and draft-context caches into page pools
        [pool][n_kv][page_size][head_dim] whose pages are handed out in a
        seeded random order (page table [S][max_pages], one table per cache
        kind shared by its layers), copying the current contents; the calls
        then address the caches through the page tables.  spare_pages adds
        unmapped pages to each pool."""
        g = torch.Generator().manual_seed(seed)
        for kind, ks, vs, cap in (("t", self.caches.tk, self.caches.tv, self.cap),
                                  ("d", self.caches.dk, self.caches.dv, self.dcap)):
            if not ks:
                continue
            assert cap % page_size == 0, "capacity must be a multiple of the page size"
            mp = cap // page_size
            S, nkv, _, d = ks[0].shape
            pool = S * mp + spare_pages
            table = torch.randperm(pool, generator=g)[:S * mp].view(S, mp).to(torch.int32)
            idx = table.view(-1).long().to(self.dev)
            for lst in (ks, vs):
                for j, c in enumerate(lst):
                    pages = c.view(S, nkv, mp, page_size, d).permute(0, 2, 1, 3, 4).reshape(S * mp, nkv, page_size, d)
                    p = torch.zeros(pool, nkv, page_size, d, dtype=c.dtype, device=self.dev)
                    p[idx] = pages
                    lst[j] = p
            self.paging[kind] = (table.to(self.dev), page_size, mp, pool)

    def unpaged_caches(self):
        """The caches' contents in the contiguous layout [S][n_kv][cap][d]
        (copies when paged)."""
        out = {}
        for kind, ks, vs, cap in (("t", self.caches.tk, self.caches.tv, self.cap),
                                  ("d", self.caches.dk, self.caches.dv, self.dcap)):
            if kind not in self.paging:
                out[kind] = ([c.clone() for c in ks], [c.clone() for c in vs])
                continue
            table, ps, mp, pool = self.paging[kind]
            idx = table.view(-1).long()
            S = table.shape[0]
            conv = lambda p: p[idx].view(S, mp, p.shape[1], ps, p.shape[3]).permute(0, 2, 1, 3, 4).reshape(
                S, p.shape[1], mp * ps, p.shape[3])
            out[kind] = ([conv(p) for p in ks], [conv(p) for p in vs])
        return out

    def draft_args(self, logits=None, rounds: int = 1, conv_rank: int | None = None):
        d = self.w.draft
        a = D.dflash_draft_args()
        a.dims = self.ddims
        a.n_layers = d.layers
        for j in range(d.layers):
            a.layers[j] = layer_weights(self.m["draft"]["layers"][j])
            a.kv_layers[j] = self._kv("d", j)
        a.final_norm = _ptr(self.m["draft"]["final_norm"])
        a.embed = _ptr(self.m["embed"])
        a.lm_head = _ptr(self.m["lm_head"])
        a.n_seqs, a.block = self.S, self.B
        a.anchor = _ptr(self.anchor)
        a.base_pos = _ptr(self.base_pos)
        a.mask_token = self.w.mask_id
        a.max_pos = self.cap
        a.rope_cs = _ptr(self.rope_d)
        a.rope_max_pos = self.rope_max
        a.drafts = _ptr(self.drafts)
        a.logits = _ptr(logits)
        if self.w.path_topk:
            a.path_topk, a.path_rank = self.w.path_topk, self.w.path_rank
            a.path_u, a.path_v = _ptr(self.m["path_u"]), _ptr(self.m["path_v"])
        a.denoise_rounds = rounds
        r = self.conv_rank if conv_rank is None else conv_rank
        if r:
            a.conv_rank = r
            for j in range(d.layers):
                L = self.m["draft"]["layers"][j]
                a.conv_w1[j], a.conv_w2[j] = _ptr(L["conv_w1"]), _ptr(L["conv_w2"])
        return a

    def verify_args(self, block: int, h, drafts=None, logits=None, update=True):
        a = D.dflash_verify_args()
        a.dims = self.tdims
        a.h = _ptr(h)
        a.final_norm = _ptr(self.m["target"]["final_norm"])
        a.lm_head = _ptr(self.m["lm_head"])
        a.n_seqs, a.block = self.S, block
        a.drafts = _ptr(drafts)
        a.argmax = _ptr(self.argmax)
        a.margin = _ptr(self.margin)
        a.accept_len = _ptr(self.accept_len)
        a.out_tokens = _ptr(self.out_tokens)
        if update:
            a.next_anchor = _ptr(self.anchor)
            a.base_pos = _ptr(self.base_pos)
            a.commit_base = _ptr(self.commit_base)
            a.commit_count = _ptr(self.commit_count)
        a.logits = _ptr(logits)
        return a

    def embed_args(self, dims, rows: int, h, first, rest=None, fill=0):
        a = D.dflash_embed_args()
        a.dims = dims
        a.embed = _ptr(self.m["embed"])
        a.n_seqs, a.rows = self.S, rows
        a.first = _ptr(first)
        a.rest = _ptr(rest)
        a.fill_token = fill
        a.h = _ptr(h)
        return a

    def _size_workspace(self, fuse_rows: int):
        need = D.dflash_workspace_bytes(D.DFLASH_OP_DRAFT, self.draft_args())
        rows_list = [self.B, 1, min(self.chunk, self.cap)]
        if fuse_rows:
            need = max(need, D.dflash_workspace_bytes(D.DFLASH_OP_FUSE, self.fuse_args(fuse_rows, self.feats,
                                                                                      self.base_pos, None)))
        for rows in rows_list:
            need = max(need, D.dflash_workspace_bytes(D.DFLASH_OP_FUSE, self.fuse_args(rows, self.feats,
                                                                                      self.base_pos, None)))
            if self.has_target:
                need = max(need, D.dflash_workspace_bytes(D.DFLASH_OP_LAYER, self.target_layer_args(0, rows, self.h)))
                need = max(need, D.dflash_workspace_bytes(D.DFLASH_OP_VERIFY, self.verify_args(rows, self.h)))
        self.ws_bytes = int(need)
        self.ws = torch.zeros(self.ws_bytes + 256, dtype=torch.uint8, device=self.dev)
        self.ws_ptr = (self.ws.data_ptr() + 255) & ~255
        D.dflash_workspace_init(self.ws_ptr, self.ws_bytes)

    # -------------------------------------------------------------- the steps

    def status(self) -> int:
        return D.dflash_read_status(self.ws_ptr)

    def target_forward(self, rows: int, first, rest=None, taps=True, base_pos=None):
        """Embed the rows and run every target layer causally; keeps tap
        features (rows x F x H) in self.feats."""
        t = self.w.target
        D.dflash_embed(self.embed_args(self.tdims, rows, self.h, first, rest), self.ws_ptr, self.ws_bytes)
        for li in range(t.layers):
            tap = None
            off = 0
            if taps and li in self.w.taps:
                tap = self.feats
                off = self.w.taps.index(li) * t.hidden
            D.dflash_decoder_layer_forward(self.target_layer_args(li, rows, self.h, tap, off, base_pos), self.ws_ptr,
                                           self.ws_bytes)

    def draft(self, logits=None, rounds: int = 1, conv_rank: int | None = None):
        D.dflash_draft_block(self.draft_args(logits, rounds, conv_rank), self.ws_ptr, self.ws_bytes)

    def verify(self, block: int, drafts=None, logits=None):
        D.dflash_verify_accept(self.verify_args(block, self.h, drafts, logits), self.ws_ptr, self.ws_bytes)

    def fuse(self, rows: int, base_pos, valid):
        D.dflash_fuse_context(self.fuse_args(rows, self.feats, base_pos, valid), self.ws_ptr, self.ws_bytes)

    def fuse_with(self, feats, rows: int, base_pos, valid):
        """Inject caller-provided tap features feats [S*rows][F][H]."""
        D.dflash_fuse_context(self.fuse_args(rows, feats, base_pos, valid), self.ws_ptr, self.ws_bytes)

    def prefill(self, prompts: torch.Tensor):
        """prompts [S][L] int32 on the device.  Runs the target over the
        prompt (chunks of prefill_chunk rows, then the last token alone),
        injects every prompt position into the draft context, and sets
        anchor = the first greedy token, base_pos = L."""
        S, L = prompts.shape
        assert S == self.S and L + self.B <= self.cap
        c0 = 0
        while c0 < L - 1:
            rows = min(self.chunk, L - 1 - c0)
            self.base_pos.fill_(c0)
            tok = prompts[:, c0:c0 + rows].contiguous()
            self.target_forward(rows, tok[:, 0].contiguous(), tok[:, 1:].contiguous() if rows > 1 else None)
            self.fuse(rows, self.base_pos, None)
            c0 += rows
        self.base_pos.fill_(L - 1)
        self.target_forward(1, prompts[:, L - 1].contiguous())
        self.fuse(1, self.base_pos, None)
        self.verify(1)  # anchor := greedy token after the prompt, base_pos := L

    def cycle(self, planted_drafts=None):
        """One draft-and-verify cycle (see the module docstring)."""
        self.draft()
        if planted_drafts is not None:
            self.drafts.copy_(planted_drafts)
        self.target_forward(self.B, self.anchor, self.drafts)
        self.verify(self.B, self.drafts)
        self.fuse(self.B, self.commit_base, self.commit_count)

    def cycle_sampled(self, T: float, seed: int, cycle: int, top_k: int = 0, top_p: float = 1.0):
        """One cycle in sampling mode (speculative sampling at temperature T,
        optionally over the top_k / top_p filtered distributions): the
        draft's logits give drafts drawn from its distribution, the target's
        logits the acceptance tests and the final draw.  `cycle` numbers the
        random draws; give every cycle its own."""
        S, B, V = self.S, self.B, self.w.vocab
        if getattr(self, "dlogits", None) is None:
            self.dlogits = torch.zeros(S * (B - 1), V, dtype=torch.float32, device=self.dev)
            self.tlogits = torch.zeros(S * B, V, dtype=torch.float32, device=self.dev)
            self.dlse = torch.zeros(S, B - 1, dtype=torch.float32, device=self.dev)
        if self.w.path_topk:
            return self._cycle_sampled_path(T, seed, cycle, top_k, top_p)
        self.draft(self.dlogits)
        a = D.dflash_sample_drafts_args()
        a.dims = self.ddims
        a.n_seqs, a.block, a.temperature, a.cycle, a.seed = S, B, T, cycle, seed
        a.base_pos, a.draft_logits = _ptr(self.base_pos), _ptr(self.dlogits)
        a.drafts, a.draft_lse = _ptr(self.drafts), _ptr(self.dlse)
        a.top_k, a.top_p = top_k, top_p
        D.dflash_sample_drafts(a, self.ws_ptr, self.ws_bytes)
        self.target_forward(B, self.anchor, self.drafts)
        D.dflash_verify_accept(self.verify_args(B, self.h, self.drafts, self.tlogits, update=False), self.ws_ptr,
                               self.ws_bytes)
        b = D.dflash_sample_accept_args()
        b.dims = self.tdims
        b.n_seqs, b.block, b.temperature, b.cycle, b.seed = S, B, T, cycle, seed
        b.target_logits, b.draft_logits, b.draft_lse = _ptr(self.tlogits), _ptr(self.dlogits), _ptr(self.dlse)
        b.drafts, b.base_pos, b.update_base_pos = _ptr(self.drafts), _ptr(self.base_pos), 1
        b.accept_len, b.out_tokens, b.next_anchor = _ptr(self.accept_len), _ptr(self.out_tokens), _ptr(self.anchor)
        b.commit_base, b.commit_count = _ptr(self.commit_base), _ptr(self.commit_count)
        b.top_k, b.top_p = top_k, top_p
        D.dflash_sample_accept(b, self.ws_ptr, self.ws_bytes)
        self.fuse(B, self.commit_base, self.commit_count)

    def _cycle_sampled_path(self, T: float, seed: int, cycle: int, top_k: int, top_p: float):
        """Sampling mode with the DFlash 2 path selector: the drafts are the
        path walked by sampling over each row's candidates, and the
        acceptance runs against that walk's sparse proposal."""
        S, B, K = self.S, self.B, self.w.path_topk
        if getattr(self, "pcand", None) is None:
            self.pcand = torch.zeros(S, B - 1, K, dtype=torch.int32, device=self.dev)
            self.plogq = torch.zeros(S, B - 1, K, dtype=torch.float32, device=self.dev)
        a = self.draft_args()
        a.path_temperature, a.path_seed, a.path_cycle = T, seed, cycle
        a.path_cand_out, a.path_logq = _ptr(self.pcand), _ptr(self.plogq)
        D.dflash_draft_block(a, self.ws_ptr, self.ws_bytes)
        self.target_forward(B, self.anchor, self.drafts)
        D.dflash_verify_accept(self.verify_args(B, self.h, self.drafts, self.tlogits, update=False), self.ws_ptr,
                               self.ws_bytes)
        b = D.dflash_sample_accept_args()
        b.dims = self.tdims
        b.n_seqs, b.block, b.temperature, b.cycle, b.seed = S, B, T, cycle, seed
        b.target_logits = _ptr(self.tlogits)
        b.draft_topk, b.draft_cand, b.draft_logq = K, _ptr(self.pcand), _ptr(self.plogq)
        b.drafts, b.base_pos, b.update_base_pos = _ptr(self.drafts), _ptr(self.base_pos), 1
        b.accept_len, b.out_tokens, b.next_anchor = _ptr(self.accept_len), _ptr(self.out_tokens), _ptr(self.anchor)
        b.commit_base, b.commit_count = _ptr(self.commit_base), _ptr(self.commit_count)
        b.top_k, b.top_p = top_k, top_p
        D.dflash_sample_accept(b, self.ws_ptr, self.ws_bytes)
        self.fuse(B, self.commit_base, self.commit_count)

    def greedy_step(self):
        """Plain autoregressive step: one target forward of the anchor."""
        self.target_forward(1, self.anchor, taps=False)
        self.verify(1)

    # ---------------------------------------------------------------- loops

    def greedy_generate(self, prompts: torch.Tensor, n_new: int):
        self.prefill(prompts)
        out = [self.anchor.clone()]
        while len(out) < n_new:
            self.greedy_step()
            out.append(self.anchor.clone())
        return torch.stack(out, 1).cpu()

    def speculative_generate(self, prompts: torch.Tensor, n_new: int):
        self.prefill(prompts)
        outs = [[int(a)] for a in self.anchor.cpu()]
        accepts = []
        while min(len(o) for o in outs) < n_new:
            self.cycle()
            k = self.accept_len.cpu()
            toks = self.out_tokens.cpu()
            accepts.append(k.clone())
            for s in range(self.S):
                outs[s].extend(int(t) for t in toks[s, :int(k[s]) + 1])
        return torch.tensor([o[:n_new] for o in outs], dtype=torch.int32), torch.stack(accepts, 1)
