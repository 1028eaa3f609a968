"""Test helpers: build oracle models from the seeded synthetic draws, and the
float64 PyTorch restatements that pin the oracle to library routines."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import torch
import torch.nn.functional as F

from block_diffusion_speculative_step_gb300 import synth
from oracle import oracle as O


def small_workload(dtype="f32", H=64, nq=4, nkv=2, d=16, I=96, V=128, t_layers=3, d_layers=2,
                   taps=(0, 1), block=4, theta=1e4, eps=1e-6, window=0, topk=0, rank=0, conv_rank=0):
    return synth.Workload(
        name="test", target=synth.Shape(t_layers, H, nq, nkv, d, I),
        draft=synth.Shape(d_layers, H, nq, nkv, d, I), vocab=V, taps=tuple(taps), block=block,
        rope_theta=theta, rms_eps=eps, dtype=dtype, window=window, path_topk=topk, path_rank=rank,
        conv_rank=conv_rank)


def ocfg(w: synth.Workload, s: synth.Shape) -> O.Cfg:
    return O.Cfg(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, w.dtype == "bf16", w.rope_theta,
                 w.rms_eps)


def ostack(w, s, st) -> O.Stack:
    c = ocfg(w, s)
    n = synth.to_numpy
    layers = [O.Layer.from_stacked(c, n(L["w_qkv"]), n(L["w_o"]), n(L["w_gu"]), n(L["w_down"]),
                                   n(L["ln1"]), n(L["ln2"]),
                                   n(L["conv_w1"]) if "conv_w1" in L else None,
                                   n(L["conv_w2"]) if "conv_w2" in L else None) for L in st["layers"]]
    return O.Stack(c, layers, n(st["final_norm"]))


def omodel(w: synth.Workload, m: dict) -> O.Model:
    n = synth.to_numpy
    return O.Model(target=ostack(w, w.target, m["target"]) if "target" in m else None,
                   draft=ostack(w, w.draft, m["draft"]), E=n(m["embed"]), Wlm=n(m["lm_head"]),
                   Wfc=n(m["fc"]), gfc=n(m["fc_norm"]), taps=list(w.taps), mask_id=w.mask_id,
                   block=w.block, window=w.window)


# ----------------------------------------------------- float64 torch restatement


def t64(a) -> torch.Tensor:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy((a.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    return torch.from_numpy(a.astype(np.float64))


def tround(x: torch.Tensor, bf16: bool) -> torch.Tensor:
    return x.to(torch.bfloat16).to(torch.float64) if bf16 else x


def trope(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """RoPE as a complex rotation z_i = x_i + j x_{i+d/2}, z_i *= exp(j pos w_i)."""
    d = x.shape[-1]
    half = d // 2
    w = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = pos.to(torch.float64)[:, None] * w[None, :]
    z = torch.complex(x[..., :half], x[..., half:])
    rot = torch.polar(torch.ones_like(ang), ang)
    while rot.dim() < z.dim():
        rot = rot.unsqueeze(1)
    z = z * rot
    return torch.cat([z.real, z.imag], dim=-1)


def tconv(c: O.Cfg, cv: O.Conv, i: int, u: torch.Tensor) -> torch.Tensor:
    """The two-tap dynamic depthwise convolution with torch ops: taps from
    F.silu / matmul, the previous row by F.pad (a zero row before row 0)."""
    ab = F.silu(u @ t64(cv.w1[i]).T) @ t64(cv.w2[i]).T
    a, b = ab[:, :c.H], ab[:, c.H:]
    prev = F.pad(u, (0, 0, 1, 0))[:-1]
    return u + a * u + b * prev


def torch_layer(c: O.Cfg, L: O.Layer, h: torch.Tensor, pos: torch.Tensor, ctx_k=None, ctx_v=None,
                causal=True, past_k=None, past_v=None, stages=None):
    """One decoder layer with F.rms_norm / F.scaled_dot_product_attention /
    F.silu.  Causal: keys = past (already rotated) ++ the rows'; bidirectional:
    keys = ctx ++ the rows', no mask.  Returns (h_out, k_rows, v_rows)."""
    M = h.shape[0]
    bf = c.bf16
    cv = L.conv
    x = tround(F.rms_norm(h, (c.H,), t64(L.g1), c.eps), bf)
    if cv is not None:
        x = tround(tconv(c, cv, 0, x), bf)
    x1 = x
    q = (x @ t64(L.wq).T).view(M, c.nq, c.d)
    k = (x @ t64(L.wk).T).view(M, c.nkv, c.d)
    v = (x @ t64(L.wv).T).view(M, c.nkv, c.d)
    q = tround(trope(q, pos, c.theta), bf)
    k = tround(trope(k, pos, c.theta), bf)
    v = tround(v, bf)
    if causal:
        K = k if past_k is None else torch.cat([past_k, k], 0)
        V = v if past_v is None else torch.cat([past_v, v], 0)
        P = K.shape[0] - M
        mask = torch.zeros(M, K.shape[0], dtype=torch.bool)
        for i in range(M):
            mask[i, :P + i + 1] = True
    else:
        K = k if ctx_k is None else torch.cat([ctx_k, k], 0)
        V = v if ctx_v is None else torch.cat([ctx_v, v], 0)
        mask = torch.ones(M, K.shape[0], dtype=torch.bool)
    grp = c.nq // c.nkv
    Kq = K.repeat_interleave(grp, dim=1).permute(1, 0, 2)
    Vq = V.repeat_interleave(grp, dim=1).permute(1, 0, 2)
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2), Kq, Vq, attn_mask=mask)
    o = tround(o.permute(1, 0, 2).reshape(M, c.nq * c.d), bf)
    y = o @ t64(L.wo).T
    h = h + (y if cv is None else tconv(c, cv, 1, y))
    x = tround(F.rms_norm(h, (c.H,), t64(L.g2), c.eps), bf)
    if cv is not None:
        x = tround(tconv(c, cv, 2, x), bf)
    a = tround(F.silu(x @ t64(L.wg).T) * (x @ t64(L.wu).T), bf)
    y = a @ t64(L.wd).T
    h = h + (y if cv is None else tconv(c, cv, 3, y))
    if stages is not None:  # the intermediates, [M][width]
        stages.update(x1=x1, q=q.reshape(M, -1), k=k.reshape(M, -1), v=v.reshape(M, -1), o=o, x2=x, act=a)
    return h, k, v
