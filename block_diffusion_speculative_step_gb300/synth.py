"""Seeded synthetic inputs for the DFlash cycle: model shapes, random-init
weights, prompts and context features.

This module holds none of the method's arithmetic.  It only draws numbers
(torch generators, seeded) in the layouts the library and the oracle both
read, so the same draws can be handed to either side as data.

Layouts (row-major, [out][in] for every projection):
  embed [V][H], lm_head [V][H]            shared by target and draft
  layer.w_qkv [(nq + 2 nkv) d][H]         rows: W_q, then W_k, then W_v
  layer.w_o   [H][nq d]
  layer.w_gu  [2 I][H]                    rows: W_gate, then W_up
  layer.w_down[H][I]
  layer.ln1, layer.ln2 [H]                RMSNorm gains (attention, MLP)
  final_norm [H]
  fc [H][F H], fc_norm [H]                context-feature fusion (draft side)
  path_u, path_v [R][H]                   path-selector low-rank factors
  draft layer.conv_w1 [4][r][H],          DFlash 2 dynamic depthwise convolution tap
  draft layer.conv_w2 [4][2H][r]          generators (attention in / out, MLP in / out)
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Shape:
    """One decoder stack's shape."""
    layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    inter: int


@dataclass(frozen=True)
class Workload:
    """A named synthetic workload: target + draft shapes and cycle sizes."""
    name: str
    target: Shape
    draft: Shape
    vocab: int
    taps: tuple
    block: int
    rope_theta: float
    rms_eps: float
    dtype: str                 # "bf16" or "f32"
    batch: int = 1
    ctx: int = 4096            # context length (uniform) or upper bound (ragged)
    ctx_min: int = 0           # >0: ragged lengths ~ U[ctx_min, ctx]
    window: int = 0            # draft-context sliding window (0 = none)
    run_target: bool = True    # False: tap features are synthesised N(0,1)
    path_topk: int = 0         # DFlash 2 path selector (0 = off)
    path_rank: int = 0
    conv_rank: int = 0         # DFlash 2 dynamic depthwise convolutions in the draft (0 = off)
    accept_mean: float = 0.0   # >0: plant drafts so accept lengths ~ Geom(mean)
    prompt: int = 0
    generate: int = 0

    @property
    def mask_id(self) -> int:
        return self.vocab - 1


_Q8 = Shape(36, 4096, 32, 8, 128, 12288)
_Q8_DRAFT = replace(_Q8, layers=5)

WORKLOADS = {
    # 4-layer causal target, 2-layer draft, fp32, block 8, 64-token prompt, 64 generated.
    "tiny-lossless": Workload(
        name="tiny-lossless", target=Shape(4, 256, 4, 4, 64, 512), draft=Shape(2, 256, 4, 4, 64, 512),
        vocab=1024, taps=(1, 2), block=8, rope_theta=1e4, rms_eps=1e-6, dtype="f32",
        ctx=64, prompt=64, generate=64),
    # Qwen3-8B-shaped draft cycle at batch 1, context 4096.
    "qwen3-8b-b1": Workload(
        name="qwen3-8b-b1", target=_Q8, draft=_Q8_DRAFT, vocab=151936, taps=(2, 9, 17, 25, 33),
        block=16, rope_theta=1e6, rms_eps=1e-6, dtype="bf16", batch=1, ctx=4096),
    # Same shapes, 32 sequences with ragged contexts U[1024, 8192], planted accept lengths.
    "qwen3-8b-b32": Workload(
        name="qwen3-8b-b32", target=_Q8, draft=_Q8_DRAFT, vocab=151936, taps=(2, 9, 17, 25, 33),
        block=16, rope_theta=1e6, rms_eps=1e-6, dtype="bf16", batch=32, ctx=8192, ctx_min=1024,
        accept_mean=5.0),
    # Coder-shaped long-context draft: 8 layers, 32k context, 4096-slot window, no target.
    "coder-long": Workload(
        name="coder-long", target=Shape(48, 2048, 32, 4, 128, 6144),
        draft=Shape(8, 2048, 32, 4, 128, 6144), vocab=151936, taps=(2, 12, 23, 34, 45), block=16,
        rope_theta=1e6, rms_eps=1e-6, dtype="bf16", batch=1, ctx=32768, window=4096,
        run_target=False),
    # Llama-3.1-8B-shaped cycle with block 10 and the path selector.
    "llama31-8b": Workload(
        name="llama31-8b", target=Shape(32, 4096, 32, 8, 128, 14336),
        draft=Shape(5, 4096, 32, 8, 128, 14336), vocab=128256, taps=(2, 8, 15, 22, 29), block=10,
        rope_theta=5e5, rms_eps=1e-5, dtype="bf16", batch=1, ctx=2048, path_topk=16, path_rank=64),
}


def torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


class _Draw:
    """Sequential seeded draws on one device."""

    def __init__(self, seed: int, device):
        self.device = torch.device(device)
        self.g = torch.Generator(device=self.device)
        self.g.manual_seed(seed)

    def normal(self, shape, std: float, dtype) -> torch.Tensor:
        t = torch.empty(shape, dtype=torch.float32, device=self.device)
        t.normal_(0.0, std, generator=self.g)
        return t.to(dtype)

    def gain(self, n: int, jitter: float, dtype) -> torch.Tensor:
        if jitter == 0.0:
            return torch.ones(n, dtype=dtype, device=self.device)
        t = torch.empty(n, dtype=torch.float32, device=self.device)
        t.normal_(0.0, jitter, generator=self.g)
        return (1.0 + t).to(dtype)


def make_stack(dr: _Draw, s: Shape, dtype, std: float, jitter: float) -> dict:
    qkv = (s.n_q + 2 * s.n_kv) * s.head_dim
    layers = []
    for _ in range(s.layers):
        layers.append(dict(
            w_qkv=dr.normal((qkv, s.hidden), std, dtype),
            w_o=dr.normal((s.hidden, s.n_q * s.head_dim), std, dtype),
            w_gu=dr.normal((2 * s.inter, s.hidden), std, dtype),
            w_down=dr.normal((s.hidden, s.inter), std, dtype),
            ln1=dr.gain(s.hidden, jitter, dtype),
            ln2=dr.gain(s.hidden, jitter, dtype)))
    return dict(layers=layers, final_norm=dr.gain(s.hidden, jitter, dtype))


def make_model(w: Workload, seed: int = 0, device="cpu", std: float = 0.02, jitter: float = 0.0,
               with_target: bool | None = None) -> dict:
    """Random-init N(0, std) weights for target + draft + shared embedding /
    LM head + fusion FC (+ path-selector factors).  `jitter` > 0 draws the
    RMSNorm gains as 1 + N(0, jitter) instead of ones."""
    dt = torch_dtype(w)
    dr = _Draw(seed, device)
    H = w.draft.hidden
    F = len(w.taps)
    m = dict(
        embed=dr.normal((w.vocab, H), std, dt),
        lm_head=dr.normal((w.vocab, H), std, dt),
        fc=dr.normal((H, F * H), std, dt),
        fc_norm=dr.gain(H, jitter, dt),
        draft=make_stack(dr, w.draft, dt, std, jitter),
    )
    if with_target is None:
        with_target = w.run_target
    if with_target:
        m["target"] = make_stack(dr, w.target, dt, std, jitter)
    if w.path_topk:
        m["path_u"] = dr.normal((w.path_rank, H), std, dt)
        m["path_v"] = dr.normal((w.path_rank, H), std, dt)
    if w.conv_rank:  # drawn last, so the other weights do not depend on it
        for L in m["draft"]["layers"]:
            L["conv_w1"] = dr.normal((4, w.conv_rank, H), std, dt)
            L["conv_w2"] = dr.normal((4, 2 * H, w.conv_rank), std, dt)
    return m


def add_conv_weights(m: dict, w: Workload, rank: int, seed: int = 1, std: float = 0.02) -> None:
    """Draw DFlash 2 convolution tap generators (conv_w1 [4][r][H], conv_w2
    [4][2H][r]) into every draft layer of an existing model dict, from a
    generator of their own on the model's device."""
    L0 = m["draft"]["layers"][0]["w_o"]
    dr = _Draw(seed, L0.device)
    H = w.draft.hidden
    for L in m["draft"]["layers"]:
        L["conv_w1"] = dr.normal((4, rank, H), std, L0.dtype)
        L["conv_w2"] = dr.normal((4, 2 * H, rank), std, L0.dtype)


def make_tokens(seed: int, n: int, vocab: int, device="cpu") -> torch.Tensor:
    """n token ids uniform over [0, vocab-1) (the mask id vocab-1 excluded)."""
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return torch.randint(0, vocab - 1, (n,), generator=g, device=device, dtype=torch.int32)


def make_features(seed: int, rows: int, F: int, H: int, dtype, device="cpu") -> torch.Tensor:
    """Tap features [rows][F][H] drawn N(0, 1)."""
    dr = _Draw(seed, device)
    return dr.normal((rows, F, H), 1.0, dtype)


def make_ctx_lengths(seed: int, w: Workload) -> list:
    """Per-sequence context lengths: all w.ctx, or U[ctx_min, ctx] when ragged."""
    if w.ctx_min <= 0:
        return [w.ctx] * w.batch
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(w.ctx_min, w.ctx + 1, (w.batch,), generator=g).tolist()


def make_accept_lengths(seed: int, w: Workload) -> list:
    """Accept lengths k ~ Geometric(p) on {0, 1, ...} with mean w.accept_mean,
    clamped to block-1."""
    g = torch.Generator()
    g.manual_seed(seed)
    p = 1.0 / (1.0 + w.accept_mean)
    u = torch.rand(w.batch, generator=g, dtype=torch.float64)
    k = torch.floor(torch.log1p(-u) / torch.log1p(torch.tensor(-p, dtype=torch.float64)))
    return k.clamp(max=w.block - 1).to(torch.int64).tolist()


def to_numpy(t: torch.Tensor):
    """Tensor -> numpy for the oracle: bf16 as its uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
