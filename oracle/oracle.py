"""CPU oracle for one DFlash draft-and-verify cycle (numpy + the plain C in
dflash_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this module.  It shares no
code with the CUDA library and never imports it; inputs arrive as numpy arrays
(weights as float32 or as bf16 bit patterns in uint16 arrays).

Sources, cited by page title and section:
  [G] "DFlash: block-diffusion accelerated LLM speculative decoding" guide
      (txtmix.com): 3.1 one forward yields the whole block; 3.2 the draft is
      conditioned on target features (taps, concat, projection, RMSNorm, K/V
      injection into every draft layer); 3.3 verification by the target;
      section 4 the cycle (draft 16 -> verify -> accept prefix -> redraft);
      section 7 the DFlash 2 path selector; FAQ Q2 the taps.
  [N] "DFlash 2 release: parallel drafts keep lowering LLM inference latency"
      (openai-hub.com): the prefix-acceptance example; lossless greedy output;
      the per-token cost example in "what it means for deployment".
  [T] llmapis.com note on DFlash, "data and technical details": the draft
      sliding window bounding draft KV growth.

Every function is the plain definition: a row's result never depends on how
many rows are processed together, so the speculative loop reproduces the plain
greedy loop exactly (the lossless property of [N] and [G] 3.3).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash_oracle.c")
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

CAUSAL = 0
BIDIR = 1


def build(force: bool = False) -> str:
    """Compile dflash_oracle.c with gcc (no fused multiply-add contraction, so
    x86 and Arm builds compute the same values)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Cfg(C.Structure):
    _fields_ = [("H", C.c_int), ("nq", C.c_int), ("nkv", C.c_int), ("d", C.c_int), ("I", C.c_int),
                ("bf16", C.c_int), ("theta", C.c_double), ("eps", C.c_double)]


class _Layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g1", "g2")]


class _Stages(C.Structure):
    _fields_ = [(n, C.POINTER(C.c_double)) for n in ("x1", "q", "k", "v", "o", "x2", "act")]


STAGES = ("x1", "q", "k", "v", "o", "x2", "act")


class _Conv(C.Structure):
    _fields_ = [("w1", C.c_void_p * 4), ("w2", C.c_void_p * 4), ("r", C.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            dp = C.POINTER(C.c_double)
            L.or_bf16_round.restype = C.c_double
            L.or_bf16_round.argtypes = [C.c_double]
            L.or_rope.argtypes = [dp, C.c_int, C.c_long, C.c_double]
            L.or_rmsnorm.argtypes = [C.POINTER(_Cfg), C.c_int, dp, C.c_void_p, dp]
            L.or_linear.argtypes = [C.POINTER(_Cfg), C.c_void_p, C.c_int, C.c_int, C.c_int, dp, dp]
            L.or_decoder_layer.argtypes = [C.POINTER(_Cfg), C.POINTER(_Layer), C.c_int, C.c_long,
                                           C.c_int, dp, dp, C.c_long, C.c_long, dp]
            L.or_decoder_layer_conv.argtypes = [C.POINTER(_Cfg), C.POINTER(_Layer), C.POINTER(_Conv), C.c_int,
                                                C.c_long, C.c_int, dp, dp, C.c_long, C.c_long, dp]
            L.or_decoder_layer_tf.argtypes = [C.POINTER(_Cfg), C.POINTER(_Layer), C.POINTER(_Conv), C.c_int,
                                              C.c_long, C.c_int, dp, dp, C.c_long, C.c_long, dp,
                                              C.POINTER(_Stages), C.POINTER(_Stages)]
            L.or_dyn_conv.argtypes = [C.POINTER(_Cfg), C.c_int, C.c_int, C.c_void_p, C.c_void_p, dp, dp]
            L.or_final_norm.argtypes = [C.POINTER(_Cfg), C.c_int, dp, C.c_void_p, dp]
            L.or_lm_head_argmax.argtypes = [C.POINTER(_Cfg), C.c_void_p, C.c_int, C.c_int, dp,
                                            C.POINTER(C.c_int), dp, C.POINTER(C.c_float)]
            L.or_accept.argtypes = [C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int),
                                    C.POINTER(C.c_int)]
            L.or_fuse_context.argtypes = [C.POINTER(_Cfg), C.c_int, C.c_void_p, C.c_void_p,
                                          C.c_int, dp, C.POINTER(C.c_long), C.c_int,
                                          C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                          C.POINTER(dp), C.POINTER(dp), C.c_long, C.c_long, dp]
            L.or_path_select.argtypes = [C.POINTER(_Cfg), C.c_int, C.c_int, C.c_int, C.c_int,
                                         C.POINTER(C.c_float), C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int), dp]
            L.or_num_threads.restype = C.c_int
            L.or_set_threads.argtypes = [C.c_int]
            u32p = C.POINTER(C.c_uint32)
            L.or_philox4x32_10.argtypes = [u32p, u32p, u32p]
            L.or_uniform.restype = C.c_double
            L.or_uniform.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint32]
            L.or_sample_row.restype = C.c_int
            L.or_sample_row.argtypes = [C.POINTER(C.c_float), C.c_int, C.c_double, C.c_uint64, C.c_int, C.c_int,
                                        C.c_int, C.c_int, dp, dp]
            u8p = C.POINTER(C.c_ubyte)
            L.or_filter_row.restype = C.c_int
            L.or_filter_row.argtypes = [C.POINTER(C.c_float), C.c_int, C.c_double, C.c_int, C.c_double, u8p, dp]
            L.or_sample_row_f.restype = C.c_int
            L.or_sample_row_f.argtypes = [C.POINTER(C.c_float), C.c_int, C.c_double, u8p, C.c_uint64, C.c_int,
                                          C.c_int, C.c_int, C.c_int, dp, dp]
            L.or_spec_sample_accept_f.restype = C.c_int
            L.or_spec_sample_accept_f.argtypes = [C.c_int, C.c_int, C.POINTER(C.c_float), C.POINTER(C.c_float), u8p,
                                                  u8p, C.POINTER(C.c_int), C.c_double, C.c_uint64, C.c_int, C.c_int,
                                                  C.c_int, C.POINTER(C.c_int), dp]
            L.or_path_walk_sample.argtypes = [C.POINTER(_Cfg), C.c_int, C.c_int, C.c_int, C.POINTER(C.c_int), C.c_void_p,
                                              C.c_void_p, C.c_void_p, C.c_int, C.c_double, C.c_uint64, C.c_int,
                                              C.c_int, C.c_int, C.POINTER(C.c_int), dp, dp]
            L.or_spec_sample_accept_sparse.restype = C.c_int
            L.or_spec_sample_accept_sparse.argtypes = [C.c_int, C.c_int, C.POINTER(C.c_float), u8p, C.c_int,
                                                       C.POINTER(C.c_int), dp, C.POINTER(C.c_int), C.c_double,
                                                       C.c_uint64, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_int), dp]
            L.or_spec_sample_accept.restype = C.c_int
            L.or_spec_sample_accept.argtypes = [C.c_int, C.c_int, C.POINTER(C.c_float), C.POINTER(C.c_float),
                                                C.POINTER(C.c_int), C.c_double, C.c_uint64, C.c_int, C.c_int,
                                                C.c_int, C.POINTER(C.c_int), dp]
            _lib = L
    return _lib


def _dp(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _vp(a: np.ndarray):
    assert a.flags.c_contiguous
    return C.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------ model data


@dataclass
class Cfg:
    """Shape and arithmetic mode of one decoder stack."""
    H: int
    nq: int
    nkv: int
    d: int
    I: int
    bf16: bool
    theta: float
    eps: float

    def c(self) -> _Cfg:
        return _Cfg(self.H, self.nq, self.nkv, self.d, self.I, int(self.bf16), self.theta, self.eps)

    def wdtype(self):
        return np.uint16 if self.bf16 else np.float32


@dataclass
class Conv:
    """The DFlash 2 dynamic depthwise convolutions of one draft layer: tap
    generators w1[i] [r][H], w2[i] [2H][r] at i = 0 attention input, 1
    attention output, 2 MLP input, 3 MLP output (see dyn_conv)."""
    w1: list
    w2: list

    def c(self) -> _Conv:
        cv = _Conv()
        for i in range(4):
            cv.w1[i] = self.w1[i].ctypes.data
            cv.w2[i] = self.w2[i].ctypes.data
        cv.r = int(self.w1[0].shape[0])
        return cv


@dataclass
class Layer:
    """One decoder layer's weights, [out][in] row-major (views are fine);
    conv: the DFlash 2 convolutions of a draft layer, or None."""
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray
    g1: np.ndarray
    g2: np.ndarray
    conv: Conv | None = None

    def c(self) -> _Layer:
        arrs = [self.wq, self.wk, self.wv, self.wo, self.wg, self.wu, self.wd, self.g1, self.g2]
        return _Layer(*[a.ctypes.data for a in arrs])

    @staticmethod
    def from_stacked(cfg: Cfg, w_qkv, w_o, w_gu, w_down, ln1, ln2, conv_w1=None, conv_w2=None) -> "Layer":
        """Split a stacked [Wq; Wk; Wv] and [W_gate; W_up] into the per-matrix
        views the definitions use; conv_w1 [4][r][H] / conv_w2 [4][2H][r]
        (optional) are the layer's convolution tap generators."""
        QD, KD = cfg.nq * cfg.d, cfg.nkv * cfg.d
        c = np.ascontiguousarray
        conv = None
        if conv_w1 is not None:
            conv = Conv([c(conv_w1[i]) for i in range(4)], [c(conv_w2[i]) for i in range(4)])
        return Layer(c(w_qkv[:QD]), c(w_qkv[QD:QD + KD]), c(w_qkv[QD + KD:QD + 2 * KD]), c(w_o),
                     c(w_gu[:cfg.I]), c(w_gu[cfg.I:]), c(w_down), c(ln1), c(ln2), conv)


def wfloat(cfg: Cfg, w: np.ndarray) -> np.ndarray:
    """Weights as float64 (bf16 bit patterns are widened exactly)."""
    if cfg.bf16:
        return (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return w.astype(np.float64)


def rnd(cfg: Cfg, x: np.ndarray) -> np.ndarray:
    """Round to bf16 (RNE) in bf16 mode; identity in fp32 mode."""
    if not cfg.bf16:
        return x
    return bf16_round_array(x)


def bf16_round_array(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (via float32, round-to-nearest-even)
    and widen back; NaN stays NaN, overflow goes to +-inf."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    r = u.astype(np.uint32).view(np.float32).astype(np.float64)
    r[np.isnan(f)] = np.nan
    return r


# ------------------------------------------------------------------ primitives


def rmsnorm(cfg: Cfg, x: np.ndarray, g: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    c = cfg.c()
    for r in range(x.shape[0]):
        lib().or_rmsnorm(C.byref(c), x.shape[1], _dp(x[r]), _vp(g), _dp(y[r]))
    return y


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of one head vector at absolute position pos."""
    v = np.array(v, dtype=np.float64)
    lib().or_rope(_dp(v), v.shape[0], int(pos), float(theta))
    return v


def linear(cfg: Cfg, W: np.ndarray, X: np.ndarray) -> np.ndarray:
    X = np.ascontiguousarray(X, dtype=np.float64)
    N, K = W.shape
    Y = np.empty((X.shape[0], N))
    lib().or_linear(C.byref(cfg.c()), _vp(W), N, K, X.shape[0], _dp(X), _dp(Y))
    return Y


def decoder_layer(cfg: Cfg, L: Layer, h: np.ndarray, p0: int, mode: int, kc: np.ndarray,
                  vc: np.ndarray, window: int = 0) -> None:
    """One decoder layer over the rows h[M][H] of one sequence at positions
    p0..p0+M-1, in place.  kc/vc: [nkv][cap][d] float64 caches."""
    assert h.dtype == np.float64 and h.flags.c_contiguous
    cap = kc.shape[1]
    if L.conv is not None:
        rc = lib().or_decoder_layer_conv(C.byref(cfg.c()), C.byref(L.c()), C.byref(L.conv.c()), h.shape[0],
                                         int(p0), int(mode), _dp(kc), _dp(vc), cap, int(window), _dp(h))
    else:
        rc = lib().or_decoder_layer(C.byref(cfg.c()), C.byref(L.c()), h.shape[0], int(p0), int(mode),
                                    _dp(kc), _dp(vc), cap, int(window), _dp(h))
    if rc != 0:
        raise ValueError(f"or_decoder_layer failed ({rc})")


def decoder_layer_tf(cfg: Cfg, L: Layer, h: np.ndarray, p0: int, mode: int, kc: np.ndarray, vc: np.ndarray,
                     window: int = 0, given: dict | None = None) -> dict:
    """The layer of decoder_layer with its stages open (teacher forcing):
    returns this oracle's own value of every stage (x1, q, k, v, o, x2, act;
    [M][width], k / v as [M][nkv*d]) computed from the stages before it, where
    each stage given in `given` (same shapes, float64) replaces the oracle's
    own value for everything after it.  h (in place) ends as the layer's
    output; in causal mode the cache receives the rows' (given) k, v."""
    assert h.dtype == np.float64 and h.flags.c_contiguous
    M = h.shape[0]
    width = dict(x1=cfg.H, q=cfg.nq * cfg.d, k=cfg.nkv * cfg.d, v=cfg.nkv * cfg.d, o=cfg.nq * cfg.d, x2=cfg.H,
                 act=cfg.I)
    out = {n: np.zeros((M, width[n])) for n in STAGES}
    keep = {}
    gv = _Stages()
    for n in STAGES:
        if given is not None and given.get(n) is not None:
            a = np.ascontiguousarray(given[n], dtype=np.float64).reshape(M, width[n])
            keep[n] = a
            setattr(gv, n, _dp(a))
    ov = _Stages(*[_dp(out[n]) for n in STAGES])
    conv = C.byref(L.conv.c()) if L.conv is not None else None
    rc = lib().or_decoder_layer_tf(C.byref(cfg.c()), C.byref(L.c()), conv, M, int(p0), int(mode), _dp(kc), _dp(vc),
                                   kc.shape[1], int(window), _dp(h), C.byref(gv), C.byref(ov))
    if rc != 0:
        raise ValueError(f"or_decoder_layer_tf failed ({rc})")
    return out


def dyn_conv(cfg: Cfg, W1: np.ndarray, W2: np.ndarray, u: np.ndarray) -> np.ndarray:
    """DFlash 2 two-tap dynamic depthwise convolution ([G] section 7) over
    the rows u [M][H] of one block: z_t = SiLU(W1 u_t), (a_t, b_t) = W2 z_t,
    y_t = u_t + a_t * u_t + b_t * u_{t-1}, u_{-1} = 0 (the reading stated in
    dflash_oracle.c, or_dyn_conv)."""
    u = np.ascontiguousarray(u, dtype=np.float64)
    y = np.empty_like(u)
    lib().or_dyn_conv(C.byref(cfg.c()), u.shape[0], W1.shape[0], _vp(W1), _vp(W2), _dp(u), _dp(y))
    return y


def final_norm(cfg: Cfg, h: np.ndarray, g: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.float64)
    x = np.empty_like(h)
    lib().or_final_norm(C.byref(cfg.c()), h.shape[0], _dp(h), _vp(g), _dp(x))
    return x


def lm_head_argmax(cfg: Cfg, Wlm: np.ndarray, x: np.ndarray, want_logits: bool = False):
    """Greedy argmax (lowest index on ties) and top1-top2 margin per row."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    M, V = x.shape[0], Wlm.shape[0]
    am = np.empty(M, dtype=np.int32)
    mg = np.empty(M, dtype=np.float64)
    lg = np.empty((M, V), dtype=np.float32) if want_logits else None
    lib().or_lm_head_argmax(C.byref(cfg.c()), _vp(Wlm), V, M, _dp(x),
                            am.ctypes.data_as(C.POINTER(C.c_int)), _dp(mg),
                            lg.ctypes.data_as(C.POINTER(C.c_float)) if lg is not None else None)
    return am, mg, lg


def accept(drafts, g) -> tuple[int, np.ndarray]:
    """Greedy longest-prefix acceptance; returns (k, out_tokens[:k+1])."""
    g = np.ascontiguousarray(g, dtype=np.int32)
    B = g.shape[0]
    d = np.ascontiguousarray(drafts, dtype=np.int32)
    assert d.shape[0] == B - 1
    out = np.zeros(B, dtype=np.int32)
    k = lib().or_accept(B, d.ctypes.data_as(C.POINTER(C.c_int)),
                        g.ctypes.data_as(C.POINTER(C.c_int)), out.ctypes.data_as(C.POINTER(C.c_int)))
    return int(k), out[:k + 1].copy()


def fuse_context(dcfg: Cfg, F: int, Wfc, gfc, feats: np.ndarray, pos, wk_list, wv_list,
                 kc_list, vc_list, window: int = 0) -> np.ndarray:
    """Fusion + K/V injection of T positions into every draft layer's context
    cache; returns c_t [T][H]."""
    feats = np.ascontiguousarray(feats, dtype=np.float64).reshape(len(pos), F * dcfg.H)
    T = feats.shape[0]
    pos_a = np.ascontiguousarray(pos, dtype=np.int64)
    n = len(wk_list)
    wk = (C.c_void_p * n)(*[w.ctypes.data for w in wk_list])
    wv = (C.c_void_p * n)(*[w.ctypes.data for w in wv_list])
    kc = (C.POINTER(C.c_double) * n)(*[_dp(a) for a in kc_list])
    vc = (C.POINTER(C.c_double) * n)(*[_dp(a) for a in vc_list])
    cout = np.empty((T, dcfg.H))
    rc = lib().or_fuse_context(C.byref(dcfg.c()), F, _vp(Wfc), _vp(gfc), T, _dp(feats),
                               pos_a.ctypes.data_as(C.POINTER(C.c_long)), n, wk, wv, kc, vc,
                               kc_list[0].shape[1], int(window), _dp(cout))
    if rc != 0:
        raise ValueError(f"or_fuse_context failed ({rc})")
    return cout


def path_select(cfg: Cfg, logits: np.ndarray, E, U, Vm, anchor: int, topk: int = 16):
    """DFlash 2 greedy path walk over the top-k candidates of each draft row."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    Bm1, Vocab = lg.shape
    R = U.shape[0]
    cand = np.zeros((Bm1, topk), dtype=np.int32)
    path = np.zeros(Bm1, dtype=np.int32)
    mg = np.zeros(Bm1)
    lib().or_path_select(C.byref(cfg.c()), Bm1 + 1, Vocab, topk, R,
                         lg.ctypes.data_as(C.POINTER(C.c_float)), _vp(E), _vp(U), _vp(Vm),
                         int(anchor), cand.ctypes.data_as(C.POINTER(C.c_int)),
                         path.ctypes.data_as(C.POINTER(C.c_int)), _dp(mg))
    return path, cand, mg


def tap_layers(n_layers: int, n_taps: int = 5, first: int = 2) -> list[int]:
    """Tap layer ids spread uniformly from layer `first` to the third-from-last
    ([G] 3.2, FAQ Q2), 0-indexed decoder-layer outputs, rounded down."""
    last = n_layers - 3
    if n_taps == 1:
        return [first]
    return [first + (i * (last - first)) // (n_taps - 1) for i in range(n_taps)]


def per_token_cost_ms(t_draft_ms: float, t_verify_ms: float, accepted: float) -> float:
    """Per-token cost of one cycle spread over the tokens it yields ([N],
    'what it means for deployment': 3 ms + 20 ms over 6 tokens ~ 3.8 ms)."""
    return (t_draft_ms + t_verify_ms) / accepted


# ------------------------------------------------------------------- the cycle


@dataclass
class Stack:
    """A decoder stack: config, layers, final norm gain."""
    cfg: Cfg
    layers: list
    g_final: np.ndarray


@dataclass
class Model:
    """Target + draft sharing the embedding E and LM head W_lm ([G] 3.1)."""
    target: Stack
    draft: Stack
    E: np.ndarray
    Wlm: np.ndarray
    Wfc: np.ndarray
    gfc: np.ndarray
    taps: list
    mask_id: int
    block: int
    window: int = 0


@dataclass
class SeqState:
    """Per-sequence caches: target KV (D1) and injected draft context KV (D2)."""
    tk: list = field(default_factory=list)
    tv: list = field(default_factory=list)
    dk: list = field(default_factory=list)
    dv: list = field(default_factory=list)


def new_state(m: Model, cap: int) -> SeqState:
    t, d = m.target.cfg, m.draft.cfg
    dcap = m.window if m.window > 0 else cap
    s = SeqState()
    s.tk = [np.zeros((t.nkv, cap, t.d)) for _ in m.target.layers]
    s.tv = [np.zeros((t.nkv, cap, t.d)) for _ in m.target.layers]
    s.dk = [np.zeros((d.nkv, dcap, d.d)) for _ in m.draft.layers]
    s.dv = [np.zeros((d.nkv, dcap, d.d)) for _ in m.draft.layers]
    return s


def embed(cfg: Cfg, E: np.ndarray, tokens) -> np.ndarray:
    return np.ascontiguousarray(wfloat(cfg, E[np.asarray(tokens, dtype=np.int64)]))


def target_forward(m: Model, st: SeqState, tokens, p0: int, want_logits: bool = False):
    """Causal target forward over tokens at positions p0.. ([G] 3.3): writes
    their K/V into the target cache, returns greedy argmax per row, margins,
    tap features [M][F*H] (rounded residual after each tap layer, in
    increasing layer order) and optionally logits."""
    cfg = m.target.cfg
    h = embed(cfg, m.E, tokens)
    taps = {}
    for li, L in enumerate(m.target.layers):
        decoder_layer(cfg, L, h, p0, CAUSAL, st.tk[li], st.tv[li])
        if li in m.taps:
            taps[li] = rnd(cfg, h.copy())
    feats = np.concatenate([taps[l] for l in m.taps], axis=1)
    x = final_norm(cfg, h, m.target.g_final)
    am, mg, lg = lm_head_argmax(cfg, m.Wlm, x, want_logits)
    return am, mg, feats, lg


def fuse(m: Model, st: SeqState, feats: np.ndarray, pos) -> np.ndarray:
    """Inject positions `pos` (tap features feats [T][F*H]) into D2."""
    d = m.draft
    wk = [L.wk for L in d.layers]
    wv = [L.wv for L in d.layers]
    return fuse_context(d.cfg, len(m.taps), m.Wfc, m.gfc, feats, pos, wk, wv, st.dk, st.dv,
                        m.window)


def draft_forward(m: Model, st: SeqState, anchor: int, P: int, want_logits: bool = False):
    """Single-step block-diffusion draft ([G] 3.1): block [anchor, mask...]
    at positions P..P+B-1, bidirectional over the injected context and the
    block; row j (j >= 1) predicts the token at position P+j.  Returns
    drafts [B-1], margins, and optionally logits [B-1][V]."""
    cfg = m.draft.cfg
    B = m.block
    tokens = [anchor] + [m.mask_id] * (B - 1)
    h = embed(cfg, m.E, tokens)
    for li, L in enumerate(m.draft.layers):
        decoder_layer(cfg, L, h, P, BIDIR, st.dk[li], st.dv[li], m.window)
    x = final_norm(cfg, h, m.draft.g_final)
    am, mg, lg = lm_head_argmax(cfg, m.Wlm, x[1:], want_logits)
    return am, mg, lg


def draft_denoise(m: Model, st: SeqState, anchor: int, P: int, rounds: int, want_logits: bool = False,
                  selector=None, init=None):
    """Multi-round block denoising ([N] "the core of DFlash 2": a block
    diffusion model settles a block in several rounds of parallel denoising
    or correction, predicting and revising every block position at once).
    Round 1 is the single-step draft on [anchor, mask...]; round r >= 2 runs
    the same forward on [anchor, drafts of round r-1] at the same positions
    P..P+B-1, every row j >= 1 predicting the token at P+j again.  With
    selector = (U, Vm, topk) every round's drafts are the DFlash 2 greedy
    path over that round's top-k candidates ([G] section 7).  Returns the
    last round's drafts, their margins (argmax or walk) and, if asked, the
    last round's logits [B-1][V].  init (optional, B-1 tokens) replaces the
    mask tokens of round 1: the rounds then continue from those drafts."""
    cfg = m.draft.cfg
    B = m.block
    rest = [m.mask_id] * (B - 1) if init is None else [int(t) for t in init]
    assert len(rest) == B - 1
    for _ in range(max(1, int(rounds))):
        h = embed(cfg, m.E, [anchor] + [int(t) for t in rest])
        for li, L in enumerate(m.draft.layers):
            decoder_layer(cfg, L, h, P, BIDIR, st.dk[li], st.dv[li], m.window)
        x = final_norm(cfg, h, m.draft.g_final)
        am, mg, lg = lm_head_argmax(cfg, m.Wlm, x[1:], want_logits or selector is not None)
        if selector is not None:
            U, Vm, topk = selector
            am, _, mg = path_select(cfg, lg, m.E, U, Vm, anchor, topk)
        rest = am
    return am, mg, (lg if want_logits else None)


def prefill(m: Model, st: SeqState, prompt):
    """Target forward over the prompt, inject every prompt position into the
    draft context; returns the first generated token (the first anchor)."""
    am, mg, feats, _ = target_forward(m, st, prompt, 0)
    fuse(m, st, feats, list(range(len(prompt))))
    return int(am[-1])


def greedy_generate(m: Model, prompt, n_new: int, cap: int):
    """Plain autoregressive greedy decoding with the target alone: one target
    forward per token.  Returns the generated tokens and the per-token argmax
    margins."""
    st = new_state(m, cap)
    am, mg, _, _ = target_forward(m, st, prompt, 0)
    out = [int(am[-1])]
    margins = [float(mg[-1])]
    P = len(prompt)
    while len(out) < n_new:
        am, mg, _, _ = target_forward(m, st, [out[-1]], P)
        out.append(int(am[0]))
        margins.append(float(mg[0]))
        P += 1
    return np.array(out, dtype=np.int32), np.array(margins)


def speculative_generate(m: Model, prompt, n_new: int, cap: int, drafter=None):
    """The DFlash loop ([G] section 4): prefill, then repeat {draft a block
    from the anchor, verify it causally with the target, accept the longest
    agreeing prefix plus the bonus token, inject the committed positions'
    features}.  `drafter(m, st, anchor, P)` may replace the draft model
    (tests plant perfect or wrong drafts).  Returns tokens, per-cycle accept
    lengths."""
    st = new_state(m, cap)
    anchor = prefill(m, st, prompt)
    out = [anchor]
    P = len(prompt)
    accepts = []
    while len(out) < n_new:
        if drafter is None:
            drafts, _, _ = draft_forward(m, st, anchor, P)
        else:
            drafts = np.asarray(drafter(m, st, anchor, P), dtype=np.int32)
        block = [anchor] + [int(t) for t in drafts]
        g, _, feats, _ = target_forward(m, st, block, P)
        k, emitted = accept(drafts, g)
        accepts.append(k)
        fuse(m, st, feats[:k + 1], list(range(P, P + k + 1)))
        out.extend(int(t) for t in emitted)
        P += k + 1
        anchor = int(emitted[-1])
    return np.array(out[:n_new], dtype=np.int32), accepts


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (results do not
    depend on it)."""
    lib().or_set_threads(int(n))


def threads() -> int:
    return int(lib().or_num_threads())


# ---------------------------------------------------------------- sampling
# Random-number purposes (the counter's low byte next to the sequence id).
RNG_DRAFT, RNG_ACCEPT, RNG_RESID, RNG_BONUS, RNG_PATH = 1, 2, 3, 4, 5


def philox4x32_10(ctr, key):
    """Philox4x32-10 (Salmon et al., SC'11): 4 x uint32 counter, 2 x uint32 key."""
    c = (C.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (C.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (C.c_uint32 * 4)()
    lib().or_philox4x32_10(c, k, o)
    return [int(x) for x in o]


def uniform(seed: int, v: int, pos: int, seq: int, purpose: int, cycle: int) -> float:
    return lib().or_uniform(seed, v, pos, seq, purpose, cycle)


def _u8(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint8).ctypes.data_as(C.POINTER(C.c_ubyte))


def filter_row(logits: np.ndarray, T: float, top_k: int = 0, top_p: float = 1.0):
    """Top-k / top-p filter of one logit row (the reading stated in
    dflash_oracle.c, or_filter_row): (keep mask [V] uint8, kept count,
    top-p boundary margin)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    keep = np.zeros(lg.shape[0], dtype=np.uint8)
    mg = C.c_double()
    n = lib().or_filter_row(lg.ctypes.data_as(C.POINTER(C.c_float)), lg.shape[0], float(T), int(top_k), float(top_p),
                            keep.ctypes.data_as(C.POINTER(C.c_ubyte)), C.byref(mg))
    return keep, n, mg.value


def sample_row(logits: np.ndarray, T: float, seed: int, pos: int, seq: int, purpose: int, cycle: int, keep=None):
    """A draw from softmax(logits / T) (over the kept entries) by Gumbel-max:
    (token, log-sum-exp over the kept entries, margin)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    lse, mg = C.c_double(), C.c_double()
    kp = None if keep is None else np.ascontiguousarray(keep, dtype=np.uint8)
    tok = lib().or_sample_row_f(lg.ctypes.data_as(C.POINTER(C.c_float)), lg.shape[0], float(T), _u8(kp), seed, pos,
                                seq, purpose, cycle, C.byref(lse), C.byref(mg))
    return tok, lse.value, mg.value


def spec_sample_accept(tl: np.ndarray, dl: np.ndarray, drafts, T: float, seed: int, seq: int, P: int, cycle: int,
                       keep_t=None, keep_d=None):
    """Speculative sampling over one sequence's block: target logits [B][V],
    draft logits [B-1][V], drafts [B-1], optional kept-entry masks of the
    target [B][V] and draft [B-1][V] rows (top-k / top-p) -> (accept length
    k, emitted tokens [k+1], smallest decision margin)."""
    tl = np.ascontiguousarray(tl, dtype=np.float32)
    dl = np.ascontiguousarray(dl, dtype=np.float32)
    B, V = tl.shape
    dr = np.ascontiguousarray(drafts, dtype=np.int32)
    out = np.zeros(B, dtype=np.int32)
    mg = C.c_double()
    kt = None if keep_t is None else np.ascontiguousarray(keep_t, dtype=np.uint8)
    kd = None if keep_d is None else np.ascontiguousarray(keep_d, dtype=np.uint8)
    k = lib().or_spec_sample_accept_f(B, V, tl.ctypes.data_as(C.POINTER(C.c_float)),
                                      dl.ctypes.data_as(C.POINTER(C.c_float)), _u8(kt), _u8(kd),
                                      dr.ctypes.data_as(C.POINTER(C.c_int)), float(T), seed, seq, P, cycle,
                                      out.ctypes.data_as(C.POINTER(C.c_int)), C.byref(mg))
    return k, out[:k + 1].copy(), mg.value



def path_walk_sample(cfg: Cfg, cand: np.ndarray, E, U, Vm, anchor: int, T: float, seed: int, seq: int, P: int,
                     cycle: int):
    """The DFlash 2 path walked by sampling ([G] section 7; the reading in
    dflash_oracle.c, or_path_walk_sample) over the candidates cand
    [B-1][topk]: (path [B-1], log q [B-1][topk], draw margins [B-1])."""
    cd = np.ascontiguousarray(cand, dtype=np.int32)
    Bm1, K = cd.shape
    path = np.zeros(Bm1, dtype=np.int32)
    lq = np.zeros((Bm1, K))
    mg = np.zeros(Bm1)
    lib().or_path_walk_sample(C.byref(cfg.c()), Bm1 + 1, K, U.shape[0], cd.ctypes.data_as(C.POINTER(C.c_int)),
                              _vp(E), _vp(U), _vp(Vm), int(anchor), float(T), seed, seq, P, cycle,
                              path.ctypes.data_as(C.POINTER(C.c_int)), _dp(lq), _dp(mg))
    return path, lq, mg


def spec_sample_accept_sparse(tl: np.ndarray, qcand: np.ndarray, qlogq: np.ndarray, drafts, T: float, seed: int,
                              seq: int, P: int, cycle: int, keep_t=None):
    """Speculative sampling with the sampled walk's sparse proposal (qcand,
    qlogq [B-1][K]) in place of the draft softmax -> (k, emitted tokens, smallest margin)."""
    tl = np.ascontiguousarray(tl, dtype=np.float32)
    B, V = tl.shape
    qc = np.ascontiguousarray(qcand, dtype=np.int32)
    lq = np.ascontiguousarray(qlogq, dtype=np.float64)
    dr = np.ascontiguousarray(drafts, dtype=np.int32)
    out = np.zeros(B, dtype=np.int32)
    mg = C.c_double()
    kt = None if keep_t is None else np.ascontiguousarray(keep_t, dtype=np.uint8)
    k = lib().or_spec_sample_accept_sparse(B, V, tl.ctypes.data_as(C.POINTER(C.c_float)), _u8(kt), qc.shape[1],
                                           qc.ctypes.data_as(C.POINTER(C.c_int)), _dp(lq),
                                           dr.ctypes.data_as(C.POINTER(C.c_int)), float(T), seed, seq, P, cycle,
                                           out.ctypes.data_as(C.POINTER(C.c_int)), C.byref(mg))
    return k, out[:k + 1].copy(), mg.value
