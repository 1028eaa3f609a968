"""Shared setup for the GPU parity tests: small seeded workloads on the
device, oracle models of the same draws, and comparison helpers."""
from __future__ import annotations

import numpy as np
import torch

from block_diffusion_speculative_step_gb300 import synth
from block_diffusion_speculative_step_gb300.engine import Engine
from tests import helpers as Hh

# Tolerances: fp32 mode 1e-4 on logits, bf16 mode 2e-2 max-abs.
LOGIT_TOL = {"f32": 1e-4, "bf16": 2e-2}
NEAR_TIE = 1e-4


def to_dev(m, device="cuda"):
    if isinstance(m, dict):
        return {k: to_dev(v, device) for k, v in m.items()}
    if isinstance(m, list):
        return [to_dev(v, device) for v in m]
    if isinstance(m, torch.Tensor):
        return m.to(device)
    return m


def setup(w: synth.Workload, seed=0, S=1, cap=256, jitter=0.1, chunk=256):
    m_cpu = synth.make_model(w, seed=seed, jitter=jitter, with_target=True)
    eng = Engine(w, to_dev(m_cpu), S, cap, prefill_chunk=chunk)
    om = Hh.omodel(w, m_cpu)
    return eng, om, m_cpu


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def check_argmax(gpu_idx, ora_idx, ora_margin, gpu_logits=None, ora_logits=None, tol=NEAR_TIE):
    """Bit-exact argmax, except rows whose oracle top1-top2 margin is below
    `tol` (near-ties, reported).  Returns the number of excluded rows."""
    gpu_idx = np.asarray(gpu_idx).ravel()
    ora_idx = np.asarray(ora_idx).ravel()
    ora_margin = np.asarray(ora_margin).ravel()
    excl = 0
    for i, (g, o, mg) in enumerate(zip(gpu_idx, ora_idx, ora_margin)):
        if g != o:
            assert mg < tol, f"row {i}: gpu argmax {g} != oracle {o} with oracle margin {mg:.3g} >= {tol}"
            excl += 1
    return excl


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """One unit in the last place of bfloat16 at |x| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_bf16_close(got, ref, ulps: float = 1.0, atol: float = 1e-3):
    """Values the GPU stores in bf16 (K/V cache, fused features): the GPU
    rounds an fp32 sum, the oracle an fp64 one, so a value sitting on a
    rounding boundary may land one bf16 step away; and a one-step difference
    of one bf16 projection input moves a projected value by up to about
    2^-8 * |x| * |w| (~1e-4 .. 1e-3) whatever the value's own size."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    tol = ulps * bf16_ulp(np.maximum(np.abs(got), np.abs(ref))) + atol
    bad = np.abs(got - ref) > tol
    if bad.any():
        idx = np.argwhere(bad)[:8]
        det = "; ".join(f"{tuple(int(v) for v in i)}: got {got[tuple(i)]:.7g} ref {ref[tuple(i)]:.7g}" for i in idx)
        raise AssertionError(f"{bad.sum()} of {bad.size} beyond {ulps} bf16 ulp: {det}")


# ---------------------------------------------------------------- teacher forcing
#
# A bf16 network compared with an fp64 oracle cannot agree element by element
# after more than a few rounding points: the GPU's fp32 sums and the oracle's
# fp64 sums differ by ~1e-6 relative, which crosses a bf16 rounding boundary
# for a fraction of the elements; each crossing is a full one-step (2^-8
# relative) difference, which the next projection spreads over every output,
# so the next rounding point crosses many more boundaries, and within one
# layer every element of the stream differs by about one bf16 step.  Measured
# at the Qwen3-8B / Llama-3.1-8B shapes: every stage fed the GPU's own inputs
# agrees to one bf16 step in <0.4% of its elements, the layer output to
# 4e-5, the LM head to 4e-4; chained from the same input, 38% of the LM
# head's inputs differ by one step and the logits by up to ~0.02.  So every
# stage is checked against the oracle fed the GPU's inputs to that stage
# (teacher forcing), at bounds derived from that arithmetic; end to end the
# tokens are checked and the logit difference is reported.

H_TOL = 1e-3          # fp32 residual stream after a teacher-forced layer (measured <= 4e-5)
STAGE_ULP_FRAC = 0.02  # share of a bf16 stage's elements that may sit one bf16 step away


def check_stage(name, got, ref, frac=STAGE_ULP_FRAC):
    """A bf16 stage output against the oracle's value computed from the same
    inputs.  Each element is within one bf16 step of max(|got|, |ref|) plus
    5e-5 of the stage's RMS, and at most `frac` of the elements differ at all
    (an fp32 sum on the other side of a rounding boundary).  The absolute
    term is the fp32 error of the sum behind a value that cancels to near
    zero: the tensor cores' fp32 sums of K = 4096 .. 14336 products carry
    errors of up to ~1e-5 of the products' scale (measured 1.3e-5 on a
    SwiGLU product of size 3e-4), which no relative bound covers."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    rms = float(np.sqrt((ref ** 2).mean())) if ref.size else 0.0
    tol = bf16_ulp(np.maximum(np.abs(got), np.abs(ref))) + 5e-5 * rms
    d = np.abs(got - ref)
    bad = d > tol
    if bad.any():
        i = tuple(int(v) for v in np.argwhere(bad)[0])
        raise AssertionError(f"stage {name}: {bad.sum()} of {bad.size} elements beyond one bf16 step; "
                             f"first {i}: got {got[i]:.7g} oracle {ref[i]:.7g}")
    diff = float((d > 0).mean())
    assert diff <= frac, f"stage {name}: {diff:.2%} of the elements differ (bound {frac:.0%})"
    return diff


def stage_buffers(shape, S, rows, bidir, dtype=torch.bfloat16, device="cuda"):
    """Device buffers for dflash_layer_args' stage outputs of one layer."""
    M = S * rows
    z = lambda *s: torch.zeros(s, dtype=dtype, device=device)
    b = dict(x1=z(M, shape.hidden), q=z(M, shape.n_q * shape.head_dim), o=z(M, shape.n_q * shape.head_dim),
             x2=z(M, shape.hidden), act=z(M, shape.inter))
    if bidir:
        b["kb"] = z(S, shape.n_kv, rows, shape.head_dim)
        b["vb"] = z(S, shape.n_kv, rows, shape.head_dim)
    return b


def attach_stages(a, bufs):
    a.out_x_attn = bufs["x1"].data_ptr()
    a.out_q = bufs["q"].data_ptr()
    a.out_attn = bufs["o"].data_ptr()
    a.out_x_mlp = bufs["x2"].data_ptr()
    a.out_act = bufs["act"].data_ptr()
    if "kb" in bufs:
        a.out_kb = bufs["kb"].data_ptr()
        a.out_vb = bufs["vb"].data_ptr()
    return a


def gpu_stages(bufs, s, rows, k_rows=None, v_rows=None):
    """Sequence s's stage values from the buffers, as [rows][width] float64
    (k / v from the block buffers, or given as [nkv][rows][d] cache rows)."""
    sl = slice(s * rows, (s + 1) * rows)
    g = {n: f64(bufs[n][sl]) for n in ("x1", "q", "o", "x2", "act")}
    kr = f64(bufs["kb"][s]) if k_rows is None else np.asarray(k_rows)
    vr = f64(bufs["vb"][s]) if v_rows is None else np.asarray(v_rows)
    g["k"] = kr.transpose(1, 0, 2).reshape(rows, -1)
    g["v"] = vr.transpose(1, 0, 2).reshape(rows, -1)
    return g


def check_layer_tf(O, cfg, L, h_in, p0, mode, kc, vc, gpu, h_out, window=0):
    """One layer's stages and output against the oracle fed the GPU's own
    input to every stage (O.decoder_layer_tf); returns the stages' mismatch
    shares and the output's max difference."""
    h = np.ascontiguousarray(h_in, dtype=np.float64).copy()
    st = O.decoder_layer_tf(cfg, L, h, p0, mode, kc.copy(), vc.copy(), window, given=gpu)
    rep = {n: check_stage(n, gpu[n], st[n]) for n in O.STAGES}
    err = float(np.abs(np.asarray(h_out, dtype=np.float64) - h).max())
    assert err <= H_TOL, f"layer output differs by {err:.3g} from the teacher-forced oracle (bound {H_TOL})"
    rep["h"] = err
    return rep


def draft_parity(O, om, eng, s, gl, gd, window=0, cap=None):
    """Sequence s of a dflash_draft_block call (its logits gl [B-1][V] and
    drafts gd [B-1]) against the oracle.  The block is run again for s alone,
    layer by layer through dflash_decoder_layer_forward (the kernels the draft
    call runs) with its stage outputs, and every layer is checked teacher-
    forced; the LM head is checked from the GPU's final residual at the
    stated logit bound, and the drafts bit for bit (near-ties reported).
    Then the oracle's whole draft forward from the same context gives the
    end-to-end logit difference, which is returned with the rest.  The
    tokens are checked against it too, a disagreement being allowed only
    where the oracle's top-2 margin is below twice that difference."""
    from block_diffusion_speculative_step_gb300 import dflash as D
    from block_diffusion_speculative_step_gb300.engine import layer_weights
    w = eng.w
    B, dsh = w.block, w.draft
    c = om.draft.cfg
    P = int(eng.base_pos[s])
    anchor = int(eng.anchor[s])
    h = torch.zeros(B, dsh.hidden, device="cuda")
    ea = eng.embed_args(eng.ddims, B, h, eng.anchor)
    ea.n_seqs = 1
    ea.first = eng.anchor.data_ptr() + 4 * s
    ea.rest = None
    ea.fill_token = w.mask_id
    D.dflash_embed(ea, eng.ws_ptr, eng.ws_bytes)
    rep = {"layers": []}
    for j in range(dsh.layers):
        h_in = f64(h)
        bufs = stage_buffers(dsh, 1, B, True)
        k, v = eng.caches.dk[j], eng.caches.dv[j]
        a = D.dflash_layer_args()
        a.dims = eng.ddims
        a.w = layer_weights(eng.m["draft"]["layers"][j])
        a.n_seqs, a.rows = 1, B
        a.base_pos = eng.base_pos.data_ptr() + 4 * s
        a.h = h.data_ptr()
        a.kv = D.dflash_kv(k.data_ptr() + s * k.stride(0) * k.element_size(),
                           v.data_ptr() + s * v.stride(0) * v.element_size(), eng.dcap, window)
        a.attn_mode = D.DFLASH_ATTN_BLOCK_BIDIR
        a.max_pos = eng.cap
        a.rope_cs = eng.rope_d.data_ptr()
        a.rope_max_pos = eng.rope_max
        attach_stages(a, bufs)
        D.dflash_decoder_layer_forward(a, eng.ws_ptr, eng.ws_bytes)
        torch.cuda.synchronize()
        rep["layers"].append(check_layer_tf(O, c, om.draft.layers[j], h_in, P, O.BIDIR, f64(k[s]), f64(v[s]),
                                            gpu_stages(bufs, 0, B), f64(h), window))
    x = O.final_norm(c, f64(h), om.draft.g_final)
    am, mg, lg = O.lm_head_argmax(c, om.Wlm, x[1:], want_logits=True)
    gl = np.asarray(gl)
    rep["head_err"] = float(np.abs(gl - lg).max())
    assert rep["head_err"] <= LOGIT_TOL["bf16"], f"LM head logits differ by {rep['head_err']} (teacher-forced)"
    if gd is not None:
        rep["head_ties"] = check_argmax(gd, am, mg, tol=max(NEAR_TIE, 2 * rep["head_err"]))
    st = O.new_state(om, cap or eng.cap)
    st.dk = [f64(t[s]) for t in eng.caches.dk]
    st.dv = [f64(t[s]) for t in eng.caches.dv]
    am2, mg2, lg2 = O.draft_forward(om, st, anchor, P, want_logits=True)
    rep["e2e_err"] = float(np.abs(gl - lg2).max())
    if gd is not None:
        rep["e2e_ties"] = check_argmax(gd, am2, mg2, tol=max(NEAR_TIE, 2 * rep["e2e_err"]))
        rep["e2e_same_tokens"] = int((np.asarray(gd) == am2).sum())
    # The oracle's own sensitivity: its draft forward again with 0.1% of the
    # first layer's attention input moved one bf16 step (the pattern of an
    # fp32 sum landing on the other side of a rounding boundary, which the
    # GPU shows at 0.002-0.4% of every stage's elements).  The rounding
    # points after it amplify that exactly as they amplify the GPU's fp32
    # arithmetic, so the GPU's end-to-end difference must be of this order;
    # a wrong term anywhere would be far above it.
    rng = np.random.default_rng(1234)
    hn = O.embed(c, om.E, [anchor] + [om.mask_id] * (B - 1))
    dk = [f64(t[s]) for t in eng.caches.dk]
    dv = [f64(t[s]) for t in eng.caches.dv]
    for j, L in enumerate(om.draft.layers):
        if j == 0:
            x1 = O.decoder_layer_tf(c, L, hn.copy(), P, O.BIDIR, dk[0].copy(), dv[0].copy(), window)["x1"]
            idx = rng.choice(x1.size, max(1, x1.size // 1000), replace=False)
            flat = x1.reshape(-1)
            flat[idx] += np.sign(flat[idx]) * bf16_ulp(flat[idx])
            O.decoder_layer_tf(c, L, hn, P, O.BIDIR, dk[0], dv[0], window, given={"x1": x1})
        else:
            O.decoder_layer(c, L, hn, P, O.BIDIR, dk[j], dv[j], window)
    xn = O.final_norm(c, hn, om.draft.g_final)
    _, _, lgn = O.lm_head_argmax(c, om.Wlm, xn[1:], want_logits=True)
    rep["oracle_noise_err"] = float(np.abs(lgn - lg2).max())
    assert rep["e2e_err"] <= 4 * max(rep["oracle_noise_err"], 1e-3), \
        f"end-to-end logit difference {rep['e2e_err']:.4g} far above the oracle's own one-step sensitivity " \
        f"{rep['oracle_noise_err']:.4g}"
    rep["tf_logits"] = lg
    return rep
