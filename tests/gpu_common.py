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


def assert_hidden_close(got, ref):
    """fp32 residual stream after one bf16 layer: bf16 rounding of the
    projection inputs (one-step differences at rounding boundaries) and of
    the attention probabilities move individual outputs by up to ~1e-2 of
    their size; bound |err| <= 0.02 * max(1, |ref|)."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    tol = 2e-2 * np.maximum(1.0, np.abs(ref))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} beyond tolerance; max err {np.abs(got - ref).max():.4g}"
