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
