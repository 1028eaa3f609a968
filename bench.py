#!/usr/bin/env python
"""Benchmark one DFlash draft-and-verify cycle on synthetic random-init
models (default: the Qwen3-8B-shaped cycle at batch 1, context 4096).

A step is one whole cycle over the batch: draft block (5 draft layers + LM
head argmax), causal target verification (36 target layers + LM head), greedy
acceptance, and context injection of the committed positions.  Each step
starts from the same state (context length and anchor restored), so every
step is the same workload.  Prints one JSON line.

  python bench.py [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on this host
Under torchrun (N > 1) every rank runs an independent replica (no data-path
collective); value = all ranks' draft-block steps / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft-block steps/s & verified tok/s at batch 1/32; HBM GB/s as % of roofline"
UNIT = "draft-block steps/s"  # one step: a whole draft-and-verify cycle of one sequence
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1700.0  # sustained bf16, the fallback for a kernel timed inside a long step


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="qwen3-8b-b1")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--trace-replays", type=int, default=5)
    p.add_argument("--no-sampling", action="store_true", help="skip the sampling-mode cycle timing")
    p.add_argument("--no-denoise", action="store_true", help="skip the multi-round denoising draft timing")
    p.add_argument("--no-conv", action="store_true", help="skip the draft-convolution timing")
    p.add_argument("--no-paged", action="store_true", help="skip the paged-KV cycle timing")
    p.add_argument("--no-b32", action="store_true", help="skip the 32-sequence record")
    p.add_argument("--layers", default="", help="T,D: shrink to T target / D draft layers (profiling captures "
                   "only; the line then names the reduced config)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9 or (self.uuid and self.uuid not in parts[0]):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload


def setup_workload(w, seed: int = 0, model=None):
    import torch

    from block_diffusion_speculative_step_gb300 import synth
    from block_diffusion_speculative_step_gb300.engine import Engine

    S, B = w.batch, w.block
    lens = synth.make_ctx_lengths(seed + 7, w)
    ctx_max = max(lens)
    cap = ((ctx_max + 2 * B + 127) // 128) * 128  # whole 128-slot pages (the paged-cache line)
    if model is None:
        model = synth.make_model(w, seed=seed, device="cuda")
    fill_rows = 256
    eng = Engine(w, model, S, cap, prefill_chunk=B, fuse_rows=fill_rows)
    dt = synth.torch_dtype(w)
    # target KV: synthetic N(0,1) keys/values in every slot
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + 11)
    for t in eng.caches.tk + eng.caches.tv:
        t.copy_(torch.randn(t.shape, generator=gen, device="cuda", dtype=torch.float32).to(dt))
    # draft context: inject N(0,1) tap features of every context position
    F, H = len(w.taps), w.draft.hidden
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    feats = torch.empty(S * fill_rows, F, H, dtype=dt, device="cuda")
    base = torch.zeros(S, dtype=torch.int32, device="cuda")
    lo = max(0, ctx_max - w.window) if w.window else 0
    for c0 in range(lo - lo % fill_rows, ctx_max, fill_rows):
        feats.normal_(0.0, 1.0, generator=gen)
        base.fill_(c0)
        valid = (lens_t - c0).clamp(0, fill_rows).to(torch.int32)
        eng.fuse_with(feats, fill_rows, base, valid)
    torch.cuda.synchronize()
    eng.base_pos.copy_(lens_t)
    eng.anchor.copy_(synth.make_tokens(seed + 13, S, w.vocab, device="cuda"))
    planted = None
    if w.accept_mean > 0 and eng.has_target:
        planted = plant_drafts(eng, w, seed)
    return eng, lens, planted


def plant_drafts(eng, w, seed):
    """Drafts that agree with the target's greedy continuation for k_s tokens
    and then differ, k_s ~ Geometric(mean w.accept_mean) clamped to B-1:
    verification then accepts exactly k_s (setup only, not timed)."""
    import torch

    from block_diffusion_speculative_step_gb300 import synth

    S, B = w.batch, w.block
    ks = synth.make_accept_lengths(seed + 17, w)
    base0, anchor0 = eng.base_pos.clone(), eng.anchor.clone()
    greedy = []
    for _ in range(B - 1):
        eng.greedy_step()
        greedy.append(eng.anchor.clone())
    greedy = torch.stack(greedy, 1)  # [S][B-1]: tokens at positions P+1 .. P+B-1
    eng.base_pos.copy_(base0)
    eng.anchor.copy_(anchor0)
    planted = greedy.clone()
    for s, k in enumerate(ks):
        if k < B - 1:
            planted[s, k] = (greedy[s, k] + 1) % (w.vocab - 1)
    return planted.to(torch.int32).contiguous(), ks


# ------------------------------------------------------- algorithmic bytes


def layer_weight_bytes(s, es: int = 2) -> float:
    """Weight bytes of one decoder layer: QKV, O, gate+up, down (each read once)."""
    qkv = (s.n_q + 2 * s.n_kv) * s.head_dim * s.hidden
    return float(es * (qkv + s.hidden * s.n_q * s.head_dim + 3 * s.hidden * s.inter))


def layer_gemm_params(s) -> float:
    """Weights of one decoder layer's four projections (QKV, O, gate+up, down)."""
    qkv = (s.n_q + 2 * s.n_kv) * s.head_dim * s.hidden
    return float(qkv + s.hidden * s.n_q * s.head_dim + 3 * s.hidden * s.inter)


def gemm_flops_per_cycle(w, rows_committed: float) -> float:
    """Algorithmic flops (2 per multiply-add) of the GEMM family in one cycle:
    every draft and target layer over all S*B block rows, and the fusion's
    FC and K/V-injection projections over the committed rows."""
    M = w.batch * w.block
    H = w.draft.hidden
    fuse = H * len(w.taps) * H + w.draft.layers * 2 * w.draft.n_kv * w.draft.head_dim * H
    return 2.0 * (M * (w.draft.layers * layer_gemm_params(w.draft) + w.target.layers * layer_gemm_params(w.target))
                  + rows_committed * fuse)


def tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a family timed inside a long step:
    the measured sustained cuBLAS figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        if "bf16_tflops_sustained" in pk:
            return float(pk["bf16_tflops_sustained"]), "measured bf16_tflops_sustained (of measured)"
    return FALLBACK_BF16_TFLOPS, "fallback bf16 TFLOP/s"


def kv_bytes(s, keys: int, es: int = 2) -> float:
    """K + V bytes of `keys` cache slots of one layer."""
    return float(2 * es * keys * s.n_kv * s.head_dim)


def draft_step_bytes(w, lens) -> float:
    """The draft-block step: every draft layer's weights, the shared LM head
    and each sequence's injected context K/V (the window's with a window),
    each read once."""
    ctx = sum(min(P, w.window) if w.window else P for P in lens)
    return (w.draft.layers * (layer_weight_bytes(w.draft) + kv_bytes(w.draft, ctx)) +
            2.0 * w.vocab * w.draft.hidden)


def attention_bytes_per_cycle(w, lens, with_target: bool) -> float:
    """K/V bytes all attention launches of one cycle read: the draft's
    context plus block, and the target's cache up to each block's last row."""
    B = w.block
    d = w.draft.layers * kv_bytes(w.draft, sum((min(P, w.window) if w.window else P) + B for P in lens))
    t = w.target.layers * kv_bytes(w.target, sum(P + B for P in lens)) if with_target else 0.0
    return d + t


def cycle_bytes(w, lens, with_target: bool) -> float:
    """One whole cycle: the draft step, the verification (target weights,
    LM head, target K/V) and the fusion (FC and K/V-injection weights)."""
    b = draft_step_bytes(w, lens)
    if with_target:
        b += w.target.layers * (layer_weight_bytes(w.target) + kv_bytes(w.target, sum(P + w.block for P in lens)))
        b += 2.0 * w.vocab * w.target.hidden
    H = w.draft.hidden
    b += 2.0 * H * len(w.taps) * H + w.draft.layers * 2.0 * 2 * w.draft.n_kv * w.draft.head_dim * H
    return b


# ------------------------------------------------------------- CPU oracle


def host_sample(w, seed: int = 0):
    """Host-side inputs for timing the oracle at the workload's shapes, drawn
    on the CPU without the GPU library: one target and one draft layer,
    the LM head, the fusion FC, context caches of N(0,1) values."""
    import dataclasses

    import numpy as np
    import torch

    from block_diffusion_speculative_step_gb300 import synth
    from oracle import oracle as O

    n = synth.to_numpy
    dt = synth.torch_dtype(w)
    dr = synth._Draw(seed, "cpu")
    F, H = len(w.taps), w.draft.hidden

    def cfg(s):
        return O.Cfg(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, w.dtype == "bf16", w.rope_theta, w.rms_eps)

    def layer(s):
        L = synth.make_stack(dr, dataclasses.replace(s, layers=1), dt, 0.02, 0.0)["layers"][0]
        return O.Layer.from_stacked(cfg(s), n(L["w_qkv"]), n(L["w_o"]), n(L["w_gu"]), n(L["w_down"]), n(L["ln1"]),
                                    n(L["ln2"]))

    smp = {"dc": cfg(w.draft), "Ld": layer(w.draft), "lm": n(dr.normal((w.vocab, H), 0.02, dt)),
           "fc": n(dr.normal((H, F * H), 0.02, dt)), "fc_norm": n(torch.ones(H, dtype=dt))}
    rng = np.random.default_rng(seed)
    P = max(synth.make_ctx_lengths(seed + 7, w))
    cap = P + 2 * w.block
    dcap = w.window if w.window else cap

    def cache(s, slots):
        return O.rnd(cfg(s), rng.standard_normal((s.n_kv, slots, s.head_dim)))

    smp["dk"], smp["dv"] = cache(w.draft, dcap), cache(w.draft, dcap)
    if w.run_target:
        smp["tc"] = cfg(w.target)
        smp["Lt"] = layer(w.target)
        smp["tk"], smp["tv"] = cache(w.target, cap), cache(w.target, cap)
    smp["P"] = P
    return smp


def oracle_units(w, smp, vocab_frac: float = 1.0):
    """Seconds of each unit of one sequence's cycle on the oracle as it
    stands: one target layer, one draft layer, the LM head (over vocab_frac of
    the vocabulary, scaled to all of it) and the fusion of one position."""
    import time as _t

    import numpy as np

    from oracle import oracle as O

    B, P = w.block, smp["P"]
    rng = np.random.default_rng(1)
    times = {}
    if "Lt" in smp:
        h = rng.standard_normal((B, w.target.hidden))
        t0 = _t.perf_counter()
        O.decoder_layer(smp["tc"], smp["Lt"], h, P, O.CAUSAL, smp["tk"].copy(), smp["tv"].copy())
        times["target_layer"] = _t.perf_counter() - t0
    h = rng.standard_normal((B, w.draft.hidden))
    t0 = _t.perf_counter()
    O.decoder_layer(smp["dc"], smp["Ld"], h, P, O.BIDIR, smp["dk"], smp["dv"], w.window)
    times["draft_layer"] = _t.perf_counter() - t0
    V = max(1, int(w.vocab * vocab_frac))
    x = O.rnd(smp["dc"], rng.standard_normal((B, w.draft.hidden)))
    t0 = _t.perf_counter()
    O.lm_head_argmax(smp["dc"], smp["lm"][:V], x)
    times["lm_head"] = (_t.perf_counter() - t0) * (w.vocab / V)
    F = len(w.taps)
    feats = O.rnd(smp["dc"], rng.standard_normal((1, F * w.draft.hidden)))
    Ld = smp["Ld"]
    kcs = [np.zeros_like(smp["dk"]) for _ in range(w.draft.layers)]
    vcs = [np.zeros_like(smp["dv"]) for _ in range(w.draft.layers)]
    t0 = _t.perf_counter()
    O.fuse_context(smp["dc"], F, smp["fc"], smp["fc_norm"], feats, [P], [Ld.wk] * w.draft.layers,
                   [Ld.wv] * w.draft.layers, kcs, vcs, w.window)
    times["fusion_row"] = _t.perf_counter() - t0
    return times


def oracle_rates(w, times) -> dict:
    """Per-unit rates of the whole batch from one sequence's unit seconds:
    the draft-block step (draft layers + LM head), the verification (target
    layers + LM head), the fusion of the accepted positions (one per
    sequence at zero acceptance) and the whole cycle, extrapolated by the
    layer counts and the batch (sequences are independent)."""
    S = w.batch
    draft = w.draft.layers * times["draft_layer"] + times["lm_head"]
    verify = (w.target.layers * times["target_layer"] + times["lm_head"]) if "target_layer" in times else 0.0
    fusion = times["fusion_row"]
    cycle = draft + verify + fusion
    return {"draft_block_s": S * draft, "verify_s": S * verify, "fusion_s": S * fusion, "cycle_s": S * cycle,
            "cycles_per_s": 1.0 / (S * cycle)}


def cpu_baseline(w, smp, lm_frac_1thread: float = 1 / 16):
    """The oracle timed on this host at one thread and at all cores, per
    unit (LM head over 1/16 of the vocabulary at one thread, scaled)."""
    import os as _os

    from oracle import oracle as O

    cores = _os.cpu_count() or 1
    out = {}
    for tag, n, frac in (("1_thread", 1, lm_frac_1thread), ("all_cores", cores, 1.0)):
        O.set_threads(n)
        t = oracle_units(w, smp, frac)
        out[tag] = {"threads": O.threads(), "unit_s": {k: round(v, 4) for k, v in t.items()},
                    **{k: v for k, v in oracle_rates(w, t).items()}}
    O.set_threads(cores)
    return out, cores


# ------------------------------------------------------------------ arms


def run_reference(args):
    """The oracle, timed on this host's cores, built from host-side inputs
    only (no GPU library).  Each step is a bounded sample of the workload:
    one target layer, one draft layer, the LM head over 1/16 of the
    vocabulary (scaled) and one fusion row of one sequence; the line's value
    is the whole cycle extrapolated from those unit times by the layer
    counts and the batch."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from block_diffusion_speculative_step_gb300 import synth
    from oracle import oracle as O

    w = synth.WORKLOADS[args.workload]
    smp = host_sample(w)
    cores = os.cpu_count() or 1
    O.set_threads(cores)
    for _ in range(args.warmup):
        oracle_units(w, smp, 1 / 16)
    t0 = time.perf_counter()
    acc = {}
    for _ in range(args.steps):
        for k, v in oracle_units(w, smp, 1 / 16).items():
            acc[k] = acc.get(k, 0.0) + v
    el = time.perf_counter() - t0
    mean = {k: v / args.steps for k, v in acc.items()}
    rates = oracle_rates(w, mean)
    value = rates["cycles_per_s"] * w.batch
    cpu = {"value": value, "unit": UNIT, "cores": O.threads(), "kind": "oracle",
           "sample": "per step: 1 target layer + 1 draft layer + LM head over 1/16 of the vocabulary (scaled "
                     "x16) + 1 fusion row of one sequence, all host cores; cycle extrapolated by layer counts "
                     "and batch", "unit_s": {k: round(v, 4) for k, v in mean.items()}}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * rates["cycle_s"] / w.batch,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random-init weights, N(0,1) context), drawn on the host",
            "config": {"workload": w.name, "batch": w.batch, "ctx": w.ctx if not w.ctx_min else [w.ctx_min, w.ctx],
                       "block": w.block},
            "extrapolated": {"value": True, "measured_sample_ms_per_step": 1000.0 * el / args.steps,
                             "how": "value and ms_per_step are the whole cycle extrapolated from the measured "
                                    "unit times; measured_sample_ms_per_step is the sampled work per step"},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": el}
    print(json.dumps(line))


def reduce_max(x: float, world: int, device: str = "cpu") -> float:
    """The largest x over the ranks (the slowest replica sets the job's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rates(world: int, S: int, steps: int, ms: float, tokens_per_step: float):
    """Whole-job draft-block steps/s and verified tokens/s: every rank runs its
    own replica of S sequences, so the job does world * S draft blocks and
    world * tokens_per_step verified tokens per step in ms per `steps` steps."""
    value = world * S * steps / (ms / 1000.0)
    verified = world * tokens_per_step * steps / (ms / 1000.0)
    return value, verified


def cost_model(t_draft_ms: float, t_cycle_ms: float, tokens_per_cycle: float) -> dict:
    """The per-token cost of a speculative cycle (DFlash 2 release news,
    'beyond speed: what DFlash 2 means for deployment'): the draft and the
    verification of one round spread over the tokens the round yields.  The
    verification share is the rest of the measured cycle (target forward,
    acceptance and context injection)."""
    return {"draft_ms": t_draft_ms, "verify_and_fusion_ms": t_cycle_ms - t_draft_ms,
            "tokens_per_cycle": tokens_per_cycle, "per_token_ms": t_cycle_ms / tokens_per_cycle}


def kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_diffusion_speculative_step_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(family: str):
    """Per-launch DRAM bytes of `family` from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(family)
    if not ent or ent.get("kernel_hash") != kernel_hash():
        return None
    return ent.get("dram_bytes_per_launch")


def time_graph(graph, n: int, warmup: int, world: int) -> float:
    """ms per replay of a captured CUDA graph (CUDA events on the stream the
    replays are launched on; the slowest rank)."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return reduce_max(e0.elapsed_time(e1), world, "cuda") / n


def capture(fn):
    import torch

    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def trace_families(fn, replays: int):
    """Per-family kernel time inside graph replays of fn: the library brackets
    every launch step with CUDA events (captured into the graph), summed per
    kernel family.  Returns {family: [launches, ms, bytes]} per replay."""
    import torch

    from block_diffusion_speculative_step_gb300 import dflash as D

    D.dflash_trace_begin(16384)
    tg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tg):
        fn()
    D.dflash_trace_pause()
    fam = {}
    reps = max(1, replays)
    for _ in range(reps):
        tg.replay()
        torch.cuda.synchronize()
        for name, (n, ms, by) in D.dflash_trace_read().items():
            a = fam.setdefault(name, [0, 0.0, 0.0])
            a[0] += n
            a[1] += ms
            a[2] += by
    D.dflash_trace_end()
    del tg
    return {k: [v[0] // reps, v[1] / reps, v[2] / reps] for k, v in fam.items() if v[0] > 0}


def roof(achieved_gbs: float, peak: float, src: str, **kw) -> dict:
    return {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s", "frac": achieved_gbs / peak,
            "peak_source": f"{src} hbm_gbs (of measured)" if src == "measured" else f"{src} hbm_gbs", **kw}


def run_b32(args, model, world: int, hbm: float, src: str) -> dict:
    """The 32-sequence workload in the same run (qwen3-8b-b32: ragged
    contexts U[1024, 8192], drafts planted so that verification accepts
    exactly k_s ~ Geometric(mean 5) tokens): whole cycle, the draft-block
    step alone, verified tokens/s, and the attention and GEMM families."""
    import torch

    from block_diffusion_speculative_step_gb300 import dflash as D
    from block_diffusion_speculative_step_gb300 import synth

    w = synth.WORKLOADS["qwen3-8b-b32"]
    eng, lens, planted = setup_workload(w, seed=0, model=model)
    planted_t, ks = planted
    base0, anchor0 = eng.base_pos.clone(), eng.anchor.clone()

    def step():
        eng.base_pos.copy_(base0)
        eng.anchor.copy_(anchor0)
        eng.cycle(planted_t)

    step()
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    acc = eng.accept_len.cpu()
    exact = [int(a) for a in acc] == [int(k) for k in ks]
    assert exact, f"planted accept lengths {ks} but verification accepted {acc.tolist()}"
    graph = capture(step)
    n = max(3, min(args.steps, 40))
    ms = time_graph(graph, n, args.warmup, world)
    tokens = float((acc + 1).sum())
    dgraph = capture(lambda: eng.draft())
    dms = time_graph(dgraph, n, args.warmup, world)
    fam = trace_families(step, 1)
    eng.base_pos.copy_(base0)
    eng.anchor.copy_(anchor0)
    S = w.batch
    attn = fam.get("attention")
    rec = {"workload": w.name, "batch": S, "ctx": [min(lens), max(lens)], "ms_per_cycle": ms,
           "cycles_per_s": world * 1000.0 / ms, "draft_block_steps_per_s": world * S * 1000.0 / dms,
           "draft_block_ms": dms, "verified_tok_s": world * tokens * 1000.0 / ms,
           "mean_accept": float(acc.float().mean()), "accept_lengths_as_planted": exact, "steps": n,
           "rooflines": {
               "cycle": roof(cycle_bytes(w, lens, True) / (ms / 1000.0) / 1e9, hbm, src,
                             bytes_per_unit=cycle_bytes(w, lens, True)),
               "draft_block_step": roof(draft_step_bytes(w, lens) / (dms / 1000.0) / 1e9, hbm, src,
                                        bytes_per_unit=draft_step_bytes(w, lens))},
           "kernels": {k: {"launches_per_step": v[0], "ms_per_step": v[1]} for k, v in fam.items()}}
    if attn:
        ab = attention_bytes_per_cycle(w, lens, True)
        rec["rooflines"]["attention"] = roof(ab / (attn[1] / 1000.0) / 1e9, hbm, src, bytes_per_cycle=ab,
                                             launches_per_cycle=attn[0], avg_launch_us=1000.0 * attn[1] / attn[0])
    gm = fam.get("gemm_tc")
    if gm:  # at 512 block rows the projections are dense contractions: tensor-bound
        fl = gemm_flops_per_cycle(w, tokens)
        tp, tsrc = tensor_peak()
        ach = fl / (gm[1] / 1000.0) / 1e12
        rec["rooflines"]["gemm_tc"] = {"bound": "tensor", "achieved": ach, "peak": tp, "unit": "TFLOP/s",
                                       "frac": ach / tp, "peak_source": tsrc, "flops_per_cycle": fl,
                                       "launches_per_cycle": gm[0], "ms_per_cycle": gm[1]}
    del graph, dgraph, eng
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist

    from block_diffusion_speculative_step_gb300 import build as b
    from block_diffusion_speculative_step_gb300 import dflash as D
    from block_diffusion_speculative_step_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if rank == 0:
        b.build()
    if world > 1:
        dist.barrier()
    b.build()
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses
        t_l, d_l = (int(x) for x in args.layers.split(","))
        w = dataclasses.replace(w, name=f"{w.name}-layers{t_l},{d_l}", target=dataclasses.replace(w.target, layers=t_l),
                                draft=dataclasses.replace(w.draft, layers=d_l))
    hbm, src = peaks()
    eng, lens, planted = setup_workload(w, seed=0)
    planted_t, ks = (planted if planted else (None, None))
    base0, anchor0 = eng.base_pos.clone(), eng.anchor.clone()

    def step():
        eng.base_pos.copy_(base0)
        eng.anchor.copy_(anchor0)
        eng.cycle(planted_t)

    step()
    torch.cuda.synchronize()
    assert eng.status() == D.DFLASH_OK
    accept = eng.accept_len.cpu()
    if ks is not None:
        assert [int(a) for a in accept] == [int(k) for k in ks], (ks, accept.tolist())
    graph = capture(step)
    fam = trace_families(step, args.trace_replays)
    launches_per_step = sum(v[0] for v in fam.values())

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    clk = ClockSampler(uuid)
    clk.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = reduce_max(e0.elapsed_time(e1), world, "cuda")
    if world > 1:
        dist.barrier()
    ms_per_step = ms / args.steps
    S = w.batch
    mean_accept = float(accept.float().mean())
    value, verified = job_rates(world, S, args.steps, ms, float((accept + 1).sum()))

    # per-step distribution: each replay between its own pair of events
    n_pct = max(3, min(args.steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_pct)]
    torch.cuda.synchronize()
    for a_ev, b_ev in evs:
        a_ev.record()
        graph.replay()
        b_ev.record()
    torch.cuda.synchronize()
    per = sorted(a_ev.elapsed_time(b_ev) for a_ev, b_ev in evs)
    step_pct = {"steps": n_pct, "p50_ms": per[len(per) // 2], "p95_ms": per[min(len(per) - 1, int(0.95 * len(per)))]}

    # the draft-block step alone (graph replay; a draft leaves the state untouched)
    n_d = max(3, min(args.steps, 50))
    dgraph = capture(lambda: eng.draft())
    draft_ms = time_graph(dgraph, n_d, args.warmup, world)
    dfam = trace_families(lambda: eng.draft(), 1)
    del dgraph

    # the same cycle in sampling mode (speculative sampling at T = 1), graph replay
    sampling = None
    if eng.has_target and not args.no_sampling:
        def step_sampled():
            eng.base_pos.copy_(base0)
            eng.anchor.copy_(anchor0)
            eng.cycle_sampled(1.0, 0x5EED, 0)

        sgraph = capture(step_sampled)
        assert eng.status() == D.DFLASH_OK
        n_s = max(3, min(args.steps, 50))
        ms_s = time_graph(sgraph, n_s, args.warmup, world)
        sampling = {"mode": "speculative sampling, temperature 1.0 (Philox4x32-10 draws)",
                    "ms_per_step": ms_s, "value": world * S * 1000.0 / ms_s, "unit": UNIT, "steps": n_s,
                    "overhead_vs_greedy": ms_s / ms_per_step - 1.0}
        del sgraph

        def step_filtered():  # top-k 50 / top-p 0.9 on the draft and target rows
            eng.base_pos.copy_(base0)
            eng.anchor.copy_(anchor0)
            eng.cycle_sampled(1.0, 0x5EED, 0, top_k=50, top_p=0.9)

        fgraph = capture(step_filtered)
        assert eng.status() == D.DFLASH_OK
        sampling["top_k50_top_p0.9_ms_per_step"] = time_graph(fgraph, n_s, args.warmup, world)
        del fgraph
        eng.base_pos.copy_(base0)
        eng.anchor.copy_(anchor0)

    # multi-round block denoising: the draft-block step alone at 2 rounds
    denoise = None
    if not args.no_denoise:
        rgraph = capture(lambda: eng.draft(rounds=2))
        assert eng.status() == D.DFLASH_OK
        denoise = {"mode": "draft-block step alone, graph replay",
                   "rounds_ms": {"1": draft_ms, "2": time_graph(rgraph, n_d, args.warmup, world)},
                   "unit": "ms per draft-block step", "steps": n_d}
        del rgraph

    # DFlash 2 draft convolutions (rank 64, four per draft layer): the
    # draft-block step alone with them (graph replay)
    conv = None
    if not args.no_conv:
        synth.add_conv_weights(eng.m, w, 64)
        if D.dflash_workspace_bytes(D.DFLASH_OP_DRAFT, eng.draft_args(conv_rank=64)) <= eng.ws_bytes:
            cgraph = capture(lambda: eng.draft(conv_rank=64))
            assert eng.status() == D.DFLASH_OK
            c_ms = time_graph(cgraph, n_d, args.warmup, world)
            del cgraph
            conv = {"mode": "draft-block step alone, graph replay", "draft_ms": {"none": draft_ms, "rank64": c_ms},
                    "steps": n_d, "overhead": c_ms / draft_ms - 1.0,
                    "params": w.draft.layers * 4 * 3 * 64 * w.draft.hidden}
        for L in eng.m["draft"]["layers"]:
            L.pop("conv_w1", None)
            L.pop("conv_w2", None)

    # per-token cost: the draft-block step alone, the rest of the cycle, over
    # the tokens a cycle emits (accepted drafts + the bonus token)
    cost = cost_model(draft_ms, ms_per_step, mean_accept + 1.0)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h_in = torch.empty(2, S, dtype=torch.int32).pin_memory()
        h_in[0].copy_(base0.cpu())
        h_in[1].copy_(anchor0.cpu())
        h_out = torch.empty(S + S * w.block, dtype=torch.int32).pin_memory()
        e2e_steps = max(3, min(args.steps, 50))

        def e2e_step():
            eng.base_pos.copy_(h_in[0], non_blocking=True)
            eng.anchor.copy_(h_in[1], non_blocking=True)
            eng.cycle(planted_t)
            h_out[:S].copy_(eng.accept_len, non_blocking=True)
            h_out[S:].copy_(eng.out_tokens.view(-1), non_blocking=True)
            torch.cuda.synchronize()

        for _ in range(2):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        el = reduce_max(time.perf_counter() - t0, world, "cuda")
        e2e = {"value": world * S * e2e_steps / el, "unit": UNIT, "h2d_bytes_per_step": int(h_in.numel() * 4),
               "d2h_bytes_per_step": int(h_out.numel() * 4), "steps": e2e_steps,
               "path": "eager C-ABI calls per step (no graph), pinned host inputs/outputs"}

    per_fam = {k: {"launches_per_step": v[0], "ms_per_step": v[1], "share": 0.0,
                   "gbs": (v[2] / (v[1] / 1000.0) / 1e9) if v[1] > 0 and v[2] > 0 else None}
               for k, v in fam.items()}
    tot = sum(v["ms_per_step"] for v in per_fam.values()) or 1.0
    for v in per_fam.values():
        v["share"] = v["ms_per_step"] / tot
    dom = max(per_fam, key=lambda k: per_fam[k]["ms_per_step"])
    dv = fam[dom]
    achieved = dv[2] / (dv[1] / 1000.0) / 1e9 if dv[1] > 0 else 0.0
    roofline = roof(achieved, hbm, src, kernel=dom, traffic=traffic_for(dom), bytes_per_launch=dv[2] / max(1, dv[0]),
                    avg_launch_us=1000.0 * dv[1] / max(1, dv[0]))
    # the units the target is stated for: the draft-block step and attention
    # (batch 1), next to the whole cycle and each weight-streaming family
    rooflines = {
        "draft_block_step": roof(draft_step_bytes(w, lens) / (draft_ms / 1000.0) / 1e9, hbm, src,
                                 bytes_per_unit=draft_step_bytes(w, lens), ms_per_unit=draft_ms,
                                 launches=sum(v[0] for v in dfam.values())),
        "cycle": roof(cycle_bytes(w, lens, eng.has_target) / (ms_per_step / 1000.0) / 1e9, hbm, src,
                      bytes_per_unit=cycle_bytes(w, lens, eng.has_target), ms_per_unit=ms_per_step)}
    if "attention" in fam:
        a = fam["attention"]
        ab = attention_bytes_per_cycle(w, lens, eng.has_target)
        rooflines["attention"] = roof(ab / (a[1] / 1000.0) / 1e9, hbm, src, bytes_per_launch=ab / a[0],
                                      avg_launch_us=1000.0 * a[1] / a[0], launches_per_cycle=a[0],
                                      traffic=traffic_for("attention"))
    for k in ("gemm_tc", "lm_head"):
        if k in fam and fam[k][2] > 0:
            rooflines[k] = roof(fam[k][2] / (fam[k][1] / 1000.0) / 1e9, hbm, src,
                                bytes_per_launch=fam[k][2] / fam[k][0], avg_launch_us=1000.0 * fam[k][1] / fam[k][0])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        units, cores = cpu_baseline(w, host_sample(w))
        cpu = {"value": units["all_cores"]["cycles_per_s"], "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "one sequence's units at the workload's shapes (1 target layer, 1 draft layer, the LM "
                         "head, 1 fusion row; at 1 thread the LM head over 1/16 of the vocabulary, scaled), timed "
                         "at 1 thread and at all cores; cycle extrapolated by layer counts and batch",
               "extrapolated": True, "per_unit": units}

    # paged KV: the same cycle with the target and draft caches moved into
    # 128-slot page pools handed out in a shuffled order (graph replay)
    paged = None
    if not args.no_paged and eng.has_target and eng.cap % 128 == 0 and eng.dcap % 128 == 0:
        eng.page_caches(128, seed=0)
        pgraph = capture(step)
        assert eng.status() == D.DFLASH_OK
        same = bool(torch.equal(eng.accept_len.cpu(), accept))
        n_p = max(3, min(args.steps, 50))
        ms_p = time_graph(pgraph, n_p, args.warmup, world)
        paged = {"mode": "the same cycle on 128-slot KV pages (shuffled page order), graph replay",
                 "ms_per_step": ms_p, "value": world * S * 1000.0 / ms_p, "unit": UNIT, "steps": n_p,
                 "overhead_vs_contiguous": ms_p / ms_per_step - 1.0, "same_accept_lengths": same}
        del pgraph

    # the 32-sequence workload, measured in the same run
    b32 = None
    if args.workload == "qwen3-8b-b1" and not args.layers and not args.no_b32:
        model = eng.m
        del graph, eng
        torch.cuda.empty_cache()
        b32 = run_b32(args, model, world, hbm, src)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded random-init weights, N(0,1) context)",
            "config": {"workload": w.name, "batch": S, "ctx": w.ctx if not w.ctx_min else [w.ctx_min, w.ctx],
                       "block": w.block, "draft_layers": w.draft.layers,
                       "target_layers": w.target.layers if w.run_target else 0,
                       "step": "one whole draft-and-verify cycle of the batch: draft block (draft layers + LM-head "
                               "argmax), target verification + acceptance, context injection",
                       "l2": "inputs larger than L2 (weights streamed each step)",
                       "parallelism": f"replicas x{world}", "timing": "CUDA graph replay, CUDA events"},
            "cycles_per_s": world * 1000.0 / ms_per_step,
            "draft_block_steps_per_s": world * S * 1000.0 / draft_ms, "draft_block_ms": draft_ms,
            "verified_tok_s": verified, "mean_accept": mean_accept,
            "roofline": roofline, "rooflines": rooflines, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "clocks": clocks, "step_ms_distribution": step_pct, "kernels": per_fam, "b32": b32,
            "sampling": sampling, "denoise": denoise, "conv": conv, "paged": paged, "cost_model": cost}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
