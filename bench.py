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
UNIT = "draft-block steps/s"
FALLBACK_HBM_GBS = 6800.0


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


def setup_workload(w, seed: int = 0):
    import torch

    from block_diffusion_speculative_step_gb300 import synth
    from block_diffusion_speculative_step_gb300.engine import Engine

    S, B = w.batch, w.block
    lens = synth.make_ctx_lengths(seed + 7, w)
    ctx_max = max(lens)
    cap = ((ctx_max + 2 * B + 127) // 128) * 128  # whole 128-slot pages (the paged-cache line)
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


# ------------------------------------------------------------- CPU oracle


def oracle_sample(w, eng, lens, vocab_frac: float = 1.0):
    """Time the CPU oracle (all host cores, as it stands) on one target layer,
    one draft layer, the LM head over vocab_frac of the vocabulary and one
    fusion at the workload's shapes, for sequence 0; extrapolate a whole
    cycle by the layer counts.  Returns (cycles/s for the batch, detail)."""
    import numpy as np

    from block_diffusion_speculative_step_gb300 import synth
    from oracle import oracle as O

    n = synth.to_numpy
    B = w.block
    P = lens[0]

    def cfg(s):
        return O.Cfg(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, w.dtype == "bf16", w.rope_theta, w.rms_eps)

    def layer(stack, s, j):
        L = stack["layers"][j]
        return O.Layer.from_stacked(cfg(s), n(L["w_qkv"]), n(L["w_o"]), n(L["w_gu"]), n(L["w_down"]), n(L["ln1"]),
                                    n(L["ln2"]))

    rng = np.random.default_rng(0)
    times = {}
    if eng.has_target:
        tc = cfg(w.target)
        Lt = layer(eng.m["target"], w.target, 0)
        kc = eng.caches.tk[0][0].float().cpu().double().numpy()
        vc = eng.caches.tv[0][0].float().cpu().double().numpy()
        h = rng.standard_normal((B, w.target.hidden))
        t0 = time.perf_counter()
        O.decoder_layer(tc, Lt, h, P, O.CAUSAL, kc, vc)
        times["target_layer"] = time.perf_counter() - t0
    dc = cfg(w.draft)
    Ld = layer(eng.m["draft"], w.draft, 0)
    dk = eng.caches.dk[0][0].float().cpu().double().numpy()
    dv = eng.caches.dv[0][0].float().cpu().double().numpy()
    h = rng.standard_normal((B, w.draft.hidden))
    t0 = time.perf_counter()
    O.decoder_layer(dc, Ld, h, P, O.BIDIR, dk, dv, w.window)
    times["draft_layer"] = time.perf_counter() - t0
    V = max(1, int(w.vocab * vocab_frac))
    Wlm = n(eng.m["lm_head"][:V])
    x = O.rnd(dc, rng.standard_normal((B, w.draft.hidden)))
    t0 = time.perf_counter()
    O.lm_head_argmax(dc, Wlm, x)
    times["lm_head"] = (time.perf_counter() - t0) * (w.vocab / V)
    F = len(w.taps)
    feats = O.rnd(dc, rng.standard_normal((1, F * w.draft.hidden)))
    wk = [layer(eng.m["draft"], w.draft, j).wk for j in range(w.draft.layers)]
    wv = [layer(eng.m["draft"], w.draft, j).wv for j in range(w.draft.layers)]
    cap = eng.dcap
    kcs = [np.zeros((w.draft.n_kv, cap, w.draft.head_dim)) for _ in range(w.draft.layers)]
    vcs = [np.zeros((w.draft.n_kv, cap, w.draft.head_dim)) for _ in range(w.draft.layers)]
    t0 = time.perf_counter()
    O.fuse_context(dc, F, n(eng.m["fc"]), n(eng.m["fc_norm"]), feats, [P], wk, wv, kcs, vcs, w.window)
    times["fusion"] = time.perf_counter() - t0
    per_seq = (w.target.layers * times.get("target_layer", 0.0) + w.draft.layers * times["draft_layer"] +
               (2 if eng.has_target else 1) * times["lm_head"] + times["fusion"])
    return w.batch / (per_seq * w.batch), times, O.threads()


# ------------------------------------------------------------------ arms


def run_reference(args):
    """The oracle, timed on this host: each step is the bounded sample of
    oracle_sample (LM head over 1/16 of the vocabulary, scaled)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    from block_diffusion_speculative_step_gb300 import synth
    from block_diffusion_speculative_step_gb300 import build as b

    b.build()
    w = synth.WORKLOADS[args.workload]
    w1 = w if w.batch == 1 else __import__("dataclasses").replace(w, batch=1, ctx_min=0, accept_mean=0.0)
    eng, lens, _ = setup_workload(w1)
    for _ in range(args.warmup):
        oracle_sample(w1, eng, lens, 1 / 16)
    t0 = time.perf_counter()
    vals = []
    for _ in range(args.steps):
        v, times, cores = oracle_sample(w1, eng, lens, 1 / 16)
        vals.append(v)
    el = time.perf_counter() - t0
    value = args.steps / sum(1.0 / v for v in vals) * w.batch / w.batch
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "ctx": w.ctx, "block": w.block},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: 1 target layer + 1 draft layer + LM head over 1/16 of the "
                                       "vocabulary (scaled x16) + 1 fusion row, sequence 0; cycle extrapolated "
                                       "by layer counts"},
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
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    # traced replays: per-kernel CUDA-event durations inside the same graph shape
    D.dflash_trace_begin(8192)
    tgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tgraph):
        step()
    D.dflash_trace_pause()
    fam = {}
    for _ in range(max(1, args.trace_replays)):
        tgraph.replay()
        torch.cuda.synchronize()
        for name, (n, ms, by) in D.dflash_trace_read().items():
            a = fam.setdefault(name, [0, 0.0, 0.0])
            a[0] += n
            a[1] += ms
            a[2] += by
    D.dflash_trace_end()
    reps = max(1, args.trace_replays)
    launches_per_step = sum(v[0] for v in fam.values()) // reps
    del tgraph

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

    # the same cycle in sampling mode (speculative sampling at T = 1), graph replay
    sampling = None
    if eng.has_target and not args.no_sampling:
        def step_sampled():
            eng.base_pos.copy_(base0)
            eng.anchor.copy_(anchor0)
            eng.cycle_sampled(1.0, 0x5EED, 0)

        step_sampled()
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        sgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sgraph):
            step_sampled()
        for _ in range(args.warmup):
            sgraph.replay()
        n_s = max(3, min(args.steps, 50))
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_s):
            sgraph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_s = reduce_max(e0.elapsed_time(e1), world, "cuda") / n_s
        sampling = {"mode": "speculative sampling, temperature 1.0 (Philox4x32-10 draws)",
                    "ms_per_step": ms_s, "value": world * S * 1000.0 / ms_s, "unit": UNIT, "steps": n_s,
                    "overhead_vs_greedy": ms_s / ms_per_step - 1.0}
        del sgraph

        # the same with top-k 50 / top-p 0.9 filtering of the draft and target rows
        def step_filtered():
            eng.base_pos.copy_(base0)
            eng.anchor.copy_(anchor0)
            eng.cycle_sampled(1.0, 0x5EED, 0, top_k=50, top_p=0.9)

        step_filtered()
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        fgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgraph):
            step_filtered()
        for _ in range(args.warmup):
            fgraph.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_s):
            fgraph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_f = reduce_max(e0.elapsed_time(e1), world, "cuda") / n_s
        sampling["top_k50_top_p0.9_ms_per_step"] = ms_f
        del fgraph
        eng.base_pos.copy_(base0)
        eng.anchor.copy_(anchor0)

    # multi-round block denoising: the draft-block step alone at 1 and 2
    # rounds (graph replay; the state is untouched by a draft)
    denoise = None
    if not args.no_denoise:
        dms = {}
        for R in (1, 2):
            eng.draft(rounds=R)
            torch.cuda.synchronize()
            assert eng.status() == D.DFLASH_OK
            dgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(dgraph):
                eng.draft(rounds=R)
            for _ in range(args.warmup):
                dgraph.replay()
            n_d = max(3, min(args.steps, 50))
            torch.cuda.synchronize()
            e0.record()
            for _ in range(n_d):
                dgraph.replay()
            e1.record()
            torch.cuda.synchronize()
            dms[str(R)] = reduce_max(e0.elapsed_time(e1), world, "cuda") / n_d
            del dgraph
        denoise = {"mode": "draft-block step alone, graph replay", "rounds_ms": dms,
                   "unit": "ms per draft-block step", "steps": n_d}
        eng.base_pos.copy_(base0)
        eng.anchor.copy_(anchor0)

    # DFlash 2 draft convolutions (rank 64, four per draft layer): the
    # draft-block step alone with and without them (graph replay)
    conv = None
    if not args.no_conv:
        synth.add_conv_weights(eng.m, w, 64)
        if D.dflash_workspace_bytes(D.DFLASH_OP_DRAFT, eng.draft_args(conv_rank=64)) <= eng.ws_bytes:
            cms = {}
            for tag, r in (("none", 0), ("rank64", 64)):
                eng.draft(conv_rank=r)
                torch.cuda.synchronize()
                assert eng.status() == D.DFLASH_OK
                cgraph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(cgraph):
                    eng.draft(conv_rank=r)
                for _ in range(args.warmup):
                    cgraph.replay()
                n_c = max(3, min(args.steps, 50))
                torch.cuda.synchronize()
                e0.record()
                for _ in range(n_c):
                    cgraph.replay()
                e1.record()
                torch.cuda.synchronize()
                cms[tag] = reduce_max(e0.elapsed_time(e1), world, "cuda") / n_c
                del cgraph
            conv = {"mode": "draft-block step alone, graph replay", "draft_ms": cms, "steps": n_c,
                    "overhead": cms["rank64"] / cms["none"] - 1.0,
                    "params": w.draft.layers * 4 * 3 * 64 * w.draft.hidden}
        for L in eng.m["draft"]["layers"]:
            L.pop("conv_w1", None)
            L.pop("conv_w2", None)
        eng.base_pos.copy_(base0)
        eng.anchor.copy_(anchor0)

    # per-token cost: the draft-block step alone, the rest of the cycle, over
    # the tokens a cycle emits (accepted drafts + the bonus token)
    cost = None
    if denoise is not None:
        cost = cost_model(denoise["rounds_ms"]["1"], ms_per_step, mean_accept + 1.0)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h_in = torch.empty(2, S, dtype=torch.int32).pin_memory()
        h_in[0].copy_(base0.cpu())
        h_in[1].copy_(anchor0.cpu())
        h_out = torch.empty(S + S * w.block, dtype=torch.int32).pin_memory()
        e2e_steps = max(3, min(args.steps, 50))
        for _ in range(2):
            eng.base_pos.copy_(h_in[0], non_blocking=True)
            eng.anchor.copy_(h_in[1], non_blocking=True)
            eng.cycle(planted_t)
            h_out[:S].copy_(eng.accept_len, non_blocking=True)
            h_out[S:].copy_(eng.out_tokens.view(-1), non_blocking=True)
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            eng.base_pos.copy_(h_in[0], non_blocking=True)
            eng.anchor.copy_(h_in[1], non_blocking=True)
            eng.cycle(planted_t)
            h_out[:S].copy_(eng.accept_len, non_blocking=True)
            h_out[S:].copy_(eng.out_tokens.view(-1), non_blocking=True)
            torch.cuda.synchronize()
        el = reduce_max(time.perf_counter() - t0, world, "cuda")
        e2e = {"value": world * S * e2e_steps / el, "unit": UNIT, "h2d_bytes_per_step": int(h_in.numel() * 4),
               "d2h_bytes_per_step": int(h_out.numel() * 4), "steps": e2e_steps,
               "path": "eager C-ABI calls per step (no graph), pinned host inputs/outputs"}

    hbm, src = peaks()
    per_fam = {k: {"launches_per_step": v[0] // reps, "ms_per_step": v[1] / reps, "share": 0.0,
                   "gbs": (v[2] / (v[1] / 1000.0) / 1e9) if v[1] > 0 and v[2] > 0 else None}
               for k, v in fam.items() if v[0] > 0}
    tot = sum(v["ms_per_step"] for v in per_fam.values()) or 1.0
    for v in per_fam.values():
        v["share"] = v["ms_per_step"] / tot
    dom = max(per_fam, key=lambda k: per_fam[k]["ms_per_step"])
    dv = fam[dom]
    achieved = dv[2] / (dv[1] / 1000.0) / 1e9 if dv[1] > 0 else 0.0
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_source": f"{src} hbm_gbs",
                "traffic": traffic_for(dom), "bytes_per_launch": dv[2] / max(1, dv[0]),
                "avg_launch_us": 1000.0 * dv[1] / max(1, dv[0])}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, times, cores = oracle_sample(w, eng, lens, 1.0 if w.vocab < 200000 else 0.5)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "sequence 0: 1 target layer + 1 draft layer + full LM head + 1 fusion row at the "
                         "workload's shapes; cycle extrapolated by layer counts; per-unit seconds " +
                         json.dumps({k: round(t, 3) for k, t in times.items()})}

    # paged KV: the same cycle with the target and draft caches moved into
    # 128-slot page pools handed out in a shuffled order (graph replay)
    paged = None
    if not args.no_paged and eng.has_target and eng.cap % 128 == 0 and eng.dcap % 128 == 0:
        eng.page_caches(128, seed=0)
        step()
        torch.cuda.synchronize()
        assert eng.status() == D.DFLASH_OK
        same = bool(torch.equal(eng.accept_len.cpu(), accept))
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph):
            step()
        for _ in range(args.warmup):
            pgraph.replay()
        n_p = max(3, min(args.steps, 50))
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_p):
            pgraph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_p = reduce_max(e0.elapsed_time(e1), world, "cuda") / n_p
        paged = {"mode": "the same cycle on 128-slot KV pages (shuffled page order), graph replay",
                 "ms_per_step": ms_p, "value": world * S * 1000.0 / ms_p, "unit": UNIT, "steps": n_p,
                 "overhead_vs_contiguous": ms_p / ms_per_step - 1.0, "same_accept_lengths": same}
        del pgraph

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded random-init weights, N(0,1) context)",
            "config": {"workload": w.name, "batch": S, "ctx": w.ctx if not w.ctx_min else [w.ctx_min, w.ctx],
                       "block": w.block, "draft_layers": w.draft.layers,
                       "target_layers": w.target.layers if eng.has_target else 0,
                       "l2": "inputs larger than L2 (weights streamed each step)",
                       "parallelism": f"replicas x{world}", "timing": "CUDA graph replay, CUDA events"},
            "verified_tok_s": verified, "mean_accept": mean_accept,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "clocks": clocks, "step_ms_distribution": step_pct, "kernels": per_fam, "sampling": sampling,
            "denoise": denoise, "conv": conv, "paged": paged, "cost_model": cost}
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
