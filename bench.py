#!/usr/bin/env python
"""Benchmark of the DFlash draft cycle on GB300: drafted tokens/s and cycle latency.

One step = one whole draft cycle on device-resident inputs: inject the
previous cycle's tau committed tokens (context fusion + K/V injection into
every draft layer) and draft a block (non-causal drafter pass + shared LM head
argmax) — one dflash_draft_cycle call, one persistent launch at small batch —
let the synthetic target answer (seeded agreement pattern), verify greedily.  value = drafted tokens/s = batch * (block - 1) / cycle time, summed
over ranks (weak scaling: each rank drafts for its own requests; requests are
independent, so there is no collective on the data path).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 8b_bs1]
    python bench.py --impl reference ...     # the CPU oracle on the host cores
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from dflash_inputs import (make_agreement, make_features, make_tokens, make_weights, seed_for,  # noqa: E402
                           synthetic_target_argmax, workloads)

METRIC = "drafted tokens/s & draft-cycle latency at bs1/bs32; % of HBM or TC roofline"
UNIT = "drafted tokens/s"
GEMM_STAGES = ("fuse", "inject", "qkv", "o", "gateup", "down", "lmhead")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="dflash", choices=["dflash", "reference"])
    ap.add_argument("--workload", default="8b_bs1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-bs32", action="store_true", help="skip the batch-32 sub-record of the default run")
    ap.add_argument("--only", choices=["verify_sampled", "packed_attention"],
                    help="run and print only this sub-benchmark (1 GPU)")
    ap.add_argument("--kv-bf16", action="store_true",
                    help="the context cache keeps one bf16 per value (else a hi and a lo bf16 plane)")
    ap.add_argument("--head-bf16", action="store_true",
                    help="the LM head reads the final normed state as one bf16 (multi-kernel path)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------- multi-rank aggregation
def max_over_ranks(value: float, device="cpu") -> float:
    """The largest `value` over all ranks (the slowest rank's time); the value
    itself when there is one rank."""
    dist = torch.distributed
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor([float(value)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return float(value)


def job_throughput(ms_per_step_max: float, drafted_per_rank_step: int, world: int) -> float:
    """Whole-job drafted tokens/s: every rank drafts for its own requests each
    step; the job's step takes as long as its slowest rank."""
    return world * drafted_per_rank_step / (ms_per_step_max / 1e3)


# ---------------------------------------------------------------- clocks
class Clocks:
    """nvidia-smi sampler running while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- algorithmic bytes
def gemm_bytes_per_cycle(cfg, B: int, block: int, inject_rows: int) -> dict:
    """Algorithmic DRAM bytes of each GEMM stage in one cycle: every weight
    byte once, activations in (4 bytes a value: fp32, or a bf16 hi/lo pair),
    outputs out (fp32; the residual stream is read and written)."""
    es, ea = cfg.elem_bytes, 4
    D, L, m = cfg.hidden, cfg.layers, cfg.n_target_feats
    hq, hk, F, V = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.ffn, cfg.vocab
    R, Rm, n = B * block, B * (block - 1), inject_rows
    return {
        "fuse": es * D * m * D + es * n * m * D + 4 * n * D,
        "inject": es * L * 2 * hk * D + ea * n * D + 4 * n * L * 2 * hk,
        "qkv": L * (es * (hq + 2 * hk) * D + ea * R * D + 4 * R * (hq + 2 * hk)),
        "o": L * (es * D * hq + ea * R * hq + 8 * R * D),
        "gateup": L * (es * 2 * F * D + ea * R * D + ea * R * F),
        "down": L * (es * D * F + ea * R * F + 8 * R * D),
        "lmhead": es * V * D + ea * Rm * D + 8 * Rm,
    }


def gemm_flops_per_cycle(cfg, B: int, block: int, inject_rows: int) -> dict:
    """Algorithmic FLOPs (2 per multiply-add) of each GEMM stage in one cycle.
    A hi/lo activation pair makes the tensor cores run twice this."""
    D, L, m = cfg.hidden, cfg.layers, cfg.n_target_feats
    hq, hk, F, V = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.ffn, cfg.vocab
    R, Rm, n = B * block, B * (block - 1), inject_rows
    return {
        "fuse": 2 * n * m * D * D,
        "inject": 2 * n * D * L * 2 * hk,
        "qkv": L * 2 * R * D * (hq + 2 * hk),
        "o": L * 2 * R * hq * D,
        "gateup": L * 2 * R * D * 2 * F,
        "down": L * 2 * R * F * D,
        "lmhead": 2 * Rm * D * V,
    }


# ---------------------------------------------------------------- measured DRAM traffic
# Committed ncu summaries of the dominant kernel's DRAM traffic; each is valid
# only for the workload and the kernel sources it was taken on.
TRAFFIC_PROFILES = {
    "gemm": (os.path.join(ROOT, "profiles", "gemm_traffic_8b_bs1.md"),
             ["gemm_tc.cu", "epilogue.cuh", "common.cuh", "ptx.cuh"]),
    "persist": (os.path.join(ROOT, "profiles", "persist_traffic_8b_bs1.md"),
                ["persist.cu", "persist.cuh", "attn_tc.cuh", "epilogue.cuh", "common.cuh", "ptx.cuh"]),
}


def source_sha1(names) -> str:
    import hashlib
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(ROOT, "block_diffusion_drafter_dflash_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kind: str, workload: str):
    """DRAM bytes (read + write) per cycle of the kernel(s) `kind` from the
    committed ncu summary, or None when it was taken on other sources or
    another workload."""
    path, sources = TRAFFIC_PROFILES[kind]
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = dict(line.split(":", 1) for line in text.splitlines() if ":" in line and line[:1].isalpha())
    try:
        if vals.get("workload", "").strip() != workload or vals.get("source_sha1", "").strip() != source_sha1(sources):
            return None
        return int(vals["traffic_bytes_per_cycle"].strip())
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- the GPU arm
class Cycle:
    """Device-resident draft cycle of one workload through the C ABI.

    Every per-cycle input lives on the device: the target features of the
    committed tokens, and a stack of seeded agreement patterns indexed by a
    device-side counter, so that one cycle can be captured in a CUDA graph and
    replayed."""

    def __init__(self, wl, total_cycles: int, rank: int):
        import block_diffusion_drafter_dflash_gb300 as df
        self.df = df
        self.wl, cfg = wl, wl.cfg
        self.cfg = cfg
        B, block = wl.batch, wl.block
        self.B, self.block = B, block
        seed = wl.seed + 100000 * rank
        self.weights = make_weights(cfg, seed, device="cuda")
        self.model = df.Model(cfg, self.weights)
        self.cap = max(wl.ctx) + block * (total_cycles + 2)
        self.cache = df.Cache(self.model, B, self.cap)
        self.rows = B * block
        setup_chunk = min(sum(wl.ctx), 16384)
        self.ws = df.dflash_workspace(self.model, B, self.cap, block, max(self.rows, setup_chunk))
        # setup injection of each request's context, in chunks of at most setup_chunk rows
        for b, c in enumerate(wl.ctx):
            for s in range(0, c, setup_chunk):
                n = min(setup_chunk, c - s)
                counts = [0] * B
                counts[b] = n
                f = make_features(cfg, n, seed=seed + 17 * b + s, device="cuda")
                df.dflash_inject_context(self.model, self.cache, f, torch.tensor(counts, dtype=torch.int32,
                                                                                 device="cuda"), counts, n, self.ws)
        torch.cuda.synchronize()
        self.feats = make_features(cfg, self.rows, seed=seed + 999, device="cuda")
        P = 16
        pats = [make_agreement(cfg, B, block, wl.accept_p, seed=seed_for(wl, i, 5) + rank, device="cuda")
                for i in range(P)]
        self.match = torch.stack([p.match for p in pats]).contiguous()
        self.off = torch.stack([p.off for p in pats]).contiguous()
        self.bonus = torch.stack([p.bonus for p in pats]).contiguous()
        self.P = P
        self.pidx = torch.zeros(1, dtype=torch.long, device="cuda")
        self.tau = torch.full((B,), wl.first_inject, dtype=torch.int32, device="cuda")
        self.tau_acc = torch.zeros(1, dtype=torch.long, device="cuda")
        self.anchor = make_tokens(cfg, B, seed=seed + 3, device="cuda")
        self.drafts = torch.empty((B, block - 1), dtype=torch.int32, device="cuda")
        self.y = torch.empty((B, block), dtype=torch.int32, device="cuda")
        self.out = torch.empty((B, block), dtype=torch.int32, device="cuda")
        self.next_anchor = self.anchor            # verification writes the next anchor in place
        self.graph = None

    def step(self):
        df = self.df
        # inject the previous cycle's tau committed tokens, then draft: one
        # persistent launch when both fit it, else the two calls in turn
        df.dflash_draft_cycle(self.model, self.cache, self.feats, self.tau, self.anchor, self.block, self.drafts,
                              None, max_rows=self.rows, workspace=self.ws)
        # the (synthetic) target's greedy tokens for this block; also adds the
        # previous cycle's accepted lengths to tau_acc
        df.dflash_synthetic_target(self.drafts, self.match, self.off, self.bonus, self.pidx, self.y,
                                   self.cfg.vocab, tau=self.tau, tau_sum=self.tau_acc)
        df.dflash_verify_greedy(self.drafts, self.y, self.tau, self.out, self.anchor)

    def capture(self):
        """Capture one cycle in a CUDA graph (after eager warm-up)."""
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        torch.cuda.synchronize()
        self.graph = g

    def replay(self):
        self.graph.replay()


def method_bytes(wl, inject_rows: int) -> dict:
    """Algorithmic DRAM bytes of one cycle as the method defines them: every
    weight matrix read once (W_K/W_V count once: injection and drafter use the
    same matrices), the context K/V of bf16 models at 2 bytes a value (20,480 B
    per token at the 8B shape), the new tokens' target features."""
    c = wl.cfg
    es = c.elem_bytes
    D, m, L = c.hidden, c.n_target_feats, c.layers
    layers = es * L * c.layer_matrix_params()
    lm = es * c.vocab * D
    wc = es * D * m * D
    kv = 2 * L * c.n_kv_heads * c.head_dim * es * sum(wl.ctx)
    feats = es * inject_rows * m * D
    return {"layers": layers, "lm_head": lm, "w_c": wc, "kv": kv, "features": feats,
            "drafter": layers + lm + kv, "cycle": layers + lm + wc + kv + feats}


def kv_storage_bytes(wl) -> int:
    """Context K/V the attention reads as stored: 4 bytes a value (fp32, or the
    hi and lo bf16 planes of bf16 models), 2 with a one-plane bf16 cache."""
    c = wl.cfg
    per = 2 if getattr(c, "kv_bf16", False) else 4
    return 2 * c.layers * c.n_kv_heads * c.head_dim * per * sum(wl.ctx)


def kv_weight_bytes(cfg) -> int:
    """Bytes of every layer's W_K and W_V (the injection's projection)."""
    return cfg.elem_bytes * cfg.layers * 2 * cfg.n_kv_heads * cfg.head_dim * cfg.hidden


def check_outputs(cyc) -> None:
    """The timed cycle's results are valid: drafts are token ids, 1 <= tau <= block."""
    d, t = cyc.drafts, cyc.tau
    V, g = cyc.cfg.vocab, cyc.block
    ok = bool(((d >= 0) & (d < V)).all().item()) and bool(((t >= 1) & (t <= g)).all().item())
    if not ok:
        raise RuntimeError("timed cycle produced invalid drafts or accepted lengths")


def measure(wl, W, K, rank, world, local, barrier, want_e2e=True):
    """Time whole cycles of workload `wl` (graph replay), then one profiled
    eager pass; returns the bench record of that workload and the Cycle."""
    import block_diffusion_drafter_dflash_gb300 as df
    total = W + 2 * K + 40
    cyc = Cycle(wl, total, rank)
    for _ in range(W):
        cyc.step()
    n0 = df.dflash_launch_count()
    cyc.capture()                                 # one cycle as a CUDA graph
    launches_per_cycle = df.dflash_launch_count() - n0
    for _ in range(2):
        cyc.replay()
    barrier()
    clocks = Clocks(local)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cyc.tau_acc.zero_()
    barrier()
    t0.record()
    for _ in range(K):
        cyc.replay()
    t1.record()
    barrier()
    launches = launches_per_cycle * K
    clk = clocks.stop()
    check_outputs(cyc)
    ms = max_over_ranks(t0.elapsed_time(t1) / K, "cuda")
    mean_tau = float(cyc.tau_acc.item()) / (K * wl.batch)
    drafted = wl.batch * (wl.block - 1)
    value = job_throughput(ms, drafted, world)

    # profiled pass (eager launches): CUDA events around each launch, per stage
    KP = min(K, 20)
    df.dflash_profile_start(cyc.model, 100 * KP)
    for _ in range(KP):
        cyc.step()
    prof = df.dflash_profile_stop(cyc.model)
    # the synthetic target (a stand-in for the target model, not part of the
    # method) timed on its own
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(KP):
        df.dflash_synthetic_target(cyc.drafts, cyc.match, cyc.off, cyc.bonus, cyc.pidx, cyc.y, cyc.cfg.vocab)
    ev1.record()
    torch.cuda.synchronize()
    target_ms = ev0.elapsed_time(ev1) / KP
    gb = gemm_bytes_per_cycle(wl.cfg, wl.batch, wl.block, cyc.rows)
    gf = gemm_flops_per_cycle(wl.cfg, wl.batch, wl.block, cyc.rows)
    mb = method_bytes(wl, int(round(mean_tau * wl.batch)))
    hbm, bf16, bf16_sus, src = load_peaks()
    extra = {}
    if prof["cycle_persist"][1] > 0:
        # one persistent launch runs the whole cycle up to the drafts: context
        # fusion, every layer (Q/K/V also projecting the injected rows' K/V),
        # attention over the context, the LM head
        kern_bytes = mb["cycle"]
        stored = sum(gb.values()) - gb["inject"] + kv_storage_bytes(wl)
        kern_ms = prof["cycle_persist"][0] / KP
        kern = "persist_kernel, injection + drafter pass (one launch a cycle)"
        traffic = measured_traffic("persist", wl.name)
    elif prof["draft_persist"][1] > 0:
        # one persistent launch runs the whole drafter pass: every layer's
        # projections and attention (context K/V read) and the LM head
        kern_bytes = mb["drafter"]
        stored = sum(gb[k] for k in ("qkv", "o", "gateup", "down", "lmhead")) + kv_storage_bytes(wl)
        kern_ms = prof["draft_persist"][0] / KP
        kern = "persist_kernel, drafter pass (one launch a cycle)"
        traffic = measured_traffic("persist", wl.name)
        if prof["inject_persist"][1] > 0:
            inj_bytes, inj_ms = mb["w_c"] + kv_weight_bytes(wl.cfg), prof["inject_persist"][0] / KP
            extra = {"injection_kernel_GBps": round(inj_bytes / (inj_ms / 1e3) / 1e9, 1),
                     "injection_kernel_ms_per_cycle": round(inj_ms, 4)}
    else:
        kern_bytes = sum(gb.values())
        stored = kern_bytes
        kern_ms = sum(prof[s][0] for s in GEMM_STAGES) / KP
        kern = "projection GEMMs (all launches of one cycle)"
        traffic = measured_traffic("gemm", wl.name)
    persistent = prof["draft_persist"][1] > 0 or prof["cycle_persist"][1] > 0
    kern_flops = sum(gf[k] for k in GEMM_STAGES) if not persistent else 0
    if kern_flops / (bf16_sus * 1e12) > kern_bytes / (hbm * 1e9):
        # many token rows: the projections are bound by the tensor cores; they
        # run back to back inside a long cycle, so the sustained peak applies
        achieved = kern_flops / (kern_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_sus, "unit": "TFLOP/s",
                    "frac": round(achieved / bf16_sus, 4), "traffic": traffic, "kernel": kern,
                    "peak_source": f"{src} (sustained bf16)", "algorithmic_flops_per_cycle": kern_flops,
                    # operands carried as hi/lo bf16 pairs run twice (the fusion's are exact bf16)
                    "tensor_pipe_flops_per_cycle": gf["fuse"] + 2 * (kern_flops - gf["fuse"]),
                    "algorithmic_bytes_per_cycle": kern_bytes, "kernel_ms_per_cycle": round(kern_ms, 4),
                    "hbm_GBps": round(kern_bytes / (kern_ms / 1e3) / 1e9, 1), **extra}
    else:
        achieved = kern_bytes / (kern_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4), "traffic": traffic, "kernel": kern, "peak_source": src,
                    "algorithmic_bytes_per_cycle": kern_bytes,
                    "stored_bytes_per_cycle": stored,
                    "frac_of_stored_bytes": round(stored / (kern_ms / 1e3) / 1e9 / hbm, 4),
                    "kernel_ms_per_cycle": round(kern_ms, 4), **extra}
    stages = {s: {"ms_per_cycle": round(v[0] / KP, 4), "launches_per_cycle": v[1] / KP} for s, v in prof.items()
              if v[1] > 0}
    cycle_roof_ms = mb["cycle"] / (hbm * 1e9) * 1e3

    e2e = run_e2e(cyc, K, wl, barrier, world) if want_e2e else None
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.cfg.dtype, "data": "synthetic (seeded N(0,0.02) weights, N(0,1) target features, "
                                       "seeded target agreement)",
        "config": {"workload": wl.name, "drafter": wl.cfg.name, "batch_per_gpu": wl.batch, "block": wl.block,
                   "ctx": wl.ctx if len(wl.ctx) <= 4 else f"{min(wl.ctx)}..{max(wl.ctx)} ({len(wl.ctx)} requests)",
                   "kv_cache": ("one bf16 per value" if getattr(wl.cfg, "kv_bf16", False)
                                else "hi and lo bf16 planes per value (fp32-level)"),
                   "lm_head_input": ("one bf16" if getattr(wl.cfg, "head_bf16", False)
                                     else "hi and lo bf16 planes"),
                   "l2": "inputs larger than L2 (weights streamed every cycle)",
                   "timing": "CUDA-graph replay of whole cycles (inject, draft, synthetic target, verify); "
                             "per-stage times from an eager pass with events",
                   "synthetic_target_ms_per_cycle": round(target_ms, 4),
                   "ms_per_cycle_without_synthetic_target": round(ms - target_ms, 4),
                   "mean_tau": round(mean_tau, 3),
                   "accepted_tokens_per_s": round(world * mean_tau * wl.batch / (ms / 1e3), 1),
                   "method_bytes_per_cycle": mb["cycle"],
                   "cycle_roofline_ms": round(cycle_roof_ms, 4),
                   "cycle_frac_of_hbm_roofline": round(cycle_roof_ms / ms, 4)},
        "roofline": roofline, "stages": stages, "gpu_launches": int(launches), "clocks": clk, "e2e": e2e,
    }
    return result, cyc


def measure_sampled_verify(K: int, W: int = 3, B: int = 32, g: int = 16, V: int = 151936) -> dict:
    """dflash_verify_sampled at the 8B shape's vocabulary and batch 32: the
    drafter's and the target's fp32 logits (603 MB, larger than L2) are read
    once for the rows' normalisers, then one or two rows per request again.
    Algorithmic bytes: the logits once."""
    import block_diffusion_drafter_dflash_gb300 as df
    gen = torch.Generator(device="cuda").manual_seed(77)
    tl = 2.0 * torch.randn((B, g, V), generator=gen, device="cuda")
    dl = (tl[:, :g - 1] + 0.5 * torch.randn((B, g - 1, V), generator=gen, device="cuda")).contiguous()
    u_d = torch.rand((B, g - 1), generator=gen, device="cuda")
    drafts = torch.empty((B, g - 1), dtype=torch.int32, device="cuda")
    df.dflash_sample_tokens(dl, 1.0, u_d, drafts)
    ua = torch.rand((B, g - 1), generator=gen, device="cuda")
    us = torch.rand((B,), generator=gen, device="cuda")
    tau = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, g), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = df.dflash_sampling_workspace(B * (2 * g - 1), B, V)
    for _ in range(W):
        df.dflash_verify_sampled(dl, tl, drafts, ua, us, 1.0, tau, out, nxt, ws)
    torch.cuda.synchronize()
    n0 = df.dflash_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        df.dflash_verify_sampled(dl, tl, drafts, ua, us, 1.0, tau, out, nxt, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    launches = (df.dflash_launch_count() - n0) // K
    nbytes = B * (2 * g - 1) * V * 4
    hbm, _, _, src = load_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    ok = bool(((tau >= 1) & (tau <= g)).all().item())
    return {"shape": f"batch {B}, block {g}, vocab {V}, temperature 1", "ms_per_call": round(ms, 4),
            "launches_per_call": int(launches), "algorithmic_bytes": nbytes, "achieved_GBps": round(gbs, 1),
            "peak_GBps": hbm, "frac": round(gbs / hbm, 4), "peak_source": src, "outputs_valid": ok,
            "mean_tau": round(float(tau.float().mean().item()), 3)}


def measure_packed_attention(K: int, W: int = 3) -> dict:
    """dflash_packed_block_attention at the training shape of paper §7.1: a
    3072-token sequence, 512 anchor blocks of 16, 32 q / 8 kv heads of 128,
    bf16 inputs.  Tensor-bound: algorithmic flops = 4 * nq * block * hd *
    sum_n (a_n + block) (Q K^T and P V over each block's visible keys)."""
    import numpy as np
    import block_diffusion_drafter_dflash_gb300 as df
    S, N, g, nq, nkv, hd = 3072, 512, 16, 32, 8, 128
    rng = np.random.default_rng(7)
    anchors = sorted(int(a) for a in rng.choice(np.arange(1, S - g), size=N, replace=False))
    gen = torch.Generator(device="cuda").manual_seed(71)
    r = lambda *shape: torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    q, kc, vc, kb, vb = r(N, g, nq, hd), r(S, nkv, hd), r(S, nkv, hd), r(N, g, nkv, hd), r(N, g, nkv, hd)
    out = torch.empty((N, g, nq, hd), device="cuda")
    ws = df.dflash_packed_attention_workspace(N, g, S, nq, nkv, hd)
    a_dev = torch.tensor(anchors, dtype=torch.int32, device="cuda")
    for _ in range(W):
        df.dflash_packed_block_attention(q, kc, vc, kb, vb, a_dev, out, ws)
    torch.cuda.synchronize()
    n0 = df.dflash_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        df.dflash_packed_block_attention(q, kc, vc, kb, vb, a_dev, out, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    flops = 4 * nq * g * hd * sum(a + g for a in anchors)
    _, _, bf16_sus, src = load_peaks()
    tf = flops / (ms / 1e3) / 1e12
    return {"shape": f"sequence {S}, {N} anchor blocks of {g}, {nq} q / {nkv} kv heads of {hd}, bf16",
            "ms_per_call": round(ms, 4), "launches_per_call": int((df.dflash_launch_count() - n0) // K),
            "algorithmic_flops": flops, "achieved_TFLOPs": round(tf, 2), "peak_TFLOPs": bf16_sus,
            "frac": round(tf / bf16_sus, 4), "peak_source": f"{src} (sustained bf16)",
            "status": df.dflash_packed_attention_status(ws), "finite": bool(torch.isfinite(out).all().item())}


def workload_for(args, name: str):
    """The named workload, with the one-bf16 options of --kv-bf16 / --head-bf16."""
    wl = workloads()[name]
    opts = {k: True for k in ("kv_bf16", "head_bf16") if getattr(args, k, False)}
    if opts:
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, **opts))
    return wl


def run_gpu(args, rank, world, local):
    torch.cuda.set_device(local)
    wl = workload_for(args, args.workload)
    dist = world > 1 and torch.distributed.is_initialized()

    def barrier():
        if dist:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    result, cyc = measure(wl, args.warmup, args.steps, rank, world, local, barrier, not args.no_e2e)
    if args.workload == "8b_bs1" and not args.no_bs32:
        # the metric's batch-32 half in the same run: the 8B-shaped drafter on
        # 32 requests of ragged context (fewer cycles: each is ~4 ms)
        result["_weights"] = cyc.weights
        cyc = None
        torch.cuda.empty_cache()
        r32, c32 = measure(workload_for(args, "8b_bs32"), 3, min(args.steps, 20), rank, world, local, barrier,
                           False)
        del c32
        torch.cuda.empty_cache()
        result["bs32"] = {k: r32[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "config",
                                               "roofline", "stages", "gpu_launches", "clocks")}
        torch.cuda.empty_cache()
        # the same batch-32 cycle with the bf16 storage options (one-bf16 cache
        # and LM-head input: the precision the method itself states)
        opts = argparse.Namespace(kv_bf16=True, head_bf16=True)
        r32b, c32b = measure(workload_for(opts, "8b_bs32"), 3, min(args.steps, 20), rank, world, local, barrier, False)
        del c32b
        result["bs32_bf16_storage"] = {k: r32b[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "config",
                                                             "roofline", "stages", "gpu_launches", "clocks")}
        torch.cuda.empty_cache()
        result["verify_sampled"] = measure_sampled_verify(min(args.steps, 50))
        torch.cuda.empty_cache()
        result["packed_attention"] = measure_packed_attention(min(args.steps, 20))
    return result, cyc


def run_e2e(cyc, K, wl, barrier, world):
    """Same cycle through the public API (graph replay of the C-ABI calls) with
    the step's inputs — target features of the committed tokens and the
    target's agreement pattern — copied from pinned host memory, and its
    results (drafts, tau, emitted tokens, next anchor) read back, every step."""
    feats_h = cyc.feats.cpu().pin_memory()
    pats_h = [(cyc.match[i].cpu().pin_memory(), cyc.off[i].cpu().pin_memory(), cyc.bonus[i].cpu().pin_memory())
              for i in range(cyc.P)]
    outs = (cyc.drafts, cyc.tau, cyc.out, cyc.next_anchor)
    out_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = feats_h.numel() * feats_h.element_size() + sum(t.numel() * t.element_size() for t in pats_h[0])
    d2h = sum(t.numel() * t.element_size() for t in out_h)
    cyc.pidx.zero_()
    barrier()
    t0 = time.perf_counter()
    for i in range(K):
        slot = i % cyc.P
        cyc.feats.copy_(feats_h, non_blocking=True)
        m, o, b = pats_h[slot]
        cyc.match[slot].copy_(m, non_blocking=True)
        cyc.off[slot].copy_(o, non_blocking=True)
        cyc.bonus[slot].copy_(b, non_blocking=True)
        cyc.replay()
        for h, d in zip(out_h, outs):
            h.copy_(d, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    barrier()
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / K, "cuda")
    return {"value": round(job_throughput(ms, wl.batch * (wl.block - 1), world), 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ---------------------------------------------------------------- the oracle (CPU)
def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


class OracleCycle:
    """The CPU oracle on one request of the workload (context injected once,
    then whole cycles: inject tau tokens, draft, argmax, verify)."""

    def __init__(self, wl, weights_gpu=None):
        import oracle
        self.o = oracle
        self.wl, self.cfg = wl, wl.cfg
        w = weights_gpu if weights_gpu is not None else make_weights(wl.cfg, wl.seed, device="cuda")
        self.hw = oracle.weights_to_host(w)
        self.cache = oracle.RequestCache(self.cfg.layers, self.cfg.n_kv_heads, self.cfg.head_dim)
        ctx = wl.ctx[0]
        feats = make_features(self.cfg, ctx, seed=wl.seed + 17, device="cuda").cpu()
        for s in range(0, ctx, 4096):
            oracle.inject_context(self.hw, self.cfg, self.cache, feats[s:s + 4096])
        self.tau = wl.first_inject
        self.anchor = int(make_tokens(self.cfg, 1, seed=wl.seed + 3).item())
        self.new = make_features(self.cfg, wl.block, seed=wl.seed + 999).cpu()
        self.i = 0

    def step(self):
        o, wl = self.o, self.wl
        r = o.draft_cycle(self.hw, self.cfg, self.cache, self.new[:self.tau], self.anchor, wl.block)
        pat = make_agreement(self.cfg, 1, wl.block, wl.accept_p[:1], seed=seed_for(wl, self.i, 5))
        y = synthetic_target_argmax(torch.tensor(r["drafts"], dtype=torch.int32).reshape(1, -1), pat, self.cfg.vocab)
        tau, _, nxt = o.verify_greedy(r["drafts"], y[0].tolist())
        self.tau, self.anchor = tau, nxt
        self.i += 1


def cpu_baseline(wl, weights_gpu=None, budget_s: float = 25.0):
    oc = OracleCycle(wl, weights_gpu)
    t0 = time.perf_counter()
    n = 0
    while True:
        oc.step()
        n += 1
        if time.perf_counter() - t0 > budget_s * 0.5 or n >= 3:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": round((wl.block - 1) / dt, 4), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
            "sample": f"{n} whole cycle(s) of request 0 of workload {wl.name} (context {wl.ctx[0]} injected "
                      f"beforehand, untimed); float64 numpy, BLAS threads on all cores", "s_per_cycle": round(dt, 3)}


def run_reference(args, rank, world, local):
    if rank != 0:
        return None
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    wl = workloads()[args.workload]
    oc = OracleCycle(wl, None)
    for _ in range(args.warmup):
        oc.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oc.step()
    dt = (time.perf_counter() - t0) / args.steps
    value = (wl.block - 1) / dt
    sample = (f"each step one whole cycle of request 0 of workload {wl.name} "
              f"({'all' if wl.batch == 1 else f'1 of {wl.batch}'} requests)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "drafter": wl.cfg.name, "batch_per_gpu": wl.batch, "block": wl.block},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if args.impl == "dflash" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    if args.only:
        torch.cuda.set_device(local)
        if rank == 0:
            fn = measure_sampled_verify if args.only == "verify_sampled" else measure_packed_attention
            print(json.dumps({"only": args.only, **fn(args.steps, max(args.warmup, 1))}), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world, local)
    else:
        res, cyc = run_gpu(args, rank, world, local)
        weights = res.pop("_weights", None)
        if weights is None and cyc is not None:
            weights = cyc.weights
        if rank == 0 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(workloads()[args.workload], weights)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
