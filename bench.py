#!/usr/bin/env python
"""Prefill and decode throughput of the decoder forward pass on GB300.

Workload (Llama-3-8B-shaped GQA model: 32 layers, hidden 4096, 32 query / 8
kv heads, head_dim 128, FFN 14336, vocab 128256 untied, RoPE base 500000 with
llama3 scaling; seeded N(0, 0.02^2) bf16 weights, norm weights 1.0, uniform
random token ids):
  * prefill: a KV-cached session prefill of 4 sequences x 4096 tokens,
    greedy next id from the last position of each (the timed "value");
  * decode: 32 sequences prefilled to 2048 tokens once (untimed), then G
    greedy decode steps per timed step (context 2048 -> 2048 + G*(W+K)).
  * decode at batch 1 from the same context length (the per-sequence
    latency case), G greedy steps per timed step.
One step = one prefill of the 4 x 4096 batch + G decode steps at batch 32 + G
at batch 1; decode steps replay the session's captured CUDA graph. The timed
steps run inside the NVTX range "timed_steps", so a profiler can keep exactly
their launches (ncu --nvtx --nvtx-include "timed_steps/").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fk|reference]
  python bench.py --all-configs     (one JSON line per other workload, below)

``--all-configs`` times the other workloads of the parity suite through the
same public API (CUDA events, after warm-up, L2 flushed between repeats):
  A  SmolLM2-135M shape, cacheless forward of 1 x 9 ids with every hidden slot
     and all logits (latency; weight bytes / latency);
  B  op-level GEMM Y = X W^T at the five (P, in, out) shapes (TFLOP/s);
  C  SmolLM2-135M shape with KV cache: 8 x 1024 session prefill (tok/s), then
     64 greedy decode steps (tok/s);
  E  Gemma3-style tower, cacheless forward at 1, 9 and 1024 ids (latency,
     tok/s);
  M  Qwen3-30B-A3B-shaped mixture-of-experts model at full depth (48 layers,
     128 experts of width 768, 8 per token): session prefill of 4 x 4096
     (tok/s, per-kernel time, tensor-core roofline of the grouped expert
     GEMM), greedy decode at batch 32 and 1 from context 2048 (tok/s, HBM
     roofline of the step). Its weights are drawn on the device (torch's
     seeded generator, N(0, 0.02^2) bf16, unit norm weights): 61 GB that the
     host generator would take minutes to make and copy.
  python bench.py --all-configs --only M   (a subset of the workloads)

N > 1 runs N independent replicas (one per GPU, launched by torchrun); the
path has no cross-sequence exchange, so there is no data-path collective.
``--impl reference`` times the CPU oracle on the host cores instead (a bounded
sample of the same workload: one sequence of 32 ids through the full model).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "prefill tok/s & decode tok/s on 1 GB300; % of bf16 TC / HBM roofline"
WORKLOAD = "llama3-8b-shaped: session prefill 4x4096 + greedy decode batch 32 at context 2048"
PREFILL_B, PREFILL_S = 4, 4096
REF_TOKENS = 32  # the oracle's bounded sample: one sequence of 32 ids through the whole model
DECODE_B, DECODE_CTX = 32, 2048


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="fk", choices=["fk", "reference"])
    ap.add_argument("--decode-steps", type=int, default=16, help="greedy decode steps per bench step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="truncate the model to this many layers (profiling of a small case only)")
    ap.add_argument("--all-configs", action="store_true", help="time the other workloads (A, B, C, E, M)")
    ap.add_argument("--only", default="", help="with --all-configs: comma-separated subset, e.g. M")
    ap.add_argument("--no-f16", action="store_true", help="skip the f16 activation-storage timing")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def source_hash(*rel_paths) -> str:
    h = hashlib.sha256()
    for r in rel_paths:
        h.update(open(os.path.join(ROOT, r), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(f"{kernel}@{workload}")
        if e and e.get("source_hash") == source_hash(*e["sources"]):
            return e["bytes_per_launch"]
    except Exception:
        return None
    return None


def nvtx_push(name: str) -> None:
    """Open an NVTX range (a marker for profilers; no effect on the timing)."""
    import torch
    try:
        torch.cuda.nvtx.range_push(name)
    except (RuntimeError, AttributeError):
        pass


def nvtx_pop() -> None:
    import torch
    try:
        torch.cuda.nvtx.range_pop()
    except (RuntimeError, AttributeError):
        pass


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings across the process group (the
    slowest replica sets the job's time); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank: float, world: int, max_ms: float) -> float:
    """Units processed by all ranks / the slowest rank's time (weak scaling)."""
    return units_per_rank * world / (max_ms / 1e3)


def host_weights(cfg, seed: int = synth.SEED_WEIGHTS) -> dict:
    return synth.make_weights(cfg, seed=seed)


def device_weights(cfg, device, seed: int = synth.SEED_WEIGHTS, sigma: float = 0.02) -> dict:
    """Weights of cfg's shapes drawn on the device: N(0, sigma^2) bf16
    matrices from torch's generator seeded with `seed`, norm weights 1.0."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = {}
    for name, shape in synth.weight_shapes(cfg).items():
        if name == "final_norm" or name.split(".")[-1] in synth.NORM_TENSORS:
            out[name] = torch.ones(shape, dtype=torch.bfloat16, device=device)
            continue
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
        step = max(1, (1 << 26) // inner)  # bound the fp32 temporary to 256 MB
        for i in range(0, shape[0], step):
            j = min(shape[0], i + step)
            t[i:j] = (torch.randn((j - i,) + tuple(shape[1:]), generator=g, device=device) * sigma).to(torch.bfloat16)
        out[name] = t
    return out


def read_profile(lib) -> dict:
    """Kernel-class timings recorded by the library: {name: (launches, ms)};
    clears them."""
    import ctypes
    prof = {}
    for i in range(lib.fk_profile_count()):
        name = ctypes.c_char_p()
        n = ctypes.c_int64()
        ms = ctypes.c_double()
        lib.fk_profile_get(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms))
        prof[name.value.decode()] = (n.value, ms.value)
    lib.fk_profile_reset()
    return prof


def upload(wbits: dict, device) -> dict:
    import torch
    out = {}
    for k, v in wbits.items():
        out[k] = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(device, non_blocking=False)
    return out


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleFullDepth:
    """The float64 oracle's session prefill through every layer of the full
    model, on a bounded sample of the workload: 1 sequence of n_tokens ids.
    The widened weights are cached once (set-up, untimed, like loading a
    checkpoint) when the host has room for them (float64: 8 bytes per
    parameter); otherwise each timed pass widens them again."""

    def __init__(self, cfg, wbits, n_tokens: int):
        import oracle
        self.oracle = oracle
        self.cfg = cfg
        params = sum(int(v.size) for v in wbits.values())
        ram = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
        self.cached = params * 8 * 2 < ram
        self.W = oracle.OracleWeights(wbits, cache_limit_bytes=params * 8 + 1 if self.cached else 2 << 30)
        self.ids = synth.make_ids(cfg, 1, n_tokens, stream=77)
        self.n = n_tokens
        t0 = time.perf_counter()
        self.run()  # widens (and caches) the weights
        self.setup_s = time.perf_counter() - t0

    def run(self) -> float:
        t0 = time.perf_counter()
        self.oracle.Session(self.cfg, self.W, 1).prefill(self.ids)
        return time.perf_counter() - t0

    def sample(self) -> str:
        return (f"float64 oracle session prefill of 1x{self.n} ids through all {self.cfg.n_layers} layers of the "
                f"full-size model (embedding, every layer, final norm, LM head); widened weights "
                f"{'cached once (untimed)' if self.cached else 'widened per pass'}")


def bench_config(world: int, decode_steps: int) -> dict:
    return {"workload": WORKLOAD, "global_batch": PREFILL_B * world, "seq_len": PREFILL_S,
            "decode_batch": DECODE_B * world, "decode_context": DECODE_CTX, "decode_steps_per_step": decode_steps,
            "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (16 GB of weights)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = synth.CONFIGS["llama3-8b"]
    ref = OracleFullDepth(cfg, synth.make_weights(cfg), REF_TOKENS)
    for _ in range(args.warmup):
        ref.run()
    secs = [ref.run() for _ in range(args.steps)]
    value = ref.n / statistics.median(secs)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.median(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(args.gpus, args.decode_steps),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": ref.sample(), "setup_s": round(ref.setup_s, 1)},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def _time_ms(fn, reps: int, flush=None) -> float:
    """Median device time of fn over reps runs (CUDA events, L2 flushed
    between runs)."""
    import torch
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def run_moe(args, fk, dev, peaks, flush, reps, emit):
    """Workload M: the Qwen3-30B-A3B-shaped MoE model (module docstring)."""
    import torch
    lib = fk.load()
    cfg = synth.CONFIGS["qwen3-moe-30b-a3b"]
    if args.layers:
        cfg = cfg.with_(n_layers=args.layers)
    G = 8
    t0 = time.time()
    wdev = device_weights(cfg, dev)
    setup_s = time.time() - t0
    B, S = PREFILL_B, PREFILL_S
    max_pos = max(S, DECODE_CTX + G * (reps + 6) + 8)
    model = fk.Model(cfg, wdev, max_positions=max_pos)
    H, L, E, k, Ie, V = cfg.hidden, cfg.n_layers, cfg.n_experts, cfg.n_experts_per_tok, cfg.expert_intermediate, cfg.vocab
    Nq, Nkv = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    T = B * S

    # prefill
    sp = model.session(B, S, max_chunk=S)
    ids_p = torch.from_numpy(synth.make_ids(cfg, B, S, stream=10)).to(dev)
    z_p = torch.empty((B, V), dtype=torch.float32, device=dev)
    n_p = torch.empty((B,), dtype=torch.int32, device=dev)

    def prefill():
        sp.reset()
        sp.prefill(ids_p, logits=z_p, next_ids=n_p)
    for _ in range(2):
        prefill()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    ms_p = _time_ms(prefill, reps, flush)
    clk = clocks.stop()
    lib.fk_profile_reset()
    lib.fk_profile_enable(1)
    prefill()
    lib.fk_profile_enable(0)
    prof = read_profile(lib)
    del sp
    torch.cuda.empty_cache()
    # algorithmic FLOPs of the prefill's GEMMs (expert rows only, no tile padding)
    fl = {"moe_gate_up": 2.0 * T * k * H * 2 * Ie, "moe_down": 2.0 * T * k * Ie * H, "moe_router": 2.0 * T * H * E,
          "gemm_qkv": 2.0 * T * H * (Nq + 2 * Nkv), "gemm_o": 2.0 * T * Nq * H}
    gemm_flops = L * sum(fl.values()) + 2.0 * B * H * V
    top = max(("moe_gate_up", "moe_down"), key=lambda n: prof.get(n, (0, 0.0))[1])
    n_top, ms_top = prof.get(top, (0, 0.0))
    ach = fl[top] * n_top / (ms_top / 1e3) / 1e12 if ms_top > 0 else None
    tot_prof = sum(m for _, m in prof.values())

    # decode at batch 32 and 1 from context 2048
    ids_d = torch.from_numpy(synth.make_ids(cfg, DECODE_B, DECODE_CTX, stream=50)).to(dev)
    dec = {}
    for Bd in (DECODE_B, 1):
        sd = model.session(Bd, max_pos, max_chunk=1024)
        sd.prefill(ids_d[:Bd].contiguous())
        z_d = torch.empty((Bd, V), dtype=torch.float32, device=dev)
        n_d = torch.empty((Bd,), dtype=torch.int32, device=dev)
        for _ in range(2 * G):  # warm-up, graph capture
            sd.decode(None, logits=z_d, next_ids=n_d)
        torch.cuda.synchronize()
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(G):
                sd.decode(None, logits=z_d, next_ids=n_d)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / G)
        ms_tok = statistics.median(times)
        # the experts a step touches: one traced step (outside the timed region)
        n_moe = sum(cfg.moe_kinds())
        tr = torch.empty((n_moe, Bd, k), dtype=torch.int32, device=dev)
        model.set_moe_routing(None, tr, None, Bd)
        sd.decode(None, logits=z_d, next_ids=n_d)
        torch.cuda.synchronize()
        model.set_moe_routing()
        uniq = float(np.mean([len(np.unique(tr[i].cpu().numpy())) for i in range(n_moe)]))
        # per-kernel times of two steps launched one by one (outside the timed region)
        lib.fk_profile_reset()
        lib.fk_profile_enable(1)
        for _ in range(2):
            sd.decode(None, logits=z_d, next_ids=n_d)
        lib.fk_profile_enable(0)
        prof_d = read_profile(lib)
        ctx = DECODE_CTX + 2 * G + G * reps // 2
        step_bytes = (2.0 * L * (H * (Nq + 2 * Nkv) + Nq * H + E * H + uniq * 3 * H * Ie) + 2.0 * V * H
                      + 2.0 * 2 * L * Nkv * Bd * ctx)
        gbs = step_bytes / (ms_tok / 1e3) / 1e9
        dec[Bd] = {"tok_s": Bd / ms_tok * 1e3, "ms_per_token_step": ms_tok, "experts_touched_per_layer": uniq,
                   "step_bytes": step_bytes, "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm"],
                   "kernels_per_2_steps": {n: {"launches": c, "ms": round(m, 3)}
                                           for n, (c, m) in sorted(prof_d.items(), key=lambda kv: -kv[1][1])}}
        del sd
        torch.cuda.empty_cache()
    st, flags = model.sync_status()
    if st != 0:
        raise RuntimeError(f"device error word set (MoE workload): {flags:#x}")
    emit({"config": "M", "workload": f"qwen3-30b-a3b-shaped MoE ({L} layers, {E} experts x {Ie}, top-{k}): "
                                     f"session prefill {B}x{S}, greedy decode batch {DECODE_B} and 1 at context {DECODE_CTX}",
          "data": "synthetic (device-drawn seeded N(0,0.02) bf16 weights, uniform ids)",
          "prefill_tok_s": T / ms_p * 1e3, "prefill_ms": ms_p,
          "prefill_tc_frac": gemm_flops / (ms_p / 1e3) / 1e12 / peaks["bf16_sustained"],
          "roofline": {"kernel": top, "bound": "tensor", "achieved": ach, "peak": peaks["bf16_sustained"],
                       "unit": "TFLOP/s", "frac": (ach / peaks["bf16_sustained"]) if ach else None,
                       "peak_src": f"{peaks['src']} bf16 sustained",
                       "flops_per_launch": fl[top], "note": "algorithmic FLOPs of the routed rows, no tile padding"},
          "decode": {"batch": DECODE_B, **dec[DECODE_B]}, "decode_b1": {"batch": 1, **dec[1]},
          "kernels_prefill": {n: {"launches": c, "ms": round(m, 3), "share": round(m / tot_prof, 4)}
                              for n, (c, m) in sorted(prof.items(), key=lambda kv: -kv[1][1])},
          "clocks": clk, "setup_s": round(setup_s, 1)})
    del model, wdev
    torch.cuda.empty_cache()


def run_all_configs(args):
    """One JSON line per workload A, B, C, E, M (see the module docstring)."""
    import torch
    import transformer_decoder_forward_bf16_gb300 as fk
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fk.load()
    peaks = load_peaks()
    hbm, tc = peaks["hbm"], peaks["bf16"]  # launches timed alone: the burst tensor-core figure
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # larger than L2
    reps = max(5, args.steps)
    only = set(args.only.split(",")) if args.only else {"A", "B", "C", "E", "M"}

    def emit(d):
        print(json.dumps(d), flush=True)

    if "M" in only:
        run_moe(args, fk, dev, peaks, flush, reps, emit)
    if not only & {"A", "B", "C", "E"}:
        return

    def weight_bytes(wbits):
        return sum(v.nbytes for v in wbits.values())

    # A: SmolLM2-135M cacheless forward, 1 x 9, all slots and logits
    cfg = synth.CONFIGS["smollm2-135m"]
    wbits = host_weights(cfg)
    model = fk.Model(cfg, upload(wbits, dev), max_positions=1100)
    ids = synth.make_ids(cfg, 1, 9)
    for _ in range(3):
        model.forward(ids, hidden=True, logits=True, argmax=True)
    ms = _time_ms(lambda: model.forward(ids, hidden=True, logits=True, argmax=True), reps, flush)
    wb = weight_bytes(wbits) - cfg.vocab * cfg.hidden * 2 + 9 * cfg.hidden * 2  # embedding: 9 rows read
    emit({"config": "A", "workload": "smollm2-135m cacheless forward 1x9, all hidden slots + logits",
          "latency_ms": ms, "weight_gbs": wb / ms / 1e6, "hbm_frac": (wb / ms / 1e6) / hbm if hbm else None,
          "note": "includes the host-to-device copy of the 9 ids and the per-call workspace set-up"})

    # C: SmolLM2-135M with KV cache, 8 x 1024 prefill then 64 greedy steps
    B, S, G = 8, 1024, 64
    prompt = torch.from_numpy(synth.make_ids(cfg, B, S)).to(dev)
    sess = model.session(B, S + G + 1, max_chunk=1024)
    z = torch.empty((B, cfg.vocab), dtype=torch.float32, device=dev)
    nxt = torch.empty((B,), dtype=torch.int32, device=dev)

    def prefill():
        sess.reset()
        sess.prefill(prompt, logits=z, next_ids=nxt)
    for _ in range(3):
        prefill()
    ms_p = _time_ms(prefill, reps, flush)

    def decode_run():
        sess.reset()
        sess.prefill(prompt, logits=z, next_ids=nxt)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(G):
            sess.decode(None, logits=z, next_ids=nxt)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)
    decode_run()
    ms_d = statistics.median(decode_run() for _ in range(3))
    kv_bytes = 2 * cfg.n_kv_heads * cfg.head_dim * 2 * cfg.n_layers * B * (S + G / 2)
    step_bytes = wb - 9 * cfg.hidden * 2 + B * cfg.hidden * 2 + kv_bytes
    emit({"config": "C", "workload": "smollm2-135m KV cache: 8x1024 prefill + 64 greedy steps",
          "prefill_tok_s": B * S / ms_p * 1e3, "prefill_ms": ms_p,
          "decode_tok_s": B * G / ms_d * 1e3, "decode_ms_per_step": ms_d / G,
          "decode_hbm_frac": (step_bytes * G / ms_d / 1e6) / hbm if hbm else None})
    del sess, model
    torch.cuda.empty_cache()

    # B: op-level GEMMs
    rows = []
    for (P, K, N) in ((16, 64, 96), (64, 512, 256), (256, 1536, 1536), (4096, 4096, 14336), (4096, 4096, 128256)):
        x = torch.randn(P, K, device=dev).to(torch.bfloat16)
        w = (0.02 * torch.randn(N, K, device=dev)).to(torch.bfloat16)
        y = torch.empty((P, N), dtype=torch.float32, device=dev)
        for _ in range(3):
            fk.gemm(x, w, out_fp32=True, out=y)
        ms = _time_ms(lambda: fk.gemm(x, w, out_fp32=True, out=y), reps, flush)
        tf = 2.0 * P * K * N / ms / 1e9
        rows.append({"P": P, "in": K, "out": N, "ms": ms, "tflops": tf, "tc_frac": tf / tc if tc else None})
        del x, w, y
    emit({"config": "B", "workload": "op-level bf16 GEMM, fp32 out", "shapes": rows})

    # E: Gemma3-style tower, cacheless forward at 1, 9, 1024 ids
    cfg = synth.CONFIGS["gemma3-tower"]
    wbits = host_weights(cfg)
    model = fk.Model(cfg, upload(wbits, dev), max_positions=1100)
    out = {"config": "E", "workload": "gemma3-style tower cacheless forward (logits, argmax)", "prompts": []}
    for S in (1, 9, 1024):
        ids = synth.make_ids(cfg, 1, S)
        for _ in range(2):
            model.forward(ids, hidden=False, logits=True, argmax=True)
        ms = _time_ms(lambda: model.forward(ids, hidden=False, logits=True, argmax=True), reps, flush)
        out["prompts"].append({"S": S, "latency_ms": ms, "tok_s": S / ms * 1e3})
    emit(out)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.all_configs:
        run_all_configs(args)
        return
    import torch
    import torch.distributed as dist
    import transformer_decoder_forward_bf16_gb300 as fk

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = fk.load()
    peaks = load_peaks()

    cfg = synth.CONFIGS["llama3-8b"]
    if args.layers:
        cfg = cfg.with_(n_layers=args.layers)
    G = args.decode_steps
    t0 = time.time()
    wbits = host_weights(cfg)
    wdev = upload(wbits, dev)
    setup_gen_s = time.time() - t0
    k16 = max(2, min(args.steps, 5))  # timed steps of the f16-storage pass (after 2 warm-up steps)
    max_pos = max(PREFILL_S, DECODE_CTX + G * max(args.warmup + args.steps, 2 + k16) + 8)
    model = fk.Model(cfg, wdev, max_positions=max_pos)
    sp = sp0 = model.session(PREFILL_B, PREFILL_S, max_chunk=PREFILL_S)
    sd = sd0 = model.session(DECODE_B, max_pos, max_chunk=1024)
    s1 = s10 = model.session(1, max_pos, max_chunk=1024)
    ids_p = torch.from_numpy(synth.make_ids(cfg, PREFILL_B, PREFILL_S, stream=10 + rank)).to(dev)
    ids_d = torch.from_numpy(synth.make_ids(cfg, DECODE_B, DECODE_CTX, stream=50 + rank)).to(dev)
    z_p = torch.empty((PREFILL_B, cfg.vocab), dtype=torch.float32, device=dev)
    n_p = torch.empty((PREFILL_B,), dtype=torch.int32, device=dev)
    z_d = torch.empty((DECODE_B, cfg.vocab), dtype=torch.float32, device=dev)
    n_d = torch.empty((DECODE_B,), dtype=torch.int32, device=dev)
    z_1 = torch.empty((1, cfg.vocab), dtype=torch.float32, device=dev)
    n_1 = torch.empty((1,), dtype=torch.int32, device=dev)
    sd.prefill(ids_d)  # contexts for the decode batches (untimed set-up)
    s1.prefill(ids_d[:1].contiguous())
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(events=None, profile_prefill=False, sessions=None):
        sp, sd, s1 = sessions or (sp0, sd0, s10)
        sp.reset()
        if events:
            events[0].record(stream)
        if profile_prefill:
            lib.fk_profile_enable(1)
        sp.prefill(ids_p, logits=z_p, next_ids=n_p)
        if profile_prefill:
            lib.fk_profile_enable(0)
        if events:
            events[1].record(stream)
        for _ in range(G):  # greedy steps, replayed from the captured decode graph
            sd.decode(None, logits=z_d, next_ids=n_d)
        if events:
            events[2].record(stream)
        for _ in range(G):
            s1.decode(None, logits=z_1, next_ids=n_1)
        if events:
            events[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    lib.fk_profile_reset()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    nvtx_push("timed_steps")  # lets a profiler keep only the timed launches (--nvtx-include "timed_steps/")
    for k in range(args.steps):
        step(ev[k], profile_prefill=True)
    nvtx_pop()
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = start.elapsed_time(stop)
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    dec1_ms = sum(e[2].elapsed_time(e[3]) for e in ev)
    import ctypes

    def read_profile():
        prof = {}
        for i in range(lib.fk_profile_count()):
            name = ctypes.c_char_p()
            n = ctypes.c_int64()
            ms = ctypes.c_double()
            lib.fk_profile_get(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms))
            prof[name.value.decode()] = (n.value, ms.value)
        lib.fk_profile_reset()
        return prof

    prof = read_profile()
    # per-kernel decode timing: one profiled pass (launched one by one, outside the timed region)
    lib.fk_profile_enable(1)
    for _ in range(2):
        sd.decode(None, logits=z_d, next_ids=n_d)
    lib.fk_profile_enable(0)
    prof_dec = read_profile()
    lib.fk_profile_enable(1)
    for _ in range(2):
        s1.decode(None, logits=z_1, next_ids=n_1)
    lib.fk_profile_enable(0)
    prof_dec1 = read_profile()
    st, flags = model.sync_status()
    if st != 0:
        raise RuntimeError(f"device error word set: {flags:#x}")

    total_ms, pre_ms, dec_ms, dec1_ms = max_over_ranks([total_ms, pre_ms, dec_ms, dec1_ms], device=dev)
    prefill_tps = job_throughput(PREFILL_B * PREFILL_S * args.steps, world, pre_ms)
    decode_tps = job_throughput(DECODE_B * G * args.steps, world, dec_ms)
    decode1_tps = job_throughput(G * args.steps, world, dec1_ms)

    # ---- roofline of the dominant kernels (algorithmic work / device time)
    H, I, V = cfg.hidden, cfg.intermediate, cfg.vocab
    Nq, Nkv = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    T = PREFILL_B * PREFILL_S
    flops_per_launch = {"gemm_gate_up": 2.0 * T * H * 2 * I, "gemm_down": 2.0 * T * I * H,
                        "gemm_qkv": 2.0 * T * H * (Nq + 2 * Nkv), "gemm_o": 2.0 * T * Nq * H}
    pre_k = max(flops_per_launch, key=lambda k: prof.get(k, (0, 0.0))[1])
    n, ms = prof.get(pre_k, (0, 0.0))
    achieved_tf = flops_per_launch[pre_k] * n / (ms / 1e3) / 1e12 if ms > 0 else None
    peak_tf = peaks["bf16_sustained"]
    bytes_per_launch_dec = {"gemm_gate_up_dec": 2.0 * 2 * I * H, "gemm_down_dec": 2.0 * I * H,
                            "gemm_qkv_dec": 2.0 * (Nq + 2 * Nkv) * H, "gemm_o_dec": 2.0 * Nq * H}
    dec_k = max(bytes_per_launch_dec, key=lambda k: prof_dec.get(k, (0, 0.0))[1])
    n2, ms2 = prof_dec.get(dec_k, (0, 0.0))
    achieved_gbs = bytes_per_launch_dec[dec_k] * n2 / (ms2 / 1e3) / 1e9 if ms2 > 0 else None
    # whole decode step: every weight once + the KV cache read + the new K/V written
    L = cfg.n_layers
    w_bytes = 2.0 * (L * (H * (Nq + 2 * Nkv) + Nq * H + 3 * H * I) + V * H)
    ctx_mid = DECODE_CTX + G * (args.warmup + args.steps // 2)
    kv_bytes = lambda B: 2.0 * 2 * L * Nkv * B * ctx_mid + 2.0 * 2 * L * Nkv * B
    step_gbs = lambda B, ms_tot: (w_bytes + kv_bytes(B)) * G * args.steps / (ms_tot / 1e3) / 1e9
    launches = sum(c * (2 if k == "attn_decode" else 1) for k, (c, _) in prof.items())
    per_dec_step = sum(c * (2 if k == "attn_decode" else 1) for k, (c, _) in prof_dec.items()) // 2 + 1
    gpu_launches = launches + 2 * G * args.steps * per_dec_step

    line = {
        "metric": METRIC, "value": prefill_tps, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) bf16 weights, uniform ids)",
        "config": bench_config(world, G),
        "decode": {"value": decode_tps, "unit": "tok/s", "batch": DECODE_B, "ms_per_token_step": dec_ms / (G * args.steps),
                   "hbm_gbs": step_gbs(DECODE_B, dec_ms), "hbm_frac": step_gbs(DECODE_B, dec_ms) / peaks["hbm"]},
        "decode_b1": {"value": decode1_tps, "unit": "tok/s", "batch": 1, "ms_per_token_step": dec1_ms / (G * args.steps),
                      "hbm_gbs": step_gbs(1, dec1_ms), "hbm_frac": step_gbs(1, dec1_ms) / peaks["hbm"]},
        "roofline": {"kernel": pre_k, "bound": "tensor", "achieved": achieved_tf, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": (achieved_tf / peak_tf) if achieved_tf else None,
                     "peak_src": f"{peaks['src']} bf16 sustained",
                     "traffic": measured_traffic(pre_k, "llama3-8b prefill 4x4096")},
        "roofline_decode": {"kernel": dec_k, "bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm"],
                            "unit": "GB/s", "frac": (achieved_gbs / peaks["hbm"]) if achieved_gbs else None,
                            "peak_src": f"{peaks['src']} hbm", "timing": "separate profiled pass (launched one by one)",
                            "traffic": measured_traffic(dec_k, "llama3-8b decode b32")},
        "step_fraction": {"prefill_tc_frac": (2.0 * T * (H * (Nq + 2 * Nkv) + Nq * H + 3 * H * I) * cfg.n_layers
                                              / (pre_ms / args.steps / 1e3) / 1e12 / peak_tf)},
        "kernels": {k: {"launches": c, "ms": round(m, 3)} for k, (c, m) in sorted(prof.items())},
        "kernels_decode_b32_per_2_steps": {k: {"launches": c, "ms": round(m, 3)} for k, (c, m) in sorted(prof_dec.items())},
        "kernels_decode_b1_per_2_steps": {k: {"launches": c, "ms": round(m, 3)} for k, (c, m) in sorted(prof_dec1.items())},
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "setup_s": round(setup_gen_s, 1),
    }

    # ---- the same step with every activation storage site in IEEE f16
    # (fk_config.f16_sites): the mode that meets the forward-parity gates on
    # this shape; same tensor-core rate, weights read from f16 copies
    if not args.no_f16:
        m16 = fk.Model(cfg.with_(f16_sites=fk.F16_ALL), wdev, max_positions=max_pos)
        s16 = (m16.session(PREFILL_B, PREFILL_S, max_chunk=PREFILL_S), m16.session(DECODE_B, max_pos, max_chunk=1024),
               m16.session(1, max_pos, max_chunk=1024))
        s16[1].prefill(ids_d)
        s16[2].prefill(ids_d[:1].contiguous())
        for _ in range(2):
            step(sessions=s16)
        ev16 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(k16)]
        torch.cuda.synchronize()
        for k in range(k16):
            step(ev16[k], sessions=s16)
        torch.cuda.synchronize()
        p16 = sum(e[0].elapsed_time(e[1]) for e in ev16)
        d16 = sum(e[1].elapsed_time(e[2]) for e in ev16)
        d116 = sum(e[2].elapsed_time(e[3]) for e in ev16)
        p16, d16, d116 = max_over_ranks([p16, d16, d116], device=dev)
        st16, fl16 = m16.sync_status()
        if st16 != 0:
            raise RuntimeError(f"device error word set (f16 storage): {fl16:#x}")
        line["f16_storage"] = {
            "f16_sites": "all", "steps": k16,
            "prefill_tok_s": job_throughput(PREFILL_B * PREFILL_S * k16, world, p16),
            "prefill_tc_frac": (2.0 * T * (H * (Nq + 2 * Nkv) + Nq * H + 3 * H * I) * cfg.n_layers
                                / (p16 / k16 / 1e3) / 1e12 / peak_tf),
            "decode_tok_s": job_throughput(DECODE_B * G * k16, world, d16),
            "decode_hbm_frac": step_gbs(DECODE_B, d16 * args.steps / k16) / peaks["hbm"],
            "decode_b1_tok_s": job_throughput(G * k16, world, d116),
            "decode_b1_hbm_frac": step_gbs(1, d116 * args.steps / k16) / peaks["hbm"]}
        gpu_launches += (launches // max(1, args.steps) + 2 * G * per_dec_step) * k16
        line["gpu_launches"] = gpu_launches
        del s16, m16

    # ---- end to end through the public API: host ids in, host result out
    if not args.no_e2e:
        ids_host = synth.make_ids(cfg, PREFILL_B, PREFILL_S, stream=10 + rank)
        res_host = torch.empty((PREFILL_B,), dtype=torch.int32, pin_memory=True)
        zl_host = torch.empty((PREFILL_B, V), dtype=torch.float32, pin_memory=True)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ke = max(1, min(3, args.steps))
        e0.record(stream)
        for _ in range(ke):
            sp.reset()
            sp.prefill(ids_host, logits=z_p, next_ids=n_p)  # host ids: copied in by the call
            res_host.copy_(n_p, non_blocking=True)
            zl_host.copy_(z_p, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / ke
        line["e2e"] = {"value": world * PREFILL_B * PREFILL_S / (e2e_ms / 1e3), "unit": "tok/s",
                       "h2d_bytes_per_step": int(ids_host.nbytes),
                       "d2h_bytes_per_step": int(res_host.numel() * 4 + zl_host.numel() * 4)}

    # ---- CPU oracle on the host cores (rank 0, N = 1 only)
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        ref = OracleFullDepth(cfg, wbits, REF_TOKENS)
        secs = [ref.run() for _ in range(2)]
        line["cpu_baseline"] = {"value": ref.n / min(secs), "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": ref.sample(), "seconds": round(sum(secs), 1),
                                "setup_s": round(ref.setup_s, 1)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
