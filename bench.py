#!/usr/bin/env python3
"""Benchmark of the GQA decode step on GB300: decode-attention HBM GB/s and decode
steps/sec at 1 GPU (N replicas under torchrun).

Headline workload: the Llama-3.1-8B-like decode, 16 sequences at 8192 cached
tokens, 32 q / 8 kv heads, head_dim 128, bf16 cache, NeoX RoPE with llama3
factor 8. One benchmark step = 64 consecutive decode steps from 8192 cached
tokens (each: RoPE/append + split-K partials in one kernel, combine), after which the lengths
return to 8192 (a 64-byte device copy) so every step times the same work. The
64 decode steps are captured once in a CUDA graph and replayed. The KV cache
(~545 MB) is larger than L2 (129 MB), so no flush is needed between steps.

The same JSON line carries `per_config`: the other four workloads of the
suite (tiny Llama-3.2-1B-like fp32 step, warm and with L2 flushed between steps;
Qwen3-8B-like ragged; Gemma-2-9B-like windowed + global; gpt-oss-like vq8 with
sinks), each measured the same way at the same --steps / --warmup, with its own
roofline, end-to-end figure, clocks and oracle baseline, and the 512-token
prefill chunk per sequence on the headline's cache (query-tiled tcgen05
kernel; roofline in TFLOP/s against the measured bf16 tensor peak; no oracle
baseline).

value       = algorithmic bytes of all timed steps / device time (CUDA events)
e2e         = the same bytes / time of K x 64 calls of DecodeLayer.step, each with
              the step's q/k/v copied from pinned host memory and out copied back
              (double-buffered, copies on a second stream overlapping the kernels)
roofline    = the split-K partial kernel alone (for bf16 / vq8 / q8 caches the kernel
              that also performs the append): its algorithmic bytes (visible KV
              rows) / its mean launch duration, against the measured HBM copy peak
              (frac) and the 8 TB/s nominal HBM3e figure (frac_of_nominal)
cpu_baseline / --impl reference = the fp64 CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import shutil
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_attention_kv_qk_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attention HBM GB/s (% of GB300 peak) and decode steps/sec at 1 GPU"
DECODES_PER_STEP = {"llama31_8b_decode": 64, "llama31_8b_q8": 64, "llama31_8b_paged": 64, "llama31_8b_verify": 16,
                    "llama32_1b_tiny": 64}
HEADLINE = "llama31_8b_decode"
# the suite's other workloads, reported beside the headline in the same line
PER_CONFIG = ("llama32_1b_tiny", "qwen3_8b_ragged", "gemma2_9b_swa", "gptoss_vq8_sink", "llama31_8b_prefill")
# the oracle takes tens of seconds per sequence of a 512-token chunk: no CPU baseline in per_config
NO_CPU_IN_PER_CONFIG = ("llama31_8b_prefill",)
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal
L2_BYTES = 129 * 2**20


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def measured_traffic(workload: str):
    """DRAM bytes per launch of the partial kernel from one ncu capture
    (profiles/traffic.json, written beside the capture's summary), or None when
    there is none or when the kernel's sources changed since the counters were
    taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    ent = json.load(open(path)).get(workload)
    if not ent:
        return None
    csrc = os.path.join(ROOT, "gqa_attention_kv_qk_gb300", "csrc")
    blob = b"".join(open(os.path.join(csrc, f), "rb").read() for f in ent["sources"])
    if hashlib.sha256(blob).hexdigest()[:16] != ent["sources_sha256_16"]:
        return None
    return int(ent["traffic_bytes_per_launch"])


# ---------------------------------------------------------------- algorithmic bytes

def _kv_row_bytes(cfg: dict) -> tuple[int, int]:
    D = cfg["head_dim"]
    kv = cfg.get("kv_dtype", "bf16")
    if kv == "f32":
        return 4 * D, 4 * D
    if kv == "bf16":
        return 2 * D, 2 * D
    if kv == "q8":
        return D + 4, D + 4  # int8 key and value rows, each with its fp32 scale
    return 2 * D, D + 4  # vq8: bf16 key row; int8 value row + fp32 scale


def visible(n: int, window: int) -> int:
    return min(n, window) if window else n


def partial_bytes(cfg: dict, lens_after: list[int]) -> int:
    """Visible K and V rows the split-K partial must read (one read per kv head):
    with T = q_len tokens per sequence and a window W, the union of the rows'
    windows, W + T - 1 keys."""
    kb, vb = _kv_row_bytes(cfg)
    T = int(cfg.get("q_len", 1) or 1)
    w = cfg.get("window", 0) or 0
    w = w + T - 1 if w else 0
    return sum(visible(n, w) for n in lens_after) * cfg["n_kv_heads"] * (kb + vb)


def attention_flops(cfg: dict, lens_before: list[int]) -> int:
    """Tensor work of one step (q_len = T tokens per sequence): every (token, query
    head) row against each key it sees (the cache and the chunk's tokens up to its
    own, within the window), 2 D flops for QK and 2 D for P.V per (row, key)."""
    T = int(cfg.get("q_len", 1) or 1)
    G = cfg["n_q_heads"] // cfg["n_kv_heads"]
    w = cfg.get("window", 0) or 0
    keys = 0
    for n in lens_before:
        for t in range(T):
            keys += visible(n + t + 1, w)
    return keys * cfg["n_kv_heads"] * G * 4 * cfg["head_dim"]


def decode_step_bytes(cfg: dict, lens_before: list[int]) -> int:
    """One step (T = q_len tokens per sequence): the partial's KV reads (each key
    once, whatever T) plus the q/k/v reads, the appended rows and the output."""
    B, Hq, Hkv, D = cfg["batch"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    T = int(cfg.get("q_len", 1) or 1)
    io = 4 if cfg.get("io_dtype") == "f32" else 2
    ob = 4 if cfg.get("out_dtype", "f32") == "f32" else 2
    kb, vb = _kv_row_bytes(cfg)
    small = T * (B * (Hq + 2 * Hkv) * D * io + B * Hkv * (kb + vb) + B * Hq * D * ob)
    return partial_bytes(cfg, [n + T for n in lens_before]) + small


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 20 ms) of the SM clock and the throttle reasons,
    each with its timestamp; mark_start / mark_end bracket the timed region, and
    summary() reports the samples taken inside it (all samples when the region
    was too short to hold one, with under_load = 0)."""
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.lines: list[str] = []
        self.t0 = self.t1 = None
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        ident = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.cmd = [exe, "-i", ident, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                    "-lms", "20"]

    def __enter__(self):
        if hasattr(self, "cmd"):
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.15)
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []  # (time or None, sm MHz, max MHz, active reasons)
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None
            rows.append((ts, sm, mx, {nm for nm, val in zip(names, parts[5:9]) if val.lower().startswith("active")}))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "under_load": 0}
        inside = [r for r in rows if self.t0 and self.t1 and r[0] and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted(set().union(*(r[3] for r in use))), "samples": len(rows),
                "under_load": len(inside)}


# ---------------------------------------------------------------- distributed

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing

def oracle_sample(cfg: dict, case: dict, budget_s: float, n_threads: int) -> dict:
    """Time the fp64 CPU oracle on whole decode steps of a prefix of the batch
    (all heads of each sequence), growing the prefix up to the time budget; a
    whole batch that takes well under the budget is stepped several times (the
    lengths put back each time, so every repetition is the same work).
    Returns bytes processed, seconds, and a description of the sample."""
    from oracle import oracle as O
    from tests.cases import oracle_arrays  # the storage arrays the parity tests give the oracle

    a = oracle_arrays(case, O)
    B = cfg["batch"]
    lens0 = a["seq_lens"].copy()

    step = O.chunk_step if int(cfg.get("q_len", 1) or 1) > 1 else O.decode_step

    def run(nb: int) -> float:
        sl = lens0[:nb].copy()
        t = time.perf_counter()
        step(cfg, a["q"][:nb].copy(), a["k_new"][:nb].copy(), a["v_new"][:nb].copy(), a["q_norm_w"],
                      a["k_norm_w"], a["sink"], a["k_cache"][:nb], a["v_cache"][:nb],
                      None if a["v_scale"] is None else a["v_scale"][:nb], sl, n_threads=n_threads,
                      k_scale=None if a["k_scale"] is None else a["k_scale"][:nb])
        return time.perf_counter() - t

    t1 = run(1)
    nb = int(max(1, min(B, budget_s / max(t1, 1e-6))))
    secs = run(nb) if nb > 1 else t1
    reps = 1
    if nb == B and secs < budget_s / 4:
        reps = int(min(1000, max(1, budget_s / 2 / max(secs, 1e-6))))
        secs = sum(run(nb) for _ in range(reps))
    lens = [int(x) for x in lens0[:nb]]
    sub = dict(cfg, batch=nb)
    T = int(cfg.get("q_len", 1) or 1)
    return {"bytes": decode_step_bytes(sub, lens) * reps, "seconds": secs, "steps": reps,
            "sample": (f"{reps} x " if reps > 1 else "") + f"one step ({T} token(s) per sequence) of {nb} of {B} "
                      f"sequences (all {cfg['n_q_heads']} q heads), {n_threads} threads"}


def cpu_baseline(name: str, cases: list, budget: float) -> dict:
    """The oracle on the host's cores (one thread per core), and on one core on a
    smaller sample of the same workload; first layer of a multi-layer workload."""
    lc = W.layer_configs(W.config(name))[0]
    n_thr = len(os.sched_getaffinity(0))
    smp = oracle_sample(lc, cases[0], budget, n_thr)
    cpu = {"value": smp["bytes"] / smp["seconds"] / 1e9, "unit": "GB/s", "cores": n_thr, "kind": "oracle",
           "sample": smp["sample"], "ms_per_decode_step": round(smp["seconds"] / smp["steps"] * 1e3, 3)}
    if n_thr > 1:
        one = oracle_sample(lc, cases[0], min(5.0, budget / 3), 1)
        cpu["one_core"] = {"value": one["bytes"] / one["seconds"] / 1e9, "sample": one["sample"]}
    return cpu


# ---------------------------------------------------------------- the workload

def workload_bytes(cfg: dict):
    """(bytes of one benchmark step, partial-kernel bytes of one benchmark step,
    decode steps per benchmark step) from the seeded lengths alone (no device)."""
    n_dec = DECODES_PER_STEP.get(cfg["name"], 1)
    T = int(cfg.get("q_len", 1) or 1)
    step_bytes = part_bytes = 0
    for lc in W.layer_configs(cfg):
        base = [int(x) for x in W.seq_lens(lc)]
        for t in range(n_dec):
            cur = [x + t * T for x in base]
            step_bytes += decode_step_bytes(lc, cur)
            part_bytes += partial_bytes(lc, [x + T for x in cur])
    return step_bytes, part_bytes, n_dec


def config_block(cfg: dict, world: int) -> dict:
    """The workload as the JSON line's `config` (the same dict on both arms)."""
    name = cfg["name"]
    lcs = W.layer_configs(cfg)
    step_bytes, part_bytes, n_dec = workload_bytes(cfg)
    kv_mb = part_bytes / n_dec / 1e6
    out = {"workload": name, "batch": cfg["batch"], "seq_len": cfg["seq_len"], "n_q_heads": cfg["n_q_heads"],
           "n_kv_heads": cfg["n_kv_heads"], "head_dim": cfg["head_dim"], "kv_dtype": cfg["kv_dtype"],
           "layers": len(lcs), "decode_steps_per_step": n_dec, "q_len": int(cfg.get("q_len", 1) or 1),
           "parallelism": f"replicas x{world}"}
    if part_bytes / n_dec > 2 * L2_BYTES:
        out["l2"] = "inputs larger than L2 (KV cache %.0f MB read per decode step)" % kv_mb
    else:
        out["l2"] = ("KV cache of %.2f MB per decode step fits in L2: warm (graph replayed back to back) "
                     "and cold (L2 flushed by a %d MB write before each step) both reported" %
                     (kv_mb, 3 * L2_BYTES // 2**20))
    return out


# ---------------------------------------------------------------- the GPU arm

def build_layers(cfg: dict, cap_extra: int, device: str):
    from gqa_attention_kv_qk_gb300.layer import DecodeLayer
    layers, cases = [], []
    for lc in W.layer_configs(cfg):
        case = W.host_case(lc, cap=W.capacity(lc, extra=cap_extra))
        layers.append(DecodeLayer.for_case(case, device))
        cases.append(case)
    return layers, cases


def measure(name: str, args, world: int, rank: int, local: int, with_cpu: bool, cpu_budget: float) -> dict | None:
    """One workload on this rank's GPU: device-timed steps (and, for a workload
    whose cache fits in L2, the same steps with L2 flushed before each), the
    partial kernel alone, the end-to-end leg with host buffers, and on rank 0 the
    oracle baseline. Returns the record on rank 0."""
    from gqa_attention_kv_qk_gb300 import binding as Bd
    device = f"cuda:{local}"
    cfg = W.config(name, seed=W.CONFIGS[name]["seed"] + 1000 * rank)
    if args.batch:
        cfg["batch"] = args.batch
    if args.reproducible:
        cfg["reproducible"] = True
    step_bytes, part_bytes, n_dec = workload_bytes(cfg)
    T = int(cfg.get("q_len", 1) or 1)  # tokens per sequence and call
    layers, cases = build_layers(cfg, cap_extra=n_dec * T + 1, device=device)
    if rank != 0:  # the seeded lengths of another rank's replica: its own bytes
        step_bytes = part_bytes = 0
        for lc, case in zip(W.layer_configs(cfg), cases):
            base = [int(x) for x in case["lens"]]
            for t in range(n_dec):
                cur = [x + t * T for x in base]
                step_bytes += decode_step_bytes(lc, cur)
                part_bytes += partial_bytes(lc, [x + T for x in cur])
    lens0 = [case["lens"].clone() for case in cases]
    lens0_dev = [l.to(device) for l in lens0]
    hint = [int(l.max()) + (n_dec - 1) * T for l in lens0]
    stream = torch.cuda.Stream(device)
    inputs = [{k: case[k].to(device) for k in ("q", "k_new", "v_new")} for case in cases]
    fits_l2 = part_bytes / n_dec <= 2 * L2_BYTES

    def reset():
        for layer, l0 in zip(layers, lens0_dev):
            layer.seq_lens.copy_(l0, non_blocking=True)

    def one_step(n=n_dec):  # one benchmark step: n decode steps of every layer, then lengths reset
        for _ in range(n):
            for li, layer in enumerate(layers):
                inp = inputs[li]
                layer.step(inp["q"], inp["k_new"], inp["v_new"], stream=stream, max_seq_len=hint[li])
        reset()

    # kernels of one call of a layer: the fused append+partial and the combine
    # (bf16 / vq8 / q8 caches, one token), one kernel for a small fp32 step, or
    # append, partial and combine
    lays = [Bd.uaa_get_workspace_layout(layer.desc, layer.batch, h, 0, T) for layer, h in zip(layers, hint)]
    fused = [lay.kernel == 1 and T == 1 for lay in lays]
    one_launch = [lay.step_splits > 0 for lay in lays]
    launches_per_step = n_dec * sum(lay.step_kernels for lay in lays)

    with torch.cuda.stream(stream):
        # warm-up, then capture one benchmark step in a graph
        for _ in range(max(1, args.warmup)):
            one_step()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one_step()
        for _ in range(args.warmup):
            graph.replay()
        stream.synchronize()

        # ---- timed region: exactly K benchmark steps (an event between steps, for
        # the per-step spread)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(local) as clocks:
            clocks.mark_start()
            evs[0].record(stream)
            for i in range(args.steps):
                graph.replay()
                evs[i + 1].record(stream)
            evs[-1].synchronize()
            clocks.mark_end()
        torch.cuda.synchronize()
        barrier(world)
        dev_s = evs[0].elapsed_time(evs[-1]) / 1e3
        per_step_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
        for layer in layers:
            st = layer.device_status(stream)
            if st:
                raise RuntimeError(f"device flags 0x{st:x} after the timed region")

        # ---- cold: K single decode steps (a graph of one step and the length reset),
        # each after a write of 1.5x L2 (untimed, and long enough that the host has
        # queued the step before the GPU reaches it), so the step finds none of its
        # cache in L2
        cold_s = None
        if fits_l2:
            graph1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph1, stream=stream):
                one_step(1)
            flush = torch.empty(3 * L2_BYTES // 2, dtype=torch.uint8, device=device)
            ce = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            barrier(world)
            torch.cuda.synchronize()
            for e0, e1 in ce:
                flush.fill_(1)
                e0.record(stream)
                graph1.replay()
                e1.record(stream)
            stream.synchronize()
            barrier(world)
            cold_s = sum(e0.elapsed_time(e1) for e0, e1 in ce) / 1e3
            del flush, graph1

        # ---- the partial kernel alone (events on the launching stream): the fused
        # append+partial kernel of the step for bf16 / vq8 caches, the partial
        # kernel after its separate append for fp32 caches; a step that is one
        # kernel takes the timed region's per-step time (events around single
        # launches of a few microseconds would time the host's launch instead)
        pe = []
        rounds = 0 if all(one_launch) else -(-20 // n_dec)  # at least 20 launches per layer
        for _ in range(rounds):
            reset()
            for _ in range(n_dec):
                for li, layer in enumerate(layers):
                    inp = inputs[li]
                    args_ = layer.args(inp["q"], inp["k_new"], inp["v_new"], max_seq_len=hint[li])
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    if one_launch[li]:  # the whole step is the one kernel
                        e0.record(stream)
                        Bd.uaa_decode_attn(layer.desc, args_, layer.ws, stream)
                        e1.record(stream)
                        pe.append((e0, e1))
                        continue
                    if fused[li]:
                        e0.record(stream)
                        Bd.uaa_decode_attn_append_partial(layer.desc, args_, layer.ws, stream)
                        e1.record(stream)
                    else:
                        Bd.uaa_rope_qk_norm_append(layer.desc, args_, layer.ws, stream)
                        e0.record(stream)
                        Bd.uaa_decode_attn_partial(layer.desc, args_, layer.ws, stream)
                        e1.record(stream)
                    Bd.uaa_decode_attn_combine(layer.desc, args_, layer.ws, stream)
                    pe.append((e0, e1))
        stream.synchronize()
        part_s = sum(a.elapsed_time(b) for a, b in pe) / 1e3
        n_part = len(pe)
        reset()
        stream.synchronize()

        # ---- end to end through the public call, host buffers
        # Every decode step copies its own q / k / v from pinned host memory and
        # reads its own output back, inside the timed region. Inputs and outputs are
        # double-buffered per layer and the copies run on a second stream, so the
        # next call's input copy and the last call's read-back overlap the current
        # call's kernels, as in a serving loop.
        # q, k_new and v_new of a call travel as one pinned buffer (one copy per call)
        names = ("q", "k_new", "v_new")
        host_in, dev_in, views = [], [], []
        for case in cases:
            parts = [case[k].contiguous() for k in names]
            nbytes = [t.numel() * t.element_size() for t in parts]
            buf = torch.empty(sum(nbytes), dtype=torch.uint8).pin_memory()
            off = 0
            for t, n in zip(parts, nbytes):
                buf[off:off + n].copy_(t.view(-1).view(torch.uint8))
                off += n
            host_in.append(buf)
            dbufs = [torch.empty_like(buf, device=device) for _ in range(2)]
            dev_in.append(dbufs)
            vs = []
            for db in dbufs:
                off, v = 0, {}
                for k, t, n in zip(names, parts, nbytes):
                    v[k] = db[off:off + n].view(t.dtype).view(t.shape)
                    off += n
                vs.append(v)
            views.append(vs)
        outs = [layer.out_for(T) for layer in layers]
        host_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)] for o in outs]
        h2d = sum(hi.numel() for hi in host_in) * n_dec
        d2h = sum(ho[0].numel() * ho[0].element_size() for ho in host_out) * n_dec
        dev_out = [[torch.empty_like(o) for _ in range(2)] for o in outs]
        copy = torch.cuda.Stream(device)
        ev = [[{n: torch.cuda.Event() for n in ("in", "done", "read")} for _ in range(2)] for _ in layers]
        # every call of the timed region: (benchmark step, decode step, layer); buffer
        # slot = the call's index among its layer's calls, mod 2
        calls = [(k, t, li) for k in range(args.steps) for t in range(n_dec) for li in range(len(layers))]
        slot = [(k * n_dec + t) % 2 for k, t, _ in calls]

        def copy_in(c):  # input copy of call c into its buffer, once the buffer's last user ran
            li, b = calls[c][2], slot[c]
            copy.wait_event(ev[li][b]["done"])
            with torch.cuda.stream(copy):
                dev_in[li][b].copy_(host_in[li], non_blocking=True)
            ev[li][b]["in"].record(copy)

        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        copy_in(0)
        for c, (k, t, li) in enumerate(calls):
            if t == 0 and li == 0:
                reset()  # lengths back to the start of the benchmark step (device copy, in stream order)
            if c + 1 < len(calls):
                copy_in(c + 1)
            b = slot[c]
            e = ev[li][b]
            stream.wait_event(e["in"])
            stream.wait_event(e["read"])  # the buffer's previous output has been read back
            d = views[li][b]
            layers[li].step(d["q"], d["k_new"], d["v_new"], stream=stream, max_seq_len=hint[li], out=dev_out[li][b])
            e["done"].record(stream)
            copy.wait_event(e["done"])
            with torch.cuda.stream(copy):
                host_out[li][b].copy_(dev_out[li][b], non_blocking=True)
            e["read"].record(copy)
        stream.synchronize()
        copy.synchronize()
        e2e_s = time.perf_counter() - t0
        barrier(world)

    dev_s = max_over_ranks(dev_s, world)
    e2e_s = max_over_ranks(e2e_s, world)
    total_bytes = sum_over_ranks(step_bytes * args.steps, world)
    if cold_s is not None:
        cold_s = max_over_ranks(cold_s, world)
    del graph, layers, inputs, dev_in, dev_out, outs
    torch.cuda.empty_cache()
    if rank != 0:
        return None
    peaks = measured_peaks()
    value = total_bytes / dev_s / 1e9
    # part_bytes covers one benchmark step (n_dec launches per layer); the timing covers all rounds
    n_layers = len(cases)
    if all(one_launch):  # the timed region: one kernel per layer and decode step (and a length reset per 64)
        part_s, n_part = dev_s, args.steps * n_dec * n_layers
    # tensor work of one benchmark step (a prefill chunk is bound by it, not by the cache bytes)
    step_flops = 0
    for lc, l0 in zip(W.layer_configs(cfg), lens0):
        base = [int(x) for x in l0]
        for t in range(n_dec):
            step_flops += attention_flops(lc, [x + t * T for x in base])
    part_gbs = (part_bytes / (n_dec * n_layers)) / (part_s / n_part) / 1e9 if n_part else None
    decodes = n_dec * args.steps * world
    rec = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(dev_s / args.steps * 1e3, 4),
        # this rank's steps one by one (ms): the spread behind the mean above
        "step_ms": {"median": round(per_step_ms[len(per_step_ms) // 2], 4), "best": round(per_step_ms[0], 4),
                    "worst": round(per_step_ms[-1], 4)} if per_step_ms else None,
        "decode_steps_per_s": round(decodes / dev_s / world, 2),
        "tokens_per_s_per_seq": round(decodes * T / dev_s / world, 2),  # q_len new tokens per sequence and step
        "pct_of_measured_copy_peak": round(100 * value / world / peaks["hbm_gbs"], 2),
        "pct_of_nominal_hbm_peak": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "dtype": {"f32": "f32", "q8": "f16"}.get(cfg["kv_dtype"], "bf16"),
        "config": config_block(cfg, world),
        "roofline": {"bound": "hbm", "achieved": round(part_gbs, 2) if part_gbs else None,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(part_gbs / peaks["hbm_gbs"], 4) if part_gbs else None,
                     "traffic": measured_traffic(name),
                     "frac_of_nominal": round(part_gbs / NOMINAL_HBM_GBS, 4) if part_gbs else None,
                     "kernel": ("fused append + split-K partial" if all(fused) else
                                "fp32 one-launch step (append, attention, merge)" if all(one_launch) else
                                "query-tiled prefill" if all(lay.kernel == 2 for lay in lays) else
                                "split-K partial"),
                     "peak_source": peaks["source"],
                     "bytes_per_launch": part_bytes // max(1, n_dec * n_layers),
                     "mean_launch_us": round(part_s / n_part * 1e6, 2) if n_part else None},
        "e2e": {"value": round(total_bytes / e2e_s / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "tflops": round(step_flops * args.steps / dev_s / 1e12, 2),
        "clocks": clocks.summary(),
        "cpu_baseline": cpu_baseline(name, cases, cpu_budget) if with_cpu else None,
    }
    if T >= 64 and n_part:  # a prefill chunk: the partial kernel against the bf16 tensor peak
        kern_tf = (step_flops / (n_dec * n_layers)) / (part_s / n_part) / 1e12
        hbm = rec["roofline"]
        rec["roofline"] = {"bound": "tensor", "achieved": round(kern_tf, 2), "peak": peaks["bf16_tflops"],
                           "unit": "TFLOP/s", "frac": round(kern_tf / peaks["bf16_tflops"], 4),
                           "traffic": hbm["traffic"], "kernel": hbm["kernel"], "peak_source": peaks["source"],
                           "flops_per_launch": step_flops // max(1, n_dec * n_layers),
                           "mean_launch_us": hbm["mean_launch_us"], "hbm_gbs": hbm["achieved"]}
    if cold_s is not None:
        first = sum(decode_step_bytes(lc, [int(x) for x in l0]) for lc, l0 in zip(W.layer_configs(cfg), lens0))
        rec["cold"] = {"value": round(first * args.steps / cold_s / 1e9, 2), "unit": "GB/s",
                       "us_per_decode_step": round(cold_s / args.steps * 1e6, 3),
                       "decode_steps_per_s": round(args.steps / cold_s, 2),
                       "l2": "one decode step per graph replay, L2 flushed before each by a %d MB write (not timed)"
                             % (3 * L2_BYTES // 2**20)}
        rec["warm_note"] = ("%d decode steps per graph replay, back to back: the cache stays in L2 between steps"
                            % n_dec)
        rec["us_per_decode_step"] = round(dev_s / (args.steps * n_dec) * 1e6, 3)
    return rec


def run_uaa(args, world, rank, local) -> dict | None:
    from gqa_attention_kv_qk_gb300 import build as ext
    ext.build()
    torch.cuda.set_device(local)
    name = args.workload
    with_cpu = world == 1 and not args.no_cpu_baseline
    head = measure(name, args, world, rank, local, with_cpu, args.cpu_budget)
    per = {}
    if name == HEADLINE and not args.no_per_config:
        for other in PER_CONFIG:
            r = measure(other, args, world, rank, local, with_cpu and other not in NO_CPU_IN_PER_CONFIG,
                        args.cpu_budget / 3)
            if r is not None:
                r.pop("dtype", None)
                per[other] = r
    if rank != 0:
        return None
    res = {"metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "step_ms": head["step_ms"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
           "data": "synthetic (seeded N(0,1) cache and inputs)",
           "decode_steps_per_s": head["decode_steps_per_s"], "tokens_per_s_per_seq": head["tokens_per_s_per_seq"],
           "pct_of_measured_copy_peak": head["pct_of_measured_copy_peak"],
           "pct_of_nominal_hbm_peak": head["pct_of_nominal_hbm_peak"],
           "config": head["config"],
           "timing": "CUDA graph of one benchmark step, replayed K times; CUDA events on the launching stream",
           "roofline": head["roofline"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
           "clocks": head["clocks"], "cpu_baseline": head["cpu_baseline"]}
    if "cold" in head:
        res["cold"] = head["cold"]
    if per:
        res["per_config"] = per
    return res


def run_reference(args, world, rank) -> dict | None:
    """The oracle as the reference arm, on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    name = args.workload
    cfg = W.config(name)
    lc = W.layer_configs(cfg)[0]
    case = W.host_case(lc, cap=W.capacity(lc, extra=2))
    n_thr = len(os.sched_getaffinity(0))
    budget = max(0.5, args.cpu_budget / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_sample(lc, case, budget / 4, n_thr)
    tot_b = tot_s = 0.0
    sample = ""
    for _ in range(args.steps):
        smp = oracle_sample(lc, case, budget, n_thr)
        tot_b += smp["bytes"]
        tot_s += smp["seconds"]
        sample = smp["sample"]
    v = tot_b / tot_s / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) cache and inputs)",
            "config": config_block(cfg, world),
            "timing": "wall clock of each sample (time.perf_counter)",
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": n_thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["uaa", "reference"], default="uaa")
    ap.add_argument("--workload", default="llama31_8b_decode", choices=list(W.CONFIGS))
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the headline workload only (not the suite's other four)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (a smaller case for profiling; not a benchmark config)")
    ap.add_argument("--reproducible", action="store_true",
                    help="uniform stream-K ranges (equal bits on every launch) instead of speed-weighted ones")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "uaa":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_setup(args.gpus)
    res = run_reference(args, world, rank) if args.impl == "reference" else run_uaa(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
