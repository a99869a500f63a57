#!/usr/bin/env python3
"""Decode-step benchmark: int4 weight-only group-wise greedy decode of the
28-layer 2B-shaped decoder on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--batch 1|4|16] [--impl kmr|reference]
    python bench.py --sweep          # standalone int4 GEMV / decode-attention sweeps
    python bench.py --prefill-only T [--prefill-mma]  # two T-token prefills (a fixed command for launch lists)

A step is one pass of the whole decode path (every layer's int4 QKV / O /
gate_up / down GEMVs, q/k norm, M-RoPE, KV write and GQA attention, final
norm, tied bf16 LM head, argmax and state advance) for the batch's rows.
Workload (synthetic, seeded): batch 1 with 512 prefilled positions, 256
greedy steps per generation (--batch 4: four continuous slots prefilled
300/512/700/900, row 2 retired at step 64, row 3 length-capped at 1024,
128 steps per generation; --batch 16: sixteen slots prefilled 256..896, 128
steps).  The timed K steps run back to back as CUDA-graph
replays; the state is rewound to the generation's start every generation.
The per-step working set (1.4 GB of weights) is far larger than L2, so
nothing survives in L2 between steps.

Prints one JSON line (rank 0).  Multi-GPU: replicas only (the decode path
does not shard); each rank runs its own model, time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "int4 decode tok/s @bs1/bs4 (2B-shaped); achieved HBM GB/s vs roofline"


# ------------------------------------------------------------------ clocks during the timed region
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int = 0, interval_ms: int = 20):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        rows = [r for t, r in self.rows if t0 - 0.05 <= t <= t1 + 0.05 and len(r) >= 9]
        if not rows:
            rows = [r for _, r in self.rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        out = {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured (MEASURED_PEAKS.json)"}
        if "bf16_tflops" in d:
            out["bf16_tflops"] = float(d["bf16_tflops"])
        return out
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def profile_traffic(summary: str):
    """DRAM bytes per launch from a committed ncu summary, if every source file it names
    (`kernel_source_sha256: <sha> (<file>), ...`) is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    line = re.search(r"kernel_source_sha256:(.*)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not line or not m_tr:
        return None
    pairs = re.findall(r"([0-9a-f]{64})\s*\(([\w.]+)\)", line.group(1))
    if not pairs:
        return None
    for sha, name in pairs:
        src = os.path.join(ROOT, "int4_weight_only_group_gb300", "csrc", name)
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != sha:
            return None
    return float(m_tr.group(1))


# ------------------------------------------------------------------ workloads
def workload(batch: int):
    from workloads import full2b_b1_workload, full2b_b4_workload, full2b_b16_workload
    return {1: full2b_b1_workload, 4: full2b_b4_workload, 16: full2b_b16_workload}[batch]()


def tokens_per_generation(wl) -> int:
    """Tokens the rows actually emit (non-pad) over one generation of wl.steps steps."""
    total = 0
    for b in range(wl.batch):
        stop = wl.finish_at.get(b, wl.steps)
        cap = wl.cfg.max_len - wl.prefill[b]
        total += min(stop, cap, wl.steps)
    return total


def kv_bytes_per_generation(wl) -> int:
    """KV bytes the attention moves over one generation (reads 0..pos-1, writes pos), all layers."""
    c = wl.cfg
    per_pos = c.n_layers * 2 * c.n_kv_heads * c.head_dim * 2
    total = 0
    for b in range(wl.batch):
        n = min(wl.finish_at.get(b, wl.steps), c.max_len - wl.prefill[b], wl.steps)
        total += per_pos * sum(wl.prefill[b] + t + 1 for t in range(n))
    return total


def weight_bytes(cfg) -> dict:
    out = {}
    for name, (N, K) in cfg.linear_shapes().items():
        out[name] = N * (K // 2 + 4 * (K // 128))
    out["lm_head"] = cfg.vocab * cfg.hidden * 2
    out["norms"] = (cfg.n_layers * (2 * cfg.hidden + 2 * cfg.head_dim) + cfg.hidden) * 2
    return out


# ------------------------------------------------------------------ GPU arm
def aggregate_ranks(torch, elapsed_ms: float, tokens: float, world: int, device: str):
    """Whole-job figures of N replicas: the slowest rank's time and the sum of every rank's
    tokens (each rank decodes its own batch on its own model; no data-path collective)."""
    t = torch.tensor([elapsed_ms, tokens], dtype=torch.float64, device=device)
    ts = [torch.zeros_like(t) for _ in range(world)]
    torch.distributed.all_gather(ts, t)
    return max(float(x[0]) for x in ts), sum(float(x[1]) for x in ts)


def percentiles(ms) -> dict:
    a = np.asarray(ms, dtype=np.float64)
    return {"mean": float(a.mean()), "p10": float(np.percentile(a, 10)), "p50": float(np.percentile(a, 50)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


def timed_steps_accounting(wl, steps: int):
    """Tokens emitted and KV bytes read (positions 0..cache_position of every active row, all
    layers, K and V) over the `steps` timed steps, generation by generation from the start."""
    c = wl.cfg
    per_pos = c.n_layers * 2 * c.n_kv_heads * c.head_dim * 2
    tokens = kv = 0
    for i in range(steps):
        t = i % wl.steps
        for b in range(wl.batch):
            n = min(wl.finish_at.get(b, wl.steps), c.max_len - wl.prefill[b], wl.steps)
            if t < n:
                tokens += 1
                kv += per_pos * (wl.prefill[b] + t + 1)
    return tokens, kv


def run_kmr(args, batch: int, rank: int, world: int, extras: bool) -> dict:
    """Decode `args.steps` timed steps of the workload of `batch` rows (after the warm-up),
    one CUDA event per step on the launching stream.  With `extras` (rank 0 of the headline
    batch) also the standalone kernel timings, prefill, slot migration and cascade attention."""
    import torch
    import int4_weight_only_group_gb300 as kmr
    from int4_weight_only_group_gb300 import driver
    from workloads import SyntheticModel
    from workloads import initial_state

    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    wl = workload(batch)
    cfg = wl.cfg
    B = wl.batch
    t_setup = time.time()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    syn = SyntheticModel(cfg, wl.seed, memo=(rank == 0 and extras and not args.no_cpu_baseline))
    model = kmr.Model.from_config(cfg, max_batch=B)
    if args.persistent_step:
        model.set_persistent_step(True)
    driver.load_weights(model, syn, cfg.n_layers, cfg.qk_norm)
    for b in range(B):
        driver.load_kv(model, syn, cfg.n_layers, wl.slot_ids[b], wl.prefill[b])
    torch.cuda.synchronize()
    memory = model.device_bytes()
    memory["mem_get_info_delta"] = int(free0 - torch.cuda.mem_get_info()[0])
    setup_s = time.time() - t_setup

    st0 = initial_state(wl)
    dev = {k: torch.tensor(np.asarray(v), device="cuda") for k, v in
           zip(("tok", "pos", "cpos", "slot", "fin"), st0)}
    saved = {k: v.clone() for k, v in dev.items()}
    stream = torch.cuda.current_stream()

    def rewind():
        for k in ("tok", "pos", "cpos", "fin"):
            dev[k].copy_(saved[k])

    def step(t_in_gen: int):
        for row, at in wl.finish_at.items():
            if at == t_in_gen:
                dev["fin"][row] = 1
        model.decode_step(dev["tok"], dev["pos"], dev["cpos"], dev["slot"], dev["fin"], B, None, stream)

    for i in range(args.warmup):
        step(i % wl.steps)
    torch.cuda.synchronize()
    assert model.sync_status(stream) == 0
    rewind()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev_index) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t0 = time.time()
    ev[0].record(stream)
    for i in range(args.steps):
        t = i % wl.steps
        if t == 0 and i > 0:
            rewind()                      # back to the generation's start (a device copy, inside the timing)
        step(t)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = ev[0].elapsed_time(ev[-1])
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    clk = None
    if clocks:
        time.sleep(0.1)
        clocks.stop()
        clk = clocks.summary(t0, t1)
    assert model.sync_status(stream) == 0, "device error during the timed region"
    tokens, kv_timed = timed_steps_accounting(wl, args.steps)

    if world > 1:
        elapsed_ms, tokens = aggregate_ranks(torch, elapsed_ms, tokens, world, "cuda")
    if rank != 0:
        model.close()
        return {}

    out = {"wl": wl, "elapsed_ms": elapsed_ms, "tokens": tokens, "setup_s": setup_s, "clocks": clk,
           "kernels_per_step": model.kernels_per_step(B), "kv_timed": kv_timed, "step_ms": percentiles(per_step),
           "memory": memory}
    if args.skip_extras:
        model.close()
        return out
    # ---- end to end through the host-buffer C ABI call
    out["e2e"] = time_e2e(torch, model, wl, st0, args.steps)
    if not extras:
        model.close()
        return out
    # ---- dominant kernel: the int4 GEMV, timed alone on rotating copies larger than L2
    out["gemv"] = time_gemv(torch, kmr, syn, cfg, B)
    # ---- slot migration: one whole cache row (every layer, K and V) per copy_row_from
    out["kv_copy"] = time_kv_copy(torch, model, cfg)
    # ---- text prefill of a 512-token prompt into slot 0 (after the timed decode region)
    out["prefill"] = time_prefill(torch, model, cfg)          # the default tcgen05 projections
    model.set_prefill_tcgen05(False)                # the warp-level mma projections, for comparison
    out["prefill_mma"] = time_prefill(torch, model, cfg)
    model.set_prefill_tcgen05(True)
    # ---- shared-prefix attention vs plain attention on the same contexts
    out["cascade"] = time_cascade(torch, kmr, cfg)
    model.close()
    if not args.no_cpu_baseline:
        out["cpu"] = cpu_baseline(wl, syn, args)
    return out


def launch_time_us(torch, fn, copies: int, reps: int) -> float:
    """Mean CUDA-event microseconds per call of fn(i % copies) over `reps` back-to-back calls on
    the current stream, after warm-up.  A sleep kernel holds the stream while the host queues
    the calls, so the events see the launches' own device time, not the host's rate of issuing
    them (a Python-side call costs several microseconds, more than a small launch runs)."""
    stream = torch.cuda.current_stream()
    for i in range(max(3, copies)):
        fn(i % copies)
    torch.cuda.synchronize()
    hold = torch.cuda.Event(enable_timing=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold.record(stream)
    torch.cuda._sleep(int(2e6 + reps * 60e3))           # ~1 ms + 30 us per queued call at ~2 GHz
    e0.record(stream)
    t0 = time.perf_counter()
    for i in range(reps):
        fn(i % copies)
    t_host = time.perf_counter() - t0
    e1.record(stream)
    torch.cuda.synchronize()
    if t_host * 1e3 > hold.elapsed_time(e0):
        print(f"launch_time_us: queueing took {t_host * 1e3:.2f} ms, longer than the hold; "
              "the figure includes host issue time", file=sys.stderr)
    return e0.elapsed_time(e1) * 1e3 / reps


def time_prefill(torch, model, cfg, T: int = 512, reps: int = 3) -> dict:
    """CUDA-event time of kmr_prefill of a T-token prompt (one chunk) into cache row 0: every
    layer's int4 projections over T rows (16-row passes), the q/k norm + M-RoPE + KV write of
    every position, causal attention, and the LM head on the last position."""
    T = min(T, cfg.max_len)
    model.reserve_prefill(T)
    g = torch.Generator(device="cuda").manual_seed(1)
    toks = torch.randint(1, cfg.vocab - 1, (T,), generator=g, device="cuda", dtype=torch.int32)
    pos = torch.arange(T, dtype=torch.int32, device="cuda").repeat(3, 1).contiguous()
    st = [torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(3, dtype=torch.int32, device="cuda"),
          torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.uint8, device="cuda")]
    stream = torch.cuda.current_stream()
    model.prefill(toks, pos, T, 0, 0, *st, None, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        model.prefill(toks, pos, T, 0, 0, *st, None, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert model.sync_status(stream) == 0
    ms = e0.elapsed_time(e1) / reps
    return {"tokens": T, "ms": ms, "tok_s": T / (ms * 1e-3)}


def time_kv_copy(torch, model, cfg, reps: int = 10) -> dict:
    """CUDA-event time of kmr_model_copy_row_from moving a full max_len row (all layers, K and
    V) from an external cache into slot 0; two alternating sources (> L2 together), so every
    copy reads HBM.  Bytes = read + write of the row.  Runs after the timed decode region
    (it overwrites slot 0)."""
    L, nkv, S, d = cfg.n_layers, cfg.n_kv_heads, cfg.max_len, cfg.head_dim
    srcs = [(torch.randint(-2 ** 15, 2 ** 15, (L, 1, nkv, S, d), dtype=torch.int16, device="cuda"),
             torch.randint(-2 ** 15, 2 ** 15, (L, 1, nkv, S, d), dtype=torch.int16, device="cuda")) for _ in range(2)]
    stream = torch.cuda.current_stream()
    for i in range(3):
        model.copy_row_from(0, S, 0, srcs[i % 2][0], srcs[i % 2][1], 1, S, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        model.copy_row_from(0, S, 0, srcs[i % 2][0], srcs[i % 2][1], 1, S, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert model.sync_status(stream) == 0
    us = e0.elapsed_time(e1) * 1e3 / reps
    nbytes = 2 * (2 * L * nkv * S * d * 2)
    return {"row_positions": S, "bytes": nbytes, "us": us, "gbs": nbytes / (us * 1e3)}


def time_cascade(torch, kmr, cfg, B: int = 16, P: int = 400, own: int = 100, copies: int = 4, reps: int = 20) -> dict:
    """Shared-prefix decode attention on one layer of the model's attention shape: B rows share
    a P-position prefix and own `own` positions each.  Timed against kmr_decode_attn over rows
    that hold the whole [prefix; own] context.  Each timed call uses the next of `copies`
    caches (> L2 together), so the KV comes from HBM."""
    import math
    nq, nkv, d, S = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.max_len
    slots = B + 1
    g = torch.Generator(device="cuda").manual_seed(0)
    caches = []
    for _ in range(copies):
        k = (torch.randn((slots, nkv, S, d), generator=g, device="cuda") * 1.0).to(torch.bfloat16).view(torch.int16)
        v = (torch.randn((slots, nkv, S, d), generator=g, device="cuda") * 1.0).to(torch.bfloat16).view(torch.int16)
        k[:B, :, :P] = k[B, :, :P]                 # the plain path's rows hold the prefix too
        v[:B, :, :P] = v[B, :, :P]
        caches.append((k, v))
    q = torch.randn((B, nq, d), generator=g, device="cuda")
    slot_ids = torch.arange(B, dtype=torch.int32, device="cuda")
    cpos = torch.tensor([P + own - 1] * B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, nq, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    ws_c = kmr.kmr_decode_attn_cascade_workspace_size(B, nq, nkv, d, P)
    wsc = torch.empty(ws_c, dtype=torch.uint8, device="cuda")
    ws_p = kmr.kmr_decode_attn_workspace_size(B, nq, nkv, d)
    wsp = torch.zeros(ws_p, dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(d)
    runs = {
        "cascade": lambda kv: kmr.kmr_decode_attn_cascade(q, kv[0], kv[1], slot_ids, cpos, B, P, B, nq, nkv, d, S, slots,
                                                          scale, out, wsc, ws_c, stream),
        "plain": lambda kv: kmr.kmr_decode_attn(q, kv[0], kv[1], slot_ids, cpos, B, nq, nkv, d, S, slots, scale, out,
                                                wsp, ws_p, stream),
    }
    row = nkv * d * 2 * 2                          # K and V bytes per position of one row
    nbytes = {"cascade": (P + B * own) * row, "plain": B * (P + own) * row}
    res = {"rows": B, "prefix": P, "own": own}
    for name, fn in runs.items():
        us = launch_time_us(torch, lambda i: fn(caches[i]), copies, reps)
        res[name] = {"us": us, "kv_bytes": nbytes[name], "gbs": nbytes[name] / (us * 1e3)}
    assert kmr.kmr_last_device_error() == 0
    return res


def time_gemv(torch, kmr, syn, cfg, M: int) -> dict:
    """Average CUDA-event duration of one int4 GEMV launch per projection shape (launches queued
    behind a hold, see launch_time_us), rotating through distinct packed copies (> 2x L2 in
    total) so every launch streams from HBM."""
    res = {}
    stream = torch.cuda.current_stream()
    for name, (N, K) in cfg.linear_shapes().items():
        q, s, z = syn.linear(0, name)
        flags = kmr.KMR_PACK_GATE_UP if name == "gate_up" else 0
        size = kmr.kmr_packed_size(N, K, 128)
        copies = max(4, int(np.ceil(300e6 / size)))
        one = torch.empty(size, dtype=torch.uint8, device="cuda")
        kmr.kmr_pack_int4(torch.from_numpy(q).cuda(), torch.from_numpy(s.view(np.int16)).cuda(),
                          torch.from_numpy(z.view(np.int16)).cuda(), N, K, 128, flags, one, size, 1, stream)
        bufs = [one] + [one.clone() for _ in range(copies - 1)]
        x = torch.randn((M, K), device="cuda")
        epi = kmr.KMR_EPI_SILU_MUL if name == "gate_up" else kmr.KMR_EPI_NONE
        y = torch.zeros((M, N), device="cuda")
        us = launch_time_us(torch, lambda i: kmr.kmr_int4_gemv(bufs[i], N, K, 128, flags, x, M, y, epi, stream),
                            copies, 200)
        nbytes = size
        res[name] = {"us": us, "bytes": nbytes, "gbs": nbytes / us / 1e3, "copies": copies}
        del bufs, one
    return res


def time_e2e(torch, model, wl, st0, steps: int) -> dict:
    """The same decode through kmr_decode_step_host: every step copies the step state in
    from pinned host memory and the emitted tokens / state back, then synchronises."""
    B = wl.batch
    pin = {k: torch.from_numpy(np.array(v, copy=True)).pin_memory() for k, v in
           zip(("tok", "pos", "cpos", "slot", "fin"), st0)}
    arrs = {k: v.numpy() for k, v in pin.items()}
    init = {k: v.copy() for k, v in arrs.items()}
    n = min(steps, wl.steps)

    def run(count):
        for k in arrs:
            arrs[k][...] = init[k]
        for t in range(count):
            for row, at in wl.finish_at.items():
                if at == t:
                    arrs["fin"][row] = 1
            model.decode_step_host(arrs["tok"], arrs["pos"], arrs["cpos"], arrs["slot"], arrs["fin"], B, None,
                                   torch.cuda.current_stream())

    run(3)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(n)
    dt = time.perf_counter() - t0
    toks = 0
    for b in range(B):
        toks += min(wl.finish_at.get(b, wl.steps), wl.cfg.max_len - wl.prefill[b], n)
    state_bytes = 25 * B   # tok, pos[3], cpos, slot (int32) + finished (uint8) per row
    return {"value": toks / dt, "unit": "tok/s", "h2d_bytes_per_step": state_bytes,
            "d2h_bytes_per_step": state_bytes, "steps": n}


# ------------------------------------------------------------------ CPU oracle legs
ORACLE_LEGS = {
    "tiny": "tiny_workload",
    "layer": "layer2b_workload",
    "b1": "full2b_b1_workload",
    "b4": "full2b_b4_workload",
}


def oracle_leg_workload(leg: str):
    import workloads
    return getattr(workloads, ORACLE_LEGS[leg])()


def warm_weights(syn, cfg) -> None:
    """Draw (and memoise) every tensor the oracle reads, outside any timed step."""
    for l in range(cfg.n_layers):
        for name in cfg.linear_shapes():
            syn.linear(l, name)
        for nm in ("in", "post", "q", "k"):
            syn.norm(l, nm)
    syn.norm(-1, "final")
    syn.embedding()


def oracle_steps(wl, syn, max_steps: int, budget_s: float) -> dict:
    """Whole oracle decode steps of `wl` from its initial state (free-running on the oracle's
    own tokens, with the workload's row retirements), each timed on its own; stops after
    `max_steps` or once `budget_s` has passed (at least one step).  Nothing is sampled or
    scaled: every timed step is the full decode step of every row."""
    from oracle import decoder as od
    o = od.OracleDecoder.for_workload(wl, syn=syn)
    tok, pos, cpos, slot, fin = od.initial_state(wl)
    times, toks = [], []
    t_start = time.perf_counter()
    for t in range(max_steps):
        fin = np.array(fin, copy=True)
        for row, at in wl.finish_at.items():
            if at == t:
                fin[row] = 1
        active = int((fin == 0).sum())
        t0 = time.perf_counter()
        res = o.step(tok, pos, cpos, slot, fin)
        times.append(time.perf_counter() - t0)
        toks.append(active)
        tok, pos, cpos, fin = res.next_ids, res.positions, res.cache_position, res.finished
        if time.perf_counter() - t_start > budget_s:
            break
    med = statistics.median(times)
    return {"workload": wl.name, "steps": len(times), "s_per_step": times, "median_s": med,
            "tok_per_s": statistics.median(toks) / med, "extrapolated": False}


def oracle_leg(leg: str, max_steps: int, budget_s: float, syn=None) -> dict:
    from workloads import SyntheticModel
    wl = oracle_leg_workload(leg)
    if syn is None:
        syn = SyntheticModel(wl.cfg, wl.seed, memo=True)
    warm_weights(syn, wl.cfg)
    return oracle_steps(wl, syn, max_steps, budget_s)


def oracle_leg_subprocess(leg: str, threads: int, max_steps: int, budget_s: float) -> dict:
    """One oracle leg in a child process with its BLAS / OpenMP pools set to `threads`."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-leg", leg, "--oracle-steps",
                        str(max_steps), "--oracle-budget-s", str(budget_s)], env=env, capture_output=True,
                       text=True, timeout=budget_s * 4 + 600)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout).strip().splitlines()[-1:] or ["failed"]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["threads"] = threads
    return d


def cpu_baseline(wl, syn, args) -> dict:
    """The oracle as it stands on the host cores: whole 28-layer steps of the headline workload
    (all cores, weights drawn before the timing), plus the smaller legs of the measurement plan
    on all cores and on one thread (--cpu-suite adds the 28-layer legs on one thread and
    batch 4 on all cores)."""
    cores = os.cpu_count()
    main = oracle_steps(wl, syn, 3, 20.0)
    main["threads"] = cores
    suite = {}
    for leg in ("tiny", "layer"):
        suite[f"{leg}_all_cores"] = oracle_leg_subprocess(leg, cores, 3, 10.0)
        suite[f"{leg}_1_thread"] = oracle_leg_subprocess(leg, 1, 3, 10.0)
    if args.cpu_suite:
        suite["b4_all_cores"] = oracle_leg_subprocess("b4", cores, 3, 60.0)
        suite["b1_1_thread"] = oracle_leg_subprocess("b1", 1, 3, 60.0)
        suite["b4_1_thread"] = oracle_leg_subprocess("b4", 1, 3, 60.0)
    tps = tokens_per_generation(wl) / wl.steps
    value = tps / main["median_s"]
    return {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"{main['steps']} whole oracle decode steps of the headline workload ({wl.name}), "
                      f"median {main['median_s']:.2f} s per step; numpy float64 with BLAS threads = host cores; "
                      "weights drawn before the timing; nothing extrapolated",
            "steps": main["steps"], "s_per_step": main["s_per_step"], "extrapolated": False, "suite": suite}


def run_reference(args) -> dict:
    """The oracle as it stands, on the host cores, on this benchmark's workloads: every timed
    step is one whole oracle decode step (all 28 layers and the full vocabulary) of the batch-1
    workload, until `--steps` are done or the time budget is spent (the line's `steps` is the
    count actually run); `bs4` times whole steps of the batch-4 workload the same way."""
    from workloads import SyntheticModel
    batches = [args.batch] if args.batch else [1, 4]
    res = {}
    for B in batches:
        wl = workload(B)
        syn = SyntheticModel(wl.cfg, wl.seed, memo=True)
        warm_weights(syn, wl.cfg)
        if args.warmup:
            oracle_steps(wl, syn, 1, 0.0)          # one whole warm-up step (numpy / BLAS first-touch)
        budget = 120.0 if B == batches[0] else 60.0
        r = oracle_steps(wl, syn, args.steps, budget)
        r["tokens_per_step"] = tokens_per_generation(wl) / wl.steps
        res[B] = (wl, r)
        del syn
    wl, r = res[batches[0]]
    value = r["tokens_per_step"] / r["median_s"]
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": r["steps"], "warmup": 1 if args.warmup else 0, "ms_per_step": r["median_s"] * 1000.0,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "kv_max_len": wl.cfg.max_len},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{r['steps']} whole oracle decode steps (median; requested {args.steps}, "
                                       "120 s budget), numpy float64, BLAS threads = host cores; nothing "
                                       "extrapolated", "extrapolated": False},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if 4 in res and batches[0] != 4:
        wl4, r4 = res[4]
        v4 = r4["tokens_per_step"] / r4["median_s"]
        line["bs4"] = {"value": v4, "unit": "tok/s", "steps": r4["steps"], "ms_per_step": r4["median_s"] * 1000.0,
                       "config": {"workload": wl4.name, "batch": 4}}
    return line


# ------------------------------------------------------------------ kernel sweeps
GEMV_SWEEP_SHAPES = [(4096, 2048), (2048, 2048), (12288, 2048), (2048, 6144), (151936, 2048)]   # (N out, K in)
ATTN_SWEEP = [(B, L) for B in (1, 4, 16) for L in (256, 1024, 4096, 8192)]


def sweep() -> None:
    """Standalone kernel sweeps of the measurement plan: kmr_int4_gemv at M in {1,2,4,8,16}
    over the decoder's projection shapes and the int4 vocabulary shape, and kmr_decode_attn
    (16 q / 8 kv heads x 128) at B in {1,4,16} rows x {256,1024,4096,8192} cached positions
    (every row full).  Each point rotates through enough distinct weight / cache copies to
    exceed L2 by 2x, so every launch streams from HBM.  Prints one JSON line: per point the
    algorithmic bytes, mean launch time and achieved GB/s against the measured copy bandwidth."""
    import math
    import torch
    import int4_weight_only_group_gb300 as kmr
    peak = measured_peaks()
    hbm = peak["hbm_gbs"]
    stream = torch.cuda.current_stream()
    g = torch.Generator(device="cuda").manual_seed(0)
    gemv = []
    for N, K in GEMV_SWEEP_SHAPES:
        size = kmr.kmr_packed_size(N, K, 128)
        q = torch.randint(0, 16, (N, K), generator=g, device="cuda", dtype=torch.uint8)
        sc = (torch.rand((N, K // 128), generator=g, device="cuda") * 0.018 + 0.002).to(torch.bfloat16).view(torch.int16)
        z = (torch.randn((N, K // 128), generator=g, device="cuda") * 0.005).to(torch.bfloat16).view(torch.int16)
        one = torch.empty(size, dtype=torch.uint8, device="cuda")
        kmr.kmr_pack_int4(q, sc, z, N, K, 128, 0, one, size, 1, stream)
        del q, sc, z
        copies = max(4, math.ceil(300e6 / size))
        bufs = [one] + [one.clone() for _ in range(copies - 1)]
        for M in (1, 2, 4, 8, 16):
            x = torch.randn((M, K), generator=g, device="cuda")
            y = torch.zeros((M, N), device="cuda")
            us = launch_time_us(torch, lambda i: kmr.kmr_int4_gemv(bufs[i], N, K, 128, 0, x, M, y, kmr.KMR_EPI_NONE,
                                                                   stream), copies, 100)
            nbytes = size + M * K * 4 + M * N * 4
            gemv.append({"N": N, "K": K, "M": M, "bytes": nbytes, "us": round(us, 2),
                         "gbs": round(nbytes / (us * 1e3), 1), "frac": round(nbytes / (us * 1e3) / hbm, 3)})
        del bufs, one
    attn = []
    nq, nkv, d = 16, 8, 128
    for B, L in ATTN_SWEEP:
        per = B * nkv * L * d * 2
        copies = max(2, math.ceil(300e6 / (2 * per)))
        caches = [(torch.randn((B, nkv, L, d), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16),
                   torch.randn((B, nkv, L, d), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16))
                  for _ in range(copies)]
        qv = torch.randn((B, nq, d), generator=g, device="cuda")
        out = torch.empty((B, nq, d), device="cuda")
        slot_ids = torch.arange(B, dtype=torch.int32, device="cuda")
        cpos = torch.full((B,), L - 1, dtype=torch.int32, device="cuda")
        ws = kmr.kmr_decode_attn_workspace_size(B, nq, nkv, d)
        wsb = torch.zeros(max(ws, 1), dtype=torch.uint8, device="cuda")
        us = launch_time_us(torch, lambda i: kmr.kmr_decode_attn(qv, caches[i][0], caches[i][1], slot_ids, cpos, B, nq,
                                                                 nkv, d, L, B, 1.0 / math.sqrt(d), out, wsb, ws,
                                                                 stream), copies, 50)
        nbytes = 2 * per
        attn.append({"B": B, "cached": L, "bytes": nbytes, "us": round(us, 2),
                     "gbs": round(nbytes / (us * 1e3), 1), "frac": round(nbytes / (us * 1e3) / hbm, 3)})
        del caches
    assert kmr.kmr_last_device_error() == 0
    print(json.dumps({"sweep": {"int4_gemv": gemv, "decode_attn": attn, "peak_gbs": hbm,
                                "peak_source": peak["source"], "l2": "rotating copies > 2x L2"}}))


# ------------------------------------------------------------------ main
def projection_flop(cfg, T: int) -> float:
    """Multiply-add flops (2 per weight and token) of every layer's int4 projections over T tokens."""
    per_token = sum(n * k for n, k in cfg.linear_shapes().values())
    return 2.0 * per_token * T * cfg.n_layers


def prefill_record(r: dict, cfg, peaks: dict) -> dict:
    """The prefill object of the JSON line: the default (tcgen05) path, its projections' achieved
    flop rate against the measured bf16 dense peak (fp16 has the same nominal tensor rate), and the
    warp-level mma path beside it."""
    pf = r["prefill"]
    flop = projection_flop(cfg, pf["tokens"])
    tflops = flop / (pf["ms"] * 1e-3) / 1e12
    return {"tokens": pf["tokens"], "ms": round(pf["ms"], 3), "tok_s": round(pf["tok_s"], 1), "kernel": "tcgen05",
            "projection_tflop": round(flop / 1e12, 4), "projection_tflops_whole_prefill": round(tflops, 1),
            "frac_of_bf16_peak": round(tflops / peaks["bf16_tflops"], 3) if peaks.get("bf16_tflops") else None,
            "warp_mma_ms": round(r["prefill_mma"]["ms"], 3),
            "speedup_over_warp_mma": round(r["prefill_mma"]["ms"] / pf["ms"], 3)}


def prefill_only(T: int, mma: bool = False) -> None:
    """Two kmr_prefill calls of T seeded tokens into slot 0 of the batch-1 model (a fixed
    command for ncu launch lists of prefill), on the tcgen05 projections if asked; prints one
    status line."""
    import torch
    import int4_weight_only_group_gb300 as kmr
    from int4_weight_only_group_gb300 import driver
    from workloads import SyntheticModel
    wl = workload(1)
    cfg = wl.cfg
    model = kmr.Model.from_config(cfg, max_batch=1)
    driver.load_weights(model, SyntheticModel(cfg, wl.seed), cfg.n_layers, cfg.qk_norm)
    T = min(T, cfg.max_len)
    model.reserve_prefill(T)
    model.set_prefill_tcgen05(not mma)
    g = torch.Generator(device="cuda").manual_seed(1)
    toks = torch.randint(1, cfg.vocab - 1, (T,), generator=g, device="cuda", dtype=torch.int32)
    pos = torch.arange(T, dtype=torch.int32, device="cuda").repeat(3, 1).contiguous()
    st = [torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(3, dtype=torch.int32, device="cuda"),
          torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.uint8, device="cuda")]
    for _ in range(2):
        model.prefill(toks, pos, T, 0, 0, *st)
    torch.cuda.synchronize()
    assert model.sync_status() == 0
    model.close()
    print(json.dumps({"prefill_tokens": T, "calls": 2, "status": "ok"}))


def device_info(torch) -> dict:
    """Name and SM count of the current CUDA device and the host's core count (None when a
    value cannot be read; never raises)."""
    info = {"gpu": None, "sms": None, "host_cores": os.cpu_count()}
    try:
        prop = torch.cuda.get_device_properties(torch.cuda.current_device())
        info["gpu"], info["sms"] = prop.name, int(prop.multi_processor_count)
    except Exception:
        pass
    return info


def start_watchdog(seconds: float, on_timeout=None) -> threading.Timer:
    """A host-side watchdog: if the run has not finished after `seconds`, report it on stderr
    and end the process with status 3 instead of leaving it hanging (device waits are bounded
    already; this covers the host).  Cancel the returned timer when the run is done."""
    def fire():
        print(json.dumps({"error": f"bench watchdog: no result after {seconds:.0f} s"}), file=sys.stderr, flush=True)
        (on_timeout or (lambda: os._exit(3)))()
    t = threading.Timer(seconds, fire)
    t.daemon = True
    t.start()
    return t


def step_figures(r, args, peaks) -> dict:
    """tok/s, per-step times and the step's algorithmic bytes against the measured peak, from
    the KV the timed steps actually read."""
    wl = r["wl"]
    cfg = wl.cfg
    ms = r["elapsed_ms"] / args.steps
    wb = weight_bytes(cfg)
    step_weight_bytes = cfg.n_layers * (wb["qkv"] + wb["o"] + wb["gate_up"] + wb["down"]) + wb["lm_head"] + wb["norms"]
    step_bytes = step_weight_bytes + r["kv_timed"] / args.steps
    return {
        "value": r["tokens"] / (r["elapsed_ms"] / 1000.0), "ms_per_step": ms,
        "step_ms": {k: (round(v, 5) if isinstance(v, float) else v) for k, v in r["step_ms"].items()},
        "step_roofline": {"bytes_per_step": step_bytes, "weight_bytes_per_step": step_weight_bytes,
                          "kv_bytes_per_step": r["kv_timed"] / args.steps, "achieved_gbs": step_bytes / (ms * 1e6),
                          "frac": step_bytes / (ms * 1e6) / peaks["hbm_gbs"],
                          "roofline_ms_per_step": step_bytes / (peaks["hbm_gbs"] * 1e6),
                          "kv": "positions 0..cache_position of every active row in the timed steps"},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--batch", type=int, default=None, choices=(1, 4, 16),
                    help="time only this batch (default: batch 1 headline plus a batch-4 'bs4' object)")
    ap.add_argument("--impl", default="kmr", choices=("kmr", "reference"))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-suite", action="store_true",
                    help="also time the 28-layer oracle legs on one thread and batch 4 on all cores")
    ap.add_argument("--persistent-step", action="store_true",
                    help="run the step's layers as the persistent kernel (opt-in) instead of one kernel per phase")
    ap.add_argument("--skip-extras", action="store_true",
                    help="time only the decode steps (no standalone GEMV timing, e2e or CPU legs; for launch lists)")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="T",
                    help="only run two T-token prefills on the batch-1 model and exit (for profiling)")
    ap.add_argument("--prefill-mma", action="store_true",
                    help="with --prefill-only: run the projections on the warp-level mma kernel")
    ap.add_argument("--sweep", action="store_true",
                    help="only run the standalone int4 GEMV and decode-attention sweeps and exit")
    ap.add_argument("--oracle-leg", choices=tuple(ORACLE_LEGS), default=None,
                    help="(internal) time whole oracle steps of one workload and print one JSON line")
    ap.add_argument("--oracle-steps", type=int, default=3)
    ap.add_argument("--oracle-budget-s", type=float, default=30.0)
    ap.add_argument("--watchdog-s", type=float, default=1800.0,
                    help="end the run with status 3 if it has not finished after this many seconds")
    args = ap.parse_args()
    watchdog = start_watchdog(args.watchdog_s)
    try:
        _main(args)
    finally:
        watchdog.cancel()


def _main(args):
    if args.oracle_leg:
        print(json.dumps(oracle_leg(args.oracle_leg, args.oracle_steps, args.oracle_budget_s)))
        return
    if args.sweep:
        sweep()
        return
    if args.prefill_only:
        prefill_only(args.prefill_only, args.prefill_mma)
        return
    if args.skip_extras:
        args.no_cpu_baseline = True
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    head_b = args.batch or 1
    r = run_kmr(args, head_b, rank, world, extras=True)
    r4 = run_kmr(args, 4, rank, world, extras=False) if args.batch is None else None
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    peaks = measured_peaks()
    if args.skip_extras:
        out = {"ms_per_step": r["elapsed_ms"] / args.steps, "steps": args.steps,
               "kernels_per_step": r["kernels_per_step"], "step_ms": r["step_ms"]}
        if r4:
            out["bs4_ms_per_step"] = r4["elapsed_ms"] / args.steps
            out["bs4_kernels_per_step"] = r4["kernels_per_step"]
        print(json.dumps(out))
        return
    wl = r["wl"]
    cfg = wl.cfg
    f = step_figures(r, args, peaks)
    g = r["gemv"]["gate_up"]
    traffic = profile_traffic("int4_gemv_gate_up.md")
    line = {
        "metric": METRIC, "value": f["value"], "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": f["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4w/bf16->f32",
        "data": "synthetic (seeded; shapes and distributions of the workload recipe)",
        "config": {"workload": wl.name, "batch": wl.batch, "kv_max_len": cfg.max_len, "prefill": wl.prefill,
                   "steps_per_generation": wl.steps, "l2": "inputs larger than L2 (1.4 GB of weights per step)",
                   "parallelism": "replicas" if args.gpus > 1 else "single-gpu"},
        "step_ms": f["step_ms"],
        "roofline": {"bound": "hbm", "kernel": "int4_gemv (gate_up shape, M=%d)" % wl.batch,
                     "achieved": g["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": g["gbs"] / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": peaks["source"]},
        "step_roofline": f["step_roofline"],
        "gemv_us": {k: round(v["us"], 2) for k, v in r["gemv"].items()},
        "gemv_gbs": {k: round(v["gbs"], 1) for k, v in r["gemv"].items()},
        "e2e": r["e2e"],
        "memory": r["memory"],
        "cascade_attn": {"rows": r["cascade"]["rows"], "prefix": r["cascade"]["prefix"], "own": r["cascade"]["own"],
                         "cascade_us": round(r["cascade"]["cascade"]["us"], 2),
                         "plain_us": round(r["cascade"]["plain"]["us"], 2),
                         "cascade_kv_bytes": r["cascade"]["cascade"]["kv_bytes"],
                         "plain_kv_bytes": r["cascade"]["plain"]["kv_bytes"]},
        "prefill": prefill_record(r, cfg, peaks),
        "kv_row_copy": {"us": round(r["kv_copy"]["us"], 2), "gbs": round(r["kv_copy"]["gbs"], 1),
                        "frac": round(r["kv_copy"]["gbs"] / peaks["hbm_gbs"], 3), "bytes": r["kv_copy"]["bytes"]},
        "gpu_launches": r["kernels_per_step"] * args.steps,
        "clocks": r["clocks"],
        "device": device_info(torch),
        "setup_s": round(r["setup_s"], 1),
        "context": {"pages_decode_tok_s": 100.6, "pages_peak_vram_gb": 2.3,
                    "note": "the pages' own figures (RTX 3050 6 GB, torch.compile + torchao, real Qwen3-VL-2B): "
                            "context only, another machine and model; vs_baseline stays null"},
    }
    if r4:
        f4 = step_figures(r4, args, peaks)
        line["bs4"] = {"value": f4["value"], "unit": "tok/s", "ms_per_step": f4["ms_per_step"],
                       "step_ms": f4["step_ms"], "step_roofline": f4["step_roofline"], "e2e": r4["e2e"],
                       "memory": r4["memory"], "clocks": r4["clocks"],
                       "gpu_launches": r4["kernels_per_step"] * args.steps,
                       "config": {"workload": r4["wl"].name, "batch": 4, "prefill": r4["wl"].prefill,
                                  "steps_per_generation": r4["wl"].steps}}
    if "cpu" in r:
        line["cpu_baseline"] = r["cpu"]
        line["cpu_baseline"]["gpu_over_cpu"] = f["value"] / r["cpu"]["value"]
    print(json.dumps(line))


if __name__ == "__main__":
    main()
