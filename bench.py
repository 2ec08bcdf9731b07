"""Decode-step benchmark: tokens/s and achieved HBM bandwidth on one GB300.

Default workload (N = 1): the full 24-layer Qwen2-0.5B-shaped model with
seeded random bf16 weights, batch 1, a 32-token prompt run through the decode
step, then greedy decoding of 64 tokens (positions 32..95) on a contiguous KV
cache. One timed step is one decode step (all layers plus the LM head and the
arg-max) through nc_decode_step, which at this batch runs the whole step as
one persistent cooperative kernel launch. The 64-token sequence is decoded
repeatedly: timed step i runs at position 32 + (i mod 64), and every 64 steps
the sequence restarts (an 8-byte host-to-device reset of token and position).

Printed (rank 0, one JSON line): the contract keys plus `roofline` (the step
kernel vs the measured HBM copy peak), `cpu_baseline` (the CPU oracle on the
host cores, bounded sample), `e2e` (host buffers, copies inside the timed
region), `hbm` (algorithmic bytes per step over step time) and `clocks`.

--workload picks one of the other measured configurations instead (batch 16
on a paged cache, W8A8, the 8B shape; see WORKLOADS): the same JSON line,
without the CPU baseline.

--workload qwen2_0p5b_b1_sampled64 is the default workload with nanoinfer's
sampler (temperature 0.7, top-k 20, top-p 0.8, the values the page reads from
Qwen2.5's config) in place of greedy: each step is nc_decode_step then
nc_sample on its logits, the sampled token fed back on the device; the line
adds the sampler kernel's own average duration.

--impl reference times the CPU oracle itself on the default workload (the
reference arm of this build).
Multi-GPU (torchrun, N > 1): replicas only, one independent model per GPU, no
collective on the data path; value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_decode_gb300 import nc, synth  # noqa: E402

METRIC = "decode tokens/s at 1 GB300 and achieved HBM GB/s as fraction of ~8 TB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "qwen3_8b_shape_b1_past4096"  # the largest single-GPU configuration
C1 = "qwen2_0p5b_b1_greedy64"            # the 0.5B model, 32-token prompt, 64 greedy


# ---------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def step_bytes(shape, batch, positions, kv_elem=4, w8a8=False, int8_head=False,
               int4_group=0):
    """Algorithmic HBM bytes of one decode step: every weight byte once, the
    embedding rows, K/V of slots 0..p read once per layer and kv head, the new
    K/V written, the logits written and tokens/positions read. kv_elem is the
    cache element size (4: fp32 cache, 2: bf16); w8a8: the seven projections
    are int8 with one fp32 scale per output row (the LM head stays bf16);
    int8_head: the tied embedding / head rows are int8 with one fp32 scale
    each too. int4_group: the projections are INT4, half a byte a weight and
    one fp32 scale per group of that many weights."""
    H, D, F, L, V = shape.hidden, shape.head_dim, shape.ffn, shape.n_layers, shape.vocab
    nqkv = shape.q_dim + 2 * shape.kv_dim
    if int4_group:
        g = int4_group
        per_layer = (nqkv * H + shape.q_dim * H + 2 * F * H + H * F) // 2 + 4 * (
            nqkv * (H // g) + H * (shape.q_dim // g) + 2 * F * (H // g) + H * (F // g))
    elif w8a8:
        per_layer = (nqkv * H + shape.q_dim * H + 2 * F * H + H * F) + 4 * (nqkv + H + 2 * F + H)
    else:
        per_layer = 2 * (nqkv * H + shape.q_dim * H + 2 * F * H + H * F)
    per_layer += 2 * 2 * H
    if shape.qkv_bias:
        per_layer += 2 * nqkv
    if shape.qk_norm:
        per_layer += 2 * 2 * D
    head = (V * H + 4 * V if int8_head else 2 * V * H) + 2 * H
    emb = (H + 4 if int8_head else 2 * H) * batch
    kv_row = 2 * shape.kv_dim * kv_elem  # K and V of one position, one layer
    kv_read = sum((p + 1) for p in positions) * L * kv_row
    kv_write = batch * L * kv_row
    return L * per_layer + head + emb + kv_read + kv_write + 4 * V * batch + 8 * batch


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.15]
        use = inside if inside else [min(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))] if rows else []
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in use for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        pw = [float(p[3]) for _, p in use if p[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(use),
                "samples_in_timed_region": len(inside)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v):
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(ws, batch, steps, local_seconds):
    """Whole-job tokens/s of `ws` independent replicas, each decoding `batch`
    sequences for `steps` steps: every rank's tokens over the slowest rank's
    time (the max over ranks). Returns (rate, max_seconds)."""
    el = max_over_ranks(ws, local_seconds)
    return ws * batch * steps / el, el


# ---------------------------------------------------------------- CPU oracle
def c1_oracle(shape, prompt, n_gen):
    """The oracle on the 0.5B prompt run: the model, and a cache that has
    taken the prompt's first 31 tokens (positions 0..30) as decode steps."""
    import oracle
    oracle.build()
    om = oracle.OracleModel(shape, cpu_weights(shape))
    kv = om.new_kv(1, len(prompt) + n_gen + 1)
    for i in range(len(prompt) - 1):
        om.decode_step(kv, np.array([prompt[i]], np.int32), np.array([i], np.int32))
    return om, kv


def cpu_baseline_c1(shape, prompt, cycle, seconds):
    """The oracle as it stands on the host cores, on the positions the GPU
    times (cycles of 65 steps at positions 31..95 after the untimed prompt):
    all cores of the affinity mask until `seconds` of work; and one thread,
    block 0 and the LM head product at position 31, scaled to a step."""
    import oracle
    n_prompt = len(prompt)
    om, kv = c1_oracle(shape, prompt, cycle - 1)
    threads = oracle.get_threads()
    cur = prompt[-1]
    t0 = time.perf_counter()
    n = 0
    while True:
        if n % cycle == 0:
            cur = prompt[-1]
        p = n_prompt - 1 + (n % cycle)
        _, nxt = om.decode_step(kv, np.array([cur], np.int32), np.array([p], np.int32))
        cur = int(nxt[0])
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    oracle.set_threads(1)
    x = synth.normal_bf16(0, 9999, (shape.hidden,), 1.0).float().numpy()
    t1 = time.perf_counter()
    om.block_decode(0, kv, 0, n_prompt - 1, x)
    t_block = time.perf_counter() - t1
    t1 = time.perf_counter()
    oracle.matvec_bf16(om.head_w, x)
    t_head = time.perf_counter() - t1
    oracle.set_threads(threads)
    return {"value": n / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "cpu": cpu_model_name(),
            "sample": f"{n} decode steps at the timed positions ({n_prompt - 1}..), "
                      f"{el:.1f} s on {threads} threads of {cpu_threads()} host cores",
            "one_thread": {"value": 1.0 / (shape.n_layers * t_block + t_head),
                           "unit": "tokens/s", "cores": 1,
                           "sample": f"block 0 ({t_block:.3f} s) and the LM head product "
                                     f"({t_head:.3f} s) on one thread, scaled to "
                                     f"{shape.n_layers} blocks + head"}}


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------- reference arm
REFERENCE_SECONDS = 150.0  # the reference arm's timed work stops here


def run_reference(args, ws, rank):
    """The CPU oracle on the bench workload, on the positions our arm times: a
    few untimed warm-up steps, then timed decode steps of the workload's cycle,
    at most args.steps of them and at most REFERENCE_SECONDS of work. For the
    0.5B prompt run the prompt's first 31 tokens run untimed first and the
    cycle is positions 31..95."""
    if rank != 0:
        return
    import oracle
    name = args.workload
    if name == SAMPLED:
        name = C1
    if name in PREFILLS:
        cfg = PREFILLS[name]
        shape = getattr(synth, cfg["shape"])
        T = cfg["T"]
        oracle.build()
        om = oracle.OracleModel(shape, cpu_weights(shape))
        okv = om.new_kv(1, T + 1)
        toks = synth.token_ids(T, shape.vocab).numpy().astype(np.int32)

        def step(i):
            om.forward_chunk(okv, 0, toks, 0)
        batch = T
        config = {"workload": name, "prompt_tokens": T, "start": 0}
    elif name == C1:
        shape = synth.QWEN2_0P5B
        n_prompt, n_gen = 32, 64
        prompt = synth.token_ids(n_prompt, shape.vocab).tolist()
        om, kv = c1_oracle(shape, prompt, n_gen)
        cycle = n_gen + 1
        cur = prompt[-1]

        def step(i):
            nonlocal cur
            if i % cycle == 0:
                cur = prompt[-1]
            p = n_prompt - 1 + (i % cycle)
            _, nxt = om.decode_step(kv, np.array([cur], np.int32), np.array([p], np.int32))
            cur = int(nxt[0])
        batch = 1
        config = {"workload": C1, "batch": 1, "prompt": n_prompt,
                  "positions": f"cycles of {cycle} steps at positions {n_prompt - 1}.."
                               f"{n_prompt + n_gen - 1}"}
    else:
        cfg = WORKLOADS[name]
        batch = cfg["batch"]
        om, okv, past = oracle_for(cfg, max(workload_past(cfg)) + cfg["gen"] + 1)

        def step(i):
            oracle_workload_steps(om, okv, cfg, past, i, 0.0, 1)
        config = {"workload": name, "batch": batch, "past": cfg["past"],
                  "positions": f"cycles of {cfg['gen']} greedy steps from the past length(s)"}
    config["note"] = "CPU oracle (plain C, fp32, OpenMP over output rows)"
    warm = min(args.warmup, 3)
    for i in range(warm):
        step(i)
    t0 = time.perf_counter()
    n = 0
    while n < args.steps:
        step(warm + n)
        n += 1
        if time.perf_counter() - t0 >= REFERENCE_SECONDS:
            break
    el = time.perf_counter() - t0
    thr = oracle.get_threads()
    value = batch * n / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": n, "steps_requested": args.steps, "warmup": warm,
        "ms_per_step": el / n * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "cpu": cpu_model_name(),
                         "sample": f"{n} timed decode steps of the workload (of "
                                   f"{args.steps} requested; at most {REFERENCE_SECONDS:.0f} s), "
                                   f"{el:.1f} s on {thr} threads of {cpu_threads()} host cores"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- our arm
PERSISTENT_SRC = os.path.join(ROOT, "transformer_decode_gb300", "csrc", "persistent.cu")


def counted_traffic(name):
    """DRAM bytes per launch of the step kernel from the committed ncu summary
    of workload `name` (dram__bytes_read.sum + dram__bytes_write.sum of one
    capture), or None when there is none or the kernel source changed since
    (the summary records the source's sha256)."""
    path = TRAFFIC_FILES.get(name)
    if not path or not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.strip().startswith(("source_sha256", "dram_bytes_per_launch")):
            k, v = line.strip().split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    src = hashlib.sha256(open(PERSISTENT_SRC, "rb").read()).hexdigest()
    if fields.get("source_sha256") != src or "dram_bytes_per_launch" not in fields:
        return None
    return float(fields["dram_bytes_per_launch"])


def run_nc(args, ws, rank, local):
    torch.cuda.set_device(local)
    shape = synth.QWEN2_0P5B
    B, n_prompt, n_gen = 1, 32, 64
    wd = synth.model_weights(shape, device="cuda")
    max_ctx = n_prompt + n_gen + 16
    model = nc.Model(shape, wd, max_batch=B, max_ctx=max_ctx)
    kv = nc.KVCache(shape, B, max_ctx=max_ctx)
    logits = torch.empty(B, shape.vocab, device="cuda")
    prompt = synth.token_ids(n_prompt, shape.vocab).tolist()
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    reset_host = torch.tensor([prompt[-1], n_prompt - 1], dtype=torch.int32).pin_memory()

    # prompt: each prompt token runs as one decode step (positions 0..30); the
    # last prompt token (position 31) opens every decode cycle below
    pos.fill_(0)
    for i in range(n_prompt - 1):
        tok.fill_(prompt[i])
        model.decode_step(tok, pos, [i], kv, logits, use_graph=True, advance=True)
    # A cycle is 65 decode steps at positions 31..95: the last prompt token
    # (set from the host, 8 bytes) then 64 greedy tokens fed back on the device.
    cycle = n_gen + 1

    def run_steps(k, off=0):
        """k decode steps of repeated cycles, from cycle step off; returns the
        positions used."""
        used = []
        for i in range(off, off + k):
            p = n_prompt - 1 + (i % cycle)
            if i % cycle == 0:
                tok.copy_(reset_host[:1], non_blocking=True)
                pos.copy_(reset_host[1:], non_blocking=True)
            model.decode_step(tok, pos, [p], kv, logits, use_graph=True, advance=True)
            used.append(p)
        return used

    run_steps(args.warmup)
    torch.cuda.synchronize()
    if args.phase_profile:
        print_phase_profile(model, shape, run_steps, model.decode_path(B, kv), args.phase_dump)

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    st = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    w0 = time.time()
    total_s, per_round, used = timed_rounds(st, run_steps, args.steps)
    w1 = time.time()
    barrier(ws)
    if rank == 0:
        time.sleep(0.2)
        sampler.stop()
    value, el = replica_rate(ws, B, args.steps, total_s)
    restarts = sum(1 for i in range(args.steps) if i % cycle == 0)
    ms = el / args.steps * 1e3
    bytes_avg = sum(step_bytes(shape, B, [p]) for p in used) / len(used)
    hbm_gbs = bytes_avg / (el / args.steps) / 1e9
    peak, peak_kind = peaks()

    # ---- e2e: public API with host buffers, copies inside the timed region
    tok_h = torch.empty(B, dtype=torch.int32).pin_memory()
    pos_h = torch.empty(B, dtype=torch.int32).pin_memory()
    nxt_h = torch.empty(B, dtype=torch.int32).pin_memory()
    nxt_d = torch.empty(B, dtype=torch.int32, device="cuda")
    # warm the (tokens, positions, logits, next) graph of this buffer set
    tok_h[0] = prompt[-1]
    pos_h[0] = n_prompt - 1
    tok.copy_(tok_h)
    pos.copy_(pos_h)
    model.decode_step(tok, pos, [n_prompt - 1], kv, logits, nxt_d, use_graph=True)
    torch.cuda.synchronize()
    k_e2e = min(args.steps, 520)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cur_tok = prompt[-1]
    for i in range(k_e2e):
        p = n_prompt - 1 + (i % cycle)
        if i % cycle == 0:
            cur_tok = prompt[-1]
        tok_h[0] = cur_tok
        pos_h[0] = p
        tok.copy_(tok_h, non_blocking=True)
        pos.copy_(pos_h, non_blocking=True)
        model.decode_step(tok, pos, [p], kv, logits, nxt_d, use_graph=True)
        nxt_h.copy_(nxt_d, non_blocking=True)
        st.synchronize()
        cur_tok = int(nxt_h[0])
    e2e_value, t_e2e = replica_rate(ws, B, k_e2e, time.perf_counter() - t0)

    # ---- the step kernel: one launch per timed step, so its average launch
    # duration is the timed region over the steps (CUDA events on its stream;
    # the region holds only these launches and the 8-byte cycle resets)
    path = model.decode_path(B, kv)
    launches_per_step = step_launches(path, shape, B, {"w8a8": False})
    dur = el / args.steps
    achieved = bytes_avg / dur / 1e9

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_c1(shape, prompt, cycle, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": C1, "batch": B, "prompt": n_prompt,
                       "positions": f"cycles of {cycle} steps at positions {n_prompt - 1}.."
                                    f"{n_prompt + n_gen - 1} ({restarts} cycles timed)",
                       "weights": "bf16 seeded N(0,0.02) stand-in, fp32 accumulate",
                       "kv": "contiguous fp32",
                       "path": ("nc_decode_step: one persistent cooperative launch per step"
                                if path == "persistent" else "nc_decode_step: stage kernels, CUDA graph"),
                       "l2": "inputs larger than L2: 988 MB of weights stream every step",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "rounds": rounds_summary(per_round),
            "hbm": {"bytes_per_step": bytes_avg, "gbs": hbm_gbs,
                    "frac_of_8tbs": hbm_gbs / NOMINAL_HBM_GBS,
                    "frac_of_measured_copy": hbm_gbs / peak, "peak_kind": peak_kind},
            "roofline": {"bound": "hbm",
                         "kernel": ("k_decode_persistent<1,64,fp32 KV> (the whole step)"
                                    if path == "persistent" else "stage kernels (whole step)"),
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": counted_traffic(C1) if path == "persistent" else None,
                         "peak_kind": peak_kind, "avg_launch_us": dur * 1e6,
                         "algorithmic_bytes_per_launch": bytes_avg},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "steps": k_e2e,
                    "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 4 * B},
            "gpu_launches": args.steps * launches_per_step,
            "clocks": sampler.summary(w0, w1),
        }
        print(json.dumps(line), flush=True)
    model.close()


SAMPLED = "qwen2_0p5b_b1_sampled64"
SAMPLER = dict(temperature=0.7, top_k=20, top_p=0.8)


def run_sampled(args, ws, rank, local):
    """The default workload, each step followed by nc_sample (temperature 0.7,
    top-k 20, top-p 0.8) whose token replaces the greedy one on the device."""
    torch.cuda.set_device(local)
    shape = synth.QWEN2_0P5B
    B, n_prompt, n_gen = 1, 32, 64
    wd = synth.model_weights(shape, device="cuda")
    max_ctx = n_prompt + n_gen + 16
    model = nc.Model(shape, wd, max_batch=B, max_ctx=max_ctx)
    kv = nc.KVCache(shape, B, max_ctx=max_ctx)
    logits = torch.empty(B, shape.vocab, device="cuda")
    prompt = synth.token_ids(n_prompt, shape.vocab).tolist()
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    reset_host = torch.tensor([prompt[-1], n_prompt - 1], dtype=torch.int32).pin_memory()
    samp = nc.Sampler(B, shape.vocab)
    n_u = args.warmup + args.steps + 256
    u = synth.uniform_f64(5, 0, n_u * B, device="cuda").view(n_u, B)
    pos.fill_(0)
    for i in range(n_prompt - 1):
        tok.fill_(prompt[i])
        model.decode_step(tok, pos, [i], kv, logits, use_graph=True, advance=True)
    cycle = n_gen + 1
    T, K, P = SAMPLER["temperature"], SAMPLER["top_k"], SAMPLER["top_p"]

    def run_steps(k, off):
        used = []
        for i in range(k):
            p = n_prompt - 1 + (i % cycle)
            if i % cycle == 0:
                tok.copy_(reset_host[:1], non_blocking=True)
                pos.copy_(reset_host[1:], non_blocking=True)
            model.decode_step(tok, pos, [p], kv, logits, use_graph=True, advance=True)
            samp(logits, T, K, P, u[off + i], tok)
            used.append(p)
        return used

    run_steps(args.warmup, 0)
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    if rank == 0:
        clk.start()
        time.sleep(0.3)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    w0 = time.time()
    e0.record(st)
    used = run_steps(args.steps, args.warmup)
    e1.record(st)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(ws)
    if rank == 0:
        time.sleep(0.2)
        clk.stop()
    value, el = replica_rate(ws, B, args.steps, e0.elapsed_time(e1) / 1e3)
    bytes_avg = sum(step_bytes(shape, B, [p]) for p in used) / len(used)
    peak, peak_kind = peaks()

    # the sampler alone, on the last step's logits (already in L2: the LM head wrote them)
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    kept = torch.empty(B, 2, dtype=torch.int32, device="cuda")
    for i in range(8):
        samp(logits, T, K, P, u[i], nxt, kept)
    n_s = 256
    torch.cuda.synchronize()
    e0.record(st)
    for i in range(n_s):
        samp(logits, T, K, P, u[i], nxt, kept)
    e1.record(st)
    torch.cuda.synchronize()
    samp_us = e0.elapsed_time(e1) / n_s * 1e3

    # e2e: host token and position in, the sampled token out, every step
    tok_h = torch.empty(B, dtype=torch.int32).pin_memory()
    pos_h = torch.empty(B, dtype=torch.int32).pin_memory()
    nxt_h = torch.empty(B, dtype=torch.int32).pin_memory()
    k_e2e = min(args.steps, 520)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cur = prompt[-1]
    for i in range(k_e2e):
        p = n_prompt - 1 + (i % cycle)
        if i % cycle == 0:
            cur = prompt[-1]
        tok_h[0] = cur
        pos_h[0] = p
        tok.copy_(tok_h, non_blocking=True)
        pos.copy_(pos_h, non_blocking=True)
        model.decode_step(tok, pos, [p], kv, logits, use_graph=True)
        samp(logits, T, K, P, u[i % n_u], nxt)
        nxt_h.copy_(nxt, non_blocking=True)
        st.synchronize()
        cur = int(nxt_h[0])
    e2e_value, t_e2e = replica_rate(ws, B, k_e2e, time.perf_counter() - t0)

    path = model.decode_path(B, kv)
    launches = (1 if path == "persistent" else 2 + 5 * shape.n_layers) + 1
    if rank == 0:
        dur = el / args.steps
        row_bytes = B * shape.vocab * 4
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dur * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": SAMPLED, "batch": B, "prompt": n_prompt,
                       "sampler": dict(SAMPLER, u="seeded uniforms, one per step"),
                       "path": f"nc_decode_step ({path}) then nc_sample",
                       "l2": "inputs larger than L2: 988 MB of weights stream every step",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": "decode step + sampler (whole step)",
                         "achieved": bytes_avg / dur / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": bytes_avg / dur / 1e9 / peak, "traffic": None,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": bytes_avg},
            "sampler": {"kernel": "k_sample (one CTA of 1024 threads per row)",
                        "avg_us": samp_us, "share_of_step": samp_us * 1e-6 / dur,
                        "logit_bytes": row_bytes, "gbs": row_bytes / (samp_us * 1e-6) / 1e9,
                        "bound": "latency (one row per CTA; the logits sit in L2)"},
            "cpu_baseline": None,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "steps": k_e2e,
                    "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 4 * B},
            "gpu_launches": args.steps * launches,
            "clocks": clk.summary(w0, w1),
        }), flush=True)
    model.close()


# Measured configurations other than the 0.5B prompt run: name -> setup.
# Past K/V are the seeded synthetic rows the tests use; each timed cycle runs
# `gen` greedy steps from the past lengths, then the host resets tokens and
# positions (B x 8 bytes). The first is the metric's workload: the largest
# single-GPU configuration, the 8B shape at 4096 past positions.
WORKLOADS = {
    "qwen3_8b_shape_b1_past4096": dict(shape="QWEN3_8B", batch=1, paged=False, past=4096,
                                       gen=64, w8a8=False),
    "qwen2_0p5b_b16_paged_past256-4096": dict(shape="QWEN2_0P5B", batch=16, paged=True,
                                              past="uniform 256..4096", gen=32, w8a8=False),
    "qwen2_0p5b_w8a8_b1_past512": dict(shape="QWEN2_0P5B", batch=1, paged=False, past=512,
                                       gen=64, w8a8=True),
    "qwen2_0p5b_w8a8_b32_b1_past512": dict(shape="QWEN2_0P5B", batch=1, paged=False, past=512,
                                           gen=64, w8a8="b32"),
    "qwen2_0p5b_int4_g128_b1_past512": dict(shape="QWEN2_0P5B", batch=1, paged=False,
                                            past=512, gen=64, w8a8=False, int4=128),
    # the 8B shape with a bf16 cache (the bytes of the 70%-of-8-TB/s target)
    "qwen3_8b_shape_b1_past4096_kvbf16": dict(shape="QWEN3_8B", batch=1, paged=False,
                                              past=4096, gen=64, w8a8=False, kv_bf16=True),
}
ROUNDS = 5  # the timed region is reported as this many equal rounds as well

# ncu DRAM summaries of the step kernel (one capture each), by workload
TRAFFIC_FILES = {
    WORKLOAD: os.path.join(ROOT, "profiles", "k_decode_persistent_qwen3_8b_shape_b1_past4096_dram.md"),
    C1: os.path.join(ROOT, "profiles", "k_decode_persistent_qwen2_0p5b_b1_dram.md"),
}


def workload_past(cfg):
    B = cfg["batch"]
    return (synth.past_lengths(B, 256, 4096).tolist() if isinstance(cfg["past"], str)
            else [cfg["past"]] * B)


def fill_past(kv, shape, past):
    """Seeded synthetic K/V rows into slots 0..p-1 of every (layer, sequence, kv head)."""
    D = shape.head_dim
    for l in range(shape.n_layers):
        for b, p in enumerate(past):
            if p == 0:
                continue
            for g in range(shape.n_kv_heads):
                kr = synth.synthetic_kv_rows(shape, l, b, g, 0, p, device="cuda")
                vr = synth.synthetic_kv_rows(shape, l, b, g, 1, p, device="cuda")
                if not kv.paged:
                    kv.k[l, b, g, :p] = kr.to(kv.k.dtype).view(p, D)
                    kv.v[l, b, g, :p] = vr.to(kv.v.dtype).view(p, D)
                else:
                    t = torch.arange(p, device="cuda")
                    blk = kv.table[b, t // kv.block_size].long()
                    kv.k[l, blk, g, t % kv.block_size] = kr.to(kv.k.dtype).view(p, D)
                    kv.v[l, blk, g, t % kv.block_size] = vr.to(kv.v.dtype).view(p, D)


def cpu_weights(shape):
    """The seeded weights as CPU tensors, drawn on the GPU when there is one
    (the generator gives the same bits on either device; drawing 8B-shaped
    weights on the host takes many minutes)."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wd = synth.model_weights(shape, device=dev)
    wc = {k: (None if v is None else v.cpu()) for k, v in wd.items() if k != "layers"}
    wc["layers"] = [{k: (None if v is None else v.cpu()) for k, v in lw.items()}
                    for lw in wd["layers"]]
    del wd
    return wc


def oracle_for(cfg, max_ctx):
    """The CPU oracle on the workload: its model and a logical cache holding
    the same synthetic past rows as the GPU cache."""
    import oracle
    oracle.build()
    shape = getattr(synth, cfg["shape"])
    if cfg.get("layers"):
        shape = shape.with_layers(cfg["layers"])
    past = workload_past(cfg)
    om = oracle.OracleModel(shape, cpu_weights(shape), w8a8=bool(cfg["w8a8"]),
                            act_block=32 if cfg["w8a8"] == "b32" else 0,
                            int8_embed=cfg["w8a8"] == "b32", int4_group=cfg.get("int4", 0))
    okv = om.new_kv(cfg["batch"], max_ctx, bf16=bool(cfg.get("kv_bf16")))
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    for l in range(shape.n_layers):
        for b, p in enumerate(past):
            if p == 0:
                continue
            for g in range(shape.n_kv_heads):
                kr = synth.synthetic_kv_rows(shape, l, b, g, 0, p, device=dev)
                vr = synth.synthetic_kv_rows(shape, l, b, g, 1, p, device=dev)
                okv.k[l, b, g, :p] = oracle_rows(kr, okv.bf16, p)
                okv.v[l, b, g, :p] = oracle_rows(vr, okv.bf16, p)
    return om, okv, past


def oracle_rows(t, bf16, p):
    """Synthetic K/V rows as the oracle cache holds them: fp32 values, or the
    bf16 bits (uint16) of a bf16 cache."""
    if bf16:
        return t.to(torch.bfloat16).contiguous().view(torch.int16).cpu().numpy().view(np.uint16).reshape(p, -1)
    return t.float().cpu().numpy().reshape(p, -1)


def cpu_model_name():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_workload_steps(om, okv, cfg, past, start, seconds, max_steps):
    """Decode steps of the workload's cycle (greedy, `gen` steps from the past
    lengths) on the oracle, from cycle step `start`, until `seconds` of work
    or `max_steps` steps. Returns (steps, elapsed_s)."""
    B, gen = cfg["batch"], cfg["gen"]
    shape = om.shape
    past_np = np.array(past, np.int32)
    tok = synth.token_ids(B, shape.vocab, stream=77).numpy().astype(np.int32)
    t0 = time.perf_counter()
    n = 0
    while n < max_steps:
        j = (start + n) % gen
        if j == 0:
            tok = synth.token_ids(B, shape.vocab, stream=77).numpy().astype(np.int32)
        _, nxt = om.decode_step(okv, tok, past_np + j)
        tok = nxt.astype(np.int32)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return n, time.perf_counter() - t0


def cpu_baseline_for(cfg, seconds):
    """The oracle as it stands on the GPU machine's host cores, on the workload's
    own positions: (a) all cores of the affinity mask, whole decode steps of
    the cycle until `seconds` of work; (b) one thread, one block and the LM
    head at the cycle's first position, scaled to a step (L blocks + head)."""
    import oracle
    om, okv, past = oracle_for(cfg, max(workload_past(cfg)) + cfg["gen"] + 1)
    shape = om.shape
    B = cfg["batch"]
    threads = oracle.get_threads()
    n, el = oracle_workload_steps(om, okv, cfg, past, 0, seconds, 10 ** 6)
    all_rate = B * n / el
    # one thread: block 0 of every sequence plus the head product, scaled
    oracle.set_threads(1)
    x = synth.normal_bf16(0, 9999, (shape.hidden,), 1.0).float().numpy()
    t0 = time.perf_counter()
    for b in range(B):
        om.block_decode(0, okv, b, past[b], x)
    t_block = time.perf_counter() - t0
    t0 = time.perf_counter()
    for b in range(B):
        oracle.matvec_bf16(om.head_w, x)
    t_head = time.perf_counter() - t0
    oracle.set_threads(threads)
    one_rate = B / (shape.n_layers * t_block + t_head)
    return {
        "value": all_rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
        "cpu": cpu_model_name(),
        "sample": f"{n} decode steps of the workload's cycle (batch {B}, from past "
                  f"{'..'.join(str(p) for p in sorted(set([min(past), max(past)])))}), "
                  f"{el:.1f} s on {threads} threads of {cpu_threads()} host cores",
        "one_thread": {"value": one_rate, "unit": "tokens/s", "cores": 1,
                       "sample": f"block 0 ({t_block:.2f} s) and the LM head product "
                                 f"({t_head:.2f} s) for {B} sequence(s) on one thread, "
                                 f"scaled to {shape.n_layers} blocks + head"},
    }


def timed_rounds(st, run_steps, steps, rounds=ROUNDS):
    """Run `steps` steps as `rounds` equal rounds inside one timed region, with
    CUDA events on stream st at every round boundary. Returns (total_s,
    [per-round ms per step], positions used)."""
    cuts = [round(steps * r / rounds) for r in range(rounds + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(rounds + 1)]
    used = []
    ev[0].record(st)
    for r in range(rounds):
        used += run_steps(cuts[r + 1] - cuts[r], cuts[r])
        ev[r + 1].record(st)
    torch.cuda.synchronize()
    per = [ev[r].elapsed_time(ev[r + 1]) / max(1, cuts[r + 1] - cuts[r])
           for r in range(rounds) if cuts[r + 1] > cuts[r]]
    return ev[0].elapsed_time(ev[rounds]) / 1e3, per, used


def rounds_summary(per):
    med = statistics.median(per)
    return {"n": len(per), "ms_per_step": [round(v, 5) for v in per], "median_ms": med,
            "min_ms": min(per), "max_ms": max(per),
            "spread": (max(per) - min(per)) / med if med > 0 else None}


def step_launches(path, shape, B, cfg):
    """Kernel launches of one decode step: the persistent kernel is one; the
    stage path is the embedding gather, five per layer (QKV, attention with
    RoPE and the K/V append, o-proj, gate|up, down) and the LM head, and at
    batch 9..16 with bf16 weights (the tensor cores) each of the five products
    follows its activation-plane kernel: 3 + 9 L."""
    if path == "persistent":
        return 1
    L = shape.n_layers
    umma = (B > 8 and not cfg.get("w8a8") and not cfg.get("int4")
            and os.environ.get("NC_UMMA", "1") != "0")
    return 3 + 9 * L if umma else 2 + 5 * L


def run_workload(args, ws, rank, local, name):
    cfg = dict(WORKLOADS[name])
    torch.cuda.set_device(local)
    shape = getattr(synth, cfg["shape"])
    if args.layers:  # a smaller case of the same shape, for profiler captures
        shape = shape.with_layers(args.layers)
        cfg["layers"] = args.layers
    B, gen = cfg["batch"], cfg["gen"]
    past = workload_past(cfg)
    wd = synth.model_weights(shape, device="cuda")
    max_ctx = max(past) + gen + 16
    model = nc.Model(shape, wd, max_batch=B, max_ctx=max_ctx, w8a8=cfg["w8a8"],
                     int4_group=cfg.get("int4", 0))
    del wd
    torch.cuda.empty_cache()
    kv_dtype = torch.bfloat16 if cfg.get("kv_bf16") else torch.float32
    if cfg["paged"]:
        table, nblk = synth.block_tables(past, gen + 1, 16)
        kv = nc.KVCache(shape, B, paged=True, block_table=table, num_blocks=nblk, dtype=kv_dtype)
    else:
        kv = nc.KVCache(shape, B, max_ctx=max_ctx, dtype=kv_dtype)
    fill_past(kv, shape, past)
    logits = torch.empty(B, shape.vocab, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    start = synth.token_ids(B, shape.vocab, stream=77).to(torch.int32)
    reset_host = torch.stack([start, torch.tensor(past, dtype=torch.int32)]).pin_memory()
    past_np = np.array(past, np.int32)

    def run_steps(k, off=0):
        used = []
        for i in range(off, off + k):
            j = i % gen
            if j == 0:
                tok.copy_(reset_host[0], non_blocking=True)
                pos.copy_(reset_host[1], non_blocking=True)
            model.decode_step(tok, pos, past_np + j, kv, logits, use_graph=True, advance=True)
            used.append(past_np + j)
        return used

    run_steps(args.warmup)
    torch.cuda.synchronize()
    path = model.decode_path(B, kv)
    if args.phase_profile:
        print_phase_profile(model, shape, run_steps, path, args.phase_dump)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    st = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    w0 = time.time()
    total_s, per_round, used = timed_rounds(st, run_steps, args.steps)
    w1 = time.time()
    barrier(ws)
    if rank == 0:
        time.sleep(0.2)
        sampler.stop()
    value, el = replica_rate(ws, B, args.steps, total_s)
    dur = el / args.steps
    bytes_avg = sum(step_bytes(shape, B, u.tolist(), kv_elem=2 if cfg.get("kv_bf16") else 4,
                               w8a8=bool(cfg["w8a8"]), int8_head=cfg["w8a8"] == "b32",
                               int4_group=cfg.get("int4", 0))
                    for u in used) / len(used)
    peak, peak_kind = peaks()

    # e2e: tokens and positions from pinned host memory, next tokens read back
    tok_h = torch.empty(B, dtype=torch.int32).pin_memory()
    pos_h = torch.empty(B, dtype=torch.int32).pin_memory()
    nxt_h = torch.empty(B, dtype=torch.int32).pin_memory()
    nxt_d = torch.empty(B, dtype=torch.int32, device="cuda")
    tok_h.copy_(start)
    pos_h.copy_(torch.tensor(past, dtype=torch.int32))
    tok.copy_(tok_h)
    pos.copy_(pos_h)
    model.decode_step(tok, pos, past_np, kv, logits, nxt_d, use_graph=True)
    torch.cuda.synchronize()
    k_e2e = min(args.steps, 4 * gen)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cur = start.clone()
    for i in range(k_e2e):
        j = i % gen
        if j == 0:
            cur = start.clone()
        tok_h.copy_(cur)
        pos_h.copy_(torch.from_numpy(past_np + j))
        tok.copy_(tok_h, non_blocking=True)
        pos.copy_(pos_h, non_blocking=True)
        model.decode_step(tok, pos, past_np + j, kv, logits, nxt_d, use_graph=True)
        nxt_h.copy_(nxt_d, non_blocking=True)
        st.synchronize()
        cur = nxt_h.clone()
    e2e_value, t_e2e = replica_rate(ws, B, k_e2e, time.perf_counter() - t0)
    launches_per_step = step_launches(path, shape, B, cfg)
    model.close()
    del kv
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_for(cfg, args.cpu_seconds)

    if rank == 0:
        if path == "persistent":
            kernel = f"k_decode_persistent<{1 if B == 1 else (2 if B == 2 else 4)}," \
                     f"{shape.head_dim},{'bf16' if cfg.get('kv_bf16') else 'fp32'} KV> (the whole step, one launch)"
            traffic = counted_traffic(name)
        else:
            kernel = "stage kernels (whole step, one CUDA graph)"
            traffic = None
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dur * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("i8/i32" if cfg["w8a8"] else "i4/f32" if cfg.get("int4") else "f32"),
            "data": "synthetic",
            "config": {"workload": name + (f" (first {args.layers} layers only)"
                                           if args.layers else ""),
                       "batch": B, "past": cfg["past"], "greedy_steps": gen,
                       "weights": ("int8 per-row scales, activations per 32, int8 tied head"
                                   if cfg["w8a8"] == "b32" else
                                   "int8 per-row scales (W8A8)" if cfg["w8a8"] else
                                   f"INT4, fp32 scale per {cfg['int4']} weights" if cfg.get("int4")
                                   else "bf16") +
                                  " from seeded N(0,0.02), fp32 accumulate",
                       "kv": ("paged (block 16, shuffled tables)" if cfg["paged"] else "contiguous")
                             + (" bf16" if cfg.get("kv_bf16") else " fp32"),
                       "positions": f"cycles of {gen} greedy steps from the past length(s)",
                       "path": ("nc_decode_step: one persistent cooperative launch per step"
                                if path == "persistent" else "nc_decode_step: stage kernels, CUDA graph"),
                       "l2": "inputs larger than L2: the weights stream every step",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "rounds": rounds_summary(per_round),
            "hbm": {"bytes_per_step": bytes_avg, "gbs": bytes_avg / dur / 1e9,
                    "frac_of_8tbs": bytes_avg / dur / 1e9 / NOMINAL_HBM_GBS,
                    "frac_of_measured_copy": bytes_avg / dur / 1e9 / peak, "peak_kind": peak_kind},
            "roofline": {"bound": "hbm", "kernel": kernel,
                         "achieved": bytes_avg / dur / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": bytes_avg / dur / 1e9 / peak, "traffic": traffic,
                         "peak_kind": peak_kind, "avg_launch_us": dur * 1e6 / launches_per_step,
                         "avg_step_us": dur * 1e6,
                         "algorithmic_bytes_per_launch": bytes_avg / launches_per_step},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "steps": k_e2e,
                    "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 4 * B},
            "gpu_launches": args.steps * launches_per_step,
            "clocks": sampler.summary(w0, w1),
        }), flush=True)


# Prefill workloads: a prompt of T tokens from position 0 as one forward pass
# (nc_prefill), repeated; the line reports prompt tokens per second and the
# tensor-core throughput of the pass.
PREFILLS = {
    "qwen2_0p5b_prefill512": dict(shape="QWEN2_0P5B", T=512),
    "qwen3_8b_shape_prefill512": dict(shape="QWEN3_8B", T=512),
}


def prefill_flops(shape, T, start=0):
    """Algorithmic FLOPs of one prefill pass: 2 per weight per token for the
    projections, 2 D per (query head, visible position) for each of the two
    attention products, and the last token's LM head."""
    H, F, L, V = shape.hidden, shape.ffn, shape.n_layers, shape.vocab
    nqkv = shape.q_dim + 2 * shape.kv_dim
    proj = L * (nqkv * H + shape.q_dim * H + 2 * F * H + H * F)
    seen = sum(start + i + 1 for i in range(T))
    attn = L * shape.n_q_heads * 4 * shape.head_dim * seen
    return 2 * proj * T + attn + 2 * V * H


def run_prefill(args, ws, rank, local, name):
    cfg = PREFILLS[name]
    torch.cuda.set_device(local)
    shape = getattr(synth, cfg["shape"])
    T = cfg["T"]
    wd = synth.model_weights(shape, device="cuda")
    model = nc.Model(shape, wd, max_batch=1, max_ctx=T + 16)
    del wd
    torch.cuda.empty_cache()
    kv = nc.KVCache(shape, 1, max_ctx=T + 16)
    tokens = synth.token_ids(T, shape.vocab).to(torch.int32).cuda()
    logits = torch.empty(shape.vocab, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(model.prefill_scratch_bytes(T), dtype=torch.uint8, device="cuda")

    def run_steps(k, off=0):
        for _ in range(k):
            model.prefill(0, tokens, 0, kv, logits, nxt, scratch=scratch)
        return [None] * k

    run_steps(args.warmup)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    st = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    w0 = time.time()
    total_s, per_round, _ = timed_rounds(st, run_steps, args.steps)
    w1 = time.time()
    barrier(ws)
    if rank == 0:
        time.sleep(0.2)
        sampler.stop()
    value, el = replica_rate(ws, T, args.steps, total_s)
    dur = el / args.steps
    flops = prefill_flops(shape, T)
    peak = 1891.1
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak_kind = "fallback"
    if os.path.exists(pk):
        peak, peak_kind = float(json.load(open(pk))["bf16_tflops"]), "measured"
    # e2e: the prompt from pinned host memory, the next token read back
    tok_h = tokens.cpu().pin_memory()
    nxt_h = torch.empty(1, dtype=torch.int32).pin_memory()
    k_e2e = min(args.steps, 16)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        tokens.copy_(tok_h, non_blocking=True)
        model.prefill(0, tokens, 0, kv, logits, nxt, scratch=scratch)
        nxt_h.copy_(nxt, non_blocking=True)
        st.synchronize()
    e2e_value, _ = replica_rate(ws, T, k_e2e, time.perf_counter() - t0)
    # embed; per layer 2 launches per projection (activation planes, GEMM),
    # RoPE/append and attention; the head
    launches = 2 + 10 * shape.n_layers
    model.close()
    if rank == 0:
        print(json.dumps({
            "metric": "prefill tokens/s at 1 GB300 (prompt as one forward pass)",
            "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dur * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x (bf16 hi + lo) -> f32",
            "data": "synthetic",
            "config": {"workload": name, "prompt_tokens": T, "start": 0,
                       "weights": "bf16 from seeded N(0,0.02)", "kv": "contiguous fp32",
                       "path": "nc_prefill: tcgen05 projections, flash-style attention",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "rounds": rounds_summary(per_round),
            "roofline": {"bound": "tensor", "kernel": "the whole prefill pass",
                         "achieved": flops / dur / 1e12, "peak": peak, "unit": "TFLOP/s",
                         "frac": flops / dur / 1e12 / peak, "traffic": None,
                         "peak_kind": peak_kind, "algorithmic_flops_per_pass": flops,
                         "note": "the tensor cores run each product twice (bf16 hi and lo "
                                 "planes of the fp32 activations); achieved counts it once"},
            "cpu_baseline": None,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "steps": k_e2e,
                    "h2d_bytes_per_step": 4 * T, "d2h_bytes_per_step": 4},
            "gpu_launches": args.steps * launches,
            "clocks": sampler.summary(w0, w1),
        }), flush=True)


def print_phase_profile(model, shape, run_steps, path, dump=None):
    """Critical-path timeline of the persistent kernel (nc_profile_phases) over
    a few steps, printed to stderr. For phase p: `handover` = the last CTA's
    input arrival minus the moment the last CTA finished phase p - 1 (the
    hand-over latency on the chain), `work` = the moment the last CTA finished
    phase p minus that input arrival. Medians over layers and steps; the two
    columns summed over all phases give the step."""
    if path != "persistent":
        print("phase profile: the stage path has no phase record", file=sys.stderr)
        return
    L = shape.n_layers
    nph = 5 * L + 1
    names = ["qkv", "attention", "o-proj", "gate|up", "down", "lm-head"]
    hand = {n: [] for n in names}
    work = {n: [] for n in names}
    sub = {k: [] for k in ("scan", "publish", "merge", "to next phase", "scan per CTA (max)",
                           "first chunk wait (max)", "last chunk wait (max)")}
    totals = []
    model.profile_phases(True)
    raw = []
    for it in range(4):
        run_steps(1, it)
        rec = model.read_phase_profile()
        raw.append({k: v.numpy() for k, v in rec.items()})
        start = rec["start"].numpy().astype(np.int64)
        inp = rec["input"].numpy().astype(np.int64)
        c0 = rec["cta_start"].numpy().astype(np.int64)
        c1 = rec["cta_end"].numpy().astype(np.int64)
        t0 = int(c0.min())
        totals.append((int(c1.max()) - t0) / 1e3)
        for p in range(nph):
            kind = names[5] if p == nph - 1 else names[p % 5]
            ok = inp[:, p] >= start[:, p]  # CTAs that ran the phase this step
            if not ok.any():
                continue
            fin_prev = start[:, p].max()
            last_in = inp[ok, p].max()
            fin = start[:, p + 1].max() if p + 1 < nph else c1.max()
            hand[kind].append((last_in - fin_prev) / 1e3)
            work[kind].append((fin - last_in) / 1e3)
            if kind == "attention":
                at = rec["attn"].numpy().astype(np.int64)[:, p // 5]
                done = ok & (at[:, 0] >= inp[:, p])
                if done.any():
                    scan = at[done, 0].max()
                    pub = at[done, 1].max()
                    merged = at[done, 2]
                    mg = merged[merged > 0].max() if (merged > 0).any() else pub
                    sub["scan"].append((scan - last_in) / 1e3)
                    sub["publish"].append((pub - scan) / 1e3)
                    sub["merge"].append((mg - pub) / 1e3)
                    sub["to next phase"].append((fin - mg) / 1e3)
                    sub["scan per CTA (max)"].append((at[done, 0] - inp[done, p]).max() / 1e3)
                    sub["first chunk wait (max)"].append((at[done, 3] - inp[done, p]).max() / 1e3)
                    sub["last chunk wait (max)"].append((at[done, 4] - inp[done, p]).max() / 1e3)
    model.profile_phases(False)
    if dump:
        np.savez_compressed(dump, **{f"{k}_{i}": v for i, r in enumerate(raw) for k, v in r.items()})
    print(f"phase profile ({len(totals)} steps, median step {statistics.median(totals):.1f} us):",
          file=sys.stderr)
    print(f"{'phase':10s} {'handover us':>12s} {'work us':>9s}", file=sys.stderr)
    for k in names:
        if hand[k]:
            print(f"{k:10s} {statistics.median(hand[k]):12.2f} {statistics.median(work[k]):9.2f}",
                  file=sys.stderr)
    if sub["scan"]:
        print("attention work, critical path (last CTA to reach each mark), us: "
              + ", ".join(f"{k} {statistics.median(v):.2f}" for k, v in sub.items()),
              file=sys.stderr)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="nc", choices=["nc", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[C1, SAMPLED] + list(WORKLOADS) + list(PREFILLS))
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload's model (a small "
                         "case for profiler captures; not a metric line)")
    ap.add_argument("--phase-dump", default=None,
                    help="with --phase-profile: also save the raw per-CTA records (.npz)")
    ap.add_argument("--phase-profile", action="store_true",
                    help="print the persistent kernel's per-phase critical path (stderr)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.workload == SAMPLED:
        run_sampled(args, ws, rank, local)
    elif args.workload == C1:
        run_nc(args, ws, rank, local)
    elif args.workload in PREFILLS:
        run_prefill(args, ws, rank, local, args.workload)
    else:
        run_workload(args, ws, rank, local, args.workload)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
