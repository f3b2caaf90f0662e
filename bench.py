#!/usr/bin/env python
"""Decode-step throughput of libg4 on GB300, with its HBM roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

A step is one greedy decode step of the whole model (embedding, per-layer embeddings, all
projections, attention with KV sharing, norms, lm_head and argmax) for the workload's batch.
Default workload: the E2B-shaped W4A16 model at batch 1 after a 128-token prompt, timed over
the 511 decode steps that produce tokens 2..512 (positions 128..638): one untimed run, then
three timed runs of K steps from the same start; the headline is their median (IQR beside
it).  Companion figures in the same line: batch 64, bf16 at batch 1 and 64, and the model
with int4 vocabulary tables and int8 cache rows.

Prints one JSON line (rank 0).  Under torchrun every rank runs an independent replica on its
own GPU (the path has no exchange step); value = tokens of all ranks / max rank time.
--impl reference times the CPU oracle (numpy) on the host cores instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tok/s at batch 1 & 64, E2B-shaped bf16/W4A16; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
RUNS = 3  # timed runs after the untimed one; the headline is their median
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ------------------------------------------------------------------------------------ helpers
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(value, world, device=None):
    """Max of a float over ranks (the barrier-bracketed timing rule)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, batch, steps, ms_max):
    """Whole-job tok/s of `world` replicas that each decode `batch` sequences for `steps`
    steps, timed by the slowest rank (ms_max)."""
    return world * batch * steps / (ms_max / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _owning(cfg):
    """Layers that keep their own K/V: below the first shared index, or sharing layers with no
    earlier layer of their type (same schedule the library and the oracle implement)."""
    L, first = cfg["num_layers"], cfg["num_layers"] - cfg["num_kv_shared_layers"]
    full = [synth.layer_is_full(cfg, l) for l in range(L)]
    return [l < first or not any(full[j] == full[l] for j in range(first)) for l in range(L)]


def algorithmic_bytes(cfg, fmt, batch, positions, count_aliased=False, tables="bf16", kv="bf16"):
    """Unique bytes one decode step must move: every weight once (int4 at 0.5 B + a bf16 scale
    per 32, or bf16), the tied lm_head (bf16, or int4 tables), and per sequence the visible K/V
    of the owning layers' caches (read once even when aliased; int8 rows add a 4-byte scale),
    the new K/V row, the per-layer-embedding row and the embedding row.  count_aliased also
    counts each KV-sharing layer's read of its source cache (the bytes the attention kernels
    actually request).  Returns (weight bytes, mean KV+row bytes per step over positions)."""
    H, P, V, L = cfg["hidden"], cfg["ple_dim"], cfg["vocab"], cfg["num_layers"]
    own = _owning(cfg)
    n_lin = L * P * H
    for l in range(L):
        sh = synth.weights.linear_shapes(cfg, l)
        for name, (n, k) in sh.items():
            if name in ("k", "v") and not own[l]:
                continue
            n_lin += n * k
    per_w = 0.5 + 2.0 / 32 if fmt == "w4a16" else 2.0
    t4 = tables == "int4"
    wbytes = n_lin * per_w + (V * H * (0.5 + 2.0 / 32) if t4 else V * H * 2)
    row = (lambda d: d + 4) if kv == "int8" else (lambda d: 2 * d)   # bytes of one cache row
    kv = []
    for p in positions:
        T = p + 1
        b = 0
        for l in range(L):
            if not own[l] and not count_aliased:
                continue
            full = synth.layer_is_full(cfg, l)
            d = cfg["head_dim_full"] if full else cfg["head_dim_sliding"]
            keys = T if full else min(T, cfg["sliding_window"])
            b += keys * row(d) * 2 + (row(d) * 2 if own[l] else 0)
        b += (L * P * 0.5 + L * 2 + H * 0.5 + H / 32 * 2) if t4 else (L * P * 2 + H * 2)
        kv.append(b * batch)
    return wbytes, float(np.mean(kv))


# DRAM traffic / algorithmic bytes of a kernel, from one ncu capture of its current code;
# traffic scales with the rows a launch streams.
# Keyed by (weight format, phase); a kernel changed since its capture has no entry.
MEASURED_TRAFFIC_RATIO = {("w4a16", "gemv.gate_up"): 10717952 / 10616832}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, f"{pre}{k}.")
                elif isinstance(x, (int, float)):
                    flat[pre[:-1]] = float(x)
            walk(d)
            for k, v in flat.items():
                if "hbm" in k.lower() and "gb" in k.lower():
                    return v, f"measured ({k})"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
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
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(power) if power else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_cores():
    return len(os.sched_getaffinity(0))


def oracle_sample(cfg, weights, batch, budget_s, n_max, start=128):
    """Time the CPU oracle's decode steps on this host at the GPU's positions: an untimed
    teacher-forced prefill of `start` tokens, then up to n_max decode steps (positions start,
    start + 1, ...) or budget_s seconds of work.  Returns (tok/s, steps, seconds, batch used)."""
    import oracle
    ob = batch
    o = oracle.Oracle(cfg, weights, max_batch=ob, max_context=start + n_max + 1)
    prompts = synth.make_prompts(cfg["vocab"], ob, start + n_max + 1, seed=0, stream=99)
    slots = np.arange(ob)
    o.prefill(slots, prompts[:, :start])                     # untimed
    t0 = time.perf_counter()
    n = 0
    while n < n_max:
        o.step(slots, prompts[:, start + n], np.full(ob, start + n))
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return ob * n / dt, n, dt, ob


# ------------------------------------------------------------------------------- GPU leg
def run_gpu(args, wl, cfg, fmt):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from accelerator_decode_gb300.runtime import Decoder

    B, P0, n_out = wl["batch"], wl["prompt"], wl["out"]
    K, W = args.steps, args.warmup
    max_ctx = ((P0 + max(K, W, n_out) + 1 + 63) // 64) * 64
    t_gen = time.perf_counter()
    weights = synth.make_model_weights(cfg, fmt, seed=args.seed)
    prompts = synth.make_prompts(cfg["vocab"], B, P0, seed=args.seed, stream=rank)
    t_gen = time.perf_counter() - t_gen
    dec = Decoder(cfg, weights, max_batch=B, max_context=max_ctx, device=local, kv_format=args.kv)
    if args.step_mode:
        dec.set_step_mode(args.step_mode)
    step_mode = dec.step_mode(B)
    if args.impl_check_only:
        return None
    st = torch.cuda.Stream()
    dev = torch.device("cuda", local)
    with torch.cuda.stream(st):
        nxt, _ = dec.prefill(list(range(B)), list(prompts), stream=st)
        st.synchronize()
        first = nxt.clone()
        slots = torch.arange(B, dtype=torch.int32, device=dev)
        tok = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(2)]
        pos = torch.empty(B, dtype=torch.int32, device=dev)

        def reset():
            tok[0].copy_(first)
            pos.fill_(P0)

        def steps(n):
            for i in range(n):
                dec.decode_step(slots, tok[i % 2], pos, tok[(i + 1) % 2], None, stream=st)
                pos.add_(1)

        reset()
        steps(W)                         # warm-up (also captures both step graphs)
        reset()
        clocks = ClockSampler(local)
        clocks.start()
        steps(min(W, 64))               # keep the GPU busy while the sampler starts
        # one untimed run (the warm-up above), then RUNS timed runs of K steps from the same
        # start; the headline is the median run, with the interquartile range beside it
        runs = []
        for r in range(RUNS):
            reset()
            st.synchronize()
            barrier(world)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.nvtx.range_push("g4_timed")
            e0.record(st)
            steps(K)
            e1.record(st)
            torch.cuda.nvtx.range_pop()
            e1.synchronize()
            barrier(world)
            runs.append(max_over_ranks(e0.elapsed_time(e1), world, dev))
        clk = clocks.stop()
        ms_max = float(np.median(runs))
        out_tokens = tok[K % 2].cpu().numpy().tolist()
        status, word = dec.device_error(stream=st)

        # e2e: host buffers through the public API; per step H2D tokens+positions, D2H next ids
        h_tok = torch.empty(B, dtype=torch.int32, pin_memory=True)
        h_pos = torch.empty(B, dtype=torch.int32, pin_memory=True)
        h_next = torch.empty(B, dtype=torch.int32, pin_memory=True)
        d_tok = torch.empty(B, dtype=torch.int32, device=dev)
        d_pos = torch.empty(B, dtype=torch.int32, device=dev)
        d_next = torch.empty(B, dtype=torch.int32, device=dev)
        h_tok.copy_(first.cpu())
        h_pos.fill_(P0)
        for i in range(3):                # warm the e2e graph
            d_tok.copy_(h_tok, non_blocking=True)
            d_pos.copy_(h_pos, non_blocking=True)
            dec.decode_step(slots, d_tok, d_pos, d_next, None, stream=st)
            h_next.copy_(d_next, non_blocking=True)
            st.synchronize()
        h_tok.copy_(first.cpu())
        h_pos.fill_(P0)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(K):
            d_tok.copy_(h_tok, non_blocking=True)
            d_pos.copy_(h_pos, non_blocking=True)
            dec.decode_step(slots, d_tok, d_pos, d_next, None, stream=st)
            h_next.copy_(d_next, non_blocking=True)
            st.synchronize()
            h_tok.copy_(h_next)
            h_pos.add_(1)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e_tokens = h_tok.numpy().tolist()

        # per-phase timing (CUDA events on this stream around every launch), mid-run position
        pos.fill_(P0 + K // 2)
        prof = dec.profile_step(slots, tok[0], pos, tok[1], None, repeats=args.profile_repeats, stream=st)

    # calibrated copy bandwidth (torch copy of 4 GiB) as a sanity line beside the measured peak
    a = torch.empty(1 << 31, dtype=torch.int16, device=dev)
    b2 = torch.empty_like(a)
    b2.copy_(a)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(5):
        b2.copy_(a)
    c1.record()
    c1.synchronize()
    copy_gbs = 5 * 2 * a.numel() * 2 / (c0.elapsed_time(c1) / 1e3) / 1e9
    del a, b2


    positions = [P0 + i for i in range(K)]
    wbytes, kvbytes = algorithmic_bytes(cfg, fmt, B, positions, kv=args.kv)
    _, kv_aliased = algorithmic_bytes(cfg, fmt, B, positions, count_aliased=True, kv=args.kv)
    peak, peak_src = measured_peak()
    step_bytes = wbytes + kvbytes
    value = replica_throughput(world, B, K, ms_max)
    reps = args.profile_repeats
    launches_per_step = sum(p["launches"] for p in prof) / reps
    prof_ms = sum(p["ms_total"] for p in prof) / reps
    dom = max(prof, key=lambda p: p["ms_total"])
    dom_name = dom["name"]
    dom_ms = dom["ms_total"] / dom["launches"]
    dom_bytes = dom["bytes_total"] / dom["launches"]
    if step_mode == 1:
        # one cooperative kernel per step: it is the dominant (only) kernel of the timed region
        dom_name, dom_ms, dom_bytes = "mega_step_kernel", ms_max / K, step_bytes
        launches_per_step = 1.0
    phases = {p["name"]: {"launches_per_step": p["launches"] / reps, "ms_per_step": p["ms_total"] / reps,
                          "share": p["ms_total"] / max(1e-9, sum(q["ms_total"] for q in prof)),
                          "weight_gb_per_step": p["bytes_total"] / reps / 1e9} for p in prof}
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_max / K, 5),
        "runs": {"timed": RUNS, "untimed": 1, "statistic": "median",
                 "ms_per_step": [round(r / K, 5) for r in runs],
                 "iqr_ms_per_step": round(float(np.percentile(runs, 75) - np.percentile(runs, 25)) / K, 5),
                 "iqr_tok_s": round(float(replica_throughput(world, B, K, np.percentile(runs, 25))
                                          - replica_throughput(world, B, K, np.percentile(runs, 75))), 2)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl["name"], "weights": fmt, "kv_cache": args.kv, "batch_per_gpu": B,
                   "prompt_tokens": P0, "decode_positions": [P0, P0 + K - 1], "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (weights streamed every step exceed 129 MB)",
                   "seed": args.seed,
                   "knobs": {k: os.environ[k] for k in ("G4_TC_MIN_BATCH", "G4_GEMV_UNSPLIT_BYTES", "G4_GEMV_STAGED",
                                                        "G4_ATTN_MQA_MIN", "G4_LMHEAD_STAGED") if k in os.environ}},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": round(dom_bytes / (dom_ms / 1e3) / 1e9, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(dom_bytes / (dom_ms / 1e3) / 1e9 / peak, 4),
                     "traffic": (round(dom_bytes * MEASURED_TRAFFIC_RATIO[(fmt, dom_name)])
                                 if (fmt, dom_name) in MEASURED_TRAFFIC_RATIO else None),
                     "bytes_per_launch": dom_bytes, "ms_per_launch": round(dom_ms, 5),
                     "peak_source": peak_src},
        "step_roofline": {"bytes_per_step": step_bytes, "weight_bytes": wbytes, "kv_and_rows_bytes": kvbytes,
                          "achieved": round(step_bytes / (ms_max / K / 1e3) / 1e9, 1), "peak": peak,
                          "frac": round(step_bytes / (ms_max / K / 1e3) / 1e9 / peak, 4), "unit": "GB/s",
                          "peak_source": peak_src, "calibrated_copy_gbs": round(copy_gbs, 1),
                          "kv_and_rows_bytes_counting_aliased_reads": kv_aliased,
                          "frac_counting_aliased_reads": round((wbytes + kv_aliased) / (ms_max / K / 1e3) / 1e9 / peak, 4)},
        "e2e": {"value": round(replica_throughput(world, B, K, e2e_s * 1e3), 2), "unit": "tok/s",
                "h2d_bytes_per_step": 2 * 4 * B,
                "d2h_bytes_per_step": 4 * B},
        "gpu_launches": int(round(launches_per_step * K)),
        "kernels_per_step": launches_per_step,
        "step_mode": "persistent" if step_mode == 1 else "launch-per-phase",
        "profile": {"repeats": reps, "ms_per_step_unfused_launches": round(prof_ms, 4), "phases": phases},
        "clocks": clk,
        "device_error": word,
        "tokens_match_e2e": out_tokens == e2e_tokens,
        "weight_gen_s": round(t_gen, 1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, dt, ob = oracle_sample(cfg, weights, B, args.cpu_budget, 64, start=P0)
        result["cpu_baseline"] = {"value": round(v, 3), "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                                  "sample": f"{n} oracle decode steps of batch {ob} at positions {P0}..{P0 + n - 1} "
                                            f"after an untimed {P0}-token prefill ({dt:.1f} s timed), same weights"}
    dec.close()
    if args.batch64 and B == 1 and world == 1:
        result["batch64"] = companion_line(args, cfg, weights, local, 64)
        if fmt == "w4a16" and args.companions:
            # the metric's bf16 half, and the int4-table / int8-cache variant of the same model
            del weights
            wb = synth.make_model_weights(cfg, "bf16", seed=args.seed)
            result["bf16_b1"] = companion_line(args, cfg, wb, local, 1)
            result["bf16_b64"] = companion_line(args, cfg, wb, local, 64)
            del wb
            wv = synth.make_model_weights(cfg, "w4a16", seed=args.seed, tables="int4")
            result["w4a16_int4_tables_int8_kv_b1"] = companion_line(args, cfg, wv, local, 1, kv="int8")
            result["w4a16_int4_tables_int8_kv_b64"] = companion_line(args, cfg, wv, local, 64, kv="int8")
            del wv
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def companion_line(args, cfg, weights, local, B, kv="bf16"):
    """Companion figure of the metric (its batch-64 half, its bf16 half, the int4-table /
    int8-cache variant): `weights` at B sequences after 128-token prompts, W >= 3 untimed
    steps, then RUNS timed runs of K = 64 steps from the same start (median and IQR), CUDA
    events on the launching stream; inputs (1.2+ GB of weights per step) exceed L2."""
    import torch
    from accelerator_decode_gb300.runtime import Decoder
    P0, K, W = 128, 64, max(3, min(args.warmup, 8))
    tables = "int4" if isinstance(weights["embed"], dict) else "bf16"
    dev = torch.device("cuda", local)
    dec = Decoder(cfg, weights, max_batch=B, max_context=((P0 + K + W + 1 + 63) // 64) * 64, device=local,
                  kv_format=kv)
    prompts = synth.make_prompts(cfg["vocab"], B, P0, seed=args.seed)
    st = torch.cuda.Stream()
    runs = []
    with torch.cuda.stream(st):
        nxt, _ = dec.prefill(list(range(B)), list(prompts), stream=st)
        slots = torch.arange(B, dtype=torch.int32, device=dev)
        tok = [nxt.clone(), torch.empty_like(nxt)]
        pos = torch.full((B,), P0, dtype=torch.int32, device=dev)
        for i in range(W):
            dec.decode_step(slots, tok[i % 2], pos, tok[(i + 1) % 2], None, stream=st)
            pos.add_(1)
        for r in range(RUNS):
            tok[0].copy_(nxt)
            pos.fill_(P0)
            st.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for i in range(K):
                dec.decode_step(slots, tok[i % 2], pos, tok[(i + 1) % 2], None, stream=st)
                pos.add_(1)
            e1.record(st)
            e1.synchronize()
            runs.append(e0.elapsed_time(e1) / K)
        status, word = dec.device_error(stream=st)
    dec.close()
    ms = float(np.median(runs))
    wbytes, kvbytes = algorithmic_bytes(cfg, weights["fmt"], B, [P0 + i for i in range(K)], tables=tables, kv=kv)
    peak, peak_src = measured_peak()
    return {"value": round(B / (ms / 1e3), 2), "unit": "tok/s", "ms_per_step": round(ms, 5),
            "iqr_ms_per_step": round(float(np.percentile(runs, 75) - np.percentile(runs, 25)), 5),
            "runs_ms_per_step": [round(r, 5) for r in runs], "steps": K, "warmup": W,
            "batch": B, "prompt_tokens": P0, "weights": weights["fmt"], "tables": tables, "kv_cache": kv,
            "step_roofline": {"bytes_per_step": wbytes + kvbytes, "frac": round((wbytes + kvbytes) / (ms / 1e3) / 1e9 / peak, 4),
                              "peak": peak, "peak_source": peak_src},
            "device_error": word}


# ------------------------------------------------------------------------- agent replay
def run_replay(args, wl, cfg, fmt):
    """Agent replay: `batch` sequences start at a `prompt`-token context; each of `turns` turns
    appends the previous turn's last output (not yet in the cache) and `turn_append` fresh
    ids by append-prefill, then runs `out` - 1 decode steps.  Reports decode tok/s per turn
    against the context length (CUDA events on the decode steps of each turn)."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from accelerator_decode_gb300.runtime import Decoder

    B, n_out, turns = wl["batch"], wl["out"], wl["turns"]
    sched = synth.replay_schedule(start=wl["prompt"], end=wl["prompt"] + turns * wl["turn_append"], turns=turns,
                                  outputs=n_out)
    max_ctx = sched[0][0] + sum(a + o for a, o in sched[1:])
    max_ctx = ((max_ctx + 63) // 64) * 64
    weights = synth.make_model_weights(cfg, fmt, seed=args.seed)
    dec = Decoder(cfg, weights, max_batch=B, max_context=max_ctx, device=local, kv_format=args.kv)
    dev = torch.device("cuda", local)
    st = torch.cuda.Stream()
    slots = list(range(B))
    ctx = [0] * B
    last = None
    rows, dec_tokens, dec_ms = [], 0, 0.0
    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(st):
        d_slots = torch.arange(B, dtype=torch.int32, device=dev)
        tok = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(2)]
        pos = torch.empty(B, dtype=torch.int32, device=dev)
        for turn, (fresh, outs) in enumerate(sched):
            ids = synth.make_prompts(cfg["vocab"], B, fresh, seed=args.seed + 1000 + turn, stream=rank)
            if last is not None:
                ids = np.concatenate([last[:, None], ids], axis=1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            nxt, _ = dec.prefill(slots, list(ids), start_pos=list(ctx), stream=st)
            e1.record(st)
            st.synchronize()
            pf_ms = e0.elapsed_time(e1)
            ctx = [c + ids.shape[1] for c in ctx]
            if outs == 0:
                continue
            tok[0].copy_(nxt)
            pos.fill_(ctx[0])
            steps = outs - 1
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(st)
            for i in range(steps):
                dec.decode_step(d_slots, tok[i % 2], pos, tok[(i + 1) % 2], None, stream=st)
                pos.add_(1)
            d1.record(st)
            d1.synchronize()
            ms = d0.elapsed_time(d1)
            rows.append({"context": ctx[0], "decode_tok_s": round(B * steps / (ms / 1e3), 1),
                         "prefill_tok_s": round(B * ids.shape[1] / (pf_ms / 1e3), 1)})
            dec_tokens += B * steps
            dec_ms += ms
            ctx = [c + steps for c in ctx]
            last = tok[steps % 2].cpu().numpy().astype(np.int32)
        status, word = dec.device_error(stream=st)
    clk = clocks.stop()
    dec.close()
    return {
        "metric": METRIC + " (agent replay: decode tok/s versus context)",
        "value": round(dec_tokens / (dec_ms / 1e3), 2),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": dec_tokens // B,
        "warmup": 0,
        "ms_per_step": round(dec_ms / max(1, dec_tokens // B), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl["name"], "weights": fmt, "kv_cache": args.kv, "batch_per_gpu": B,
                   "start_context": sched[0][0],
                   "final_context": ctx[0], "turns": turns, "outputs_per_turn": n_out},
        "by_context": rows,
        "clocks": clk,
        "device_error": word,
    }


# ------------------------------------------------------------------------- reference arm
def run_reference(args, wl, cfg, fmt):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    weights = synth.make_model_weights(cfg, fmt, seed=args.seed)
    B = wl["batch"]
    # bounded sample: the whole run (warm-up + steps) must end within a few minutes
    budget = args.ref_budget
    total_steps = args.steps + args.warmup
    v, n, dt, ob = oracle_sample(cfg, weights, B, budget, total_steps, start=wl["prompt"])
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 3),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": n,
        "warmup": 1,
        "ms_per_step": round(dt / max(n, 1) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl["name"], "weights": fmt, "batch_per_gpu": B, "prompt_tokens": wl["prompt"],
                   "decode_positions": [wl["prompt"], wl["prompt"] + n - 1]},
        "cpu_baseline": {"value": round(v, 3), "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{n} oracle decode steps of batch {ob} at positions {wl['prompt']}.."
                                   f"{wl['prompt'] + n - 1} after an untimed {wl['prompt']}-token prefill "
                                   f"(bounded to {budget:.0f} s of {total_steps} requested)"},
        "e2e": {"value": round(v, 3), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=511)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--workload", default="e2b-w4a16-b1", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--step-mode", type=int, default=0, choices=[0, 1],
                    help="0: one launch per phase (CUDA graph); 1: persistent single-launch step (batch <= 2)")
    ap.add_argument("--profile-repeats", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-batch64", dest="batch64", action="store_false",
                    help="skip the companion figures (batch 64, bf16, int4 tables + int8 cache)")
    ap.add_argument("--no-companions", dest="companions", action="store_false",
                    help="keep the batch-64 figure, skip the bf16 and int4-table / int8-cache ones")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "int8"], help="KV cache rows (default bf16)")
    ap.add_argument("--impl-check-only", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = synth.get_workload(args.workload)
    cfg = synth.get_config(wl["config"])
    fmt = wl["fmt"]
    rank, world, _ = dist_env()
    if world != args.gpus and rank == 0:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        res = run_reference(args, wl, cfg, fmt)
    elif "turns" in wl:
        res = run_replay(args, wl, cfg, fmt)
    else:
        res = run_gpu(args, wl, cfg, fmt)
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
