"""Decode throughput of the 2.3B lane model on GB300 (batch 1, FP16).

Workload (the single-step microbench): full shape (15 layers, d=4096, 32 q /
16 KV heads of 128, FFN 7168, vocab 32000, 8 lanes, delay 2), FP16 weights
N(0, 0.02) from seed 1, KV cache slots 0..511 of every layer filled with
N(0, 1) FP16 values, one decode step of a random token at position 512.  A
timed "step" is one such decode step (the whole hot path: 15 layers, the
delayed lane sum, LM head, argmax); the position is set back to 512 before
every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload e2e|long|sweep|prefill|passn|passn_batch|batch   # further workloads, one line each

Under torchrun (N > 1) every rank decodes its own replica on its own GPU (the
path needs no exchange between GPUs); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "batch-1 decode tokens/s (2.3B lane model, FP16) and % of HBM roofline"
UNIT = "tokens/s"
POS = 512
SEED = 1
PROFILE = os.path.join(ROOT, "profiles", "decode_kernel_full_p512.txt")
# the sources that decide what the decode kernel reads and writes
KERNEL_SRCS = [os.path.join(ROOT, "decode_persistent_sm_gb300", "csrc", f)
               for f in ("lf_kernel.cu", "lf_kernel.cuh", "lf_ptx.cuh", "lf_common.h", "lf_plan.cpp")]


def kernel_sources_hash():
    h = hashlib.sha256()
    for f in KERNEL_SRCS:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def algorithmic_bytes(shape, pos: int) -> int:
    """Bytes one decode step must move at position `pos`: every parameter but
    the embedding table (one 8 KB row of it), plus the live KV cache
    sum_l min(pos+1, W_l) keys * n_kv * head_dim * (K, V) * 2 bytes."""
    d = shape.d_model
    weights = (shape.n_params - shape.vocab * d) * 2
    kv = 0
    for w in shape.swa_window:
        keys = pos + 1 if w == 0 else min(pos + 1, w)
        kv += keys * shape.n_kv_heads * shape.head_dim * 2 * 2
    return weights + kv


def workload_config(shape):
    return {
        "workload": f"single decode step at position {POS} (KV pre-filled N(0,1)), full 2.3B lane "
                    "model: 15 layers, d_model 4096, 32 q / 16 KV heads x 128, FFN 7168, vocab 32000, "
                    "8 lanes, DTP delay 2, SWA 1024 on 10 layers",
        "batch": 1, "position": POS, "n_lanes": shape.n_lanes, "dtp_delay": shape.dtp_delay,
        "l2": "no flush: inputs larger than L2 (4.4 GB streamed per step vs 129 MB L2)",
        "seed": SEED,
    }


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = None

    def start(self):
        if not shutil.which("nvidia-smi"):
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen(
            ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits", "-lms", "50"],
            stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


def profile_traffic():
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since the counters were taken."""
    if not os.path.exists(PROFILE):
        return None
    kv = {}
    for line in open(PROFILE):
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_sources_sha256_16") != kernel_sources_hash():
        return None
    try:
        return int(float(kv["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def peak_tensor(sustained: bool):
    """Measured dense bf16 tensor throughput (FP16 has the same nominal rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    return (1700.0 if sustained else 1900.0), "fallback"


def prefill_flops(shape, n: int, p0: int = 0):
    """Algorithmic FLOPs of a batched prefill of n positions from p0: the
    projections (2 per weight per position) plus attention (QK and PV, 2 per
    key per head dimension each) over each position's visible keys; the LM
    head of the last position."""
    d, dh = shape.d_model, shape.head_dim
    qkvn = (shape.n_q_heads + 2 * shape.n_kv_heads) * dh
    per_tok = 2 * (qkvn * d + d * shape.n_q_heads * dh + 2 * shape.ffn_dim * d + d * shape.ffn_dim)
    gemm = per_tok * n * shape.n_layers
    attn = 0
    for w in shape.swa_window:
        keys = 0
        for p in range(p0, p0 + n):
            keys += p + 1 if w == 0 else min(p + 1, w)
        attn += 4 * shape.n_q_heads * dh * keys
    return gemm, attn, 2 * shape.vocab * d


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def read_stream_gbs(nbytes: int, stream, reps: int = 20):
    """Read-only HBM bandwidth of the decode kernel's copy pattern (lf_stream_read)
    over a buffer of nbytes (rounded up to 32 KB tiles), best of `reps` launches
    timed one by one with CUDA events; None if a device-side wait ran out."""
    import torch
    from decode_persistent_sm_gb300 import stream_read
    n = -(-nbytes // 32768) * 32768
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    n_sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sink = torch.empty(n_sm, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    best = None
    for i in range(reps + 3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        stream_read(buf.data_ptr(), n, sink.data_ptr(), n_sm, status.data_ptr(), stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
    if int(status.item()) != 0:
        return None
    del buf
    return n / (best / 1e3) / 1e9


def oracle_rate(shape, blob, kv, tokens, budget_s: float, max_steps: int, pos: int = POS):
    """Decode steps/s of the CPU oracle at position `pos` (cache filled with
    `kv` up to there) on a bounded sample."""
    import oracle
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, pos)
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        orc.set_pos(pos)
        orc.step(int(tokens[n % len(tokens)]))
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt, oracle.threads()


def oracle_prompt_rate(shape, blob, prompt, budget_s: float):
    """Positions/s of the CPU oracle over a prompt: it computes a prompt one
    position at a time (exact under causality), so a bounded sample of
    positions spread evenly over the prompt, each with the cache filled up to
    it, has the prompt's mean cost per position."""
    import oracle
    import synth
    n = len(prompt)
    kv = synth.make_kv(shape, SEED, n)
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, n)
    grid = np.linspace(0, n - 1, 64).astype(int)
    # bit-reversed order: whenever the budget ends the sample, the positions
    # done so far are spread evenly over the prompt
    order = [grid[int(format(i, "06b")[::-1], 2)] for i in range(64)]
    done, t0 = 0, time.perf_counter()
    for p in order:
        orc.set_pos(int(p))
        orc.step(int(prompt[p]))
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt, oracle.threads()


OP_NAMES = {0: "embed", 1: "add", 2: "norm", 3: "qkv", 4: "gateup", 5: "down", 6: "attn",
            7: "oproj", 8: "reduce", 9: "lmhead"}


def write_trace(eng, path, tokens, shape):
    """One traced step at position 512: per op type, the mean over CTAs of the
    time spent in the op, blocked on cross-CTA counters and blocked on tiles."""
    eng.trace(True)
    for i in range(3):
        eng.set_position(POS)
        eng.decode_step_async(int(tokens[i]))
    eng.synchronize()
    tr, ops = eng.read_trace()
    eng.trace(False)
    tr = tr.astype(np.int64)
    t0 = tr[:, 0, 0].min()  # EMBED, written by every CTA
    step_ns = int(tr[:, -1, 1].max() - t0)
    dur = tr[:, :, 1] - tr[:, :, 0]
    by = {}
    # a REDUCE slot is written only by the CTAs that sum a chunk (others: 0)
    rows = [np.nonzero(tr[:, j, 0])[0] for j in range(len(ops))]
    for j, op in enumerate(ops):
        name = OP_NAMES[int(op) & 0xFF]
        b = by.setdefault(name, [0.0, 0.0, 0.0, 0, 0.0])
        r = rows[j]
        b[0] += dur[r, j].mean()
        b[1] += tr[r, j, 2].mean()
        b[2] += tr[r, j, 3].mean()
        b[3] += 1
        b[4] += tr[r, j, 4].mean()
    start_skew = int(tr[:, 0, 0].max() - t0)
    end_spread = int(tr[:, -1, 1].max() - tr[:, -1, 1].min())
    lm = [j for j, op in enumerate(ops) if int(op) & 0xFF == 9][0]
    out = {"step_ns": step_ns, "cta_start_skew_ns": start_skew, "cta_end_spread_ns": end_spread,
           "lmhead_start_ns_mean": float((tr[:, lm, 0] - t0).mean()),
           "by_op": {k: {"count": v[3], "mean_ns": v[0], "sync_wait_ns": v[1], "tile_wait_ns": v[2],
                         "copy_warp_blocked_ns": v[4]} for k, v in by.items()},
           "per_op": [{"op": OP_NAMES[int(op) & 0xFF], "arg": (int(op) >> 8) & 0xFF,
                       "ctas": int(len(rows[j])),
                       "start_ns_mean": float((tr[rows[j], j, 0] - t0).mean()),
                       "end_ns_max": int((tr[rows[j], j, 1] - t0).max()),
                       "dur_ns_mean": float(dur[rows[j], j].mean()), "dur_ns_max": int(dur[rows[j], j].max()),
                       "sync_ns_mean": float(tr[rows[j], j, 2].mean()),
                       "tile_ns_mean": float(tr[rows[j], j, 3].mean()),
                       "copy_blocked_ns_mean": float(tr[rows[j], j, 4].mean())} for j, op in enumerate(ops)]}
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    np.savez_compressed(os.path.splitext(path)[0] + "_raw.npz", trace=tr, ops=ops)
    print(f"traced step: {step_ns / 1e3:.1f} us; CTA start skew {start_skew / 1e3:.1f} us", file=sys.stderr)
    for k, v in out["by_op"].items():
        print(f"  {k:7s} x{v['count']:3d}  {v['mean_ns'] / 1e3:8.1f} us  sync {v['sync_wait_ns'] / 1e3:7.1f}"
              f"  tiles {v['tile_wait_ns'] / 1e3:7.1f}  copy warp blocked {v['copy_warp_blocked_ns'] / 1e3:7.1f}",
              file=sys.stderr)


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """The largest x over all ranks of the process group (each rank passes
    its own); x itself when there is one rank."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: int, worst_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (every rank runs the same work on its own GPU)."""
    return world * units_per_rank / (worst_ms / 1e3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    import synth
    if rank != 0:
        return
    shape = synth.FULL
    blob = synth.make_weights(shape, SEED)
    kv = synth.make_kv(shape, SEED, POS)
    tokens = synth.make_tokens(SEED, args.steps + args.warmup, shape.vocab)
    import oracle
    orc = oracle.Oracle(shape, blob)
    orc.load_kv(kv, POS)
    for i in range(args.warmup):
        orc.set_pos(POS)
        orc.step(int(tokens[i]))
    t0 = time.perf_counter()
    for i in range(args.steps):
        orc.set_pos(POS)
        orc.step(int(tokens[args.warmup + i]))
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{args.steps} decode steps at position {POS} (each step a full "
                                   "pass of the fp64 oracle over the same workload)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch
    import synth
    from decode_persistent_sm_gb300 import Engine

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    shape = synth.FULL
    if args.layers:  # a smaller model of the same width, for profiler captures only
        shape = shape.replace(n_layers=args.layers, swa_window=shape.swa_window[:args.layers])
    blob = synth.make_weights(shape, SEED)
    kv = synth.make_kv(shape, SEED, POS)
    tokens = synth.make_tokens(SEED + rank, args.steps + args.warmup, shape.vocab)

    stream = torch.cuda.current_stream()
    eng = Engine.from_shape(shape)
    eng.set_stream(stream.cuda_stream)
    eng.load_weights(blob)
    eng.load_kv(kv, POS)
    if args.idle_prefetch_kb >= 0:
        eng.set_idle_prefetch(args.idle_prefetch_kb * 1024, args.idle_after_ns)
    if args.l2_prefetch_kb >= 0 or args.lm_prefetch_kb >= 0:
        eng.set_l2_prefetch(max(args.l2_prefetch_kb, 0) * 1024 if args.l2_prefetch_kb >= 0 else 128 * 1024,
                            args.lm_prefetch_kb * 1024 if args.lm_prefetch_kb >= 0 else 128 * 1024)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for i in range(max(args.warmup, 3)):
        eng.set_position(POS)
        eng.decode_step_async(int(tokens[i % len(tokens)]))
    eng.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    launches0 = eng.info()["launches"]
    ev0.record(stream)
    for i in range(args.steps):
        eng.set_position(POS)
        eng.decode_step_async(int(tokens[args.warmup + i]))
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    eng.synchronize()  # raises if any timed step failed
    launches = eng.info()["launches"] - launches0
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms = total_ms / args.steps
    value = job_rate(world, args.steps, total_ms)

    # end to end through the C ABI: token in by value, logits + argmax back
    # into pinned host memory, every step synchronous
    n_e2e = min(args.steps, 300)
    host_logits = torch.empty(shape.vocab, dtype=torch.float32, pin_memory=True)
    barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        eng.set_position(POS)
        eng.decode_step_into(int(tokens[i]), host_logits.data_ptr())
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": job_rate(world, n_e2e, e2e_s * 1e3), "unit": UNIT, "h2d_bytes_per_step": 4,
           "d2h_bytes_per_step": shape.vocab * 4 + 4 * 8}

    if args.trace:
        write_trace(eng, args.trace, tokens, shape)

    nbytes = algorithmic_bytes(shape, POS)
    peak, peak_kind = peak_hbm()
    achieved = nbytes / (ms / 1e3) / 1e9
    read_gbs = read_stream_gbs(nbytes, stream)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                # the committed capture covers the full-shape launch at position 512 only
                "traffic": profile_traffic() if POS == 512 and not args.layers else None,
                "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": nbytes,
                # the copy figure counts a read and a write; a read-only stream in
                # the kernel's own copy pattern, measured in this run, and the
                # vendor's nominal bandwidth are the other two denominators
                "read_stream_gbs": read_gbs,
                "frac_of_read_stream": achieved / read_gbs if read_gbs else None,
                "frac_of_nominal_7900": achieved / 7900.0}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt, cores = oracle_rate(shape, blob, kv, tokens, args.cpu_budget_s, 200)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n} decode steps at position {POS} of the same workload ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16 weights, fp32 accumulate",
            "data": "synthetic (seeded N(0,0.02) FP16 weights, N(0,1) KV fill)",
            "config": workload_config(shape) if not args.layers else
            {"workload": f"profiling case: {args.layers} layers of the full width"},
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "parallelism": "replicas only" if world > 1 else "1 GPU, 8 lanes = SM groups",
        }
        print(json.dumps(line), flush=True)
    eng.close()
    if world > 1:
        torch.distributed.destroy_process_group()


# Generation workloads (not the default line): the end-to-end and long-context
# runs and the delay x lane sweep, each timed step by step with CUDA events.
GEN_WORKLOADS = {
    "e2e": (128, 512, "end to end: prompt of 128 random ids (prefilled by decode steps), then 512 greedy "
                      "tokens chained on the device (positions 128..639), full 2.3B lane model, 8 lanes, delay 2"),
    "long": (3584, 512, "long context: prompt of 3584 random ids (prefilled by decode steps), then 512 greedy "
                        "tokens chained on the device (positions 3584..4095), full 2.3B lane model, 8 lanes, "
                        "delay 2"),
}
SWEEP_CTX, SWEEP_STEPS = 2048, 256
PREFILL_N = 3584
PASSN = (128, 8, 256, 0.8, 0.95)  # prompt, samples, tokens per sample, temperature, top_p
BATCH_SWEEP = (512, 64, (1, 2, 4, 8, 16))  # KV fill (--position), greedy steps per batch size, batch sizes


def timed_generation(eng, stream, first_token: int, n: int):
    """n chained greedy steps from the engine's position, an event between
    every two; returns (tokens, per-step ms, total ms)."""
    import torch
    buf = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    buf[0] = int(first_token)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    base = buf.data_ptr()
    torch.cuda.synchronize()
    for i in range(n):
        evs[i].record(stream)
        eng.decode_step_chained(base + 4 * i, base + 4 * (i + 1))
    evs[n].record(stream)
    torch.cuda.synchronize()
    eng.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return buf[1:].cpu().numpy(), per, evs[0].elapsed_time(evs[n])


def timed_generate_fused(eng, stream, first_token: int, n: int):
    """lf_generate (all n steps in one launch of the persistent kernel) timed
    with CUDA events around the call; per-step latencies from the steps'
    completion stamps.  Returns (tokens, per-step ms, total ms)."""
    import torch
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    toks, _ = eng.generate(int(first_token), n)
    e1.record(stream)
    torch.cuda.synchronize()
    stamps = eng.generate_stamps(n).astype(np.int64)
    per = list(np.diff(stamps) / 1e6)
    return toks, per, e0.elapsed_time(e1)


def latency_summary(per_ms):
    a = np.sort(np.asarray(per_ms))
    return {"p50_ms": float(np.percentile(a, 50)), "p99_ms": float(np.percentile(a, 99)),
            "max_ms": float(a[-1]), "mean_ms": float(a.mean())}


def gen_roofline(shape, pos0: int, n: int, ms_per_step: float, batch: int = 1):
    """Roofline of n steps from pos0 at ms_per_step; a batch of B samples
    streams the weights once per step and reads B live KV caches."""
    kv = lambda p: algorithmic_bytes(shape, p) - algorithmic_bytes(shape, -1)
    nbytes = sum(algorithmic_bytes(shape, p) + (batch - 1) * kv(p) for p in range(pos0, pos0 + n)) / n
    peak, peak_kind = peak_hbm()
    achieved = nbytes / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": None, "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
            "algorithmic_bytes_per_launch": nbytes}


def run_generation(args, world, rank, local):
    import torch
    import synth
    from decode_persistent_sm_gb300 import Engine

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def worst(x):  # max over ranks
        return max_over_ranks(x, world)

    base = synth.FULL
    if args.layers:  # a smaller model of the same width, for profiler captures only
        base = base.replace(n_layers=args.layers, swa_window=base.swa_window[:args.layers])
    blob = synth.make_weights(base, SEED)
    stream = torch.cuda.current_stream()
    data = "synthetic (seeded N(0,0.02) FP16 weights, uniform random token ids)"
    common = {"n_gpus": world, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "fp16 weights, fp32 accumulate", "unit": UNIT,
              "parallelism": "replicas only" if world > 1 else "1 GPU, 8 lanes = SM groups"}

    if args.workload == "prefill":
        shape = base
        prompt = synth.make_tokens(SEED + rank, PREFILL_N, shape.vocab)
        with Engine.from_shape(shape) as eng:
            eng.set_stream(stream.cuda_stream)
            eng.load_weights(blob)
            for _ in range(max(args.warmup, 3)):
                eng.reset()
                eng.prefill_batched(prompt, logits=False)
            clocks = ClockSampler(local)
            clocks.start()
            times = []
            reps = max(1, min(args.steps, 10))
            for _ in range(reps):
                eng.reset()
                torch.cuda.synchronize()
                if world > 1:
                    torch.distributed.barrier()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                eng.prefill_batched(prompt, logits=False)
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(worst(e0.elapsed_time(e1)))
            clk = clocks.stop()
            eng.reset()
            t0 = time.perf_counter()
            _, am = eng.prefill_batched(prompt, logits=True)
            e2e_s = worst(time.perf_counter() - t0)
        ms = float(np.median(times))
        gemm, attn, lm = prefill_flops(shape, PREFILL_N)
        peak, kind = peak_tensor(sustained=False)
        achieved = (gemm + attn + lm) / (ms / 1e3) / 1e12
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            rate, n_o, dt, cores = oracle_prompt_rate(shape, blob, prompt, args.cpu_budget_s)
            cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                   "sample": f"{n_o} prompt positions spread evenly over 0..{PREFILL_N - 1}, each computed by "
                             f"the oracle as one step of the prompt (cache filled up to it), {dt:.1f} s; "
                             "the positions' mean cost stands for the prompt's"}
        if rank == 0:
            line = {"metric": "batched prefill tokens/s (prompt of 3584 ids, 2.3B lane model, FP16)",
                    "value": world * PREFILL_N / (ms / 1e3), "steps": reps, "warmup": max(args.warmup, 3),
                    "ms_per_step": ms, "ttft_ms": ms, "data": data,
                    "config": {"workload": "prefill of a 3584-id prompt from an empty cache (batched: one pass "
                                           "per sub-block, tensor-core GEMMs), full 2.3B lane model, 8 lanes, "
                                           "delay 2", "prompt": PREFILL_N, "seed": SEED,
                               "l2": "no flush: 4.4 GB of weights per pass vs 129 MB L2"},
                    "flops": {"gemm": gemm, "attention": attn, "lm_head": lm},
                    "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                                 "frac": achieved / peak, "traffic": None,
                                 "peak_source": f"{kind} dense bf16 burst (MEASURED_PEAKS.json bf16_tflops); "
                                                "FP16 has the same nominal rate"},
                    "cpu_baseline": cpu,
                    "e2e": {"value": world * PREFILL_N / e2e_s, "unit": "tokens/s",
                            "h2d_bytes_per_step": PREFILL_N * 4, "d2h_bytes_per_step": shape.vocab * 4 + 4,
                            "call": "lf_prefill_batched with host token ids and host logits"},
                    "gpu_launches": None, "clocks": clk, **common}
            if args.layers:
                line["config"] = {"workload": f"profiling case: {args.layers} layers of the full width"}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == "gemm":  # the prefill's tensor-core GEMM on its QKV shape
        from decode_persistent_sm_gb300 import matmul_f16, matmul_f16_async
        M, N, K = PREFILL_N, 8192, 4096
        g = torch.Generator(device="cuda").manual_seed(SEED)
        a = torch.randn(M, K, device="cuda", generator=g).half()
        b = (0.02 * torch.randn(N, K, device="cuda", generator=g)).half()
        c = torch.empty(M, N, device="cuda", dtype=torch.float32)
        errw = torch.zeros(1, dtype=torch.int32, device="cuda")
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")  # > the 129 MB L2
        for _ in range(max(args.warmup, 3)):
            matmul_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, stream.cuda_stream)
        reps = max(1, min(args.steps, 50))
        clocks = ClockSampler(local)
        clocks.start()
        times, calls = [], []
        for _ in range(reps):  # the kernel alone, L2 flushed before each launch (outside the events)
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            matmul_f16_async(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, errw.data_ptr(), stream.cuda_stream)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        for _ in range(min(reps, 10)):  # through the synchronous call (status set and read back)
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            matmul_f16(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, stream.cuda_stream)
            calls.append((time.perf_counter() - t0) * 1e3)
        clk = clocks.stop()
        if int(errw.item()) != 0:
            raise SystemExit("GEMM: a device-side wait ran out")
        ms = worst(float(np.median(times)))
        flop = 2.0 * M * N * K
        peak, kind = peak_tensor(sustained=False)
        ach = flop / (ms / 1e3) / 1e12
        call_ms = worst(float(np.median(calls)))
        if rank == 0:
            print(json.dumps({
                "metric": "tensor-core GEMM TFLOP/s (prefill QKV shape, FP16 in, fp32 out)", "value": world * ach,
                "unit": "TFLOP/s", "steps": reps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16 x fp16 -> fp32",
                "data": "synthetic N(0,1) x N(0,0.02)", "n_gpus": world,
                "config": {"workload": f"C[{M}][{N}] = A[{M}][{K}] . B[{N}][{K}]^T: median of single launches "
                                       "(lf_matmul_f16_async) timed by CUDA events",
                           "l2": "flushed before every launch (256 MB written outside the timed region)"},
                "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                             "frac": ach / peak, "traffic": None,
                             "peak_source": f"{kind} dense bf16 burst (MEASURED_PEAKS.json bf16_tflops)"},
                "e2e": {"value": world * flop / (call_ms / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 4, "call": "lf_matmul_f16 (synchronous, status read back), host-timed"},
                "cpu_baseline": None, "gpu_launches": reps, "clocks": clk}), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == "passn":
        n_prompt, n_samp, n_tok, temp, top_p = PASSN
        shape = base
        prompt = synth.make_tokens(SEED + rank, n_prompt, shape.vocab)
        with Engine.from_shape(shape) as eng:
            eng.set_stream(stream.cuda_stream)
            eng.load_weights(blob)
            eng.prefill_batched(prompt[:-1], logits=False)
            eng.generate_sampled(int(prompt[-1]), max(args.warmup, 3), temp, top_p, SEED, sample=999)
            clocks = ClockSampler(local)
            clocks.start()
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            outs = []
            for k in range(n_samp):
                eng.set_position(n_prompt - 1)
                toks, _ = eng.generate_sampled(int(prompt[-1]), n_tok, temp, top_p, SEED, sample=k)
                outs.append(toks)
            e1.record(stream)
            torch.cuda.synchronize()
            clk = clocks.stop()
            total = worst(e0.elapsed_time(e1))
        ms = total / (n_samp * n_tok)
        distinct = len({tuple(o) for o in outs})
        if rank == 0:
            line = {"metric": "batch-1 sampled decode tokens/s for pass@N (2.3B lane model, FP16)",
                    "value": world * n_samp * n_tok / (total / 1e3), "steps": n_samp * n_tok,
                    "warmup": max(args.warmup, 3), "ms_per_step": ms, "data": data,
                    "config": {"workload": f"pass@{n_samp}: prompt of {n_prompt} random ids (batched prefill), then "
                                           f"{n_samp} samples of {n_tok} tokens, temperature {temp}, top-p {top_p}, "
                                           "each sample restarting at the prompt's end; samples run one after "
                                           "another (no batch-N decode)", "seed": SEED,
                               "l2": "no flush: inputs larger than L2"},
                    "distinct_samples": distinct,
                    "roofline": gen_roofline(shape, n_prompt - 1, n_tok, ms), "cpu_baseline": None,
                    "e2e": {"value": world * n_samp * n_tok / (total / 1e3), "unit": UNIT, "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 4 + 32 / n_tok,
                            "call": "lf_generate_sampled per sample (tokens copied back once per sample)"},
                    "gpu_launches": 2 * n_samp * n_tok, "clocks": clk, **common}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == "passn_batch":
        n_prompt, n_samp, n_tok, temp, top_p = PASSN
        shape = base
        prompt = synth.make_tokens(SEED + rank, n_prompt, shape.vocab)
        with Engine.from_shape(shape) as eng:
            eng.set_stream(stream.cuda_stream)
            eng.load_weights(blob)
            eng.prefill_batched(prompt[:-1], logits=False)
            eng.batch_begin(n_samp)
            eng.batch_generate([int(prompt[-1])] * n_samp, max(args.warmup, 3), temp, top_p, SEED + 999)
            clocks = ClockSampler(local)
            clocks.start()
            eng.batch_begin(n_samp)  # back to the prompt's end
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            toks = eng.batch_generate([int(prompt[-1])] * n_samp, n_tok, temp, top_p, SEED)
            e1.record(stream)
            torch.cuda.synchronize()
            clk = clocks.stop()
            total = worst(e0.elapsed_time(e1))
        ms = total / n_tok  # one batch step: every sample advances one token
        distinct = len({tuple(o) for o in toks})
        if rank == 0:
            rate = world * n_samp * n_tok / (total / 1e3)
            line = {"metric": "sampled decode tokens/s for pass@N, N samples decoded as one batch (2.3B lane model, "
                              "FP16)",
                    "value": rate, "steps": n_tok, "warmup": max(args.warmup, 3), "ms_per_step": ms, "data": data,
                    "config": {"workload": f"pass@{n_samp}: prompt of {n_prompt} random ids (batched prefill), then "
                                           f"{n_samp} samples of {n_tok} tokens decoded together (lf_batch_generate: "
                                           f"one weight stream per step for all samples), temperature {temp}, "
                                           f"top-p {top_p}", "batch": n_samp, "seed": SEED,
                               "l2": "no flush: inputs larger than L2"},
                    "distinct_samples": distinct,
                    "roofline": gen_roofline(shape, n_prompt - 1, n_tok, ms, batch=n_samp), "cpu_baseline": None,
                    "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 4 * n_samp / n_tok,
                            "d2h_bytes_per_step": 4 * n_samp + 4 / n_tok,
                            "call": "lf_batch_generate (first tokens in, all tokens and the status word out once)"},
                    "gpu_launches": n_tok * (7 * shape.n_layers + 6), "clocks": clk, **common}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == "batch":
        _, n_tok, sizes = BATCH_SWEEP
        fill = POS  # --position: the KV fill every sample starts from (default 512)
        if args.batch:  # one batch size, at most 64 steps (profiling runs)
            sizes, n_tok = (args.batch,), min(args.steps, n_tok)
        shape = base
        kv = synth.make_kv(shape, SEED, fill)
        first = synth.make_tokens(SEED + rank, 16, shape.vocab)
        variants = {}
        clocks = ClockSampler(local)
        clocks.start()
        with Engine.from_shape(shape) as eng:
            eng.set_stream(stream.cuda_stream)
            eng.load_weights(blob)
            eng.load_kv(kv, fill)
            for B in sizes:
                eng.batch_begin(B)
                eng.batch_generate([int(t) for t in first[:B]], max(args.warmup, 3), 0.0, 1.0, 0)
                eng.batch_begin(B)
                if world > 1:
                    torch.distributed.barrier()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                eng.batch_generate([int(t) for t in first[:B]], n_tok, 0.0, 1.0, 0)
                e1.record(stream)
                torch.cuda.synchronize()
                total = worst(e0.elapsed_time(e1))
                ms = total / n_tok
                variants[f"B{B}"] = {"value": world * B * n_tok / (total / 1e3), "ms_per_step": ms,
                                     "roofline_frac": gen_roofline(shape, fill, n_tok, ms, batch=B)["frac"]}
            eng.batch_end()
        clk = clocks.stop()
        main_b = 8 if "B8" in variants else sizes[0]
        main_v = variants[f"B{main_b}"]
        if rank == 0:
            line = {"metric": "batched greedy decode tokens/s (all samples) per batch size", "value": main_v["value"],
                    "steps": n_tok, "warmup": max(args.warmup, 3), "ms_per_step": main_v["ms_per_step"],
                    "data": data + ", N(0,1) KV fill",
                    "config": {"workload": f"batched decode: KV pre-filled N(0,1) to {fill} and shared by every "
                                           f"sample, then {n_tok} greedy steps of B samples together "
                                           f"(lf_batch_generate) for B in {list(sizes)}; value at B = {main_b}",
                               "seed": SEED, "l2": "no flush: inputs larger than L2"},
                    "variants": variants,
                    "roofline": gen_roofline(shape, fill, n_tok, main_v["ms_per_step"], batch=main_b),
                    "cpu_baseline": None, "e2e": None,
                    "gpu_launches": len(sizes) * n_tok * (7 * shape.n_layers + 6), "clocks": clk, **common}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    if args.workload == "sweep":
        variants = {}
        kv = synth.make_kv(base, SEED, SWEEP_CTX)
        first = int(synth.make_tokens(SEED + rank, 1, base.vocab)[0])
        clocks = ClockSampler(local)
        clocks.start()
        launches = 0
        for delay, lanes, own in [(d, n, o) for d in (0, 1, 2) for n in (1, 8) for o in (0, 1) if d > 0 or o == 0]:
            shape = base.replace(n_lanes=lanes, dtp_delay=delay, own_lane_immediate=own)
            with Engine.from_shape(shape) as eng:
                eng.set_stream(stream.cuda_stream)
                eng.load_weights(blob)
                eng.load_kv(kv, SWEEP_CTX)
                eng.generate(first, max(args.warmup, 3))
                eng.set_position(SWEEP_CTX)
                if world > 1:
                    torch.distributed.barrier()
                _, per, total = timed_generate_fused(eng, stream, first, SWEEP_STEPS)
                total = worst(total)
                launches += 1
            variants[f"delay{delay}_lanes{lanes}" + ("_own" if own else "")] = {
                "value": world * SWEEP_STEPS / (total / 1e3), "ms_per_step": total / SWEEP_STEPS,
                **latency_summary(per)}
        clk = clocks.stop()
        main_v = variants["delay2_lanes8"]
        if rank == 0:
            line = {"metric": "batch-1 greedy decode tokens/s per delay x lane variant", "value": main_v["value"],
                    "steps": SWEEP_STEPS, "warmup": max(args.warmup, 3), "ms_per_step": main_v["ms_per_step"],
                    "data": data + ", N(0,1) KV fill",
                    "config": {"workload": f"sweep: KV pre-filled N(0,1) to {SWEEP_CTX}, then {SWEEP_STEPS} greedy "
                                           "tokens in one lf_generate launch for delay in {0,1,2} x lanes in {1,8}, "
                                           "both readings of the delayed sum for delay > 0 (_own: each lane "
                                           "adds its own partial at once); value = delay 2, 8 lanes", "seed": SEED,
                               "l2": "no flush: inputs larger than L2"},
                    "variants": variants,
                    "roofline": gen_roofline(base, SWEEP_CTX, SWEEP_STEPS, main_v["ms_per_step"]),
                    "cpu_baseline": None, "e2e": None, "gpu_launches": launches, "clocks": clk, **common}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    n_prompt, n_gen, desc = GEN_WORKLOADS[args.workload]
    shape = base
    prompt = synth.make_tokens(SEED + rank, n_prompt, shape.vocab)
    pos0 = n_prompt - 1  # first decode position of the generation
    eng = Engine.from_shape(shape)
    eng.set_stream(stream.cuda_stream)
    eng.load_weights(blob)
    eng.generate(int(prompt[0]), max(args.warmup, 3))  # warm-up
    eng.reset()
    t0 = time.perf_counter()
    eng.prefill(prompt[:-1], logits=False)
    loop_prefill_ms = (time.perf_counter() - t0) * 1e3
    eng.reset()
    t0 = time.perf_counter()
    eng.prefill_batched(prompt[:-1], logits=False)
    prefill_ms = (time.perf_counter() - t0) * 1e3
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    gen, per, total = timed_generate_fused(eng, stream, int(prompt[-1]), n_gen)
    clk = clocks.stop()
    total = worst(total)
    # the same steps as separate launches (one per token, chained on the device)
    eng.reset()
    eng.prefill_batched(prompt[:-1], logits=False)
    gen_sep, per_sep, total_sep = timed_generation(eng, stream, int(prompt[-1]), n_gen)
    total_sep = worst(total_sep)
    # end to end through lf_generate: tokens back in host memory
    eng.reset()
    eng.prefill_batched(prompt[:-1], logits=False)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    gen2, _ = eng.generate(int(prompt[-1]), n_gen)
    e2e_s = worst(time.perf_counter() - t0)
    eng.close()
    ms = total / n_gen
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kv = synth.make_kv(shape, SEED, pos0)
        rate, n, dt, cores = oracle_rate(shape, blob, kv, prompt, args.cpu_budget_s, 200, pos=pos0)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n} decode steps at position {pos0} of the same model, cache filled with N(0,1) "
                         f"({dt:.1f} s)"}
    if rank == 0:
        line = {"metric": "batch-1 greedy decode tokens/s (2.3B lane model, FP16)",
                "value": world * n_gen / (total / 1e3), "steps": n_gen, "warmup": max(args.warmup, 3),
                "ms_per_step": ms, "data": data,
                "config": {"workload": desc, "prompt": n_prompt, "generated": n_gen, "seed": SEED,
                           "l2": "no flush: inputs larger than L2 (4.4 GB streamed per step)"},
                "latency": latency_summary(per),
                "prefill_ms": prefill_ms, "prefill": f"{n_prompt - 1} positions, lf_prefill_batched, host-timed",
                "prefill_ms_decode_loop": loop_prefill_ms,
                "timing": "lf_generate: all steps in one launch of the persistent kernel, CUDA events "
                          "around the call; latency from the steps' completion stamps",
                "separate_launches": {"value": world * n_gen / (total_sep / 1e3), "ms_per_step": total_sep / n_gen,
                                      **latency_summary(per_sep),
                                      "tokens_match": bool(np.array_equal(gen, gen_sep))},
                "chain_matches_lf_generate": bool(np.array_equal(gen, gen2)),
                "roofline": gen_roofline(shape, pos0, n_gen, ms), "cpu_baseline": cpu,
                "e2e": {"value": world * n_gen / e2e_s, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 4 + 32 / n_gen,
                        "call": "lf_generate (first token by value, tokens and status copied back once)"},
                "gpu_launches": 1, "clocks": clk, **common}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    global POS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--l2-prefetch-kb", type=int, default=-1,
                    help="weight-stream L2 prefetch distance per SM (default: the engine's)")
    ap.add_argument("--lm-prefetch-kb", type=int, default=-1,
                    help="LM-head L2 prefetch distance per SM (default: the engine's)")
    ap.add_argument("--trace", default="", help="write a one-step op trace (JSON) to this path")
    ap.add_argument("--position", type=int, default=POS,
                    help="step workload: decode position (KV pre-filled up to it); 512 is the default line")
    ap.add_argument("--workload", choices=["step", "e2e", "long", "sweep", "prefill", "passn", "passn_batch", "batch",
                                           "gemm"],
                    default="step",
                    help="step: the single-step microbench (default line); e2e / long / sweep: the "
                         "generation workloads")
    ap.add_argument("--batch", type=int, default=0,
                    help="--workload batch: one batch size instead of the sweep (steps = min(--steps, 64))")
    ap.add_argument("--idle-prefetch-kb", type=int, default=-1,
                    help="step workload: L2 lead (KiB per SM) the copy warp builds while it waits for a stage")
    ap.add_argument("--idle-after-ns", type=int, default=4000,
                    help="step workload: wait before the idle prefetch starts")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: same width with fewer layers (not a bench number)")
    args = ap.parse_args()
    POS = args.position
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        if args.steps > 50:
            args.steps = 20  # each oracle step takes a fraction of a second
        run_reference(args, world, rank)
    elif args.workload != "step":
        run_generation(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
