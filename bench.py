#!/usr/bin/env python3
"""Benchmark of the P-EAGLE draft + verify step on GB300.

One step = one parallel draft pass (pe_draft: FC fusion, row build, 4 drafter
layers over the paged KV cache, LM head + fused argmax) followed by one fused
greedy verify / batch-metadata rebuild (pe_verify_rebuild), on seeded
synthetic inputs with a random-init drafter. Inputs stay resident in HBM; the
weights alone (1.12 GB for the Qwen3-Coder-shaped drafter) exceed the 126 MB
L2, so every step streams them from HBM again without an explicit flush.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, time-boxed

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the workload (the path shards by request with no
exchange step) and the whole-job value is N * K steps / max-over-ranks time.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft+verify steps/s & draft tok/s at B=1..128, K=3/7/11; % HBM / TC roofline"
DEFAULT_WORKLOAD = "qwen-b1-k7"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the K sweep, the cold-L2 line and the workload sweep")
    ap.add_argument("--max-prefix", type=int, default=0,
                    help="cap the workload's prefix lengths (same GEMM shapes, smaller KV cache: for small ncu captures)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0, help="time box of the oracle CPU baseline")
    ap.add_argument("--fp8", action="store_true",
                    help="the main line with FP8 (E4M3) GEMM weights and per-row scales (bf16 activations and KV)")
    ap.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--worker-warmup", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ------------------------------------------------------------------ shared helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(wl):
    s = wl.shape
    lo, hi = wl.prefix
    prefix = str(lo) if lo == hi else f"U[{lo},{hi}]"
    return (f"{s.name} drafter (H={s.hidden}, {s.n_q_heads}q/{s.n_kv_heads}kv x {s.head_dim}, F={s.ffn}, "
            f"V={s.vocab}, 4 layers, {s.dtype}), B={wl.B}, K={wl.K}, prefix {prefix} in 16-token pages")


def algorithmic_work(kind, wl, seq_lens, chained=False, fp8=False):
    """Algorithmic HBM bytes and FLOPs of ONE launch of a kernel kind,
    averaged over that kind's launches in a step. `chained`: the step runs
    O, gate/up, down and the next QKV (or the LM head) as one persistent
    layer-chain launch per layer. `fp8`: the GEMM weights are E4M3 codes
    (one byte each) with one fp32 scale per output row."""
    s = wl.shape
    e = 2 if s.dtype == "bf16" else 4
    H, F, V, hd, nq, nkv = s.hidden, s.ffn, s.vocab, s.head_dim, s.n_q_heads, s.n_kv_heads
    B, K = wl.B, wl.K
    R = B * K
    qd, qkv = nq * hd, s.qkv_rows

    def wb(rows, cols):      # bytes of one weight matrix
        return rows * cols + 4 * rows if fp8 else rows * cols * e

    def qkv_work(kin):       # + q out and the new K/V rows
        return wb(qkv, kin) + R * kin * e + R * qd * e + R * 2 * nkv * hd * e, 2 * R * qkv * kin

    def o_work():            # + residual read/write and the folded RMSNorm's gain * r output
        return wb(H, qd) + R * qd * e + 2 * R * H * 4 + R * H * e, 2 * R * H * qd

    def gu_work():
        return 2 * wb(F, H) + R * H * e + R * F * e, 2 * R * 2 * F * H

    def down_work():
        return wb(H, F) + R * F * e + 2 * R * H * 4 + R * H * e, 2 * R * H * F

    def lm_work():
        return wb(V, H) + R * H * e + R * 8, 2 * R * V * H

    def add(*ws):
        return sum(w[0] for w in ws), sum(w[1] for w in ws)

    if kind == "fc":
        return wb(H, 3 * H) + B * 3 * H * e + B * H * 4, 2 * B * 3 * H * H
    if kind == "qkv":
        if chained:          # only layer 0's QKV (2H inputs) runs on its own
            return qkv_work(2 * H)
        b, f = add(qkv_work(2 * H), qkv_work(H), qkv_work(H), qkv_work(H))
        return b / 4.0, f / 4.0
    if kind == "attention":
        ctx = sum(int(S) + K for S in seq_lens)
        kv = ctx * nkv * hd * 2 * e
        flops = sum(4 * nq * hd * (int(S) + j + 1) for S in seq_lens for j in range(K))
        return kv + 2 * R * qd * e, flops
    if kind == "o_proj":
        return o_work()
    if kind == "gate_up":
        return gu_work()
    if kind == "down":
        return down_work()
    if kind == "lm_head":
        return lm_work()
    if kind == "layer_chain":   # three launches end with a QKV, the last with the LM head
        mid = add(o_work(), gu_work(), down_work(), qkv_work(H))
        last = add(o_work(), gu_work(), down_work(), lm_work())
        return (3 * mid[0] + last[0]) / 4.0, (3 * mid[1] + last[1]) / 4.0
    if kind == "row_build":
        return R * (3 * H * e + H * 4) + B * H * 4, 8 * R * H
    return R * 12, R


def gemm_weight_shapes(s):
    """(rows, cols) of every GEMM weight matrix of the drafter."""
    H, F, qd = s.hidden, s.ffn, s.n_q_heads * s.head_dim
    mats = [(H, 3 * H), (s.vocab, H)]
    for layer in range(s.n_layers):
        mats += [(s.qkv_rows, 2 * H if layer == 0 else H), (H, qd), (F, H), (F, H), (H, F)]
    return mats


def step_bytes(wl, seq_lens, fp8=False):
    """Algorithmic HBM bytes of one whole step: every weight matrix once,
    except the token embedding, of which only the B gathered rows are read;
    plus the KV cache read (prefix and new entries) and the new entries
    written. `fp8`: GEMM weights at one byte each plus a 4-byte scale per
    row."""
    s = wl.shape
    e = 2 if s.dtype == "bf16" else 4
    R = wl.B * wl.K
    weights = (s.param_count() - s.vocab * s.hidden + wl.B * s.hidden) * e
    if fp8:
        gemm = gemm_weight_shapes(s)
        weights += sum(r * c + 4 * r - r * c * e for r, c in gemm)
    kv_read = sum(int(S) + wl.K for S in seq_lens) * s.n_kv_heads * s.head_dim * 2 * e * s.n_layers
    kv_write = R * s.n_kv_heads * s.head_dim * 2 * e * s.n_layers
    return weights + kv_read + kv_write


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read-only)."""

    def __init__(self, gpu_index, out_path=None, interval_ms=50):
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(interval_ms), "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.out_path = out_path

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.strip() == "Active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x, device=None):
    """Largest value of x over all ranks of the default process group (the
    timing every rank reports is the slowest rank's); x itself when there is
    no group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_steps_per_s(world, steps, elapsed_ms):
    """Replicas: every rank runs `steps` steps of its own batch; the job
    processed world * steps steps in the slowest rank's time."""
    return world * steps / (elapsed_ms / 1e3)


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)

def oracle_worker(args):
    """Runs in a child process: time the oracle's step on the host cores."""
    import numpy as np
    import torch

    import oracle
    from speculative_drafting_pe_gb300 import synth

    torch.set_num_threads(max(1, len(os.sched_getaffinity(0))))
    wl = synth.WORKLOADS[args.workload]
    W = synth.make_weights(wl.shape, wl.seed)
    inp = synth.make_step_inputs(wl)
    if args.fp8:
        Wq, sc = synth.quantize_weights_fp8(W)
        Wn = oracle.dequant_weights(*synth.fp8_to_numpy(Wq, sc))
        del Wq, sc
    else:
        Wn = synth.weights_to_numpy(W)
    del W
    a = dict(last_token=inp.last_token.numpy(), target_hidden=inp.target_hidden.float().numpy(),
             positions=inp.positions.numpy(), seq_lens=inp.seq_lens.numpy(), page_table=inp.page_table.numpy(),
             k_cache=inp.k_cache.float().numpy(), v_cache=inp.v_cache.float().numpy())
    K = wl.K

    def step():
        out = oracle.draft_pass(wl.shape, Wn, a["last_token"], a["target_hidden"], a["positions"], a["seq_lens"],
                                a["page_table"], a["k_cache"], a["v_cache"], K)
        g = synth.plant_targets(out["drafts"], inp.alpha, wl.shape.vocab, wl.seed)
        acc, bonus = oracle.verify(out["drafts"], g)
        oracle.rebuild_metadata(acc, K, a["seq_lens"], a["positions"], a["page_table"], inp.num_pages)

    for _ in range(args.worker_warmup):   # untimed
        step()
    times = []
    budget = args.cpu_seconds
    t_start = time.time()
    max_steps = args.steps
    while len(times) < max_steps:
        t0 = time.time()
        step()
        times.append(time.time() - t0)
        if time.time() - t_start > budget:
            break
    print(json.dumps({"steps": len(times), "seconds": sum(times), "step_s": times,
                      "warmup": args.worker_warmup, "cores": len(os.sched_getaffinity(0))}))


def run_oracle_subprocess(workload, seconds, max_steps, fp8=False, warmup=0):
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker", "--workload", workload,
           "--cpu-seconds", str(seconds), "--steps", str(max_steps),
           "--worker-warmup", str(warmup)] + (["--fp8"] if fp8 else [])
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=seconds * 6 + 600)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_obj(res, wl):
    steps_s = res["steps"] / res["seconds"]
    return {"value": steps_s, "unit": "steps/s", "cores": res["cores"], "kind": "oracle",
            "sample": f"{res['steps']} full float64 oracle step(s) (draft pass + verify + rebuild) of the same "
                      f"workload, time-boxed, {res['seconds']:.1f} s of CPU work, BLAS threads = cores",
            "draft_tok_s": steps_s * wl.B * wl.K}


# ------------------------------------------------------------------ our arm

FP8_WORKLOADS = ("qwen-b1-k3", "qwen-b1-k7", "qwen-b1-k11", "qwen-b8-k7", "qwen-b32-k11", "qwen-b128-k11",
                 "gptoss-b64-k10")
SWEEP_WORKLOADS = (["qwen-b1-k3", "qwen-b1-k7", "qwen-b1-k11"]
                   + [f"qwen-b{B}-k{K}" for B in (4, 8, 32, 128) for K in (3, 7, 11)]
                   + ["gptoss-b64-k10"])


def roofline_of(kind, wl, seq_np, avg_launch_s, peaks, chained=False, fp8=False):
    """Roofline of one kernel kind: its algorithmic bytes (or FLOPs) per
    launch over its measured average launch time, against the measured peak
    of whichever resource bounds it at these sizes."""
    b, f = algorithmic_work(kind, wl, seq_np, chained=chained, fp8=fp8)
    t_hbm = b / (peaks["hbm_gbs"] * 1e9)
    t_tc = f / (peaks["bf16_tflops_sustained"] * 1e12)
    if t_hbm >= t_tc:
        a = b / avg_launch_s / 1e9
        return {"bound": "hbm", "achieved": a, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": a / peaks["hbm_gbs"]}
    a = f / avg_launch_s / 1e12
    return {"bound": "tensor", "achieved": a, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "frac": a / peaks["bf16_tflops_sustained"]}


def sweep_workload(name, dev, weights_cache, peaks, replays, fp8=False):
    """Steps/s, draft tok/s, step HBM fraction and the dominant kernel's
    roofline for one workload: per-kind CUDA events over three direct steps
    (shares and per-launch times), then `replays` timed step-graph replays.
    `fp8`: the drafter's GEMM weights as E4M3 codes with per-row scales."""
    import torch

    from speculative_drafting_pe_gb300 import binding, synth

    wl = synth.WORKLOADS[name]
    key = (wl.shape.name, wl.seed, fp8)
    if key not in weights_cache:
        weights_cache.clear()
        torch.cuda.empty_cache()
        W0 = synth.make_weights(wl.shape, wl.seed, device=dev)
        weights_cache[key] = synth.quantize_weights_fp8(W0) if fp8 else (W0, None)
        del W0
    W, scales = weights_cache[key]
    inp = synth.make_step_inputs(wl, device=dev)
    seq_np = inp.seq_lens.cpu().numpy()
    drafter = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=wl.K, fp8_scales=scales)
    B, K = wl.B, wl.K
    drafts = torch.empty(B, K, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    drafter.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table, inp.num_pages,
                  inp.k_cache, inp.v_cache, K, drafts=drafts, status=status)
    torch.cuda.synchronize()
    g = torch.as_tensor(synth.plant_targets(drafts.cpu().numpy(), inp.alpha, wl.shape.vocab, wl.seed), device=dev)
    vout = {}

    def step():
        drafter.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                      inp.num_pages, inp.k_cache, inp.v_cache, K, drafts=drafts, status=status)
        binding.verify_rebuild(drafts, g, inp.page_table, inp.num_pages, inp.positions, inp.seq_lens, out=vout)

    for _ in range(3):
        step()
    per_kind = {}
    for kind in binding.KERNEL_KINDS:
        drafter.profile_start(kind, 64)
        for _ in range(3):
            step()
        ms, n = drafter.profile_stop()
        if n > 0:
            per_kind[kind] = (ms / 3.0, (ms / 1e3) / n)
    dominant = max(per_kind, key=lambda k: per_kind[k][0])
    sg = drafter.step_graph(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                            inp.num_pages, inp.k_cache, inp.v_cache, K, g)
    for _ in range(3):
        sg.launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(replays):
        sg.launch()
    e1.record(stream)
    torch.cuda.synchronize()
    assert drafter.device_errors() == 0
    ms_step = e0.elapsed_time(e1) / replays
    roof = roofline_of(dominant, wl, seq_np, per_kind[dominant][1], peaks, fp8=fp8)
    out = {"steps_s": 1e3 / ms_step, "ms_per_step": ms_step, "draft_tok_s": 1e3 / ms_step * B * K,
           "step_bytes": step_bytes(wl, seq_np, fp8=fp8),
           "step_hbm_frac": step_bytes(wl, seq_np, fp8=fp8) / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"],
           "dominant": dominant, "dominant_us_per_launch": per_kind[dominant][1] * 1e6,
           "dominant_roofline": {k: roof[k] for k in ("bound", "achieved", "unit", "frac")},
           "kernel_ms_per_step": {k: round(v[0], 4) for k, v in sorted(per_kind.items(), key=lambda x: -x[1][0])}}
    sg.close()
    drafter.close()
    del inp
    return out



def bench_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from speculative_drafting_pe_gb300 import binding, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    binding.load()

    wl = synth.WORKLOADS[args.workload]
    if args.max_prefix > 0:
        import dataclasses
        cap = args.max_prefix
        wl = dataclasses.replace(wl, prefix=(min(wl.prefix[0], cap), min(wl.prefix[1], cap)))
    K_max = max(wl.K, 11) if wl.B == 1 and wl.shape.name.startswith("qwen") else wl.K
    W = synth.make_weights(wl.shape, wl.seed, device=dev)
    scales = None
    if args.fp8:
        W, scales = synth.quantize_weights_fp8(W)
    inp = synth.make_step_inputs(wl, device=dev)
    drafter = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=K_max, fp8_scales=scales)
    stream = torch.cuda.current_stream()
    B, K = wl.B, wl.K
    seq_np = inp.seq_lens.cpu().numpy()

    drafts = torch.empty(B, K, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    drafter.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                  inp.num_pages, inp.k_cache, inp.v_cache, K, drafts=drafts, status=status)
    torch.cuda.synchronize()
    g = torch.as_tensor(synth.plant_targets(drafts.cpu().numpy(), inp.alpha, wl.shape.vocab, wl.seed), device=dev)
    vout = {}

    def step():
        drafter.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                      inp.num_pages, inp.k_cache, inp.v_cache, K, drafts=drafts, status=status)
        binding.verify_rebuild(drafts, g, inp.page_table, inp.num_pages, inp.positions, inp.seq_lens,
                               out=vout)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert drafter.device_errors() == 0

    # per-kernel shares (untimed): each kind profiled over a few steps
    shares = {}
    for kind in binding.KERNEL_KINDS:
        drafter.profile_start(kind, 64)
        for _ in range(3):
            step()
        ms, n = drafter.profile_stop()
        shares[kind] = ms / 3.0
    dominant = max(shares, key=shares.get)

    # ---------------- timed region A: step-graph replays (value, clocks)
    sg = drafter.step_graph(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                            inp.num_pages, inp.k_cache, inp.v_cache, K, g)
    for _ in range(max(3, args.warmup)):
        sg.launch()
    torch.cuda.synchronize()
    launches_per_step = sg.launch_count()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_id = vis.split(",")[local] if vis.strip() else str(local)
    sampler = ClockSampler(smi_id)
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        sg.launch()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_steps_per_s(world, args.steps, elapsed_ms)
    acc = sg.out["accepted"].cpu().numpy()
    assert (sg.out["drafts"] == drafts).all().item()

    # ---------------- timed region B: the same K steps launched directly, the
    # dominant kernel bracketed by CUDA events on its launch stream (roofline)
    drafter.profile_start(dominant, args.steps * 8 + 8)
    torch.cuda.synchronize()
    d_start = torch.cuda.Event(enable_timing=True)
    d_end = torch.cuda.Event(enable_timing=True)
    d_start.record(stream)
    for _ in range(args.steps):
        step()
    d_end.record(stream)
    torch.cuda.synchronize()
    direct_ms = d_start.elapsed_time(d_end) / args.steps
    dom_ms, dom_n = drafter.profile_stop()
    assert drafter.device_errors() == 0

    # ---------------- the same step with L2 cold: a buffer larger than L2 is
    # written between timed steps (outside the events), so no weight or KV
    # byte of the previous step is still cached when a step starts
    cold = None
    if not args.no_sweep:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        n_cold = max(args.steps, 20)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_cold)]
        for _ in range(3):
            flush.fill_(1)
            sg.launch()
        torch.cuda.synchronize()
        for i in range(n_cold):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            sg.launch()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        cold_ms = sum(a.elapsed_time(b) for a, b in evs) / n_cold
        cold = {"ms_per_step": cold_ms, "steps_s": 1e3 / cold_ms,
                "step_hbm_frac": step_bytes(wl, seq_np, fp8=args.fp8) / (cold_ms / 1e3) / 1e9 /
                                 load_peaks()[0]["hbm_gbs"],
                "steps": n_cold, "flush": "256 MB buffer written between timed steps, outside the timed events"}
        del flush

    # ---------------- flatness in K at B=1 (step graphs of the draft pass
    # followed by the verify/rebuild, ~3 us of the step)
    k_sweep = None
    k_sweep_seq = None
    if not args.no_sweep and wl.B == 1 and wl.shape.name.startswith("qwen"):
        k_sweep, k_sweep_seq = {}, {}
        for Ks in (3, 7, 11):
            inp_k = synth.make_step_inputs(wl, device=dev, K=Ks)
            g_k = torch.zeros(1, Ks + 1, dtype=torch.int32, device=dev)
            for sequential, out in ((False, k_sweep), (True, k_sweep_seq)):
                sg_k = drafter.step_graph(inp_k.last_token, inp_k.target_hidden, inp_k.positions, inp_k.seq_lens,
                                          inp_k.page_table, inp_k.num_pages, inp_k.k_cache, inp_k.v_cache, Ks, g_k,
                                          sequential=sequential)
                for _ in range(10):
                    sg_k.launch()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                n = 100 if sequential else 300
                e0.record(stream)
                for _ in range(n):
                    sg_k.launch()
                e1.record(stream)
                torch.cuda.synchronize()
                out[str(Ks)] = e0.elapsed_time(e1) / n
                sg_k.close()
            del inp_k

    # ---------------- end to end through the public API with pinned host buffers:
    # every step copies its inputs host->device (one pinned staging buffer
    # holding every input, 256-byte aligned, in one copy), replays the step
    # graph and copies all of the step's results (the graph's packed int32
    # output buffer) device->host in one copy
    srcs = (("last_token", inp.last_token), ("target_hidden", inp.target_hidden), ("positions", inp.positions),
            ("seq_lens", inp.seq_lens), ("page_table", inp.page_table), ("targets", g))
    in_offs, in_total = {}, 0
    for n, t in srcs:
        in_offs[n] = in_total
        in_total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_flat = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    dev_flat = torch.empty(in_total, dtype=torch.uint8, device=dev)

    def typed_view(flat, n, t):
        return flat.narrow(0, in_offs[n], t.numel() * t.element_size()).view(t.dtype).view(t.shape)

    host_in = {n: typed_view(host_flat, n, t) for n, t in srcs}
    dev_in = {n: typed_view(dev_flat, n, t) for n, t in srcs}
    for n, t in srcs:
        host_in[n].copy_(t)
    sg_e = drafter.step_graph(dev_in["last_token"], dev_in["target_hidden"], dev_in["positions"],
                              dev_in["seq_lens"], dev_in["page_table"], inp.num_pages, inp.k_cache, inp.v_cache, K,
                              dev_in["targets"])
    host_out_flat = torch.empty(sg_e.out_packed.shape, dtype=torch.int32).pin_memory()
    drafts_off = (sg_e.out["drafts"].data_ptr() - sg_e.out_packed.data_ptr()) // 4
    host_drafts = host_out_flat.narrow(0, drafts_off, sg_e.out["drafts"].numel()).view(sg_e.out["drafts"].shape)

    def e2e_step():
        dev_flat.copy_(host_flat, non_blocking=True)
        sg_e.launch()
        host_out_flat.copy_(sg_e.out_packed, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    assert torch.equal(host_drafts, drafts.cpu())
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    h2d = host_flat.numel() * host_flat.element_size()
    d2h = host_out_flat.numel() * host_out_flat.element_size()

    # ---------------- every workload of the metric (C2, C3, C4): one line each
    sweep = None
    fp8_lines = None
    if not args.no_sweep and world == 1 and args.max_prefix == 0 and not args.fp8:
        peaks0, _ = load_peaks()
        del sg, sg_e
        drafter.close()
        cache = {(wl.shape.name, wl.seed, False): (W, None)}
        sweep = {}
        for name in SWEEP_WORKLOADS:
            sweep[name] = sweep_workload(name, dev, cache, peaks0, max(args.steps, 50))
        fp8_lines = {}
        for name in FP8_WORKLOADS:
            fp8_lines[name] = sweep_workload(name, dev, cache, peaks0, max(args.steps, 50), fp8=True)
        cache.clear()

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peaks, peaks_src = load_peaks()
    dom_bytes, dom_flops = algorithmic_work(dominant, wl, seq_np, chained=shares.get("layer_chain", 0.0) > 0.0,
                                            fp8=args.fp8)
    dom_avg_s = (dom_ms / 1e3) / max(dom_n, 1)
    t_hbm = dom_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = dom_flops / (peaks["bf16_tflops_sustained"] * 1e12)
    if t_hbm >= t_tc:
        achieved = dom_bytes / dom_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    else:
        achieved = dom_flops / dom_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops_sustained"]}
    if dominant == "lm_head":
        # the LM head loads its first 40 MB of weight rows evict-last, so that
        # they stay in L2 from one step to the next: the fraction without the
        # bytes that window serves from L2
        e_w = 1 if args.fp8 else (2 if wl.shape.dtype == "bf16" else 4)
        keep_tiles = (40 << 20) // (128 * wl.shape.hidden * e_w)
        window = min(keep_tiles * 128, wl.shape.vocab) * wl.shape.hidden * e_w
        roof["l2_window_bytes"] = window
        roof["frac_without_l2_window"] = (dom_bytes - window) / dom_avg_s / 1e9 / peaks["hbm_gbs"]
    roof.update({"traffic": None if args.fp8 else read_profile_traffic(dominant, args.workload), "kernel": dominant,
                 "launches_timed": dom_n, "avg_launch_us": dom_avg_s * 1e6,
                 "algorithmic_bytes_per_launch": dom_bytes, "algorithmic_flops_per_launch": dom_flops,
                 "timed_in": "a second timed region of the same steps launched directly (events cannot sit inside "
                             "a graph replay)",
                 "peak_source": f"{peaks_src} (MEASURED_PEAKS.json)" if peaks_src == "measured" else "fallback"})
    total_share = sum(shares.values())
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8w" if args.fp8 else wl.shape.dtype,
        "data": "synthetic (seeded inputs, random-init drafter weights)",
        "config": {"workload": workload_desc(wl) + (", FP8 (E4M3) GEMM weights with per-row scales" if args.fp8 else ""),
                   "name": wl.name, "B": B, "K": K,
                   "l2": "no flush: each step streams >1 GB of weights, larger than the 126 MB L2",
                   "parallelism": f"replicas x{world} (requests shard with no exchange)" if world > 1 else "1 GPU"},
        "draft_tok_s": value * B * K,
        "step_hbm_gbs": step_bytes(wl, seq_np, fp8=args.fp8) / (ms_per_step / 1e3) / 1e9,
        "step_hbm_frac": step_bytes(wl, seq_np, fp8=args.fp8) / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
        "mean_accepted": float(acc.mean()),
        "direct_launch_ms_per_step": direct_ms,
        "roofline": roof,
        "kernel_share": {k: round(v / total_share, 4) for k, v in sorted(shares.items(), key=lambda x: -x[1])},
        "kernel_ms_per_step": {k: round(v, 4) for k, v in sorted(shares.items(), key=lambda x: -x[1])},
        "clocks": clocks,
        "e2e": {"value": whole_job_steps_per_s(world, args.steps, e2e_ms), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
    }
    if k_sweep:
        line["k_sweep_step_ms"] = k_sweep
        line["k_sweep_note"] = "ms per step-graph replay (draft pass + verify/rebuild) at B=1, K = 3 / 7 / 11"
        line["k11_over_k3"] = k_sweep["11"] / k_sweep["3"]
    if k_sweep_seq:
        line["k_sweep_sequential_step_ms"] = k_sweep_seq
        line["k_sweep_sequential_note"] = ("the same steps with sequential EAGLE-style drafting (K one-row passes "
                                           "on the same kernels, pe_draft_sequential) in place of the parallel pass")
        line["sequential_k11_over_k3"] = k_sweep_seq["11"] / k_sweep_seq["3"]
        line["parallel_speedup_over_sequential"] = {k: k_sweep_seq[k] / k_sweep[k] for k in k_sweep}
    if cold:
        line["cold_l2"] = cold
    if sweep:
        line["sweep"] = sweep
    if fp8_lines:
        line["fp8_weights"] = fp8_lines
        line["fp8_note"] = ("the same workloads with FP8 (E4M3) GEMM weights and per-row fp32 scales (bf16 "
                            "activations and KV); step_bytes counts one byte per weight plus the scales")
    if world == 1 and not args.no_cpu_baseline:
        try:
            res = run_oracle_subprocess(args.workload, args.cpu_seconds, 1000, fp8=args.fp8)
            line["cpu_baseline"] = cpu_baseline_obj(res, wl)
        except Exception as exc:  # the baseline is reported, never required
            line["cpu_baseline"] = {"value": None, "unit": "steps/s", "cores": len(os.sched_getaffinity(0)),
                                    "kind": "oracle", "sample": f"failed: {exc}"[:300]}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def read_profile_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    profiles/traffic_<kernel>_<workload>.md, if that summary was taken on the
    current kernel sources (its source_hash line); else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("source_hash", "dram_bytes_per_launch")):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_hash") != kernel_source_hash():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_hash(csrc=None):
    """Hash of the kernel sources (all of csrc) with comments and whitespace
    removed: a comment edit does not change the kernels the profile counters
    were taken on, any code edit does."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "speculative_drafting_pe_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            text = re.sub(r"\s+", " ", text).strip()
            h.update(name.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ reference arm

def bench_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from speculative_drafting_pe_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    res = run_oracle_subprocess(args.workload, max(args.cpu_seconds, 60.0), args.steps, warmup=args.warmup)
    value = res["steps"] / res["seconds"]
    base = cpu_baseline_obj(res, wl)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": res["steps"],
        "steps_requested": args.steps,
        "warmup": res["warmup"],
        "ms_per_step": 1e3 / value,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded inputs, random-init drafter weights)",
        "config": {"workload": workload_desc(wl), "name": wl.name, "B": wl.B, "K": wl.K,
                   "l2": "host run (no GPU)", "parallelism": "host cores"},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the CPU float64 oracle as it stands, time-boxed: each step is one full oracle step of the workload",
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.oracle_worker:
        oracle_worker(args)
        return
    if args.impl == "reference":
        bench_reference(args)
        return
    bench_ours(args)


if __name__ == "__main__":
    main()
