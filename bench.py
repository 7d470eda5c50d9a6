"""Benchmark of the split-KV attention path on GB300: one JSON line on rank 0.

A step is one pass of the whole path over one batch of resident synthetic
input: block costs -> LPT plan -> work lists (host) -> work upload ->
partial attention -> merge (device).  Default workload: the largest single-GPU
shape (B=1, Hq=32, Hkv=8, d=128, 256 causal queries after a 1,048,576-token
context, bf16, paged block_len 2048, 64 shards), bound by the bf16 tensor pipe:
its value is TFLOP/s.  A workload bound by HBM (decode) reports GB/s of K/V read.
The same run also times the decode, short-query and variable-length forward
workloads and the short-query backward pass, each under ``per_workload``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload largest]
                    [--impl ours|reference] [--kernel auto|simt|decode|tc]
                    [--per-workload decode,shortq,varlen] [--per-backward shortq]

--gpus N > 1 runs one process per GPU under torch.distributed.run (bench.py
relaunches itself that way when started without WORLD_SIZE; a WORLD_SIZE that
differs from N is an error).  Every rank solves its own copy of the workload
(replicas; the path has no cross-GPU exchange on one device): value = all
ranks' work / max-over-ranks time.
--impl reference times the fp64 CPU oracle on the host cores instead.
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Split-KV attn fwd TFLOP/s & KV-read GB/s vs GB300 roofline, short-Q/long-KV"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SUSTAINED_REGION_S = 1.0  # timed regions at least this long compare with the sustained bf16 peak
L2_BYTES = 129 * 1024 * 1024


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="largest")
    ap.add_argument("--per-workload", default="decode,shortq,varlen,specdec",
                    help="forward workloads also timed in the same run (comma list, '' for none)")
    ap.add_argument("--per-backward", default="shortq,largest,varlen",
                    help="workloads whose backward pass is also timed in the same run ('' for none)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "decode", "tc"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--fused", action="store_true",
                    help="splitkv_attn_fused (one launch with the decode and tensor-core kernels) instead of partial + merge")
    ap.add_argument("--planner", choices=["lpt", "dcp"], default="lpt",
                    help="lpt: cost-aware LPT onto all shards; dcp: shard count chosen by the attention + "
                         "reduction completion model (splitkv_plan_dcp)")
    ap.add_argument("--tail-pieces", type=int, default=None,
                    help="cut the items of the last partial wave of CTAs into this many pieces "
                         "(splitkv_build_work_tail; 0: no cut; default: the runner's choice, 4 when the last "
                         "wave of CTAs is at most half full)")
    ap.add_argument("--item-blocks", type=int, default=0,
                    help="cut work items into runs of at most this many blocks (0: one item per shard and "
                         "sequence)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (delta, per-shard dK/dV + partial dQ, dQ reduce) instead")
    ap.add_argument("--context", type=int, default=None,
                    help="override the context length (smaller cases for profiling)")
    return ap.parse_args(argv)


# --------------------------------------------------------------- distributed


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def finish(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(dist_ctx, local_seconds, local_units, device=None):
    """Max of the per-rank times and sum of the per-rank units over all ranks."""
    if dist_ctx.pg is None:
        return local_seconds, local_units
    import torch

    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    dist_ctx.pg.all_reduce(t, op=dist_ctx.pg.ReduceOp.MAX)
    dist_ctx.pg.all_reduce(u, op=dist_ctx.pg.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# -------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 20 ms, time-stamped); only the samples taken
    inside the timed region (mark_start .. mark_end, host clock) are summarised."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id, path):
        self.gpu_id, self.path, self.proc = gpu_id, path, None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        return self.summary()

    @staticmethod
    def _stamp(text):
        import datetime

        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((self._stamp(parts[0]), float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if r[0] is not None and self.t0 is not None and self.t1 is not None
                  and self.t0 <= r[0] <= self.t1 + 0.02]
        window = "timed region"
        if not inside:  # region shorter than the sampling period: the samples closest to it
            mid = 0.5 * (self.t0 + self.t1) if self.t0 is not None and self.t1 is not None else None
            inside = sorted(rows, key=lambda r: abs(r[0] - mid) if (r[0] is not None and mid is not None) else 0)[:2]
            window = "nearest samples (region shorter than the 20 ms sampling period)"
        reasons = sorted({n for r in inside for n, v in zip(names, r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "power_w_max": max(r[3] for r in inside),
                "window": window}


def gpu_nvsmi_id(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # pragma: no cover - older torch
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


# -------------------------------------------------------------- accounting


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def unit_pairs(q_len, kv_len, causal):
    """Visible (query token, key) pairs of one sequence: q_len x kv_len without a mask; with
    the causal tail token t sees kv_len - q_len + t + 1 keys."""
    q_len, kv_len = int(q_len), int(kv_len)
    if not causal:
        return q_len * kv_len
    return q_len * (kv_len - q_len) + q_len * (q_len + 1) // 2


def workload_accounting(w, q_len, kv_len, block_cost, part_rows):
    """Algorithmic flops and bytes of one pass: flops = 4 d Hq x (visible query-key pairs,
    the sum of the block costs); K/V bytes = sum(kv_len) Hkv d x 2 tensors x element size,
    each read once; Q bytes likewise; partial bytes = part_rows Hq (d + 1) x 4 (fp32 O_i and
    L_i, written by the partial kernel and read by the merge)."""
    pairs = int(np.sum(block_cost))  # visible (query token, key) pairs, per query head
    flops = 4.0 * w.d * w.Hq * pairs
    kv_bytes = float(sum(kv_len)) * w.Hkv * w.d * 2 * w.elem_bytes
    q_bytes = float(sum(q_len)) * w.Hq * w.d * w.elem_bytes
    part_bytes = float(part_rows) * w.Hq * (w.d + 1) * 4
    return {"flops": flops, "kv_bytes": kv_bytes, "q_bytes": q_bytes, "part_bytes": part_bytes,
            "partial_bytes": kv_bytes + q_bytes + part_bytes}


def traffic_for(kernel_name, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel_name}/{workload}")
    if not e:
        return None
    src = os.path.join(ROOT, e["source"])
    import hashlib

    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != e["sha256"]:
        return None
    return float(e["bytes_per_launch"])


def dcp_model(w):
    """Costs of the split-selection model for a context-parallel deployment of this
    workload: alpha = seconds per unit of block cost on one rank (4*d*Hq flops at
    1200 TFLOP/s, the tensor-core kernel's measured rate), gamma = seconds per K/V
    token streamed (Hkv*d*2 elements at 5.7 TB/s, the decode kernel's measured rate),
    beta = seconds per partial row exchanged and merged (Hq*(d+1)*4 bytes at 900 GB/s
    of NVLink)."""
    return (4.0 * w.d * w.Hq / 1.2e15, w.Hq * (w.d + 1) * 4.0 / 0.9e12,
            w.Hkv * w.d * 2.0 * w.elem_bytes / 5.7e12)


# -------------------------------------------------------------- our arm


def _binding(w, acc, peaks):
    """The roofline that binds the partial kernel: HBM when its algorithmic intensity is
    below the ridge (peak flops / peak bytes), the bf16 tensor pipe above it."""
    return "hbm" if acc["flops"] / acc["partial_bytes"] < 1e3 * peaks["bf16_tflops"] / peaks["hbm_gbs"] else "tensor"


def _timed_steps(torch, n, step, stream, sampler):
    """n steps, each bracketed by events; returns (total s, mean per-step event deltas, clocks)."""
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(n)]
    if sampler is not None:
        sampler.start()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.mark_start()
    t0.record(stream)
    for i in range(n):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.mark_end()
    clocks = sampler.stop() if sampler is not None else None
    return t0.elapsed_time(t1) / 1e3, evs, clocks


def measure_forward(args, dctx, name, dev, headline=False):
    """Times the forward path of one workload; returns (bench fields, objects for e2e / cpu)."""
    import torch

    from context_long_attention_lpt_gb300 import splitkv as K
    from context_long_attention_lpt_gb300 import workloads as wl
    from context_long_attention_lpt_gb300.runner import SplitKVAttention

    w = wl.WORKLOADS[name]
    if args.context and headline:
        w = wl.custom(w, context=args.context)
    kernel = {"auto": K.KERNEL_AUTO, "simt": K.KERNEL_SIMT, "decode": K.KERNEL_DECODE,
              "tc": K.KERNEL_TC}[args.kernel if headline else "auto"]
    inp = wl.make_inputs(w, device=f"cuda:{dev}")
    alpha, beta, gamma = dcp_model(w)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, device=f"cuda:{dev}", kernel=kernel, fused=args.fused,
                           planner=args.planner, dcp_alpha=alpha, dcp_beta=beta, dcp_gamma=gamma,
                           item_blocks=args.item_blocks if headline else 0,
                           tail_pieces=args.tail_pieces if headline else None)
    fused_one_launch = run.fused and run.fuses_in_one_launch()
    out = torch.empty((run.total_q, w.Hq, w.d), dtype=inp.q.dtype, device=f"cuda:{dev}")
    lse = torch.empty((run.total_q, w.Hq), dtype=torch.float32, device=f"cuda:{dev}")
    acc = workload_accounting(w, inp.q_len, inp.kv_len, run.block_cost, run.part_rows)
    stream = torch.cuda.current_stream()

    # One step = the device calls on the plan made at the end of the previous step, then the
    # next step's plan (block costs, LPT, work lists, descriptor upload).  Planning after the
    # launches lets the host work overlap the kernels, so the events around each launch time
    # the kernel and not a device waiting for the host; every step still plans once.  The
    # upload goes on its own stream into the descriptor buffer the running step does not read.
    upload_stream = torch.cuda.Stream()
    run.plan(stream=upload_stream)

    def step(ev=None):
        run.wait_plan(stream)  # the upload's cross-stream wait stays out of the kernel's events
        if ev is not None:
            ev[0].record(stream)
        if run.fused:
            run.fused_call(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse)
            if ev is not None:
                ev[1].record(stream)
                ev[2].record(stream)
        else:
            run.partial(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
            if ev is not None:
                ev[1].record(stream)
            run.merge(out, lse)
            if ev is not None:
                ev[2].record(stream)
        run.plan(stream=upload_stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_nvsmi_id(torch, dev), os.path.join(ROOT, f".bench_clocks_{dctx.rank}.csv"))
    dctx.barrier()
    host0 = time.perf_counter()
    local_s, evs, clocks = _timed_steps(torch, args.steps, step, stream, sampler)
    host_s = time.perf_counter() - host0
    dctx.barrier()
    try:
        os.remove(sampler.path)
    except OSError:
        pass
    kernel_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)  # the dominant kernel's launch
    merge_ms = None if run.fused else sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)

    peaks, peak_src = load_peaks()
    kname = K.KERNEL_NAMES[run.kernel_used()] + ("_fused" if fused_one_launch else "")
    if fused_one_launch:  # the same launch also reads the partials back and writes the output
        acc["partial_bytes"] += acc["part_bytes"] + float(run.total_q) * w.Hq * (w.d * w.elem_bytes + 4)
    bound = _binding(w, acc, peaks)
    if bound == "hbm":
        achieved = acc["partial_bytes"] / (kernel_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
        units_local, unit, scale = acc["kv_bytes"] * args.steps, "GB/s", 1e9
    else:
        achieved = acc["flops"] / (kernel_ms / 1e3) / 1e12
        # A kernel timed inside a timed region of a second or more runs into the power limiter,
        # as the sustained GEMM figure did; a shorter region is compared with the burst figure.
        kind = "sustained" if local_s >= SUSTAINED_REGION_S else "burst"
        peak = peaks["bf16_tflops_sustained"] if kind == "sustained" else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                "frac": achieved / peak, "frac_of_burst": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}
        units_local, unit, scale = acc["flops"] * args.steps, "TFLOP/s", 1e12
    roof.update({"traffic": traffic_for(f"partial_{kname}", w.name), "kernel": f"partial_{kname}",
                 "kernel_ms": kernel_ms, "merge_ms": merge_ms, "peak_source": peak_src,
                 "algorithmic_per_launch": acc["partial_bytes"] if bound == "hbm" else acc["flops"]})
    t_max, units = aggregate(dctx, local_s, units_local, device=f"cuda:{dev}")
    _, kv_all = aggregate(dctx, local_s, acc["kv_bytes"] * args.steps, device=f"cuda:{dev}")
    _, fl_all = aggregate(dctx, local_s, acc["flops"] * args.steps, device=f"cuda:{dev}")
    fields = {
        "value": units / t_max / scale, "unit": unit, "ms_per_step": 1e3 * t_max / args.steps,
        "steps": args.steps, "kv_gbs": kv_all / t_max / 1e9, "tflops": fl_all / t_max / 1e12,
        "shape": w.description, "kernel": kname, "n_items": run.n_items, "tail_pieces": run.tail_pieces,
        "lpt_imbalance": run.imbalance,
        "planner": args.planner, "shards_used": run.n_shards_used, "part_rows": run.part_rows,
        "host_s": host_s, "roofline": roof, "clocks": clocks,
        "gpu_launches": (1 if fused_one_launch else 2) * args.steps,
        "l2": (f"inputs larger than L2 (K/V {acc['kv_bytes'] / 1e9:.2f} GB vs L2 {L2_BYTES / 1e6:.0f} MB); "
               "no flush") if acc["kv_bytes"] > L2_BYTES else "inputs smaller than L2; not flushed",
    }
    return fields, (w, inp, run, acc, bound)


def measure_backward(args, dctx, name, dev):
    """Times the backward pass of one workload (delta, per-shard dK/dV + partial dQ, dQ
    reduction) over its LPT plan; the forward output is computed once, untimed."""
    import torch

    from context_long_attention_lpt_gb300 import splitkv as K
    from context_long_attention_lpt_gb300 import workloads as wl
    from context_long_attention_lpt_gb300.runner import SplitKVAttention

    w = wl.WORKLOADS[name]
    if args.context and args.backward:
        w = wl.custom(w, context=args.context)
    inp = wl.make_inputs(w, device=f"cuda:{dev}")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, device=f"cuda:{dev}")
    out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    acc = workload_accounting(w, inp.q_len, inp.kv_len, run.block_cost, run.part_rows)
    g = torch.Generator(device=out.device).manual_seed(0)
    dout = torch.randn(out.shape, generator=g, device=out.device, dtype=torch.float32).to(out.dtype)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)

    for _ in range(max(2, min(args.warmup, 5))):
        step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    sampler = ClockSampler(gpu_nvsmi_id(torch, dev), os.path.join(ROOT, f".bench_clocks_{dctx.rank}.csv"))
    dctx.barrier()
    local_s, _, clocks = _timed_steps(torch, n, step, stream, sampler)
    dctx.barrier()
    try:
        os.remove(sampler.path)
    except OSError:
        pass
    flops = 2.5 * acc["flops"]
    t_max, units = aggregate(dctx, local_s, flops * n, device=f"cuda:{dev}")
    s = t_max / n
    peaks, src = load_peaks()
    code = K.SPLITKV_BF16 if w.dtype == "bf16" else K.SPLITKV_F32
    tc = K.splitkv_backward_kernel(w.Hq, w.Hkv, w.d, w.block_len, code) == K.KERNEL_TC
    achieved = flops / (local_s / n) / 1e12
    if tc:
        kind = "sustained" if local_s >= SUSTAINED_REGION_S else "burst"
        peak = peaks["bf16_tflops_sustained"] if kind == "sustained" else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                "frac": achieved / peak, "frac_of_burst": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"], "peak_source": src,
                "note": "whole backward step: delta, dQ and dK/dV tensor-core kernels, dQ reduction"}
    else:
        roof = {"bound": "fp32_fma", "achieved": achieved, "unit": "TFLOP/s",
                "note": "CUDA-core kernel: bf16 inputs, fp32 FMA arithmetic"}
    return {"value": units / t_max / 1e12, "unit": "TFLOP/s", "ms_per_step": 1e3 * s, "steps": n,
            "shape": w.description, "kernel": "backward_tcgen05" if tc else "backward_simt",
            "lpt_imbalance": run.imbalance, "roofline": roof, "clocks": clocks,
            "gpu_launches": (4 if tc else 5) * n,
            "accounting": "flops = 2.5 x forward (QK^T recomputed, dP, dV, dQ, dK)"}


def run_ours(args, dctx):
    import torch

    from context_long_attention_lpt_gb300 import splitkv as K

    dctx.init("nccl")
    dev = dctx.local_rank
    torch.cuda.set_device(dev)
    K.lib()
    if args.backward:
        f = measure_backward(args, dctx, args.workload, dev)
        line = {"metric": METRIC + " (backward pass)", "value": f["value"], "unit": f["unit"],
                "n_gpus": dctx.world, "steps": f["steps"], "warmup": args.warmup, "ms_per_step": f["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": args.workload, "shape": f["shape"],
                                                "kernel": f["kernel"], "parallelism": f"replicas x{dctx.world}"},
                "roofline": f["roofline"], "clocks": f["clocks"], "gpu_launches": f["gpu_launches"]}
        if dctx.rank == 0:
            print(json.dumps(line), flush=True)
        dctx.finish()
        return

    f, (w, inp, run, acc, bound) = measure_forward(args, dctx, args.workload, dev, headline=True)
    # planner time alone (host), for the report
    tp = time.perf_counter()
    for _ in range(20):
        K.splitkv_plan(K.splitkv_block_costs(run._q_len_np, run._kv_len_np, w.block_len, w.causal), w.n_shards)
    planner_us = (time.perf_counter() - tp) / 20 * 1e6
    # end to end: host inputs -> device, the path, result -> host, every step
    e2e = run_e2e(args, w, inp, run, dev, acc, bound) if args.e2e_steps > 0 else None
    cpu = None
    if dctx.rank == 0 and dctx.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, args.cpu_seconds, bound)
    del inp, run
    torch.cuda.empty_cache()

    per = {}
    for name in [x for x in args.per_workload.split(",") if x and x != args.workload]:
        pf, objs = measure_forward(args, dctx, name, dev)
        del objs
        torch.cuda.empty_cache()
        per[name] = {k: pf[k] for k in ("value", "unit", "ms_per_step", "steps", "kv_gbs", "tflops", "shape",
                                        "kernel", "n_items", "tail_pieces", "lpt_imbalance", "shards_used",
                                        "part_rows",
                                        "roofline", "clocks", "gpu_launches", "l2")}
    for name in [x for x in args.per_backward.split(",") if x]:
        per[f"backward/{name}"] = measure_backward(args, dctx, name, dev)
        torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": f["value"], "unit": f["unit"], "n_gpus": dctx.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": f["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "kv_gbs": f["kv_gbs"], "tflops": f["tflops"],
        "config": {"workload": w.name, "shape": f["shape"], "kernel": f["kernel"], "n_items": f["n_items"],
                   "tail_pieces": f["tail_pieces"],
                   "lpt_imbalance": f["lpt_imbalance"], "planner": f["planner"], "shards_used": f["shards_used"],
                   "part_rows": f["part_rows"], "planner_us": planner_us, "host_s": f["host_s"], "l2": f["l2"],
                   "parallelism": f"replicas x{dctx.world}"},
        "roofline": f["roofline"],
        "gpu_launches": f["gpu_launches"],
        "clocks": f["clocks"],
        "e2e": e2e,
        "per_workload": per,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if dctx.rank == 0:
        print(json.dumps(line), flush=True)
    dctx.finish()


def run_e2e(args, w, inp, run, dev, acc, bound):
    import torch

    d = f"cuda:{dev}"
    host = {k: getattr(inp, k).cpu().pin_memory() for k in ("q", "k_pool", "v_pool", "block_table")}
    out_h = torch.empty((run.total_q, w.Hq, w.d), dtype=inp.q.dtype).pin_memory()
    lse_h = torch.empty((run.total_q, w.Hq), dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * 4
    # Two device copies of the inputs, used in turn: step i+1's inputs cross the host link
    # on a copy stream while step i computes on the compute stream (each step still copies
    # all of its inputs in and its result out inside the timed region).
    comp = torch.cuda.current_stream(d)
    copy_stream = torch.cuda.Stream(device=d)
    dbuf = [{k: torch.empty_like(v, device=d) for k, v in host.items()} for _ in range(2)]
    dout = [(torch.empty((run.total_q, w.Hq, w.d), dtype=inp.q.dtype, device=d),
             torch.empty((run.total_q, w.Hq), dtype=torch.float32, device=d)) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def one(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if used[b]:
                copy_stream.wait_event(ev_free[b])  # the step that last read this copy is done
            # block costs, LPT, work lists and their upload, as every step: the upload goes on
            # the copy stream ahead of the inputs, so it never queues behind the next step's copy
            run.plan(stream=copy_stream)
            for k, v in host.items():
                dbuf[b][k].copy_(v, non_blocking=True)
            ev_in[b].record(copy_stream)
        comp.wait_event(ev_in[b])
        out, lse = run(dbuf[b]["q"], dbuf[b]["k_pool"], dbuf[b]["v_pool"], dbuf[b]["block_table"], w.scale,
                       out=dout[b][0], lse=dout[b][1], stream=comp)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        ev_free[b].record(comp)
        used[b] = True

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    n = args.e2e_steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    copy_stream.wait_event(t0)  # the copies of the timed steps start inside the timed region
    for i in range(3, 3 + n):
        one(i)
    t1.record(comp)  # after the last step's result has been read back
    torch.cuda.synchronize()
    s = t0.elapsed_time(t1) / 1e3
    h2d += run.work_host.size * 4
    del dbuf, dout
    if bound == "hbm":
        value, unit = acc["kv_bytes"] * n / s / 1e9, "GB/s"
    else:
        value, unit = acc["flops"] * n / s / 1e12, "TFLOP/s"
    return {"value": value, "unit": unit, "ms_per_step": 1e3 * s / n, "steps": n,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------- oracle on the host


def _oracle_unit(w, inp_cpu, b, kvh, n_keys=None):
    """The oracle's unsharded attention for sequence b, K/V head kvh (its G query heads).

    ``n_keys`` truncates the sequence to its first n_keys keys (a bounded sample;
    the queries keep their place at the end of the truncated sequence).  Returns the
    (K/V bytes, flops) of the sample."""
    import oracle

    cu = int(sum(inp_cpu["q_len"][:b]))
    lq = inp_cpu["q_len"][b]
    g = w.G
    kv = inp_cpu["kv_len"][b] if n_keys is None else max(lq, min(n_keys, inp_cpu["kv_len"][b]))
    q = inp_cpu["q"][cu: cu + lq, kvh * g: (kvh + 1) * g]
    kp = inp_cpu["k_pool"][:, :, kvh: kvh + 1]
    vp = inp_cpu["v_pool"][:, :, kvh: kvh + 1]
    table = inp_cpu["block_table"][b: b + 1]
    oracle.attention(q, kp, vp, table, [lq], [kv], w.block_len, w.causal, w.scale)
    return float(kv) * w.d * 2 * w.elem_bytes, 4.0 * w.d * g * unit_pairs(lq, kv, w.causal)


def _pick(bound, nbytes, flops, seconds):
    return (nbytes / seconds / 1e9, "GB/s") if bound == "hbm" else (flops / seconds / 1e12, "TFLOP/s")


def _sample_keys(w, cpu, budget_s):
    """Keys per (sequence, K/V head) unit so that one unit of the oracle takes about budget_s."""
    b0 = 0
    probe = max(w.block_len, min(cpu["kv_len"][b0], 8192))
    t0 = time.perf_counter()
    _oracle_unit(w, cpu, b0, 0, n_keys=probe)
    per_key = max((time.perf_counter() - t0) / probe, 1e-9)
    n = int(budget_s / per_key)
    return max(w.block_len, (n // w.block_len) * w.block_len)


def cpu_baseline(w, inp, seconds, bound):
    """Times the fp64 oracle as it stands on the host cores over a bounded sample: the
    workload's (sequence, K/V head) units in order, each truncated to at most n_keys keys,
    until about ``seconds`` have passed."""
    import torch

    torch.set_num_threads(os.cpu_count() or 1)
    cpu = {"q": inp.q.cpu(), "k_pool": inp.k_pool.cpu(), "v_pool": inp.v_pool.cpu(),
           "block_table": inp.block_table.cpu(), "q_len": inp.q_len, "kv_len": inp.kv_len}
    units = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    n_keys = _sample_keys(w, cpu, seconds / 6)
    t0 = time.perf_counter()
    done, nbytes, flops = 0, 0.0, 0.0
    for b, h in units:
        nb, fl = _oracle_unit(w, cpu, b, h, n_keys=n_keys)
        nbytes += nb
        flops += fl
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    s = time.perf_counter() - t0
    value, unit = _pick(bound, nbytes, flops, s)
    return {"value": value, "unit": unit, "cores": torch.get_num_threads(), "kind": "oracle", "seconds": s,
            "sample": f"{done} of {len(units)} (sequence, K/V head) units of the workload, each truncated to "
                      f"its first {n_keys} keys (queries at the end), fp64 unsharded attention"}


def run_reference(args, dctx):
    """The oracle as the reference arm: rank 0 only, bounded sample per step."""
    import torch

    from context_long_attention_lpt_gb300 import workloads as wl

    if dctx.rank != 0:
        return
    torch.set_num_threads(os.cpu_count() or 1)
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w, device="cpu")
    cpu = {"q": inp.q, "k_pool": inp.k_pool, "v_pool": inp.v_pool, "block_table": inp.block_table,
           "q_len": inp.q_len, "kv_len": inp.kv_len}
    units = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    peaks, _ = load_peaks()
    q_len, kv_len = inp.q_len, inp.kv_len
    flops_all = sum(4.0 * w.d * w.Hq * unit_pairs(a, b, w.causal) for a, b in zip(q_len, kv_len))
    kv_all = float(sum(kv_len)) * w.Hkv * w.d * 2 * w.elem_bytes
    bound = "hbm" if flops_all / kv_all < 1e3 * peaks["bf16_tflops"] / peaks["hbm_gbs"] else "tensor"
    # size each step (one truncated (sequence, K/V head) unit) so the whole run fits the budget
    budget = 150.0
    n_keys = _sample_keys(w, cpu, budget / (args.steps + args.warmup))
    for i in range(args.warmup):
        _oracle_unit(w, cpu, *units[i % len(units)], n_keys=n_keys)
    t0 = time.perf_counter()
    nbytes, flops = 0.0, 0.0
    for i in range(args.steps):
        b, h = units[i % len(units)]
        nb, fl = _oracle_unit(w, cpu, b, h, n_keys=n_keys)
        nbytes += nb
        flops += fl
    s = time.perf_counter() - t0
    value, unit = _pick(bound, nbytes, flops, s)
    sample = (f"per step one (sequence, K/V head) unit of the workload truncated to its first {n_keys} "
              f"keys, fp64 unsharded attention")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": dctx.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "shape": w.description},
            "cpu_baseline": {"value": value, "unit": unit, "kind": "oracle",
                             "cores": torch.get_num_threads(), "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def relaunch_or_check(args, argv):
    """--gpus N > 1 without WORLD_SIZE: run N ranks under torch.distributed.run and return
    their exit code.  WORLD_SIZE set but different from N: an error.  Otherwise None."""
    world = os.environ.get("WORLD_SIZE")
    if world is None:
        if args.gpus <= 1:
            return None
        import socket

        with socket.socket() as s:
            s.bind(("127.0.0.1", 0))
            port = s.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + list(argv)
        return subprocess.call(cmd)
    if int(world) != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one rank per GPU "
              f"(torch.distributed.run --nproc-per-node {args.gpus})", file=sys.stderr)
        return 2
    return None


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse_args(argv)
    rc = relaunch_or_check(args, argv)
    if rc is not None:
        sys.exit(rc)
    dctx = Dist()
    if args.impl == "reference":
        run_reference(args, dctx)
        return
    run_ours(args, dctx)


if __name__ == "__main__":
    main()
