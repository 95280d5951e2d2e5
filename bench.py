"""Benchmark: paged-KV attention forward on GB300.

Default workload: the dynamic bf16 decode batch (B=64, Hq=32, Hkv=8, D=128,
64-token pages, NHD, KV lengths log-uniform in [128, 32768], q_len = 1+MTP
with MTP=1).  One step = Assign + split-K decode + Combine over the whole
batch.  Metric: achieved HBM GB/s = algorithmic bytes (every visible K/V
element once, Q in, O and LSE out, block-table entries) / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload decode_bf16|decode_fp8|prefill_dense|prefill_sparse|hybrid]

Under torchrun each rank processes its own independent batch (seed + rank)
on its own GPU with no data-path collective (weak scaling); the barrier and
the max-over-ranks of the step time are the only communication.
--impl reference times the fp64 CPU oracle on bounded samples of the same
workload on the host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn achieved HBM GB/s; prefill attn TFLOP/s; both as % of GB300 roofline"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def make_workload(name: str, rank: int, shrink: int = 1, mtp: int = 0):
    """The workload's batch for `rank`: every rank draws its own independent
    batch of the same shape (weak scaling).  shrink > 1 divides batch and
    lengths (small profiling cases only; bench lines use shrink = 1).  mtp
    (decode workloads) sets q_len = 1 + mtp; 0 keeps the default (1 for bf16,
    2 for E4M3)."""
    from paged_attention_gb300 import workloads as W
    from paged_attention_gb300.dist import rank_seed
    if name == "decode_bf16":
        return W.decode_bf16(mtp=mtp or 1, seed=rank_seed(1002, rank), shrink=shrink)
    if name == "decode_fp8":
        return W.decode_fp8(seed=rank_seed(1003, rank), shrink=shrink, mtp=mtp or 2)
    if name == "prefill_dense":
        return W.prefill_bf16(sparse=False, seed=rank_seed(1004, rank), shrink=shrink)
    if name == "prefill_sparse":
        return W.prefill_bf16(sparse=True, seed=rank_seed(1004, rank), shrink=shrink)
    if name == "hybrid":
        return W.hybrid_bf16(seed=rank_seed(1005, rank), shrink=shrink)
    raise SystemExit(f"unknown workload {name}")


def workload_config(w, name):
    cfg = {"workload": name, "batch": w.num_seqs, "num_q_heads": w.num_q_heads,
           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
           "layout": "NHD" if w.layout == 0 else "HND",
           "kv_dtype": "bf16" if w.kv_dtype == 0 else "e4m3",
           "total_q_tokens": w.total_q, "total_kv_tokens": int(w.context_lens.sum())}
    if "mtp" in w.meta:
        cfg["mtp"] = w.meta["mtp"]
    if w.window:
        cfg["window"] = w.window
    return cfg


def is_decode(name):
    return name.startswith("decode")


def work_of(w, name):
    from paged_attention_gb300 import workloads as W
    if is_decode(name) or name == "hybrid":
        return W.decode_algorithmic_bytes(w), "bytes"
    return W.prefill_algorithmic_flops(w), "flops"


# --------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")
        self.uuid = uuid

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle

def oracle_sample_rate(w, name, target_s):
    """Time the fp64 oracle on the first sequences of the workload (all heads,
    all new tokens) until about target_s seconds of work; returns
    (value in the metric's unit, sample description, cores)."""
    import oracle
    from paged_attention_gb300 import workloads as W
    oracle.build()
    cores = oracle.max_threads()
    Hq = w.num_q_heads
    ql = [int(x) for x in w.q_lens]
    cu = np.concatenate([[0], np.cumsum(ql)])
    done_rows = 0
    runs = 0          # sequence runs; the batch is walked again when it runs out
    t_total = 0.0
    work = 0
    n = w.num_seqs
    decode_like = is_decode(name) or name == "hybrid"
    while runs < 100 * n and (runs == 0 or t_total < target_s):
        b = runs % n
        rows = np.arange(cu[b] * Hq, cu[b + 1] * Hq, dtype=np.int64)
        if not decode_like and len(rows) > 4096:
            rows = rows[:: max(1, len(rows) // 4096)]
        t0 = time.perf_counter()
        oracle.attention(w, rows=rows)
        t_total += time.perf_counter() - t0
        done_rows += len(rows)
        c = int(w.context_lens[b])
        if decode_like:
            e = 2 if w.kv_dtype == 0 else 1
            work += c * w.num_kv_heads * w.head_dim * 2 * e + ql[b] * Hq * (w.head_dim * 4 + 4)
        else:
            frac = len(rows) / (ql[b] * Hq)
            pairs = ql[b] * (c - ql[b]) + ql[b] * (ql[b] + 1) // 2
            work += int(4 * w.head_dim * Hq * pairs * frac)
        runs += 1
    if decode_like:
        value = work / t_total / 1e9
        unit = "GB/s"
    else:
        value = work / t_total / 1e12
        unit = "TFLOP/s"
    if runs <= n:
        what = f"sequences 0..{runs - 1} of the workload"
    else:
        what = f"the whole batch ({n} sequences) {runs / n:.1f} times over"
    sample = f"oracle on {what} ({done_rows} query rows, {t_total:.1f} s)"
    return value, unit, sample, cores, t_total


# ------------------------------------------------------------------ native

def launches_per_step(w, mode):
    from paged_attention_gb300 import binding as B
    if mode == B.PA_MODE_DECODE:
        return 3
    G = w.num_q_heads // w.num_kv_heads
    return 5 + (3 if w.block_mask is None and G <= 16 else 0)


def run_native(args, rank, world, dist):
    import torch
    from paged_attention_gb300 import binding as B
    from paged_attention_gb300 import build as build_mod
    build_mod.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    name = args.workload
    w_cpu = make_workload(name, rank, args.shrink, args.mtp)
    if args.window:
        if not is_decode(name) or w_cpu.kv_dtype != 0:
            raise SystemExit("--window: bf16 decode workloads only")
        w_cpu.window = args.window
    w = w_cpu.to(dev)
    work, kind = work_of(w_cpu, name)
    mode = B.PA_MODE_DECODE if is_decode(name) else B.PA_MODE_PREFILL
    bufs = B.make_buffers(w, mode)
    stream = torch.cuda.current_stream()
    runner = B.run_decode if mode == B.PA_MODE_DECODE else B.run_prefill

    def step(ev=None):
        p = bufs.problem
        B.pa_assign(p, mode, w.context_lens, w.q_lens,
                    w.block_mask if mode == B.PA_MODE_PREFILL else None, bufs.assign_ws)
        if ev is not None:
            ev[0].record(stream)
        if mode == B.PA_MODE_DECODE:
            B.pa_decode_splitk(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens,
                               w.q_lens, w.k_scale, w.v_scale, bufs.assign_ws, bufs.partial_ws,
                               bufs.out, bufs.lse)
        else:
            B.pa_prefill(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.q_lens,
                         w.k_scale, w.v_scale, w.block_mask, bufs.assign_ws, bufs.partial_ws,
                         bufs.out, bufs.lse)
        if ev is not None:
            ev[1].record(stream)
        B.pa_combine(p, mode, bufs.assign_ws, bufs.partial_ws, bufs.out, bufs.lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if B.pa_last_device_error(bufs.assign_ws) != 0:
        raise SystemExit("device error during warm-up")

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # the step as a user runs it: nothing between the launches (events recorded
    # between kernels would keep the dependent launches from overlapping)
    t0.record(stream)
    for i in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    # the compute kernel alone, bracketed by events, for the roofline
    for i in range(args.steps):
        step(kev[i])
    torch.cuda.synchronize()
    kern_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps

    # end-to-end through the public API: every step copies its inputs from
    # pinned host memory (Q, block table, lengths; the KV cache is resident
    # state), runs Assign + compute + Combine, and reads its outputs (O, LSE)
    # back to pinned host memory.  As in a serving loop, the copies run on
    # their own streams with two sets of device buffers, so step k+1's upload
    # and step k-1's read-back overlap step k's compute.
    import copy
    hq = w_cpu.q.pin_memory()
    hbt = w_cpu.block_table.pin_memory()
    hctx = w_cpu.context_lens.pin_memory()
    hql = w_cpu.q_lens.pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hbt, hctx, hql))
    sets = []
    for k in range(2):
        wk = copy.copy(w)
        if k == 1:
            wk.q = torch.empty_like(w.q)
            wk.block_table = torch.empty_like(w.block_table)
            wk.context_lens = torch.empty_like(w.context_lens)
            wk.q_lens = torch.empty_like(w.q_lens)
        bk = bufs if k == 0 else B.make_buffers(w, mode)
        hout = torch.empty(bk.out.shape, dtype=bk.out.dtype).pin_memory()
        hlse = torch.empty(bk.lse.shape, dtype=bk.lse.dtype).pin_memory()
        sets.append((wk, bk, hout, hlse))
    d2h = sets[0][2].numel() * sets[0][2].element_size() + \
        sets[0][3].numel() * sets[0][3].element_size()
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        k = i % 2
        wk, bk, hout, hlse = sets[k]
        with torch.cuda.stream(up):
            up.wait_event(ev_done[k])          # step i-2 no longer reads this set
            wk.q.copy_(hq, non_blocking=True)
            wk.block_table.copy_(hbt, non_blocking=True)
            wk.context_lens.copy_(hctx, non_blocking=True)
            wk.q_lens.copy_(hql, non_blocking=True)
            ev_in[k].record(up)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])           # step i-2's outputs have been read back
        runner(wk, bk)
        ev_done[k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[k])
            hout.copy_(bk.out, non_blocking=True)
            hlse.copy_(bk.lse, non_blocking=True)
            ev_out[k].record(down)

    for i in range(max(3, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_event(ev_out[0])
    stream.wait_event(ev_out[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    for wk, bk, hout, hlse in sets:
        if B.pa_last_device_error(bk.assign_ws) != 0:
            raise SystemExit("device error during the end-to-end run")
    for wk, bk, hout, hlse in sets:
        if not torch.equal(hout, bufs.out.cpu()):
            raise SystemExit("end-to-end outputs differ from the device-timed run")
    # the same device-resident step captured once in a CUDA graph and replayed
    # (the launch chain without host launch overhead)
    graph = None
    try:
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            step()   # warm on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / args.steps
        graph = {"ms_per_step": round(graph_ms, 4), "value": None}
    except Exception as exc:   # report, do not fail the bench line
        graph = {"unavailable": f"{type(exc).__name__}: {str(exc)[:120]}"}
    clk = clocks.stop()
    if dist is not None:
        from paged_attention_gb300.dist import max_over_ranks
        ms, e2e_ms, kern_ms = max_over_ranks([ms, e2e_ms, kern_ms])
    if B.pa_last_device_error(bufs.assign_ws) != 0:
        raise SystemExit("device error during the timed region")

    peaks = load_peaks()
    if kind == "bytes":
        value = work * world / (ms * 1e-3) / 1e9
        unit = "GB/s"
        e2e_val = work * world / (e2e_ms * 1e-3) / 1e9
        achieved = work / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"]}
    else:
        value = work * world / (ms * 1e-3) / 1e12
        unit = "TFLOP/s"
        e2e_val = work * world / (e2e_ms * 1e-3) / 1e12
        achieved = work / (kern_ms * 1e-3) / 1e12
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk,
                "unit": "TFLOP/s", "frac": round(achieved / pk, 4),
                "peak_source": peaks["source"]}
    if graph is not None and "ms_per_step" in graph:
        scale = 1e9 if kind == "bytes" else 1e12
        graph["value"] = round(work * world / (graph["ms_per_step"] * 1e-3) / scale, 2)
    roof["kernel"] = "pa_decode_splitk" if mode == B.PA_MODE_DECODE else "pa_prefill"
    roof["kernel_ms"] = round(kern_ms, 4)
    roof["traffic"] = load_traffic(roof["kernel"], name)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == 0 else "e4m3-kv/bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, paged, NaN decoy pages)",
        "config": dict(workload_config(w_cpu, name),
                       l2="inputs larger than L2" if args.shrink == 1 else f"shrink {args.shrink}",
                       parallelism=f"independent batch per GPU x{world}"),
        "e2e": {"value": round(e2e_val, 2), "unit": unit, "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "uploads and read-backs on their own streams, two buffer sets"},
        "roofline": roof,
        # decode mode: Assign, compute, Combine.  Prefill mode: Assign (3) +
        # prefill kernel + Combine, and without a block mask (G <= 16) the
        # decode part too: its Assign, the decode kernel and its Combine
        "gpu_launches": launches_per_step(w_cpu, mode) * args.steps,
        "clocks": clk,
        "graph": graph,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, u, sample, cores, _ = oracle_sample_rate(w_cpu, name, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": u, "cores": cores,
                                "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        from paged_attention_gb300 import build as build_mod
        entry = d.get(f"{kernel}:{workload}")
        if not entry or entry.get("source_hash") != build_mod.kernel_fingerprint(kernel):
            return None
        return entry.get("dram_bytes_per_launch")
    except Exception:
        return None


# --------------------------------------------------------------- reference

def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload
    w = make_workload(name, 0, 1, args.mtp)
    if args.window:
        w.window = args.window
    per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    vals = []
    sample = ""
    cores = 1
    unit = "GB/s"
    for i in range(args.warmup + args.steps):
        v, unit, sample, cores, t = oracle_sample_rate(w, name, per_step)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": dict(workload_config(w, name), l2="inputs larger than L2",
                       parallelism="host cores"),
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="decode_bf16",
                    choices=["decode_bf16", "decode_fp8", "prefill_dense", "prefill_sparse",
                             "hybrid"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window (bf16 decode workloads): keys p - window < j <= p")
    ap.add_argument("--mtp", type=int, default=0,
                    help="decode workloads: q_len = 1 + MTP (default: 1 for bf16, 2 for E4M3)")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide batch and lengths (profiling of small cases only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        run_native(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
