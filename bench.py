"""Benchmark: paged-KV attention forward on GB300.

Headline workload: the dynamic bf16 decode batch (B=64, Hq=32, Hkv=8, D=128,
64-token pages, NHD, KV lengths log-uniform in [128, 32768], q_len = 1+MTP
with MTP=1).  One step = Assign + split-K decode + Combine over the whole
batch.  Metric: achieved HBM GB/s = algorithmic bytes (every visible K/V
element once, Q in, O and LSE out, block-table entries) / step time; for the
prefill workloads TFLOP/s = algorithmic FLOPs (4 * D * Hq per visible
query-key pair) / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload decode_bf16|decode_fp8|prefill_dense|prefill_sparse|hybrid|
                              tiny_mixed|decode_bf16_static|prefill_fp8_dense|
                              prefill_fp8_sparse|prefill_fp8_dense_q0_hnd]
                  [--configs all|none]

With no --workload (N = 1), the one JSON line also carries a "configs" object:
every other workload of the metric (tiny mixed batch, bf16 decode with q_len
3 and 4, E4M3 decode with q_len 3 and 4, dense and block-sparse prefill, the
hybrid batch, the static split-K decode, and the E4M3 prefill: dense and
block-sparse with Q scales per (token, head), dense HND with one Q scale), each timed on the same contract (W warm-up steps, K timed
steps, CUDA events on the launching stream) with its own roofline, clocks, CPU
baseline and a parity check of sampled rows against the oracle leg's output.

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
WORKLOADS = ["decode_bf16", "decode_fp8", "prefill_dense", "prefill_sparse", "hybrid",
             "tiny_mixed", "decode_bf16_static", "prefill_fp8_dense", "prefill_fp8_sparse",
             "prefill_fp8_dense_q0_hnd"]
# the "configs" object of the default line: (key, workload, mtp)
CONFIG_SET = [
    ("tiny_mixed", "tiny_mixed", 0),
    ("decode_bf16_mtp2", "decode_bf16", 2),
    ("decode_bf16_mtp3", "decode_bf16", 3),
    ("decode_fp8_mtp2", "decode_fp8", 2),
    ("decode_fp8_mtp3", "decode_fp8", 3),
    ("prefill_dense", "prefill_dense", 0),
    ("prefill_sparse", "prefill_sparse", 0),
    ("hybrid", "hybrid", 0),
    ("decode_bf16_static", "decode_bf16_static", 1),
    ("prefill_fp8_dense", "prefill_fp8_dense", 0),
    ("prefill_fp8_sparse", "prefill_fp8_sparse", 0),
    ("prefill_fp8_dense_q0_hnd", "prefill_fp8_dense_q0_hnd", 0),
]
PARALLELISM = "independent batch per GPU x{world}"
# pa_problem.unit_cost for every Assign of the run (0 = the library's choice)
UNIT_COST = 0


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
    if name in ("decode_bf16", "decode_bf16_static"):
        return W.decode_bf16(mtp=mtp or 1, seed=rank_seed(1002, rank), shrink=shrink)
    if name == "decode_fp8":
        return W.decode_fp8(seed=rank_seed(1003, rank), shrink=shrink, mtp=mtp or 2)
    if name == "prefill_dense":
        return W.prefill_bf16(sparse=False, seed=rank_seed(1004, rank), shrink=shrink)
    if name == "prefill_sparse":
        return W.prefill_bf16(sparse=True, seed=rank_seed(1004, rank), shrink=shrink)
    if name == "hybrid":
        return W.hybrid_bf16(seed=rank_seed(1005, rank), shrink=shrink)
    if name.startswith("prefill_fp8_"):
        # E4M3 Q/K/V; quant type 1 (Q per token and head) unless "_q0"
        return W.prefill_fp8(quant_type=0 if "_q0" in name else 1, sparse="_sparse" in name,
                             layout=W.HND if name.endswith("_hnd") else W.NHD,
                             seed=rank_seed(1006, rank), shrink=shrink)
    if name == "tiny_mixed":
        return W.tiny_mixed(seed=rank_seed(1001, rank))
    raise SystemExit(f"unknown workload {name}")


def workload_config(w, name, world):
    cfg = {"workload": name, "batch": w.num_seqs, "num_q_heads": w.num_q_heads,
           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "page_size": w.page_size,
           "layout": "NHD" if w.layout == 0 else "HND",
           "kv_dtype": "bf16" if w.kv_dtype == 0 else "e4m3",
           "q_dtype": "bf16" if w.q_dtype == 0 else "e4m3",
           "total_q_tokens": w.total_q, "total_kv_tokens": int(w.context_lens.sum()),
           "l2": "inputs larger than L2" if w.meta.get("shrink", 1) == 1 and
           name != "tiny_mixed" else "inputs smaller than L2 (launch-bound case)",
           "parallelism": PARALLELISM.format(world=world)}
    if "mtp" in w.meta:
        cfg["mtp"] = w.meta["mtp"]
        cfg["q_len"] = 1 + w.meta["mtp"]
    if w.window:
        cfg["window"] = w.window
    if w.q_dtype != 0:
        cfg["quant_type"] = w.q_scale_mode
        cfg["sparse"] = w.block_mask is not None
    return cfg


def is_decode(name):
    return name.startswith("decode")


def is_static(name):
    """The static split-K path (pa_decode_static) on a decode workload."""
    return name.endswith("_static")


def bytes_metric(name):
    """Decode-shaped workloads report HBM GB/s, prefill ones TFLOP/s."""
    return is_decode(name) or name in ("hybrid", "tiny_mixed")


def work_of(w, name):
    from paged_attention_gb300 import workloads as W
    if bytes_metric(name):
        return W.decode_algorithmic_bytes(w), "bytes"
    return W.prefill_algorithmic_flops(w), "flops"


# --------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None, path=None):
        self.proc = None
        self.keep = path is not None
        if path is None:
            import tempfile
            fd, path = tempfile.mkstemp(prefix="pa_clocks_", suffix=".csv")
            os.close(fd)
        self.path = path
        self.uuid = uuid

    def start(self):
        try:
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
        self.proc = None
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
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle

def visible_keys_per_row(w, b, toks):
    """Visible keys of query tokens `toks` (local indices) of sequence b, per
    q head: causal (bottom-right), sliding window, block mask."""
    c, q = int(w.context_lens[b]), int(w.q_lens[b])
    toks = np.asarray(toks, dtype=np.int64)
    p = c - q + toks                                   # absolute positions
    hi = np.minimum(p, c - 1)
    lo = np.maximum(0, p - w.window + 1) if w.window > 0 else np.zeros_like(p)
    if w.block_mask is None:
        return np.clip(hi - lo + 1, 0, None)
    T = w.mask_tile
    m = w.block_mask[b].numpy().astype(np.int64)
    mq = toks // T
    out = np.zeros_like(p)
    for kt in range(min(m.shape[1], c // T + 1)):
        a = np.maximum(lo, kt * T)
        e = np.minimum(hi, kt * T + T - 1)
        keep = np.where(mq < m.shape[0], m[np.minimum(mq, m.shape[0] - 1), kt], 0)
        out += np.clip(e - a + 1, 0, None) * keep
    return out


def oracle_sample(w, name, target_s, keep_first=True):
    """Time the fp64 oracle, as it stands, on the workload's sequences in order
    (every row of a decode sequence; at most 4096 evenly spaced rows of a long
    prefill chunk), walking the batch again if it runs out, until about
    target_s seconds of work.  Returns a dict with the value in the metric's
    unit, the sample description, the threads used, and (keep_first) the rows
    and oracle outputs of the first walk over the batch, for a parity check."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    Hq, D = w.num_q_heads, w.head_dim
    ql = [int(x) for x in w.q_lens]
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int64)
    kind = "bytes" if bytes_metric(name) else "flops"
    e = 2 if w.kv_dtype == 0 else 1
    done_rows, runs, t_total, work, n = 0, 0, 0.0, 0.0, w.num_seqs
    first = []
    while runs < 100 * n and (runs == 0 or t_total < target_s):
        b = runs % n
        runs += 1
        if ql[b] == 0:
            continue
        toks = np.arange(ql[b], dtype=np.int64)
        nrows = ql[b] * Hq
        if nrows > 4096:
            toks = toks[:: max(1, nrows // 4096)]
        rows = ((cu[b] + toks)[:, None] * Hq + np.arange(Hq)[None, :]).reshape(-1)
        t0 = time.perf_counter()
        ref_o, ref_l = oracle.attention(w, rows=rows)
        t_total += time.perf_counter() - t0
        if keep_first and runs <= n:
            first.append((rows, ref_o, ref_l))
        done_rows += len(rows)
        vis = visible_keys_per_row(w, b, toks)
        if kind == "bytes":
            # the sequence's algorithmic bytes, scaled by the fraction of its rows computed
            lo = max(0, int(w.context_lens[b]) - ql[b] - w.window + 1) if w.window > 0 else 0
            c = int(w.context_lens[b])
            pages = (c + w.page_size - 1) // w.page_size - lo // w.page_size
            seq = ((c - lo) * w.num_kv_heads * D * 2 * e + ql[b] * Hq * (D * 4 + 4) + pages * 4
                   + (pages * w.num_kv_heads * 8 if w.kv_dtype == 1 else 0))
            work += seq * len(rows) / nrows
        else:
            work += 4.0 * D * Hq * float(vis.sum())
    value = work / max(t_total, 1e-9) / (1e9 if kind == "bytes" else 1e12)
    unit = "GB/s" if kind == "bytes" else "TFLOP/s"
    what = (f"sequences 0..{runs - 1} of the workload" if runs <= n else
            f"the whole batch ({n} sequences) {runs / n:.1f} times over")
    if first:
        first = tuple(np.concatenate([f[i] for f in first]) for i in range(3))
    return {"value": value, "unit": unit, "cores": cores, "seconds": t_total,
            "sample": f"oracle on {what} ({done_rows} query rows, {t_total:.1f} s)",
            "first": first or None}


# ------------------------------------------------------------------ native

def launches_per_step(w, mode, static=False):
    """Kernels one step launches.  Decode mode: Assign and the decode kernel
    (bf16: it finalizes its split units and pa_combine launches nothing;
    E4M3: also Combine).  Prefill mode: Assign (3 kernels), the prefill kernel
    and Combine, and without a block mask (G <= 16) the decode part's Assign
    and decode kernel."""
    from paged_attention_gb300 import binding as B
    if static:
        return 1
    if mode == B.PA_MODE_DECODE:
        return 2 if w.kv_dtype == 0 else 3
    G = w.num_q_heads // w.num_kv_heads
    return 5 + (2 if w.block_mask is None and G <= 16 and w.q_dtype == 0 else 0)


class Case:
    """One workload on the device: its buffers, one step of the hot path
    (Assign + compute + Combine), and the timed loops."""

    def __init__(self, name, mtp, rank, shrink, window, dev):
        import torch
        from paged_attention_gb300 import binding as B
        self.B = B
        self.name = name
        self.w_cpu = make_workload(name, rank, shrink, mtp)
        if window:
            if not is_decode(name):
                raise SystemExit("--window: decode workloads only")
            self.w_cpu.window = window
        self.w = self.w_cpu.to(dev)
        self.work, self.kind = work_of(self.w_cpu, name)
        self.mode = B.PA_MODE_DECODE if is_decode(name) else B.PA_MODE_PREFILL
        self.stream = torch.cuda.current_stream()
        if is_static(name):
            self.bufs = B.StaticBuffers(self.w, 0)
            self.splits = B.pa_static_num_splits(self.bufs.problem, 0)
            self.runner = lambda w, bufs: B.run_decode_static(w, bufs)
        else:
            self.bufs = B.make_buffers(self.w, self.mode, unit_cost=UNIT_COST)
            self.runner = B.run_decode if self.mode == B.PA_MODE_DECODE else B.run_prefill

    def step(self, ev=None, w=None, bufs=None):
        B = self.B
        w = w or self.w
        bufs = bufs or self.bufs
        if is_static(self.name):
            # one call: the error-word memset and the kernel (no Assign, no Combine)
            if ev is not None:
                ev[0].record(self.stream)
            B.run_decode_static(w, bufs)
            if ev is not None:
                ev[1].record(self.stream)
            return
        p, mode = bufs.problem, self.mode
        B.pa_assign(p, mode, w.context_lens, w.q_lens,
                    w.block_mask if mode == B.PA_MODE_PREFILL else None, bufs.assign_ws)
        if ev is not None:
            ev[0].record(self.stream)
        if mode == B.PA_MODE_DECODE:
            B.pa_decode_splitk(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens,
                               w.q_lens, w.k_scale, w.v_scale, bufs.assign_ws, bufs.partial_ws,
                               bufs.out, bufs.lse)
        elif p.q_dtype == B.PA_FP8_E4M3:
            B.pa_prefill_fp8(p, w.q, w.q_scale, w.k_cache, w.v_cache, w.block_table,
                             w.context_lens, w.q_lens, w.k_scale, w.v_scale, w.block_mask,
                             bufs.assign_ws, bufs.partial_ws, bufs.out, bufs.lse)
        else:
            B.pa_prefill(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.q_lens,
                         w.k_scale, w.v_scale, w.block_mask, bufs.assign_ws, bufs.partial_ws,
                         bufs.out, bufs.lse)
        if ev is not None:
            ev[1].record(self.stream)
        B.pa_combine(p, mode, bufs.assign_ws, bufs.partial_ws, bufs.out, bufs.lse)

    def balance(self):
        """One extra step (outside every timed region) with the task trace on:
        how evenly the persistent CTAs share the compute launch.  Per CTA the
        busy time runs from its first task's start to its last task's end."""
        import torch
        B = self.B
        if is_static(self.name):
            return None
        cap = int(self.bufs.assign_ws.numel() // 16) + 1024
        trace = torch.full((cap, 3), -1, dtype=torch.int64, device=self.bufs.out.device)
        B.pa_set_task_trace(trace)
        try:
            self.step()
            torch.cuda.synchronize()
        finally:
            B.pa_set_task_trace(None)
        tm = B.pa_read_task_map(self.bufs.problem, self.mode, self.bufs.assign_ws)
        T = tm["num_tasks"]
        if T == 0 or T > cap:
            return None
        tr = trace[:T].cpu().numpy()
        cp = tm["cta_ptr"]
        busy = []
        for c in range(len(cp) - 1):
            if cp[c + 1] > cp[c]:
                seg = tr[cp[c]:cp[c + 1]]
                busy.append((seg[:, 1].max() - seg[:, 0].min()) / 1000.0)
        busy = np.array(busy)
        t0 = tr[:, 0].min()
        return {"tasks": int(T), "ctas_with_tasks": int(len(busy)),
                "cta_busy_us": {"min": round(float(busy.min()), 1),
                                "mean": round(float(busy.mean()), 1),
                                "max": round(float(busy.max()), 1)},
                "max_over_mean": round(float(busy.max() / busy.mean()), 3),
                "last_end_us": round(float((tr[:, 1].max() - t0) / 1000.0), 1),
                "how": "task trace (pa_set_task_trace) of one extra step"}

    def device_error(self):
        ws = self.bufs.ws if is_static(self.name) else self.bufs.assign_ws
        return self.B.pa_last_device_error(ws)

    def timed(self, args, dist, uuid):
        """W warm-up steps, then exactly K steps bracketed by a barrier and a
        synchronize (the step as a user runs it: nothing recorded between its
        launches), then K steps with events around the compute call (the
        kernel's own time, for the roofline).  Clocks are sampled from an
        untimed soak of about 0.3 s before the timed region to its end."""
        import torch
        for _ in range(args.warmup):
            self.step()
        torch.cuda.synchronize()
        if self.device_error() != 0:
            raise SystemExit(f"{self.name}: device error during warm-up")
        clocks = ClockSampler(uuid)
        clocks.start()
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            self.step()
            torch.cuda.synchronize()
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record(self.stream)
        for _ in range(args.steps):
            self.step()
        t1.record(self.stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        ms = t0.elapsed_time(t1) / args.steps
        for i in range(args.steps):
            self.step(kev[i])
        torch.cuda.synchronize()
        kern_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps
        clk = clocks.stop()
        if self.device_error() != 0:
            raise SystemExit(f"{self.name}: device error during the timed region")
        return ms, kern_ms, clk

    def rate(self, ms, world=1):
        scale = 1e9 if self.kind == "bytes" else 1e12
        return self.work * world / (ms * 1e-3) / scale

    def unit(self):
        return "GB/s" if self.kind == "bytes" else "TFLOP/s"

    def roofline(self, kern_ms, peaks):
        achieved = self.rate(kern_ms)
        if self.kind == "bytes":
            roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
        else:
            # E4M3 contractions: the measured bf16 peak x the nominal 2x of fp8
            ratio = 2.0 if self.w_cpu.q_dtype == 1 else 1.0
            pk = peaks["bf16_tflops"] * ratio
            roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk,
                    "unit": "TFLOP/s", "frac": round(achieved / pk, 4),
                    "frac_of_sustained": round(
                        achieved / (peaks["bf16_tflops_sustained"] * ratio), 4)}
            if ratio != 1.0:
                roof["peak_dtype"] = "e4m3 (measured bf16 x 2, the nominal fp8/bf16 ratio)"
        roof["peak_source"] = peaks["source"]
        roof["kernel"] = ("pa_decode_static" if is_static(self.name) else
                          "pa_decode_splitk" if self.mode == self.B.PA_MODE_DECODE else
                          "pa_prefill")
        roof["kernel_ms"] = round(kern_ms, 4)
        roof["algorithmic_" + self.kind + "_per_launch"] = int(self.work)
        if self.name == "hybrid":
            # the batch's two parts run one after the other, each on its own
            # roofline: the decode part's bytes at HBM rate, the chunk's FLOPs
            # at the bf16 rate
            from paged_attention_gb300 import workloads as W
            dec_bytes, pre_flops = W.mixed_batch_parts(self.w_cpu)
            bound_ms = (dec_bytes / (peaks["hbm_gbs"] * 1e9) +
                        pre_flops / (peaks["bf16_tflops"] * 1e12)) * 1e3
            roof["parts"] = {"decode_part_bytes": int(dec_bytes),
                             "prefill_part_flops": int(pre_flops),
                             "bound_ms": round(bound_ms, 4),
                             "frac": round(bound_ms / kern_ms, 4),
                             "how": "bytes at the measured HBM rate plus FLOPs at the "
                                    "measured bf16 peak, against the kernel pair's time"}
        roof["traffic"] = load_traffic(roof["kernel"], self.name,
                                       self.w_cpu.meta.get("mtp"))
        return roof

    def parity(self, first):
        """Sampled rows of the last timed step's output against the oracle
        leg's output for the same rows."""
        import torch
        if first is None:
            return None
        rows, ref_o, ref_l = first
        idx = torch.as_tensor(rows, device=self.bufs.out.device)
        o = self.bufs.out.reshape(-1, self.w.head_dim).index_select(0, idx).float().cpu().numpy()
        lg = self.bufs.lse.reshape(-1).index_select(0, idx).cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_l)
        tol = 6e-2 if self.w.kv_dtype == 1 else 2e-2
        err_o = float(np.abs(o - ref_o).max()) if o.size else 0.0
        err_l = float(np.abs(lg[fin] - ref_l[fin]).max()) if fin.any() else 0.0
        ok = bool(np.isfinite(o).all() and np.array_equal(np.isfinite(lg), fin)
                  and err_o <= tol and err_l <= 1e-3)
        return {"rows": int(len(rows)), "max_abs_out": round(err_o, 6),
                "max_abs_lse": round(err_l, 7), "tol_out": tol, "tol_lse": 1e-3, "ok": ok}


def gpu_uuid(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


def e2e_measure(case, args, dist, dev):
    """The same metric through the public C-ABI calls, with each step's
    inputs copied from pinned host memory (Q, block table, lengths; the K/V
    cache is resident state) and its outputs (O, LSE) read back to pinned host
    memory.  As in a serving loop, uploads and read-backs run on their own
    streams with two sets of device buffers, so step k+1's upload and step
    k-1's read-back overlap step k's compute.  Also the serial latency of one
    step with its copies (upload, compute, read-back, synchronize)."""
    import copy
    import torch
    B = case.B
    w, w_cpu, stream = case.w, case.w_cpu, case.stream
    hq = w_cpu.q.pin_memory()
    hbt = w_cpu.block_table.pin_memory()
    hctx = w_cpu.context_lens.pin_memory()
    hql = w_cpu.q_lens.pin_memory()
    # an E4M3 Q comes with its scales (one, or one per token and q head)
    hqs = w_cpu.q_scale.pin_memory() if w_cpu.q_scale is not None else None
    h2d = sum(t.numel() * t.element_size() for t in (hq, hbt, hctx, hql, hqs) if t is not None)
    sets = []
    for k in range(2):
        wk = copy.copy(w)
        if k == 1:
            wk.q = torch.empty_like(w.q)
            wk.block_table = torch.empty_like(w.block_table)
            wk.context_lens = torch.empty_like(w.context_lens)
            wk.q_lens = torch.empty_like(w.q_lens)
            if hqs is not None:
                wk.q_scale = torch.empty_like(w.q_scale)
        bk = case.bufs if k == 0 else (B.StaticBuffers(w, 0) if is_static(case.name)
                                       else B.make_buffers(w, case.mode, unit_cost=UNIT_COST))
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
            if hqs is not None:
                wk.q_scale.copy_(hqs, non_blocking=True)
            ev_in[k].record(up)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])           # step i-2's outputs have been read back
        case.runner(wk, bk)
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
        ws = bk.ws if is_static(case.name) else bk.assign_ws
        if B.pa_last_device_error(ws) != 0:
            raise SystemExit("device error during the end-to-end run")
    ref = case.bufs.out.cpu()
    for wk, bk, hout, hlse in sets:
        if not torch.equal(hout, ref):
            raise SystemExit("end-to-end outputs differ from the device-timed run")
    # serial: one step at a time, copies not overlapped with anything
    wk, bk, hout, hlse = sets[1]
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(args.steps):
        wk.q.copy_(hq, non_blocking=True)
        wk.block_table.copy_(hbt, non_blocking=True)
        wk.context_lens.copy_(hctx, non_blocking=True)
        wk.q_lens.copy_(hql, non_blocking=True)
        if hqs is not None:
            wk.q_scale.copy_(hqs, non_blocking=True)
        case.runner(wk, bk)
        hout.copy_(bk.out, non_blocking=True)
        hlse.copy_(bk.lse, non_blocking=True)
    s1.record(stream)
    torch.cuda.synchronize()
    serial_ms = s0.elapsed_time(s1) / args.steps
    return e2e_ms, serial_ms, h2d, d2h


def graph_measure(case, args, dev):
    """The device-resident step captured once in a CUDA graph and replayed."""
    import torch
    try:
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(case.stream)
        with torch.cuda.stream(gs):
            case.step()   # warm on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            case.step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(case.stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(case.stream)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / args.steps
        return {"ms_per_step": round(graph_ms, 4), "value": round(case.rate(graph_ms), 2)}
    except Exception as exc:   # report, do not fail the bench line
        return {"unavailable": f"{type(exc).__name__}: {str(exc)[:120]}"}


def config_entry(key, name, mtp, args, dev, peaks, uuid):
    """One entry of the "configs" object (N = 1 only)."""
    import torch
    case = Case(name, mtp, 0, 1, 0, dev)
    ms, kern_ms, clk = case.timed(args, None, uuid)
    entry = {"workload": name, "value": round(case.rate(ms), 2), "unit": case.unit(),
             "ms_per_step": round(ms, 4), "kernel_ms": round(kern_ms, 4),
             "roofline": case.roofline(kern_ms, peaks), "clocks": clk,
             "gpu_launches": launches_per_step(case.w_cpu, case.mode, is_static(name))
             * args.steps,
             "config": workload_config(case.w_cpu, name, 1)}
    if name == "tiny_mixed":
        entry["note"] = "launch-bound: parity workload, time reported only"
    bal = case.balance()
    if bal is not None:
        entry["balance"] = bal
    if is_static(name):
        entry["static_splits"] = case.splits
        entry["note"] = ("static split-K (no Assign, no Combine; splits of a unit on one "
                         "cluster, merged through DSM when S is 2, 4 or 8); the step is one "
                         "memset and one kernel, timed whole as kernel_ms")
    if not args.no_cpu_baseline:
        s = oracle_sample(case.w_cpu, name, args.config_cpu_seconds)
        entry["cpu_baseline"] = {"value": round(s["value"], 4), "unit": s["unit"],
                                 "cores": s["cores"], "kind": "oracle", "sample": s["sample"]}
        entry["parity"] = case.parity(s["first"])
    del case
    torch.cuda.empty_cache()
    return entry


def run_native(args, rank, world, dist):
    import torch
    from paged_attention_gb300 import build as build_mod
    build_mod.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    uuid = gpu_uuid(dev)
    peaks = load_peaks()
    name = args.workload or "decode_bf16"
    case = Case(name, args.mtp, rank, args.shrink, args.window, dev)
    ms, kern_ms, clk = case.timed(args, dist, uuid)
    e2e_ms, serial_ms, h2d, d2h = e2e_measure(case, args, dist, dev)
    graph = graph_measure(case, args, dev)
    if dist is not None:
        from paged_attention_gb300.dist import max_over_ranks
        ms, e2e_ms, kern_ms, serial_ms = max_over_ranks([ms, e2e_ms, kern_ms, serial_ms])
    unit = case.unit()
    line = {
        "metric": METRIC, "value": round(case.rate(ms, world), 2), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if case.w.kv_dtype == 0 else "e4m3-kv/bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V, paged, NaN decoy pages)",
        "config": workload_config(case.w_cpu, name, world),
        "e2e": {"value": round(case.rate(e2e_ms, world), 2), "unit": unit,
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "uploads and read-backs on their own streams, two buffer sets",
                "serial_ms_per_step": round(serial_ms, 4),
                "serial_value": round(case.rate(serial_ms, world), 2)},
        "roofline": case.roofline(kern_ms, peaks),
        "gpu_launches": launches_per_step(case.w_cpu, case.mode, is_static(name)) * args.steps,
        "clocks": clk,
        "graph": graph,
    }
    bal = case.balance()
    if bal is not None:
        line["balance"] = bal
    first = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(case.w_cpu, name, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(s["value"], 4), "unit": s["unit"],
                                "cores": s["cores"], "kind": "oracle", "sample": s["sample"]}
        first = s["first"]
        line["parity"] = case.parity(first)
    del case
    torch.cuda.empty_cache()
    want_configs = args.configs == "all" or (args.configs is None and args.workload is None)
    if world == 1 and want_configs:
        configs = {}
        for key, wname, mtp in CONFIG_SET:
            configs[key] = config_entry(key, wname, mtp, args, dev, peaks, uuid)
        line["configs"] = configs
    if rank == 0:
        print(json.dumps(line), flush=True)


def load_traffic(kernel, workload, mtp=None):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        from paged_attention_gb300 import build as build_mod
        entry = d.get(f"{kernel}:{workload}" + (f":mtp{mtp}" if mtp is not None else ""))
        if entry is None:
            entry = d.get(f"{kernel}:{workload}")
            # an entry without a q_len is the workload's default q_len only
            if entry is not None and mtp is not None and entry.get("mtp", mtp) != mtp:
                entry = None
        if not entry or entry.get("source_hash") != build_mod.kernel_fingerprint(kernel):
            return None
        return entry.get("dram_bytes_per_launch")
    except Exception:
        return None


# --------------------------------------------------------------- reference

def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload or "decode_bf16"
    w = make_workload(name, 0, 1, args.mtp)
    if args.window:
        w.window = args.window
    per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    vals = []
    s = None
    for i in range(args.warmup + args.steps):
        s = oracle_sample(w, name, per_step, keep_first=False)
        if i >= args.warmup:
            vals.append(s["value"])
    value = statistics.median(vals)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": s["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(w, name, world),
        "cpu_baseline": {"value": round(value, 4), "unit": s["unit"], "cores": s["cores"],
                         "kind": "oracle", "sample": s["sample"]},
        "e2e": {"value": round(value, 4), "unit": s["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=None, choices=WORKLOADS,
                    help="headline workload (default decode_bf16); giving one skips the "
                         "configs object unless --configs all")
    ap.add_argument("--configs", default=None, choices=["all", "none"],
                    help="time every other workload into a configs object (default: all "
                         "when no --workload is given; N = 1 only)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window (bf16 decode workloads): keys p - window < j <= p")
    ap.add_argument("--unit-cost", type=int, default=0,
                    help="Assign's fixed cost per unit (pa_problem.unit_cost; 0 = the library's "
                         "choice, < 0 = none)")
    ap.add_argument("--mtp", type=int, default=0,
                    help="decode workloads: q_len = 1 + MTP (default: 1 for bf16, 2 for E4M3)")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide batch and lengths (profiling of small cases only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    global UNIT_COST
    UNIT_COST = args.unit_cost
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
