"""ctypes binding of the C ABI in include/pa.h (argument marshalling only).

Each ``pa_*`` function here has the name and argument order of the C entry
point, takes torch tensors (device memory) instead of raw pointers, passes
``torch.cuda.current_stream()`` unless a stream is given, and raises
:class:`PaError` on a non-OK status.  Every step of the computation runs in
the CUDA library; there is no fallback: if the library is missing or cannot
be loaded, the first call raises.

``run_decode`` / ``run_prefill`` chain Assign -> compute -> Combine for a
:class:`paged_attention_gb300.workloads.Workload` already on the device.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np
import torch

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE = 1, 2, 3
PA_NHD, PA_HND = 0, 1
PA_BF16, PA_FP8_E4M3 = 0, 1
PA_SCALE_PER_TENSOR, PA_SCALE_PER_ROW = 0, 1
PA_MODE_DECODE, PA_MODE_PREFILL = 0, 1
PA_MAP_DECODE_PART = 2   # pa_read_task_map: decode part of a prefill-mode workspace
PA_DEV_OK, PA_DEV_BAD_LENGTHS, PA_DEV_BAD_PAGE, PA_DEV_WAIT_TIMEOUT = 0, 1, 2, 4

EXPORTED = (
    "pa_status_string", "pa_version", "pa_num_ctas", "pa_assign_workspace_size",
    "pa_partial_workspace_size", "pa_assign", "pa_decode_splitk", "pa_combine", "pa_prefill",
    "pa_read_task_map", "pa_last_device_error", "pa_decode_noalloc",
    "pa_test_inject_wait_timeout", "pa_static_workspace_size", "pa_static_num_splits",
    "pa_decode_static", "pa_prefill_fp8", "pa_set_task_trace",
)

PA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # size of the library's fixed scratch
# pa_problem.unit_cost = 0 takes these (PA_DEFAULT_UNIT_COST_DECODE / _PREFILL)
PA_DEFAULT_UNIT_COST_DECODE = 6
PA_DEFAULT_UNIT_COST_PREFILL = 4


def effective_unit_cost(unit_cost: int, mode: int) -> int:
    """The fixed cost per unit Assign uses for pa_problem.unit_cost in `mode`
    (the decode part of a mixed batch takes the decode value)."""
    if unit_cost > 0:
        return unit_cost
    if unit_cost < 0:
        return 0
    return PA_DEFAULT_UNIT_COST_DECODE if mode == PA_MODE_DECODE else PA_DEFAULT_UNIT_COST_PREFILL


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {status_string(status)} ({status})")


class PaProblem(ctypes.Structure):
    """Field-for-field copy of ``pa_problem`` in include/pa.h."""

    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("total_q_tokens", ctypes.c_int32),
        ("max_q_len", ctypes.c_int32),
        ("max_context_len", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("mask_q_tiles", ctypes.c_int32),
        ("mask_kv_tiles", ctypes.c_int32),
        ("num_ctas", ctypes.c_int32),
        ("balance_rows", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
        ("window", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("q_scale_mode", ctypes.c_int32),
        ("unit_cost", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Load the shared library (building it first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {path}")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        PP = ctypes.POINTER(PaProblem)
        sig = {
            "pa_status_string": (ctypes.c_char_p, [i32]),
            "pa_version": (ctypes.c_char_p, []),
            "pa_num_ctas": (i32, [PP, i32, ctypes.POINTER(ctypes.c_int32)]),
            "pa_assign_workspace_size": (sz, [PP, i32]),
            "pa_partial_workspace_size": (sz, [PP, i32]),
            "pa_assign": (i32, [PP, i32, vp, vp, vp, vp, sz, vp]),
            "pa_decode_splitk": (i32, [PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp,
                                       vp, vp]),
            "pa_combine": (i32, [PP, i32, vp, sz, vp, sz, vp, vp, vp]),
            "pa_prefill": (i32, [PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp, vp,
                                 vp]),
            "pa_read_task_map": (i32, [PP, i32, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pa_last_device_error": (i32, [vp, ctypes.POINTER(ctypes.c_int32), vp]),
            "pa_decode_noalloc": (i32, [PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pa_test_inject_wait_timeout": (i32, [ctypes.c_int32, ctypes.c_int64]),
            "pa_set_task_trace": (i32, [vp, ctypes.c_int64]),
            "pa_static_workspace_size": (sz, [PP, ctypes.c_int32]),
            "pa_static_num_splits": (i32, [PP, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
            "pa_decode_static": (i32, [PP, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                       vp, vp, vp]),
            "pa_prefill_fp8": (i32, [PP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz,
                                     vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != PA_OK:
        raise PaError(status, where)


def problem_from(w, num_ctas: int = 0, balance_rows: int = 0, unit_cost: int = 0) -> PaProblem:
    """pa_problem for a Workload (shapes only)."""
    ql = [int(x) for x in w.q_lens]
    ctx = [int(x) for x in w.context_lens]
    bm = w.block_mask
    return PaProblem(
        num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, page_size=w.page_size, num_pages=w.num_pages,
        max_pages_per_seq=w.max_pages_per_seq, total_q_tokens=sum(ql),
        max_q_len=max(ql) if ql else 0, max_context_len=max(ctx) if ctx else 0,
        layout=w.layout, kv_dtype=w.kv_dtype,
        mask_q_tiles=(bm.shape[1] if bm is not None else 0),
        mask_kv_tiles=(bm.shape[2] if bm is not None else 0),
        num_ctas=num_ctas, balance_rows=balance_rows, sm_scale=float(w.sm_scale),
        window=int(getattr(w, "window", 0)), q_dtype=int(getattr(w, "q_dtype", PA_BF16)),
        q_scale_mode=int(getattr(w, "q_scale_mode", PA_SCALE_PER_TENSOR)),
        unit_cost=int(unit_cost))


# ------------------------------------------------------------ entry points

def pa_version() -> str:
    return load().pa_version().decode()


def pa_num_ctas(problem: PaProblem, mode: int) -> int:
    n = ctypes.c_int32(0)
    _check(load().pa_num_ctas(ctypes.byref(problem), mode, ctypes.byref(n)), "pa_num_ctas")
    return int(n.value)


def pa_assign_workspace_size(problem: PaProblem, mode: int) -> int:
    return int(load().pa_assign_workspace_size(ctypes.byref(problem), mode))


def pa_partial_workspace_size(problem: PaProblem, mode: int) -> int:
    return int(load().pa_partial_workspace_size(ctypes.byref(problem), mode))


def pa_assign(problem, mode, context_lens, q_lens, block_mask, assign_ws, stream=None):
    _check(load().pa_assign(ctypes.byref(problem), mode, _p(context_lens), _p(q_lens),
                            _p(block_mask), _p(assign_ws), _nbytes(assign_ws), _stream(stream)),
           "pa_assign")


def pa_decode_splitk(problem, q, k_cache, v_cache, block_table, context_lens, q_lens, k_scale,
                     v_scale, assign_ws, partial_ws, out, lse, stream=None):
    _check(load().pa_decode_splitk(
        ctypes.byref(problem), _p(q), _p(k_cache), _p(v_cache), _p(block_table),
        _p(context_lens), _p(q_lens), _p(k_scale), _p(v_scale), _p(assign_ws),
        _nbytes(assign_ws), _p(partial_ws), _nbytes(partial_ws), _p(out), _p(lse),
        _stream(stream)), "pa_decode_splitk")


def pa_combine(problem, mode, assign_ws, partial_ws, out, lse, stream=None):
    _check(load().pa_combine(ctypes.byref(problem), mode, _p(assign_ws), _nbytes(assign_ws),
                             _p(partial_ws), _nbytes(partial_ws), _p(out), _p(lse),
                             _stream(stream)), "pa_combine")


def pa_decode_noalloc(problem, q, k_cache, v_cache, block_table, context_lens, q_lens, k_scale,
                      v_scale, out, lse, device_error=None, stream=None):
    """Whole decode with the library's fixed scratch (no workspace arguments)."""
    status = load().pa_decode_noalloc(
        ctypes.byref(problem), _p(q), _p(k_cache), _p(v_cache), _p(block_table),
        _p(context_lens), _p(q_lens), _p(k_scale), _p(v_scale), _p(out), _p(lse),
        _p(device_error), _stream(stream))
    if status == PA_ERR_WORKSPACE:
        raise PaError(status, f"pa_decode_noalloc (the problem needs more than the "
                              f"{PA_NOALLOC_SCRATCH_BYTES} bytes of fixed scratch)")
    _check(status, "pa_decode_noalloc")


def pa_static_workspace_size(problem: PaProblem, num_splits: int = 0) -> int:
    return int(load().pa_static_workspace_size(ctypes.byref(problem), int(num_splits)))


def pa_static_num_splits(problem: PaProblem, num_splits: int = 0) -> int:
    n = ctypes.c_int32(0)
    _check(load().pa_static_num_splits(ctypes.byref(problem), int(num_splits), ctypes.byref(n)),
           "pa_static_num_splits")
    return int(n.value)


def pa_decode_static(problem, num_splits, q, k_cache, v_cache, block_table, context_lens, q_lens,
                     k_scale, v_scale, ws, out, lse, stream=None):
    _check(load().pa_decode_static(
        ctypes.byref(problem), int(num_splits), _p(q), _p(k_cache), _p(v_cache), _p(block_table),
        _p(context_lens), _p(q_lens), _p(k_scale), _p(v_scale), _p(ws), _nbytes(ws), _p(out),
        _p(lse), _stream(stream)), "pa_decode_static")


def pa_prefill(problem, q, k_cache, v_cache, block_table, context_lens, q_lens, k_scale, v_scale,
               block_mask, assign_ws, partial_ws, out, lse, stream=None):
    _check(load().pa_prefill(
        ctypes.byref(problem), _p(q), _p(k_cache), _p(v_cache), _p(block_table),
        _p(context_lens), _p(q_lens), _p(k_scale), _p(v_scale), _p(block_mask), _p(assign_ws),
        _nbytes(assign_ws), _p(partial_ws), _nbytes(partial_ws), _p(out), _p(lse),
        _stream(stream)), "pa_prefill")


def pa_prefill_fp8(problem, q, q_scale, k_cache, v_cache, block_table, context_lens, q_lens,
                   k_scale, v_scale, block_mask, assign_ws, partial_ws, out, lse, stream=None):
    _check(load().pa_prefill_fp8(
        ctypes.byref(problem), _p(q), _p(q_scale), _p(k_cache), _p(v_cache), _p(block_table),
        _p(context_lens), _p(q_lens), _p(k_scale), _p(v_scale), _p(block_mask), _p(assign_ws),
        _nbytes(assign_ws), _p(partial_ws), _nbytes(partial_ws), _p(out), _p(lse),
        _stream(stream)), "pa_prefill_fp8")


def pa_set_task_trace(trace: Optional[torch.Tensor]):
    """Record per-task start/end times of the following launches into
    ``trace`` (int64 [capacity, 3] on the device), or stop with None."""
    if trace is None:
        _check(load().pa_set_task_trace(None, 0), "pa_set_task_trace")
        return
    if trace.dtype != torch.int64 or trace.dim() != 2 or trace.shape[1] != 3:
        raise ValueError("trace must be int64 [capacity, 3]")
    _check(load().pa_set_task_trace(_p(trace), int(trace.shape[0])), "pa_set_task_trace")


def pa_read_task_map(problem, mode, assign_ws, stream=None) -> dict:
    """Copy the task map out of the Assign workspace (synchronises)."""
    lib = load()
    counts = np.zeros(4, np.int32)
    c = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    _check(lib.pa_read_task_map(ctypes.byref(problem), mode, _p(assign_ws), _nbytes(assign_ws),
                                c(counts), None, None, None, None, None, None, None,
                                _stream(stream)), "pa_read_task_map")
    U, T, S, N = (int(x) for x in counts)
    kv_tile = 64 if mode in (PA_MODE_DECODE, PA_MAP_DECODE_PART) else 128
    max_kv_tiles = max(1, -(-max(1, problem.max_context_len) // kv_tile))
    out = dict(num_units=U, num_tasks=T, num_slots=S, num_ctas=N,
               cta_ptr=np.zeros(N + 1, np.int32), tasks=np.zeros((T, 4), np.int32),
               units=np.zeros((U, 4), np.int32), unit_ntiles=np.zeros(U, np.int32),
               unit_nsplit=np.zeros(U, np.int32), unit_slot0=np.zeros(U, np.int32),
               active=np.zeros((U, max_kv_tiles), np.int32) if problem.mask_q_tiles > 0 else None)
    _check(lib.pa_read_task_map(
        ctypes.byref(problem), mode, _p(assign_ws), _nbytes(assign_ws), c(counts),
        c(out["cta_ptr"]), c(out["tasks"]), c(out["units"]), c(out["unit_ntiles"]),
        c(out["unit_nsplit"]), c(out["unit_slot0"]),
        c(out["active"]) if out["active"] is not None else None, _stream(stream)),
        "pa_read_task_map")
    return out


def pa_test_inject_wait_timeout(skip_entry: int, wait_limit_ns: int = 20_000_000):
    """Test hook: the next compute launch leaves one K/V ring entry unfilled in
    CTA 0 and limits its waits to wait_limit_ns (see include/pa.h)."""
    _check(load().pa_test_inject_wait_timeout(int(skip_entry), int(wait_limit_ns)),
           "pa_test_inject_wait_timeout")


def pa_last_device_error(assign_ws, stream=None) -> int:
    code = ctypes.c_int32(0)
    load().pa_last_device_error(_p(assign_ws), ctypes.byref(code), _stream(stream))
    return int(code.value)


# ----------------------------------------------------- convenience wrappers

class Buffers:
    """Workspaces and outputs for one problem (device memory from torch)."""

    def __init__(self, problem: PaProblem, mode: int, device, total_q: int, Hq: int, D: int):
        self.problem = problem
        self.mode = mode
        a = pa_assign_workspace_size(problem, mode)
        p = pa_partial_workspace_size(problem, mode)
        if a == 0 or p == 0:
            raise PaError(1, "workspace size query")
        self.assign_ws = torch.empty(a, dtype=torch.uint8, device=device)
        self.partial_ws = torch.empty(p, dtype=torch.uint8, device=device)
        self.out = torch.empty((total_q, Hq, D), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((total_q, Hq), dtype=torch.float32, device=device)


def make_buffers(w, mode: Optional[int] = None, num_ctas: int = 0, balance_rows: int = 0,
                 unit_cost: int = 0):
    if mode is None:
        mode = PA_MODE_DECODE if w.mode == "decode" else PA_MODE_PREFILL
    prob = problem_from(w, num_ctas=num_ctas, balance_rows=balance_rows, unit_cost=unit_cost)
    return Buffers(prob, mode, w.q.device, w.total_q, w.num_q_heads, w.head_dim)


def run_decode(w, bufs: Optional[Buffers] = None, stream=None) -> Buffers:
    """Assign + split-K decode + Combine for a device-resident workload."""
    if bufs is None:
        bufs = make_buffers(w, PA_MODE_DECODE)
    p = bufs.problem
    pa_assign(p, PA_MODE_DECODE, w.context_lens, w.q_lens, None, bufs.assign_ws, stream)
    pa_decode_splitk(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.q_lens,
                     w.k_scale, w.v_scale, bufs.assign_ws, bufs.partial_ws, bufs.out, bufs.lse,
                     stream)
    pa_combine(p, PA_MODE_DECODE, bufs.assign_ws, bufs.partial_ws, bufs.out, bufs.lse, stream)
    return bufs


class StaticBuffers:
    """Workspace and outputs of the static split-K path (device memory from torch)."""

    def __init__(self, w, num_splits: int = 0, num_ctas: int = 0):
        self.problem = problem_from(w, num_ctas=num_ctas)
        self.num_splits = num_splits
        n = pa_static_workspace_size(self.problem, num_splits)
        if n == 0:
            raise PaError(1, "pa_static_workspace_size")
        self.ws = torch.empty(n, dtype=torch.uint8, device=w.q.device)
        self.out = torch.empty((w.total_q, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                               device=w.q.device)
        self.lse = torch.empty((w.total_q, w.num_q_heads), dtype=torch.float32,
                               device=w.q.device)


def run_decode_static(w, bufs: Optional["StaticBuffers"] = None, num_splits: int = 0,
                      stream=None) -> "StaticBuffers":
    """Static split-K decode (one call, no Assign) for a device-resident workload."""
    if bufs is None:
        bufs = StaticBuffers(w, num_splits)
    pa_decode_static(bufs.problem, bufs.num_splits, w.q, w.k_cache, w.v_cache, w.block_table,
                     w.context_lens, w.q_lens, w.k_scale, w.v_scale, bufs.ws, bufs.out, bufs.lse,
                     stream)
    return bufs


def run_prefill(w, bufs: Optional[Buffers] = None, stream=None) -> Buffers:
    """Assign + prefill / mixed-batch compute + Combine for a device-resident workload."""
    if bufs is None:
        bufs = make_buffers(w, PA_MODE_PREFILL)
    p = bufs.problem
    pa_assign(p, PA_MODE_PREFILL, w.context_lens, w.q_lens, w.block_mask, bufs.assign_ws, stream)
    if p.q_dtype == PA_FP8_E4M3:
        pa_prefill_fp8(p, w.q, w.q_scale, w.k_cache, w.v_cache, w.block_table, w.context_lens,
                       w.q_lens, w.k_scale, w.v_scale, w.block_mask, bufs.assign_ws,
                       bufs.partial_ws, bufs.out, bufs.lse, stream)
    else:
        pa_prefill(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.q_lens,
                   w.k_scale, w.v_scale, w.block_mask, bufs.assign_ws, bufs.partial_ws, bufs.out,
                   bufs.lse, stream)
    pa_combine(p, PA_MODE_PREFILL, bufs.assign_ws, bufs.partial_ws, bufs.out, bufs.lse, stream)
    return bufs
