"""fp64 CPU oracle for paged-KV-cache attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference leg may import this package.  It is
a ctypes wrapper around ``pa_oracle.c`` (plain C, fp64, OpenMP); it shares no
code with the CUDA library and the CUDA library never calls it.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` and ``tests/test_oracle_assign.py``.

Pages cited (by title and section):
  "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Assign / Split-K /
  Combine, block-table paging, block mask), 二.1 (active-tile list), 三.3
  (softmax-aware merge); the xdnf.cn "Chunked Prefill" hybrid-batch article
  (causal chunk over unmasked history); "vLLM Triton Attention Backend Deep
  Dive", "Q Blocks" (GQA grouping).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

INT64_MAX = (1 << 63) - 1


class OracleProblem(ctypes.Structure):
    """Field-for-field copy of ``oracle_problem`` in pa_oracle.c."""

    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("mask_q_tiles", ctypes.c_int32),
        ("mask_kv_tiles", ctypes.c_int32),
        ("mask_tile", ctypes.c_int32),
        ("sm_scale", ctypes.c_double),
        ("window", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("q_scale_mode", ctypes.c_int32),
        ("kv_scale_mode", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into a shared library (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            vp = ctypes.c_void_p
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [
                P(OracleProblem), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, ctypes.c_int]
            lib.oracle_assign.restype = ctypes.c_int
            lib.oracle_assign.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, vp, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int64, vp, vp, vp,
                ctypes.c_int64, ctypes.c_int, ctypes.c_int]
            lib.oracle_combine.restype = None
            lib.oracle_combine.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _arr(x, dtype):
    """numpy array with dtype ``dtype`` holding the same bytes as ``x``.

    Torch tensors of 16-/8-bit float types are reinterpreted bit for bit (the
    oracle decodes bf16 and E4M3 itself); same-width types are viewed, other
    integer / float arrays converted."""
    if x is None:
        return None
    dtype = np.dtype(dtype)
    if hasattr(x, "detach"):
        import torch
        t = x.detach().contiguous().cpu()
        if t.dtype.is_floating_point and t.dtype not in (torch.float32, torch.float64):
            t = t.view(torch.int16 if t.element_size() == 2 else torch.uint8)
        elif t.dtype == torch.bool:
            t = t.view(torch.uint8)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == dtype:
        return a
    if a.dtype.itemsize == dtype.itemsize and (a.dtype.kind in "iub") == (dtype.kind in "iub"):
        return a.view(dtype)
    return np.ascontiguousarray(a.astype(dtype))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_to_double(byte: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(byte) & 0xFF))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def attention(w, rows=None, key_lo=0, key_hi=INT64_MAX, mask=True, num_threads=0):
    """fp64 attention of workload ``w`` (see paged_attention_gb300.workloads).

    rows: None for all (token, q-head) rows, else int64 array of token*Hq+h.
    Returns (out [n_rows, D] float64, lse [n_rows] float64).
    """
    lib = _load()
    q_dtype = int(getattr(w, "q_dtype", 0))
    q = _arr(w.q, np.uint16 if q_dtype == 0 else np.uint8)
    qs = _arr(w.q_scale, np.float32) if q_dtype == 1 else None
    kc = _arr(w.k_cache, np.uint16 if w.kv_dtype == 0 else np.uint8)
    vc = _arr(w.v_cache, np.uint16 if w.kv_dtype == 0 else np.uint8)
    ks = _arr(w.k_scale, np.float32) if w.kv_dtype == 1 else None
    vs = _arr(w.v_scale, np.float32) if w.kv_dtype == 1 else None
    bt = _arr(w.block_table, np.int32)
    ctx = _arr(w.context_lens, np.int32)
    ql = _arr(w.q_lens, np.int32)
    bm = _arr(w.block_mask, np.uint8) if (mask and w.block_mask is not None) else None
    total = int(ql.sum())
    if rows is None:
        n_rows = total * w.num_q_heads
        rows_a = None
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_a.shape[0]
    prob = OracleProblem(
        num_seqs=w.num_seqs, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, page_size=w.page_size, num_pages=w.num_pages,
        max_pages_per_seq=bt.shape[1], layout=w.layout, kv_dtype=w.kv_dtype,
        mask_q_tiles=(bm.shape[1] if bm is not None else 0),
        mask_kv_tiles=(bm.shape[2] if bm is not None else 0),
        mask_tile=w.mask_tile, sm_scale=float(w.sm_scale), window=int(getattr(w, "window", 0)),
        q_dtype=q_dtype,
        q_scale_mode=int(getattr(w, "q_scale_mode", 0)),
        kv_scale_mode=int(getattr(w, "kv_scale_mode", 0)))
    out = np.zeros((n_rows, w.head_dim), dtype=np.float64)
    lse = np.zeros((n_rows,), dtype=np.float64)
    rc = lib.oracle_attention(ctypes.byref(prob), _ptr(q), _ptr(qs), _ptr(kc), _ptr(vc), _ptr(ks),
                              _ptr(vs), _ptr(bt), _ptr(ctx), _ptr(ql), _ptr(bm), _ptr(rows_a),
                              n_rows, int(key_lo), int(key_hi), _ptr(out), _ptr(lse),
                              int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with status {rc}")
    return out, lse


def combine(o_parts, lse_parts):
    """Merge split-K partials of one row: o_parts [S, D], lse_parts [S]."""
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, D = o_parts.shape
    o = np.zeros((D,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    lib.oracle_combine(S, D, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    return o, float(lse[0])


class TaskMap:
    """Result of oracle Assign (all int32 numpy arrays)."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def assign(mode, num_seqs, num_q_heads, num_kv_heads, num_ctas, kv_tile, balance_rows,
           context_lens, q_lens, block_mask=None, mask_tile=128, window=0, unit_cost=0):
    """Oracle Assign (the tile-by-tile procedure written in pa_oracle.c).

    mode 0 = decode units (b, hk); mode 1 = prefill / mixed units (b, hk, q tile).
    window > 0: a unit's tiles start at the first one its first query can see.
    unit_cost: the fixed cost of a unit with tiles, in tile-weight units.
    """
    lib = _load()
    ctx = _arr(context_lens, np.int32)
    ql = _arr(q_lens, np.int32)
    bm = _arr(block_mask, np.uint8) if block_mask is not None else None
    G = num_q_heads // num_kv_heads
    if mode == 0:
        unit_cap = num_seqs * num_kv_heads
    else:
        qtok = 128 if (bm is not None and G == 1) else max(1, 256 // G)
        unit_cap = num_kv_heads * int(sum((int(x) + qtok - 1) // qtok for x in ql))
    unit_cap = max(unit_cap, 1)
    max_ctx = int(ctx.max()) if ctx.size else 0
    max_kv_tiles = max(1, (max_ctx + kv_tile - 1) // kv_tile)
    task_cap = unit_cap + num_ctas + 1
    units = np.zeros((unit_cap, 4), np.int32)
    ntiles = np.zeros((unit_cap,), np.int32)
    active = np.zeros((unit_cap, max_kv_tiles), np.int32)
    cta_ptr = np.zeros((num_ctas + 1,), np.int32)
    tasks = np.zeros((task_cap, 4), np.int32)
    nsplit = np.zeros((unit_cap,), np.int32)
    slot0 = np.zeros((unit_cap,), np.int32)
    counts = np.zeros((3,), np.int32)
    rc = lib.oracle_assign(
        int(mode), int(num_seqs), int(num_q_heads), int(num_kv_heads), int(num_ctas),
        int(kv_tile), int(balance_rows), _ptr(ctx), _ptr(ql), _ptr(bm),
        (bm.shape[1] if bm is not None else 0), (bm.shape[2] if bm is not None else 0),
        int(mask_tile), _ptr(units), _ptr(ntiles), _ptr(active), int(max_kv_tiles),
        _ptr(cta_ptr), _ptr(tasks), int(task_cap), _ptr(nsplit), _ptr(slot0), _ptr(counts),
        int(unit_cap), int(window), int(unit_cost))
    if rc != 0:
        raise ValueError(f"oracle_assign failed with status {rc}")
    U, n_tasks, n_slots = (int(x) for x in counts)
    return TaskMap(num_units=U, num_tasks=n_tasks, num_slots=n_slots,
                   units=units[:U], unit_ntiles=ntiles[:U], active=active[:U],
                   cta_ptr=cta_ptr, tasks=tasks[:n_tasks], unit_nsplit=nsplit[:U],
                   unit_slot0=slot0[:U], max_kv_tiles=max_kv_tiles)


# A prefill-mode batch without a block mask sends every sequence with
# 1 <= G * q_len <= MIXED_DECODE_ROWS to a decode-mode map (the decode steps of a
# mixed chunked-prefill + decode batch) and the others to the prefill-mode map.
MIXED_DECODE_ROWS = 16


def assign_prefill(num_seqs, num_q_heads, num_kv_heads, num_ctas, balance_rows,
                   context_lens, q_lens, block_mask=None, decode_ctas=None, window=0,
                   unit_cost=0, decode_unit_cost=None):
    """Prefill-mode Assign as pa_assign(PA_MODE_PREFILL) defines it.

    Returns (prefill_map, decode_map).  Each map is the plain Assign over the
    whole batch with the other part's q_lens taken as 0: such a sequence has no
    prefill units, and its decode units hold no query and no tile.  decode_map
    is None when the batch has a block mask or G > MIXED_DECODE_ROWS (every
    sequence then stays in the prefill map).  decode_ctas: the decode map's CTA
    count (default num_ctas).  window: the sliding window, passed to both maps
    (a unit's tiles start at the first one its first query can see).  unit_cost /
    decode_unit_cost: the fixed cost per unit of the prefill / decode map (the
    decode map's defaults to unit_cost)."""
    if decode_unit_cost is None:
        decode_unit_cost = unit_cost
    G = num_q_heads // num_kv_heads
    ql = [int(x) for x in q_lens]
    if block_mask is not None or G > MIXED_DECODE_ROWS:
        return assign(1, num_seqs, num_q_heads, num_kv_heads, num_ctas, 128, balance_rows,
                      context_lens, ql, block_mask, window=window,
                      unit_cost=unit_cost), None
    small_q = MIXED_DECODE_ROWS // G
    ql_pre = [q if q > small_q else 0 for q in ql]
    ql_dec = [q if q <= small_q else 0 for q in ql]
    pre = assign(1, num_seqs, num_q_heads, num_kv_heads, num_ctas, 128, balance_rows,
                 context_lens, ql_pre, window=window, unit_cost=unit_cost)
    dec = assign(0, num_seqs, num_q_heads, num_kv_heads, decode_ctas or num_ctas, 64,
                 balance_rows, context_lens, ql_dec, window=window, unit_cost=decode_unit_cost)
    return pre, dec
