"""The C-ABI library builds, loads on the host and exports every entry point
declared in include/pa.h; host-side validation works without a GPU (only
calls that never reach the device are made here)."""
import ctypes
import os
import re

import pytest

from paged_attention_gb300 import binding as B
from paged_attention_gb300 import build as build_mod
from paged_attention_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("pa_assign", "pa_decode_splitk", "pa_combine", "pa_prefill"):
        assert name in syms
    assert set(syms) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert B.status_string(0) == "PA_OK"
    assert B.status_string(3) == "PA_ERR_WORKSPACE"
    assert "sm_103a" in B.pa_version()


def test_workspace_sizes_host_only(lib):
    w = W.decode_bf16(mtp=1, shrink=16)
    p = B.problem_from(w, num_ctas=152)
    a = B.pa_assign_workspace_size(p, B.PA_MODE_DECODE)
    part = B.pa_partial_workspace_size(p, B.PA_MODE_DECODE)
    assert a > 0 and a % 256 == 0
    # partial slots = units + CTAs, rows rounded to 16, (D + 1) floats per row
    U = w.num_seqs * w.num_kv_heads
    assert part == (U + 152) * 16 * (128 + 1) * 4
    wp = W.prefill_bf16(sparse=True, shrink=32)
    pp = B.problem_from(wp, num_ctas=152)
    assert B.pa_assign_workspace_size(pp, B.PA_MODE_PREFILL) > 0
    assert B.pa_partial_workspace_size(pp, B.PA_MODE_PREFILL) % (128 * 129 * 4) == 0
    # without a mask, prefill mode adds a decode part: one 16-row slot per
    # (sequence, KV head) and per CTA, after the prefill partials
    wd = W.prefill_bf16(sparse=False, shrink=32)
    pd = B.problem_from(wd, num_ctas=152)
    extra = (wd.num_seqs * wd.num_kv_heads + 152) * 16 * (128 + 1) * 4
    assert (B.pa_partial_workspace_size(pd, B.PA_MODE_PREFILL)
            == B.pa_partial_workspace_size(pp, B.PA_MODE_PREFILL) + extra)
    assert (B.pa_assign_workspace_size(pd, B.PA_MODE_PREFILL)
            > B.pa_assign_workspace_size(pp, B.PA_MODE_PREFILL))


def test_invalid_problems_rejected_on_host(lib):
    w = W.decode_bf16(mtp=1, shrink=16)
    p = B.problem_from(w, num_ctas=8)
    bad = B.PaProblem.from_buffer_copy(p)
    bad.num_kv_heads = 7                      # Hq % Hkv != 0
    assert B.pa_assign_workspace_size(bad, B.PA_MODE_DECODE) == 0
    bad = B.PaProblem.from_buffer_copy(p)
    bad.head_dim = 96                         # not built
    assert B.pa_assign_workspace_size(bad, B.PA_MODE_DECODE) == 0
    bad = B.PaProblem.from_buffer_copy(p)
    bad.max_context_len = max(bad.max_context_len, 17)
    bad.max_q_len = 9                         # G * q_len = 36 rows > 32 per D=128 decode unit
    assert B.pa_assign_workspace_size(bad, B.PA_MODE_DECODE) == 0
    ok = B.PaProblem.from_buffer_copy(p)
    ok.max_q_len = 8                          # 32 rows: built
    assert B.pa_assign_workspace_size(ok, B.PA_MODE_DECODE) > 0
    win = B.PaProblem.from_buffer_copy(p)
    win.window = 100                          # sliding window: bf16 decode is built
    assert B.pa_assign_workspace_size(win, B.PA_MODE_DECODE) > 0
    assert B.pa_assign_workspace_size(win, B.PA_MODE_PREFILL) > 0    # and prefill
    win.kv_dtype = 1                          # E4M3 decode with a window: built
    assert B.pa_assign_workspace_size(win, B.PA_MODE_DECODE) > 0
    bad = B.PaProblem.from_buffer_copy(p)
    bad.window = -1
    assert B.pa_assign_workspace_size(bad, B.PA_MODE_DECODE) == 0
    bad = B.PaProblem.from_buffer_copy(p)
    bad.mask_q_tiles, bad.mask_kv_tiles = 1, 1  # masks are prefill-only
    assert B.pa_assign_workspace_size(bad, B.PA_MODE_DECODE) == 0
    bad = B.PaProblem.from_buffer_copy(p)
    bad.page_size = 48
    assert B.pa_assign_workspace_size(bad, B.PA_MODE_DECODE) == 0
    # null device pointers are refused before any CUDA call
    st = lib.pa_assign(ctypes.byref(p), 0, None, None, None, None, 0, None)
    assert st == 1


def test_noalloc_host_checks(lib):
    """pa_decode_noalloc refuses, before any CUDA call, null pointers and
    problems whose task map + partials exceed the fixed scratch."""
    w = W.decode_bf16(mtp=1, shrink=16)
    p = B.problem_from(w, num_ctas=152)
    fake = ctypes.c_void_p(1 << 20)           # aligned, never dereferenced
    args = [fake] * 10
    st = lib.pa_decode_noalloc(ctypes.byref(p), None, *args[:9], None, None)
    assert st == 1
    need = (-(-B.pa_assign_workspace_size(p, B.PA_MODE_DECODE) // 256) * 256
            + B.pa_partial_workspace_size(p, B.PA_MODE_DECODE))
    assert need <= B.PA_NOALLOC_SCRATCH_BYTES
    big = B.PaProblem.from_buffer_copy(p)
    big.num_seqs = 4096                       # (4096 * 8 + 152) slots x 16 rows x 129 x 4 B
    big.num_ctas = 152
    big_need = (-(-B.pa_assign_workspace_size(big, B.PA_MODE_DECODE) // 256) * 256
                + B.pa_partial_workspace_size(big, B.PA_MODE_DECODE))
    assert big_need > B.PA_NOALLOC_SCRATCH_BYTES
    st = lib.pa_decode_noalloc(ctypes.byref(big), *args, None, None)
    assert st == B.PA_ERR_WORKSPACE
    assert B.PA_NOALLOC_SCRATCH_BYTES == 32 * 1024 * 1024
    header = open(os.path.join(ROOT, "include", "pa.h")).read()
    assert "#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)" in header
    # the binding's copy of the default fixed cost per unit
    assert f"#define PA_DEFAULT_UNIT_COST_DECODE {B.PA_DEFAULT_UNIT_COST_DECODE}\n" in header
    assert f"#define PA_DEFAULT_UNIT_COST_PREFILL {B.PA_DEFAULT_UNIT_COST_PREFILL}\n" in header


def test_static_workspace_sizes_host_only(lib):
    """Static split-K: a 256-byte header and 4 completion counters per unit
    (one per 16-row tile; 256-byte aligned), then U * S partial slots of 16
    rows x (D + 1) floats for S > 1."""
    w = W.decode_bf16(mtp=1, shrink=16)
    p = B.problem_from(w, num_ctas=152)
    U = w.num_seqs * w.num_kv_heads
    head = -(-(256 + U * 4 * 4) // 256) * 256
    assert B.pa_static_workspace_size(p, 1) == head
    assert B.pa_static_workspace_size(p, 4) == head + U * 4 * 16 * 129 * 4
    assert B.pa_static_num_splits(p, 3) == 3
    assert B.pa_static_num_splits(p, 0) >= 1
    assert B.pa_static_workspace_size(p, 65) == 0          # beyond 64 splits


def test_fp8_prefill_host_checks(lib):
    """E4M3 prefill problems: accepted in prefill mode only, with E4M3 K/V and
    head_dim 128; every sequence on the tensor-core map (no decode part)."""
    w = W.prefill_fp8(quant_type=1, shrink=32)
    p = B.problem_from(w, num_ctas=152)
    assert p.q_dtype == B.PA_FP8_E4M3 and p.q_scale_mode == B.PA_SCALE_PER_ROW
    assert B.pa_assign_workspace_size(p, B.PA_MODE_PREFILL) > 0
    assert B.pa_assign_workspace_size(p, B.PA_MODE_DECODE) == 0    # decode takes bf16 Q
    wd = W.prefill_bf16(sparse=False, shrink=32)
    pd = B.problem_from(wd, num_ctas=152)
    extra = (wd.num_seqs * wd.num_kv_heads + 152) * 16 * (128 + 1) * 4
    assert (B.pa_partial_workspace_size(p, B.PA_MODE_PREFILL)
            == B.pa_partial_workspace_size(pd, B.PA_MODE_PREFILL) - extra)
    for field, value in (("head_dim", 64), ("kv_dtype", B.PA_BF16), ("q_dtype", 2),
                         ("q_scale_mode", 2)):
        bad = B.PaProblem.from_buffer_copy(p)
        setattr(bad, field, value)
        assert B.pa_assign_workspace_size(bad, B.PA_MODE_PREFILL) == 0, field
    fake = ctypes.c_void_p(1 << 20)           # aligned, never dereferenced
    # pa_prefill takes no Q scales: an E4M3 Q is refused
    st = lib.pa_prefill(ctypes.byref(p), *([fake] * 8), None, fake, 1 << 30, fake, 1 << 30,
                        fake, fake, None)
    assert st == B.PA_ERR_INVALID_ARG
    # pa_prefill_fp8 needs E4M3 Q and K/V, and its scales
    st = lib.pa_prefill_fp8(ctypes.byref(pd), *([fake] * 9), None, fake, 1 << 30, fake,
                            1 << 30, fake, fake, None)
    assert st == B.PA_ERR_UNSUPPORTED
    st = lib.pa_prefill_fp8(ctypes.byref(p), fake, None, *([fake] * 7), None, fake, 1 << 30,
                            fake, 1 << 30, fake, fake, None)
    assert st == B.PA_ERR_INVALID_ARG


def test_task_trace_host_checks(lib):
    """pa_set_task_trace: a buffer with a capacity, or NULL with 0."""
    fake = ctypes.c_void_p(1 << 20)
    assert lib.pa_set_task_trace(None, 5) == B.PA_ERR_INVALID_ARG
    assert lib.pa_set_task_trace(fake, 0) == B.PA_ERR_INVALID_ARG
    assert lib.pa_set_task_trace(fake, -1) == B.PA_ERR_INVALID_ARG
    assert lib.pa_set_task_trace(ctypes.c_void_p((1 << 20) + 4), 3) == B.PA_ERR_INVALID_ARG
    assert lib.pa_set_task_trace(fake, 3) == B.PA_OK         # never dereferenced here
    assert lib.pa_set_task_trace(None, 0) == B.PA_OK
