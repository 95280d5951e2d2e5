"""GPU Assign task maps and active-tile lists are bit-exact with the oracle's.

"基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 Assign (load-balanced task
map) and 二.1 (active-KV-tile compaction of the block mask)."""
import copy

import numpy as np
import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import task_map_equal

pytestmark = pytest.mark.gpu


def check(w, mode, num_ctas=0, balance_rows=0, unit_cost=0):
    wd = w.to("cuda")
    bufs = B.make_buffers(wd, mode, num_ctas=num_ctas, balance_rows=balance_rows,
                          unit_cost=unit_cost)
    h = B.effective_unit_cost(unit_cost, mode)
    hd = B.effective_unit_cost(unit_cost, B.PA_MODE_DECODE)
    N = B.pa_num_ctas(bufs.problem, mode)
    B.pa_assign(bufs.problem, mode, wd.context_lens, wd.q_lens,
                wd.block_mask if mode == B.PA_MODE_PREFILL else None, bufs.assign_ws)
    gpu = B.pa_read_task_map(bufs.problem, mode, bufs.assign_ws)
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    if mode == B.PA_MODE_DECODE:
        tm = oracle.assign(mode, w.num_seqs, w.num_q_heads, w.num_kv_heads, N, 64,
                           balance_rows or 128, w.context_lens, w.q_lens,
                           window=int(getattr(w, "window", 0)), unit_cost=h)
        task_map_equal(gpu, tm, with_active=False)
        return gpu
    # prefill mode: the prefill map and the decode part (its own CTA count: the
    # decode kernel's, for at most MIXED_DECODE_ROWS rows per unit)
    G = w.num_q_heads // w.num_kv_heads
    pd = copy.copy(bufs.problem)
    pd.max_q_len = min(pd.max_q_len, max(1, oracle.MIXED_DECODE_ROWS // G))
    has_part = w.block_mask is None and G <= oracle.MIXED_DECODE_ROWS
    Nd = B.pa_num_ctas(pd, B.PA_MODE_DECODE) if has_part else N
    pre, dec = oracle.assign_prefill(w.num_seqs, w.num_q_heads, w.num_kv_heads, N,
                                     balance_rows or 128, w.context_lens, w.q_lens,
                                     w.block_mask, decode_ctas=Nd,
                                     window=int(getattr(w, "window", 0)), unit_cost=h,
                                     decode_unit_cost=hd)
    task_map_equal(gpu, pre, with_active=w.block_mask is not None)
    gpu_d = B.pa_read_task_map(bufs.problem, B.PA_MAP_DECODE_PART, bufs.assign_ws)
    if dec is None:
        assert gpu_d["num_units"] == 0 and gpu_d["num_tasks"] == 0
    else:
        task_map_equal(gpu_d, dec, with_active=False)
    return gpu


@pytest.mark.parametrize("mtp", [1, 2, 3])
def test_decode_map_full_size(mtp):
    check(W.decode_bf16(mtp=mtp), B.PA_MODE_DECODE)


def test_decode_map_fp8_full_size():
    check(W.decode_fp8(), B.PA_MODE_DECODE)


@pytest.mark.parametrize("n", [1, 7, 152, 1000])
def test_decode_map_any_cta_count(n):
    check(W.decode_bf16(mtp=1, shrink=8), B.PA_MODE_DECODE, num_ctas=n)


@pytest.mark.parametrize("sparse", [False, True])
def test_prefill_map_full_size(sparse):
    check(W.prefill_bf16(sparse=sparse), B.PA_MODE_PREFILL)


def test_hybrid_map_full_size():
    check(W.hybrid_bf16(), B.PA_MODE_PREFILL)


@pytest.mark.parametrize("rbal", [16, 64, 288])
def test_weighted_map(rbal):
    check(W.hybrid_bf16(shrink=8), B.PA_MODE_PREFILL, balance_rows=rbal)


def test_tiny_mixed_map():
    check(W.tiny_mixed(), B.PA_MODE_PREFILL, num_ctas=5)


@pytest.mark.parametrize("window", [1, 100, 4096])
def test_decode_map_with_sliding_window(window):
    w = W.decode_bf16(mtp=2)
    w.window = window
    check(w, B.PA_MODE_DECODE)


def test_bad_lengths_flagged():
    w = W.decode_bf16(mtp=1, shrink=16).to("cuda")
    bufs = B.make_buffers(w, B.PA_MODE_DECODE)
    ql = w.q_lens.clone()
    ql[0] = int(w.context_lens[0]) + 1          # more new tokens than context
    B.pa_assign(bufs.problem, B.PA_MODE_DECODE, w.context_lens, ql, None, bufs.assign_ws)
    assert B.pa_last_device_error(bufs.assign_ws) & B.PA_DEV_BAD_LENGTHS
    gpu = B.pa_read_task_map(bufs.problem, B.PA_MODE_DECODE, bufs.assign_ws)
    assert gpu["num_units"] == 0 and gpu["num_tasks"] == 0


def test_decode_map_many_short_sequences():
    """3000 sequences (24000 units, some with no query token, some one token
    long): the one-launch decode Assign at scale."""
    g = torch.Generator().manual_seed(77)
    B_ = 3000
    ctx = torch.randint(1, 300, (B_,), generator=g).tolist()
    ql = [min(c, int(q)) for c, q in zip(ctx, torch.randint(0, 3, (B_,), generator=g).tolist())]
    w = W.make_workload("many", ctx, ql, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        page_size=16, seed=77, mode="decode")
    check(w, B.PA_MODE_DECODE)
    check(w, B.PA_MODE_DECODE, num_ctas=7)


def test_prefill_map_beyond_the_shared_memory_cache():
    """24,000 prefill units: more than the map pass keeps in shared memory, so
    it reads unit data from the workspace (the other path of the same pass)."""
    g = torch.Generator().manual_seed(78)
    B_ = 3000
    ctx = torch.randint(40, 200, (B_,), generator=g).tolist()
    ql = [min(c, 5 + int(q)) for c, q in zip(ctx, torch.randint(0, 20, (B_,), generator=g).tolist())]
    w = W.make_workload("manyp", ctx, ql, num_q_heads=32, num_kv_heads=8, head_dim=64,
                        page_size=16, seed=78, mode="prefill")
    check(w, B.PA_MODE_PREFILL)


@pytest.mark.parametrize("window,sparse", [(1, False), (300, False), (1000, True), (4096, True)])
def test_prefill_map_with_sliding_window(window, sparse):
    """Prefill-mode maps with a sliding window: each unit's tiles (or its
    active list under a block mask) start at the first tile its first query
    can see; bit-exact with the oracle, decode part included."""
    w = W.prefill_bf16(sparse=sparse, shrink=4)
    w.window = window
    check(w, B.PA_MODE_PREFILL)
    h = W.hybrid_bf16(shrink=8)
    h.window = window
    check(h, B.PA_MODE_PREFILL, num_ctas=37)


@pytest.mark.parametrize("unit_cost", [-1, 1, 3, 16])
def test_decode_map_unit_cost(unit_cost):
    """Explicit fixed costs per unit (and none): bit-exact with the oracle."""
    check(W.decode_bf16(mtp=1), B.PA_MODE_DECODE, unit_cost=unit_cost)


@pytest.mark.parametrize("unit_cost", [-1, 2, 5])
def test_prefill_maps_unit_cost(unit_cost):
    check(W.hybrid_bf16(shrink=4), B.PA_MODE_PREFILL, unit_cost=unit_cost)
    check(W.prefill_bf16(sparse=True, shrink=4), B.PA_MODE_PREFILL, unit_cost=unit_cost)
