"""Mixed batches through pa_prefill: the decode-shaped sequences (1 <= G *
q_len <= 16) run on the decode kernel over a decode-mode map of their own, the
others on the tensor-core prefill kernel ("Chunked Prefill" hybrid batch
article: decode rows and prefill chunks in one batch).  Outputs are compared
with the oracle element by element; the two maps with oracle.assign_prefill."""
import copy

import numpy as np
import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import compare, task_map_equal

pytestmark = pytest.mark.gpu


def run(w, num_ctas=0):
    wd = w.to("cuda")
    bufs = B.make_buffers(wd, B.PA_MODE_PREFILL, num_ctas=num_ctas)
    B.run_prefill(wd, bufs)
    torch.cuda.synchronize()
    return wd, bufs


def check(w, num_ctas=0):
    wd, bufs = run(w, num_ctas)
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    ref_o, ref_l = oracle.attention(w)
    compare(w, bufs.out, bufs.lse, ref_o, ref_l)
    # both task maps, bit-exact
    G = w.num_q_heads // w.num_kv_heads
    N = B.pa_num_ctas(bufs.problem, B.PA_MODE_PREFILL)
    pd = copy.copy(bufs.problem)
    pd.max_q_len = min(pd.max_q_len, max(1, oracle.MIXED_DECODE_ROWS // G))
    split = G <= oracle.MIXED_DECODE_ROWS
    Nd = B.pa_num_ctas(pd, B.PA_MODE_DECODE) if split else N
    pre, dec = oracle.assign_prefill(
        w.num_seqs, w.num_q_heads, w.num_kv_heads, N, 128, w.context_lens, w.q_lens,
        decode_ctas=Nd, unit_cost=B.effective_unit_cost(bufs.problem.unit_cost, B.PA_MODE_PREFILL),
        decode_unit_cost=B.effective_unit_cost(bufs.problem.unit_cost, B.PA_MODE_DECODE))
    task_map_equal(B.pa_read_task_map(bufs.problem, B.PA_MODE_PREFILL, bufs.assign_ws), pre,
                   with_active=False)
    gd = B.pa_read_task_map(bufs.problem, B.PA_MAP_DECODE_PART, bufs.assign_ws)
    if dec is None:
        assert gd["num_units"] == 0
    else:
        task_map_equal(gd, dec, with_active=False)
    return pre, dec


def test_rows_at_the_split_boundary():
    """G = 4: q_len 4 (16 rows) is decode-shaped, q_len 5 (20 rows) is not."""
    ctx = [900, 33, 400, 17, 260, 700]
    ql = [4, 5, 1, 16, 3, 200]
    w = W.make_workload("edge", ctx, ql, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        page_size=16, seed=61, mode="prefill")
    pre, dec = check(w, num_ctas=19)
    assert sorted({int(u[0]) for u in pre.units}) == [1, 3, 5]
    assert sorted({int(u[0]) for u, n in zip(dec.units, dec.unit_ntiles) if u[3] > 0}) == [0, 2, 4]


def test_every_sequence_decode_shaped():
    """The prefill map is empty: only the decode kernel writes."""
    ctx = [5000, 64, 1, 777, 2049]
    ql = [2, 1, 1, 2, 1]
    w = W.make_workload("alldec", ctx, ql, num_q_heads=16, num_kv_heads=2, head_dim=128,
                        page_size=32, seed=62, mode="prefill")
    pre, dec = check(w)
    assert pre.num_units == 0 and dec.num_tasks > 0


def test_no_decode_shaped_sequence():
    """Every sequence takes the prefill kernel; the decode part is empty."""
    ctx = [300, 1000]
    ql = [300, 40]
    w = W.make_workload("nodec", ctx, ql, num_q_heads=8, num_kv_heads=1, head_dim=64,
                        page_size=64, seed=63, mode="prefill")
    pre, dec = check(w, num_ctas=11)
    assert dec.num_tasks == 0


@pytest.mark.parametrize("G", [16, 32])
def test_group_width_at_the_limit(G):
    """G = 16: one query token is 16 rows (decode part); G = 32: 32 rows, so
    the batch has no decode part at all."""
    ctx = [1500, 90, 3000]
    ql = [1, 1, 64]
    w = W.make_workload(f"g{G}", ctx, ql, num_q_heads=G, num_kv_heads=1, head_dim=128,
                        page_size=64, seed=64 + G, mode="prefill")
    pre, dec = check(w, num_ctas=31)
    if G == 16:
        assert dec.num_tasks > 0 and sorted({int(u[0]) for u in pre.units}) == [2]
    else:
        assert dec is None


def test_bad_page_in_the_decode_part_is_reported():
    """A block-table entry outside the pool, read by the decode kernel, lands
    in the error word that pa_last_device_error reads."""
    w = W.make_workload("badpg", [500, 40], [1, 40], num_q_heads=8, num_kv_heads=2,
                        head_dim=128, page_size=16, seed=65, mode="prefill")
    w.block_table[0, 3] = w.num_pages + 50   # sequence 0 is decode-shaped
    wd, bufs = run(w, num_ctas=9)
    assert B.pa_last_device_error(bufs.assign_ws) & B.PA_DEV_BAD_PAGE
