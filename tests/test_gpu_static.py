"""Static split-K decode (pa_decode_static) against the fp64 oracle.

"基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (the Static Split-K
paragraph: a fixed split count, no dynamic Assign, a shorter launch chain) and
三.3 (the regular split mapping resolved from the program id).  Every unit is
cut into S equal splits; split units are finalized in the kernel.  Tolerances
as for the dynamic path: bf16 outputs 2e-2, E4M3 6e-2, LSE 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import compare

pytestmark = pytest.mark.gpu


def run_and_compare(w, num_splits, rows=None, num_ctas=0):
    wd = w.to("cuda")
    bufs = B.StaticBuffers(wd, num_splits, num_ctas=num_ctas)
    bufs.out.fill_(float("nan"))
    B.run_decode_static(wd, bufs)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.ws) == 0
    ref_o, ref_l = oracle.attention(w, rows=rows)
    compare(w, bufs.out, bufs.lse, ref_o, ref_l, rows=rows)
    return bufs


@pytest.mark.parametrize("S", [1, 2, 3, 8, 64])
def test_static_bf16_shrunk(S):
    """Split counts from one to more than most units have tiles (empty splits)."""
    run_and_compare(W.decode_bf16(mtp=2, shrink=16), S)


@pytest.mark.parametrize("S,n", [(4, 1), (2, 5), (5, 37)])
def test_static_any_cta_count(S, n):
    run_and_compare(W.decode_bf16(mtp=1, shrink=8), S, num_ctas=n)


def test_static_fp8_and_windows():
    run_and_compare(W.decode_fp8(shrink=16), 4)
    w = W.decode_fp8(shrink=16)
    w.window = 300
    run_and_compare(w, 3)
    w = W.decode_bf16(mtp=3, shrink=8)
    w.window = 100
    run_and_compare(w, 8)


def test_static_edge_cases():
    # ctx < page, q_len 0, one long sequence, head_dim 64, pages of 16
    ctx = [1, 5, 64, 128, 129, 4, 3000, 63]
    ql = [1, 5, 2, 4, 1, 4, 3, 0]
    w = W.make_workload("sedge", ctx, ql, num_q_heads=16, num_kv_heads=4, head_dim=128,
                        page_size=64, seed=31)
    run_and_compare(w, 4, num_ctas=11)
    w = W.make_workload("sd64", [300, 17, 4096], [2, 1, 4], num_q_heads=8, num_kv_heads=1,
                        head_dim=64, page_size=16, seed=32)
    run_and_compare(w, 8, num_ctas=9)


def test_static_many_sequences():
    """Query offsets come from a prefix over q_lens computed in the kernel:
    3000 short sequences, a third of them without a query token."""
    g = torch.Generator().manual_seed(79)
    n = 3000
    ctx = torch.randint(1, 300, (n,), generator=g).tolist()
    ql = [min(c, int(q)) for c, q in zip(ctx, torch.randint(0, 3, (n,), generator=g).tolist())]
    w = W.make_workload("smany", ctx, ql, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        page_size=16, seed=79, mode="decode")
    run_and_compare(w, 2)


def test_static_full_size_default_splits():
    """The bf16 decode workload at full size with the library's split count,
    checked on every row."""
    w = W.decode_bf16(mtp=1)
    bufs = run_and_compare(w, 0)
    assert B.pa_static_num_splits(bufs.problem, 0) >= 1


def test_static_fp8_full_size_sampled():
    w = W.decode_fp8()
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(w.total_q * w.num_q_heads, size=4096, replace=False))
    run_and_compare(w, 4, rows=rows)


def test_static_bad_lengths_reported_and_next_call_clean():
    good = W.decode_bf16(mtp=1, shrink=16)
    bad = W.decode_bf16(mtp=1, shrink=16)
    bad.context_lens[2] = 1                      # q_len 2 > context length 1
    wb = bad.to("cuda")
    bufs = B.StaticBuffers(wb, 2)
    B.run_decode_static(wb, bufs)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.ws) & B.PA_DEV_BAD_LENGTHS
    wg = good.to("cuda")
    B.run_decode_static(wg, bufs)                # the call clears the error word itself
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.ws) == 0
    ref_o, ref_l = oracle.attention(good)
    compare(good, bufs.out, bufs.lse, ref_o, ref_l)


def test_static_is_deterministic_and_replays_from_a_graph():
    w = W.decode_bf16(mtp=2, shrink=8).to("cuda")
    bufs = B.StaticBuffers(w, 4)
    B.run_decode_static(w, bufs)
    torch.cuda.synchronize()
    o1, l1 = bufs.out.clone(), bufs.lse.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.run_decode_static(w, bufs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.run_decode_static(w, bufs)
    bufs.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bufs.out, o1) and torch.equal(bufs.lse, l1)


@pytest.mark.parametrize("S,n", [(2, 38), (4, 152), (8, 16), (8, 0), (2, 0)])
def test_static_cluster_dsm_merge(S, n):
    """S in {2, 4, 8} with a grid that is a multiple of S: the splits of a
    unit run on the S CTAs of one hardware cluster and merge through
    distributed shared memory ("基于Triton-TLE…", 三.3).  bf16 (8 and 16 rows
    per unit) and E4M3 (24 rows), windows, q_len 0, units with fewer tiles
    than S."""
    run_and_compare(W.decode_bf16(mtp=1, shrink=8), S, num_ctas=n)
    run_and_compare(W.decode_bf16(mtp=3, shrink=16), S, num_ctas=n)
    run_and_compare(W.decode_fp8(shrink=16), S, num_ctas=n)
    w = W.make_workload("cl", [1, 70, 5, 900, 3000, 64], [1, 2, 0, 3, 3, 3], num_q_heads=32,
                        num_kv_heads=8, head_dim=128, page_size=16, seed=S + n)
    w.window = 200
    run_and_compare(w, S, num_ctas=n)


def test_static_cluster_and_partials_agree():
    """The same static split through DSM (grid a multiple of S) and through the
    partial workspace (a grid that is not) give outputs within rounding."""
    w = W.decode_bf16(mtp=2, shrink=8).to("cuda")
    a = B.StaticBuffers(w, 4, num_ctas=40)
    b = B.StaticBuffers(w, 4, num_ctas=41)
    # the partial area (after the header and counters, i.e. the whole S = 1
    # workspace) is filled with a sentinel: the DSM path never writes it
    head = B.pa_static_workspace_size(a.problem, 1)
    a.ws[head:].fill_(0xA5)
    b.ws[head:].fill_(0xA5)
    B.run_decode_static(w, a)
    B.run_decode_static(w, b)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(a.ws) == 0 and B.pa_last_device_error(b.ws) == 0
    assert bool((a.ws[head:] == 0xA5).all()), "cluster mode wrote partials"
    assert not bool((b.ws[head:] == 0xA5).all()), "partial mode wrote no partials"
    assert (a.out.float() - b.out.float()).abs().max().item() <= 1e-2
    assert (a.lse - b.lse).abs().max().item() <= 1e-5
