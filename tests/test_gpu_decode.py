"""GPU split-K decode (Assign + Split-K + Combine) against the fp64 oracle.

"基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Dynamic Split-K decode,
Combine equal to full attention), 三.1 (GQA x MTP rows share a KV tile).
Tolerances: bf16 outputs max-abs 2e-2, LSE 1e-3, FP8-KV outputs 6e-2."""
import numpy as np
import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import compare

pytestmark = pytest.mark.gpu


def run_and_compare(w, rows=None, num_ctas=0):
    wd = w.to("cuda")
    bufs = B.make_buffers(wd, B.PA_MODE_DECODE, num_ctas=num_ctas)
    B.run_decode(wd, bufs)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    ref_o, ref_l = oracle.attention(w, rows=rows)
    return compare(w, bufs.out, bufs.lse, ref_o, ref_l, rows=rows), bufs


@pytest.mark.parametrize("mtp", [1, 2, 3])
def test_decode_bf16_shrunk(mtp):
    run_and_compare(W.decode_bf16(mtp=mtp, shrink=16))


def test_decode_fp8_shrunk():
    run_and_compare(W.decode_fp8(shrink=16))


@pytest.mark.parametrize("n", [1, 3, 37, 500])
def test_decode_any_cta_count(n):
    """Many / few CTAs change how units split; the result must not change."""
    run_and_compare(W.decode_bf16(mtp=2, shrink=16), num_ctas=n)


def test_decode_mixed_edge_cases():
    # ctx < page, ctx a page multiple, ctx = ql, one long sequence, q_len 0
    ctx = [1, 5, 64, 128, 129, 4, 3000, 63]
    ql = [1, 5, 2, 4, 1, 4, 3, 0]
    w = W.make_workload("edge", ctx, ql, num_q_heads=16, num_kv_heads=4, head_dim=128,
                        page_size=64, seed=21)
    run_and_compare(w, num_ctas=11)


@pytest.mark.parametrize("ps,layout", [(16, W.NHD), (32, W.HND), (128, W.NHD), (256, W.HND)])
def test_decode_page_sizes_and_layouts(ps, layout):
    w = W.make_workload("pages", [33, 700, 1025, 64, 2], [1, 2, 1, 2, 1], num_q_heads=8,
                        num_kv_heads=2, head_dim=128, page_size=ps, layout=layout, seed=ps)
    run_and_compare(w, num_ctas=13)


def test_decode_head_dim_64_and_gqa_variants():
    w = W.make_workload("d64", [300, 17, 4096], [2, 1, 4], num_q_heads=8, num_kv_heads=1,
                        head_dim=64, page_size=16, seed=5)
    run_and_compare(w, num_ctas=9)
    w = W.make_workload("mha", [300, 17], [1, 1], num_q_heads=4, num_kv_heads=4, head_dim=128,
                        page_size=64, seed=6)
    run_and_compare(w)


def test_decode_rows_up_to_64_head_dim_64():
    w = W.make_workload("rows64", [500, 90], [8, 5], num_q_heads=16, num_kv_heads=2,
                        head_dim=64, page_size=64, seed=8)
    run_and_compare(w, num_ctas=10)


def test_decode_rows_32_head_dim_128():
    w = W.make_workload("rows32", [500, 90, 1200], [4, 3, 4], num_q_heads=16, num_kv_heads=2,
                        head_dim=128, page_size=64, seed=10)
    run_and_compare(w, num_ctas=10)


def test_decode_fp8_mtp4_and_small_pages():
    w = W.make_workload("fp8b", [100, 1000, 2049], [4, 4, 4], num_q_heads=32, num_kv_heads=4,
                        head_dim=128, page_size=16, layout=W.NHD, kv_dtype=W.FP8_E4M3, seed=9)
    run_and_compare(w, num_ctas=7)


def test_decode_bf16_full_size_mtp1():
    """The benchmark workload, in the launch configuration the bench times,
    checked on every row."""
    run_and_compare(W.decode_bf16(mtp=1))


@pytest.mark.parametrize("mtp", [2, 3])
def test_decode_bf16_full_size_mtp(mtp):
    """The bf16 decode workload at q_len 3 and 4 at full size (12 and 16 rows
    per unit), checked on every row."""
    run_and_compare(W.decode_bf16(mtp=mtp))


def test_decode_fp8_full_size_sampled():
    w = W.decode_fp8()
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(w.total_q * w.num_q_heads, size=4096, replace=False))
    run_and_compare(w, rows=rows)


def test_decode_fp8_q_len_4_full_size_sampled():
    """The E4M3 workload with four query tokens per sequence (MTP 3 here;
    the pages' "MTP4" row counts the tokens): 32 rows per unit, the
    four-tile variant, sampled rows at full size."""
    w = W.decode_fp8(mtp=3)
    rng = np.random.default_rng(4)
    rows = np.sort(rng.choice(w.total_q * w.num_q_heads, size=4096, replace=False))
    run_and_compare(w, rows=rows)


@pytest.mark.parametrize("window,ps,ql,D", [(1, 64, 1, 128), (64, 64, 2, 128), (100, 16, 3, 128),
                                             (1000, 32, 4, 128), (5000, 64, 2, 128),
                                             (300, 16, 2, 64)])
def test_decode_sliding_window(window, ps, ql, D):
    """Sliding window ("HiLS-Attention", 二.1 local branch): each query sees
    the keys p - window < j <= p.  Windows shorter than a tile, a tile long,
    across page boundaries, past some contexts; MTP rows whose windows start
    at different keys; split units (19 CTAs)."""
    ctx = [37, 700, 1500, 4096, 129, 9000]
    w = W.make_workload(f"win{window}", ctx, [ql] * 6, num_q_heads=32, num_kv_heads=8,
                        head_dim=D, page_size=ps, seed=window + ps + ql)
    w.window = window
    run_and_compare(w, num_ctas=19)


@pytest.mark.parametrize("window,ps,ql,G,layout", [(1, 64, 1, 8, W.HND), (64, 64, 3, 8, W.HND),
                                                    (100, 16, 2, 4, W.NHD),
                                                    (1000, 32, 4, 8, W.HND),
                                                    (5000, 64, 3, 8, W.NHD),
                                                    (37, 128, 4, 4, W.NHD)])
def test_decode_fp8_sliding_window(window, ps, ql, G, layout):
    """The sliding window on the E4M3 decode kernel: every row-tile variant
    (8 to 32 rows), windows below, at and far above a 64-token tile, MTP rows
    whose windows start at different keys, pages of 16 to 128 tokens, both
    layouts, split units (19 CTAs)."""
    ctx = [37, 700, 1500, 4096, 129, 9000]
    w = W.make_workload(f"win8_{window}", ctx, [ql] * 6, num_q_heads=8 * G, num_kv_heads=8,
                        head_dim=128, page_size=ps, layout=layout, kv_dtype=W.FP8_E4M3,
                        seed=7 * window + ps + ql)
    w.window = window
    run_and_compare(w, num_ctas=19)


def test_decode_fp8_window_full_size_sampled():
    """The E4M3 workload (q_len 3) with a 2048-key window at full size."""
    w = W.decode_fp8()
    w.window = 2048
    rng = np.random.default_rng(12)
    rows = np.sort(rng.choice(w.total_q * w.num_q_heads, size=4096, replace=False))
    run_and_compare(w, rows=rows)


def test_decode_is_deterministic():
    w = W.decode_bf16(mtp=3, shrink=8).to("cuda")
    a = B.run_decode(w)
    o1, l1 = a.out.clone(), a.lse.clone()
    B.run_decode(w, a)
    torch.cuda.synchronize()
    assert torch.equal(o1, a.out) and torch.equal(l1, a.lse)


def test_bad_page_is_reported_not_faulted():
    w = W.decode_bf16(mtp=1, shrink=16)
    w.block_table[1, 0] = w.num_pages + 100   # out of the pool
    wd = w.to("cuda")
    bufs = B.run_decode(wd)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) & B.PA_DEV_BAD_PAGE


def test_decode_fp8_page_scales_spread():
    """Per-page K/V scales that differ by up to 2^6 between the pages of one
    sequence (P carries v_scale relative to the first page a warp sees)."""
    w = W.make_workload("fp8s", [900, 3000, 130], [3, 3, 3], num_q_heads=64, num_kv_heads=8,
                        head_dim=128, page_size=64, layout=W.HND, kv_dtype=W.FP8_E4M3, seed=41)
    g = torch.Generator().manual_seed(41)
    mult_k = torch.pow(2.0, -torch.randint(0, 7, w.k_scale.shape, generator=g).float())
    mult_v = torch.pow(2.0, -torch.randint(0, 7, w.v_scale.shape, generator=g).float())
    w.k_scale = (w.k_scale * mult_k).contiguous()
    w.v_scale = (w.v_scale * mult_v).contiguous()
    run_and_compare(w, num_ctas=17)


@pytest.mark.parametrize("ql,G,layout,ps", [(1, 8, W.HND, 64), (2, 8, W.NHD, 32), (1, 4, W.NHD, 16),
                                            (3, 4, W.HND, 128)])
def test_decode_fp8_row_tiles(ql, G, layout, ps):
    """Every E4M3 row-tile variant (8, 16, 24 and 32 rows per unit hit NT = 1..4
    across this and the other FP8 tests), both layouts, small and large pages."""
    hkv = 4
    w = W.make_workload(f"fp8r{ql}{G}", [37, 700, 1500, 64, 129], [ql] * 5, num_q_heads=G * hkv,
                        num_kv_heads=hkv, head_dim=128, page_size=ps, layout=layout,
                        kv_dtype=W.FP8_E4M3, seed=50 + ql * 10 + G)
    run_and_compare(w, num_ctas=19)


def test_decode_step_replays_from_a_cuda_graph():
    """Assign + split-K + Combine captured once in a CUDA graph and replayed give
    the eager result bit for bit, also after the inputs change in place."""
    w = W.decode_bf16(mtp=2, shrink=16).to("cuda")
    bufs = B.make_buffers(w, B.PA_MODE_DECODE)
    B.run_decode(w, bufs)
    torch.cuda.synchronize()
    eager_o, eager_l = bufs.out.clone(), bufs.lse.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.run_decode(w, bufs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.run_decode(w, bufs)
    bufs.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bufs.out, eager_o) and torch.equal(bufs.lse, eager_l)
    # new query values in place: the replay reads them
    w.q.mul_(-1.0)
    B.run_decode(w, bufs)
    torch.cuda.synchronize()
    eager2 = bufs.out.clone()
    bufs.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bufs.out, eager2)
    assert B.pa_last_device_error(bufs.assign_ws) == 0


def test_decode_many_short_sequences():
    """3000 short sequences, a third of them without a query token."""
    g = torch.Generator().manual_seed(78)
    B_ = 3000
    ctx = torch.randint(1, 300, (B_,), generator=g).tolist()
    ql = [min(c, int(q)) for c, q in zip(ctx, torch.randint(0, 3, (B_,), generator=g).tolist())]
    w = W.make_workload("many", ctx, ql, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        page_size=16, seed=78, mode="decode")
    run_and_compare(w)


def test_decode_and_prefill_without_query_tokens():
    """A batch where no sequence has a new token: nothing to compute, no error."""
    w = W.make_workload("noq", [5, 300, 64], [0, 0, 0], num_q_heads=8, num_kv_heads=2,
                        head_dim=128, page_size=64, seed=79, mode="decode")
    wd = w.to("cuda")
    bufs = B.run_decode(wd)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    bufs = B.run_prefill(wd)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
