"""GPU E4M3 prefill (pa_prefill_fp8: Assign + tcgen05 kind::f8f6f4 prefill +
Combine) against the fp64 oracle on the same quantised inputs.

"基于Triton-TLE优化Tencent HPC-Ops Attention", 二 (FP8 prefill over NHD and
HND caches, two quantisation types, dense or block-sparse) and 三 (quant type
0: one scale for Q, K and V each; quant type 1: Q scaled per (token, q head),
K and V per tensor).  The oracle dequantises the E4M3 bytes exactly and
computes in fp64, so the tolerance covers only the kernel's own rounding (the
probabilities as two E4M3 terms, fp32 accumulation, bf16 output): max-abs
6e-2 on outputs, 1e-3 on the natural-log LSE."""
import numpy as np
import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import BF16_OUT_ATOL, compare
from test_gpu_prefill import kv_head_rows, sample_rows

pytestmark = pytest.mark.gpu


def run_and_compare(w, rows=None, num_ctas=0):
    wd = w.to("cuda")
    bufs = B.make_buffers(wd, B.PA_MODE_PREFILL, num_ctas=num_ctas)
    B.run_prefill(wd, bufs)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    ref_o, ref_l = oracle.attention(w, rows=rows)
    return compare(w, bufs.out, bufs.lse, ref_o, ref_l, rows=rows), bufs


def fp8_workload(name, ctx, ql, G, ps, quant_type, layout=W.NHD, seed=0, mask=None,
                 num_kv_heads=2):
    return W.make_workload(name, ctx, ql, num_q_heads=G * num_kv_heads,
                           num_kv_heads=num_kv_heads, head_dim=128, page_size=ps,
                           layout=layout, kv_dtype=W.FP8_E4M3, seed=seed, block_mask=mask,
                           mode="prefill", q_dtype=W.FP8_E4M3, quant_type=quant_type)


@pytest.mark.parametrize("quant_type", [0, 1])
@pytest.mark.parametrize("layout", [W.NHD, W.HND])
@pytest.mark.parametrize("sparse", [False, True])
def test_fp8_prefill_shrunk(quant_type, layout, sparse):
    """The E4M3 prefill workload at 1/16 size (2 x 512 causal), every row."""
    run_and_compare(W.prefill_fp8(quant_type=quant_type, sparse=sparse, layout=layout,
                                  shrink=16))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("quant_type", [0, 1])
def test_fp8_gqa_ratios_and_ragged_chunks(G, quant_type):
    """Ragged chunks over cached history, decode-shaped sequences (one new
    token: they stay on the tensor-core kernel here), a sequence with no new
    token, split units (few CTAs)."""
    ctx = [300, 77, 129, 1000, 40, 513]
    ql = [300, 5, 100, 37, 1, 0]
    run_and_compare(fp8_workload(f"f8g{G}", ctx, ql, G, 32, quant_type, seed=60 + G),
                    num_ctas=17)


@pytest.mark.parametrize("ps,layout", [(16, W.HND), (64, W.HND), (128, W.NHD), (256, W.NHD),
                                       (16, W.NHD)])
def test_fp8_page_sizes_and_layouts(ps, layout):
    w = fp8_workload("f8pl", [515, 64, 300, 1], [200, 64, 1, 1], 8, ps, 1, layout=layout,
                     seed=ps + 7, num_kv_heads=1)
    run_and_compare(w, num_ctas=23)


@pytest.mark.parametrize("n", [1, 5, 300])
def test_fp8_any_cta_count(n):
    run_and_compare(W.prefill_fp8(quant_type=1, sparse=True, shrink=32), num_ctas=n)


def test_fp8_mask_with_empty_query_tiles():
    """Query tiles whose every reachable tile is masked produce O = 0, LSE = -inf."""
    L = 512
    g = torch.Generator().manual_seed(5)
    m = W.causal_block_mask(2, 4, 4, 0.3, g)
    m[1, 1, :] = 0                      # query tile 1 of sequence 1 keeps nothing
    w = fp8_workload("f8emptyq", [L, L], [L, L], 4, 64, 0, seed=15, mask=m)
    (err, _), bufs = run_and_compare(w)
    lse = bufs.lse.reshape(-1, w.num_q_heads).cpu()
    assert torch.isinf(lse[L + 128:L + 256]).all()


def test_fp8_chunk_over_history_with_mask():
    ctx, ql = [1000, 333], [300, 200]
    g = torch.Generator().manual_seed(9)
    m = (torch.rand((2, 3, 8), generator=g) < 0.5).to(torch.uint8)
    run_and_compare(fp8_workload("f8hist", ctx, ql, 4, 16, 1, seed=16, mask=m), num_ctas=7)


@pytest.mark.parametrize("window,G,ps,masked", [(1, 4, 64, False), (100, 8, 16, False),
                                                (333, 4, 64, True), (1000, 2, 128, False)])
def test_fp8_prefill_sliding_window(window, G, ps, masked):
    """Sliding window ("HiLS-Attention", 二.1 local branch) on the E4M3 path."""
    ctx = [1000, 700, 300, 2000, 57]
    ql = [300, 5, 100, 1000, 1]
    mask = None
    if masked:
        g = torch.Generator().manual_seed(window)
        mask = (torch.rand((5, -(-max(ql) // 128), -(-max(ctx) // 128)), generator=g)
                < 0.6).to(torch.uint8)
    w = fp8_workload(f"f8win{window}", ctx, ql, G, ps, window % 2, seed=window + G, mask=mask)
    w.window = window
    run_and_compare(w, num_ctas=23)


def test_fp8_scales_enter_exactly():
    """Scales by powers of two act exactly: Q's times 2 with K's times 1/2
    leaves every logit's bits unchanged, and V's times 2 doubles every output
    exactly (LSE unchanged)."""
    w = fp8_workload("f8sc", [700, 300], [700, 100], 4, 64, 1, seed=21)
    wd = w.to("cuda")
    a = B.run_prefill(wd)
    o1 = a.out.float().clone()
    wd.q_scale = wd.q_scale * 2
    wd.k_scale = wd.k_scale * 0.5
    wd.v_scale = wd.v_scale * 2
    b = B.run_prefill(wd)
    torch.cuda.synchronize()
    assert torch.equal(b.out.float(), 2 * o1)
    assert torch.equal(b.lse, a.lse)


def test_fp8_prefill_dense_full_size_kv_head_rows():
    """The E4M3 dense prefill workload (4 x 8192, quant type 1) at full size in
    the bench's launch configuration: all 8192 x 8 rows of one KV head per
    sequence."""
    w = W.prefill_fp8(quant_type=1, sparse=False)
    run_and_compare(w, rows=kv_head_rows(w, seed=3))


def test_fp8_prefill_sparse_full_size_sampled():
    w = W.prefill_fp8(quant_type=1, sparse=True)
    run_and_compare(w, rows=sample_rows(w, per_seq=1024, seed=4))


def test_fp8_prefill_dense_q0_hnd_full_size_sampled():
    w = W.prefill_fp8(quant_type=0, sparse=False, layout=W.HND)
    run_and_compare(w, rows=sample_rows(w, per_seq=1024, seed=5))


def test_fp8_masked_tiles_never_loaded():
    """E4M3 NaN bytes (0x7F) in every tile the mask drops for all query tiles
    leave the output bit-identical."""
    w = W.prefill_fp8(quant_type=1, sparse=True, shrink=16)
    a = B.run_prefill(w.to("cuda"))
    o1 = a.out.clone()
    T = w.mask_tile
    for b in range(w.num_seqs):
        for kt in range(w.block_mask.shape[2]):
            if int(w.block_mask[b, :, kt].max()) == 0:
                for j in range(kt * T, min((kt + 1) * T, int(w.context_lens[b]))):
                    pg = int(w.block_table[b, j // w.page_size])
                    w.k_cache[pg, j % w.page_size] = 0x7F
                    w.v_cache[pg, j % w.page_size] = 0x7F
    b2 = B.run_prefill(w.to("cuda"))
    torch.cuda.synchronize()
    assert torch.equal(o1, b2.out)


def test_fp8_prefill_deterministic():
    w = W.prefill_fp8(quant_type=0, sparse=False, shrink=8).to("cuda")
    a = B.run_prefill(w)
    o1, l1 = a.out.clone(), a.lse.clone()
    B.run_prefill(w, a)
    torch.cuda.synchronize()
    assert torch.equal(o1, a.out) and torch.equal(l1, a.lse)


def test_fp8_short_rows_at_bf16_accuracy():
    """Rows that see one to eight keys, where one E4M3 rounding of P (3
    mantissa bits) would move an output by up to ~3% of a V difference: with
    P as two E4M3 terms they stay within the bf16 path's tolerance."""
    w = fp8_workload("f8p2", [256, 256], [256, 256], 8, 64, 1, seed=33)
    rows = np.concatenate([np.arange(8 * 16), 256 * 16 + np.arange(8 * 16)]).astype(np.int64)
    (err_o, _), _ = run_and_compare(w, rows=rows)
    assert err_o <= BF16_OUT_ATOL
