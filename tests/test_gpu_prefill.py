"""GPU prefill / mixed batch (Assign + tcgen05 prefill + Combine; the
decode-shaped sequences of an unmasked batch run on the decode kernel) against
the fp64 oracle.

"基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 Prefill (causal,
block-sparse over paged KV) and 二.1 (only kept tiles are computed); the
xdnf.cn "Chunked Prefill" article (a chunk causal over its own tokens and
unmasked over cached history, batched with decode rows).
Tolerances: bf16 outputs max-abs 2e-2, LSE 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import compare

pytestmark = pytest.mark.gpu


def run_and_compare(w, rows=None, num_ctas=0, balance_rows=0):
    wd = w.to("cuda")
    bufs = B.make_buffers(wd, B.PA_MODE_PREFILL, num_ctas=num_ctas, balance_rows=balance_rows)
    B.run_prefill(wd, bufs)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    ref_o, ref_l = oracle.attention(w, rows=rows)
    return compare(w, bufs.out, bufs.lse, ref_o, ref_l, rows=rows), bufs


def sample_rows(w, per_seq=256, seed=0):
    """Rows (token*Hq + head) spread over every sequence, always including the
    first and last new token of each."""
    rng = np.random.default_rng(seed)
    ql = [int(x) for x in w.q_lens]
    cu = np.concatenate([[0], np.cumsum(ql)])
    rows = []
    for b in range(w.num_seqs):
        if ql[b] == 0:
            continue
        toks = np.unique(np.concatenate([[cu[b], cu[b + 1] - 1],
                                         rng.integers(cu[b], cu[b + 1], size=per_seq)]))
        heads = rng.integers(0, w.num_q_heads, size=toks.shape[0])
        rows.append(toks * w.num_q_heads + heads)
    return np.sort(np.concatenate(rows)).astype(np.int64)


def test_tiny_mixed():
    run_and_compare(W.tiny_mixed())


def test_tiny_mixed_split_everywhere():
    run_and_compare(W.tiny_mixed(), num_ctas=40)


@pytest.mark.parametrize("sparse", [False, True])
def test_prefill_shrunk(sparse):
    run_and_compare(W.prefill_bf16(sparse=sparse, shrink=16))


@pytest.mark.parametrize("sparse", [False, True])
def test_prefill_quarter_size(sparse):
    w = W.prefill_bf16(sparse=sparse, shrink=4)
    run_and_compare(w, rows=sample_rows(w, per_seq=512))


def test_hybrid_shrunk():
    run_and_compare(W.hybrid_bf16(shrink=16))


@pytest.mark.parametrize("n", [1, 5, 300])
def test_prefill_any_cta_count(n):
    run_and_compare(W.prefill_bf16(sparse=True, shrink=32), num_ctas=n)


@pytest.mark.parametrize("G", [1, 2, 4, 16])
def test_gqa_ratios_and_ragged_chunks(G):
    ctx = [300, 77, 129, 1000]
    ql = [300, 5, 100, 37]
    w = W.make_workload(f"g{G}", ctx, ql, num_q_heads=2 * G, num_kv_heads=2, head_dim=128,
                        page_size=32, seed=40 + G, mode="prefill")
    run_and_compare(w, num_ctas=17)


@pytest.mark.parametrize("ps,layout", [(16, W.HND), (64, W.HND), (128, W.NHD), (256, W.NHD)])
def test_page_sizes_and_layouts(ps, layout):
    w = W.make_workload("pl", [515, 64, 300], [200, 64, 1], num_q_heads=8, num_kv_heads=1,
                        head_dim=128, page_size=ps, layout=layout, seed=ps + 3, mode="prefill")
    run_and_compare(w, num_ctas=23)


def test_head_dim_64():
    w = W.make_workload("d64", [700, 50], [650, 50], num_q_heads=8, num_kv_heads=2,
                        head_dim=64, page_size=64, seed=77, mode="prefill")
    run_and_compare(w, num_ctas=29)


def test_mask_with_empty_query_tiles():
    """Query tiles whose every reachable tile is masked produce O = 0, LSE = -inf."""
    L = 512
    g = torch.Generator().manual_seed(5)
    m = W.causal_block_mask(2, 4, 4, 0.3, g)
    m[0, 2, :] = 0                      # query tile 2 of sequence 0 keeps nothing
    w = W.make_workload("emptyq", [L, L], [L, L], num_q_heads=8, num_kv_heads=2, head_dim=128,
                        page_size=64, seed=13, block_mask=m, mode="prefill")
    (err, _), bufs = run_and_compare(w)
    lse = bufs.lse.cpu()
    assert torch.isinf(lse[256:384]).all()


def test_chunk_over_history_with_mask():
    """A chunk over cached history with a block mask (mask rows = local query
    tiles, columns = absolute key tiles)."""
    ctx, ql = [1000], [300]
    g = torch.Generator().manual_seed(8)
    m = (torch.rand((1, 3, 8), generator=g) < 0.5).to(torch.uint8)
    w = W.make_workload("hist", ctx, ql, num_q_heads=4, num_kv_heads=1, head_dim=128,
                        page_size=16, seed=14, block_mask=m, mode="prefill")
    run_and_compare(w, num_ctas=7)


def kv_head_rows(w, seed=0):
    """Every row of one (sequence, KV head) per sequence: all new tokens x the
    G q heads of a KV head picked per sequence (so every 256-row unit and
    both 128-row tensor-core halves of that head are checked end to end)."""
    rng = np.random.default_rng(seed)
    G = w.num_q_heads // w.num_kv_heads
    ql = [int(x) for x in w.q_lens]
    cu = np.concatenate([[0], np.cumsum(ql)])
    rows = []
    for b in range(w.num_seqs):
        hk = int(rng.integers(0, w.num_kv_heads))
        toks = np.arange(cu[b], cu[b + 1], dtype=np.int64)
        heads = hk * G + np.arange(G, dtype=np.int64)
        rows.append((toks[:, None] * w.num_q_heads + heads[None, :]).reshape(-1))
    return np.sort(np.concatenate(rows))


def all_head_rows(w, per_seq=64, seed=0):
    """Sampled tokens of every sequence (first and last included) with all
    their q heads."""
    rng = np.random.default_rng(seed)
    ql = [int(x) for x in w.q_lens]
    cu = np.concatenate([[0], np.cumsum(ql)])
    rows = []
    for b in range(w.num_seqs):
        if ql[b] == 0:
            continue
        toks = np.unique(np.concatenate([[cu[b], cu[b + 1] - 1],
                                         rng.integers(cu[b], cu[b + 1], size=per_seq)]))
        rows.append((toks[:, None] * w.num_q_heads
                     + np.arange(w.num_q_heads)[None, :]).reshape(-1))
    return np.sort(np.concatenate(rows)).astype(np.int64)


def test_prefill_dense_full_size_kv_head_rows():
    """The dense prefill workload at full size, in the launch configuration
    the bench times: all 8192 x 8 rows of one KV head per sequence."""
    w = W.prefill_bf16(sparse=False)
    run_and_compare(w, rows=kv_head_rows(w, seed=0))


def test_prefill_sparse_full_size_kv_head_rows():
    w = W.prefill_bf16(sparse=True)
    run_and_compare(w, rows=kv_head_rows(w, seed=1))


def test_hybrid_full_size_sampled():
    """Full-size hybrid batch: every head of every decode sequence's token,
    and sampled chunk tokens with all their heads."""
    w = W.hybrid_bf16()
    run_and_compare(w, rows=all_head_rows(w, per_seq=64, seed=2))


def test_masked_tiles_never_loaded():
    """NaN in every tile the mask drops for all query tiles leaves the output
    bit-identical: such tiles are never loaded."""
    w = W.prefill_bf16(sparse=True, shrink=16)
    wd = w.to("cuda")
    a = B.run_prefill(wd)
    o1 = a.out.clone()
    T = w.mask_tile
    for b in range(w.num_seqs):
        for kt in range(w.block_mask.shape[2]):
            if int(w.block_mask[b, :, kt].max()) == 0:
                for j in range(kt * T, min((kt + 1) * T, int(w.context_lens[b]))):
                    pg = int(w.block_table[b, j // w.page_size])
                    w.k_cache[pg, j % w.page_size] = float("nan")
                    w.v_cache[pg, j % w.page_size] = float("nan")
    wd2 = w.to("cuda")
    b2 = B.run_prefill(wd2)
    torch.cuda.synchronize()
    assert torch.equal(o1, b2.out)


@pytest.mark.parametrize("num_ctas", [0, 300])
def test_prefill_outputs_only_16_byte_aligned(num_ctas):
    """The epilogue stores 32 bytes at a time where out and the partials are
    32-byte aligned, 16 bytes otherwise: both give the same bits (300 CTAs
    split every unit, so the partials' stores are covered too)."""
    w = W.hybrid_bf16(shrink=16).to("cuda")
    a = B.make_buffers(w, B.PA_MODE_PREFILL, num_ctas=num_ctas)
    B.run_prefill(w, a)
    b = B.make_buffers(w, B.PA_MODE_PREFILL, num_ctas=num_ctas)
    big_o = torch.empty(b.out.numel() + 8, dtype=torch.bfloat16, device="cuda")
    b.out = big_o[8:].view(b.out.shape)                  # 16 bytes past a 32-byte boundary
    big_p = torch.empty(b.partial_ws.numel() + 48, dtype=torch.uint8, device="cuda")
    b.partial_ws = big_p[16:16 + b.partial_ws.numel()]
    assert b.out.data_ptr() % 32 == 16 and b.partial_ws.data_ptr() % 32 == 16
    B.run_prefill(w, b)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(a.assign_ws) == 0 and B.pa_last_device_error(b.assign_ws) == 0
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)


def test_prefill_deterministic():
    w = W.hybrid_bf16(shrink=8).to("cuda")
    a = B.run_prefill(w)
    o1, l1 = a.out.clone(), a.lse.clone()
    B.run_prefill(w, a)
    torch.cuda.synchronize()
    assert torch.equal(o1, a.out) and torch.equal(l1, a.lse)


@pytest.mark.parametrize("window,G,ps,masked", [(1, 4, 64, False), (100, 8, 16, False),
                                                (128, 1, 32, False), (333, 4, 64, True),
                                                (1000, 2, 128, False), (4096, 8, 64, True)])
def test_prefill_sliding_window(window, G, ps, masked):
    """Sliding window on the tensor-core prefill path ("HiLS-Attention", 二.1
    local branch: query p sees the keys p - window < j <= p): windows shorter
    than a row of a tile, a tile long and across many tiles, chunks over
    history, decode-shaped sequences (their own kernel), block masks, split
    units."""
    ctx = [1000, 700, 300, 2000, 57]
    ql = [300, 5, 100, 1000, 1]
    mask = None
    if masked:
        g = torch.Generator().manual_seed(window)
        mask = (torch.rand((5, -(-max(ql) // 128), -(-max(ctx) // 128)), generator=g)
                < 0.6).to(torch.uint8)
    w = W.make_workload(f"pwin{window}", ctx, ql, num_q_heads=2 * G, num_kv_heads=2,
                        head_dim=128, page_size=ps, seed=window + G, block_mask=mask,
                        mode="prefill")
    w.window = window
    run_and_compare(w, num_ctas=23)


def test_prefill_window_quarter_size_sampled():
    """The dense prefill workload at quarter size with a 1000-key window."""
    w = W.prefill_bf16(sparse=False, shrink=4)
    w.window = 1000
    run_and_compare(w, rows=sample_rows(w, per_seq=512, seed=5))
