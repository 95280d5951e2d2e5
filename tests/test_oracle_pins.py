"""Pins for the fp64 attention oracle (CPU only).

Each test ties the oracle to something other than itself: a library routine
(torch scaled_dot_product_attention / logsumexp on explicitly gathered K/V),
closed forms, causal invariants, the split-K merge identity, invariance to
layout and page placement, and the E4M3 code points of the OCP FP8
specification.  A plausible mistake in the oracle (dropped scale, wrong
causal offset, wrong page index, transposed layout, wrong GQA map, wrong LSE
base) fails at least one of them.

Pages: "基于Triton-TLE优化Tencent HPC-Ops Attention" 一.2 (paged KV through
a block table, block mask, Combine equal to full attention), 三.3 (merge of
partial softmax states); the xdnf.cn "Chunked Prefill" article (decode rows
unmasked, chunk causal on its own tokens, unmasked over history); "vLLM
Triton Attention Backend Deep Dive", "Q Blocks" (GQA grouping).
"""
import math
import os

import numpy as np
import pytest
import torch

from paged_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers

def dense_kv(w, b, hk, which):
    """float64 [ctx, D] of sequence b / KV head hk, gathered with torch indexing."""
    ctx = int(w.context_lens[b])
    npg = (ctx + w.page_size - 1) // w.page_size
    pages = w.block_table[b, :npg].long()
    cache = w.k_cache if which == "k" else w.v_cache
    if w.kv_dtype == W.BF16:
        vals = cache.double()
    else:
        vals = cache.view(torch.float8_e4m3fn).double()
    if w.layout == W.NHD:
        x = vals[pages][:, :, hk, :]          # [npg, page, D]
    else:
        x = vals[pages][:, hk, :, :]
    if w.kv_dtype == W.FP8_E4M3:
        scales = w.k_scale if which == "k" else w.v_scale
        if w.kv_scale_mode == 1:                 # one scale for the cache
            x = x * scales.reshape(-1)[0].double()
        else:                                    # one per (page, KV head)
            x = x * scales[pages, hk].double()[:, None, None]
    return x.reshape(-1, w.head_dim)[:ctx]


def dense_q(w):
    """float64 [total_q, Hq, D]: bf16 Q, or E4M3 bytes times their scale."""
    if w.q_dtype == W.BF16:
        return w.q.double()
    q = w.q.view(torch.float8_e4m3fn).double()
    if w.q_scale_mode == 1:                      # one per (token, q head)
        return q * w.q_scale.double()[:, :, None]
    return q * w.q_scale.reshape(-1)[0].double()


def visibility(w, b):
    """bool [ql, ctx]: key j visible to local query i (causal + block mask)."""
    ctx, ql = int(w.context_lens[b]), int(w.q_lens[b])
    i = torch.arange(ql)[:, None]
    j = torch.arange(ctx)[None, :]
    vis = j <= (ctx - ql + i)
    if w.window > 0:                         # sliding window: p - window < j <= p
        vis = vis & (j > (ctx - ql + i) - w.window)
    if w.block_mask is not None:
        m = w.block_mask[b].bool()
        qt = (i // w.mask_tile).expand(ql, ctx)
        kt = (j // w.mask_tile).expand(ql, ctx)
        inb = (qt < m.shape[0]) & (kt < m.shape[1])
        vis = vis & inb & m[qt.clamp(max=m.shape[0] - 1), kt.clamp(max=m.shape[1] - 1)]
    return vis


def library_reference(w):
    """(out [total*Hq, D], lse [total*Hq]) from torch SDPA + logsumexp."""
    G = w.gqa
    outs, lses = [], []
    cu = 0
    qd = dense_q(w)
    for b in range(w.num_seqs):
        ql = int(w.q_lens[b])
        q = qd[cu:cu + ql]                                 # [ql, Hq, D]
        vis = visibility(w, b)
        o_b = torch.zeros(ql, w.num_q_heads, w.head_dim, dtype=torch.float64)
        l_b = torch.zeros(ql, w.num_q_heads, dtype=torch.float64)
        for hk in range(w.num_kv_heads):
            K = dense_kv(w, b, hk, "k")
            V = dense_kv(w, b, hk, "v")
            qh = q[:, hk * G:(hk + 1) * G, :].transpose(0, 1)  # [G, ql, D]
            o = torch.nn.functional.scaled_dot_product_attention(
                qh, K[None].expand(G, -1, -1), V[None].expand(G, -1, -1),
                attn_mask=vis[None], scale=w.sm_scale)
            s = torch.matmul(qh, K.T) * w.sm_scale
            s = s.masked_fill(~vis[None], float("-inf"))
            o_b[:, hk * G:(hk + 1) * G, :] = o.transpose(0, 1)
            l_b[:, hk * G:(hk + 1) * G] = torch.logsumexp(s, dim=-1).transpose(0, 1)
        outs.append(o_b.reshape(-1, w.head_dim))
        lses.append(l_b.reshape(-1))
        cu += ql
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


def small_workloads():
    return [
        W.tiny_mixed(),
        W.decode_bf16(mtp=1, shrink=32),
        W.decode_bf16(mtp=3, shrink=32),
        W.decode_fp8(shrink=32),
        W.prefill_bf16(sparse=False, shrink=32),
        W.prefill_bf16(sparse=True, shrink=32),
        W.hybrid_bf16(shrink=32),
        W.make_workload("hnd_gqa2", [5, 64, 130], [5, 2, 3], num_q_heads=4, num_kv_heads=2,
                        head_dim=64, page_size=16, layout=W.HND, seed=7),
        W.prefill_fp8(quant_type=0, shrink=64),
        W.prefill_fp8(quant_type=1, sparse=True, layout=W.HND, shrink=64),
    ]


# ------------------------------------------------- 1. library special case

@pytest.mark.parametrize("idx", range(8))
def test_matches_torch_sdpa(oracle_mod, idx):
    w = small_workloads()[idx]
    out, lse = oracle_mod.attention(w)
    ref_o, ref_l = library_reference(w)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_row_subset_equals_full(oracle_mod):
    w = W.hybrid_bf16(shrink=32)
    out, lse = oracle_mod.attention(w)
    rng = np.random.default_rng(0)
    rows = rng.choice(out.shape[0], size=50, replace=False).astype(np.int64)
    o2, l2 = oracle_mod.attention(w, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


# ------------------------------------------------------- 2. closed forms

def _decode_ws(ctx, ql, seed=3, **kw):
    base = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16)
    base.update(kw)
    return W.make_workload("cf", ctx, ql, seed=seed, **base)


def test_single_key_gives_its_value(oracle_mod):
    w = _decode_ws([1, 1], [1, 1])
    out, lse = oracle_mod.attention(w)
    for b in range(2):
        for h in range(4):
            hk = h // 2
            v = dense_kv(w, b, hk, "v")[0].numpy()
            k = dense_kv(w, b, hk, "k")[0].numpy()
            r = b * 4 + h
            assert np.array_equal(out[r], v)
            q = w.q[b, h].double().numpy()
            assert lse[r] == pytest.approx(w.sm_scale * float(np.dot(q, k)), abs=1e-12)


def test_constant_v_gives_that_row(oracle_mod):
    w = _decode_ws([77, 200], [1, 3])
    row = torch.linspace(-2, 2, w.head_dim).to(torch.bfloat16)
    if w.layout == W.NHD:
        w.v_cache[:] = row
    out, _ = oracle_mod.attention(w)
    np.testing.assert_allclose(out, np.broadcast_to(row.double().numpy(), out.shape),
                               rtol=0, atol=1e-14)


@pytest.mark.parametrize("how", ["zero_q", "zero_scale"])
def test_uniform_weights(oracle_mod, how):
    w = _decode_ws([50, 130], [1, 4])
    if how == "zero_q":
        w.q.zero_()
    else:
        w.sm_scale = 0.0
    out, lse = oracle_mod.attention(w)
    r = 0
    for b in range(2):
        ctx, ql = int(w.context_lens[b]), int(w.q_lens[b])
        for i in range(ql):
            n_vis = ctx - ql + i + 1
            for h in range(4):
                V = dense_kv(w, b, h // 2, "v")[:n_vis].numpy()
                np.testing.assert_allclose(out[r], V.mean(axis=0), rtol=0, atol=1e-13)
                assert lse[r] == pytest.approx(math.log(n_vis), abs=1e-13)
                r += 1


def test_constant_k_gives_uniform_weights(oracle_mod):
    w = _decode_ws([40], [2])
    krow = torch.linspace(-1, 1, w.head_dim).to(torch.bfloat16)
    w.k_cache[:] = krow
    out, lse = oracle_mod.attention(w)
    r = 0
    for i in range(2):
        n_vis = 40 - 2 + i + 1
        for h in range(4):
            V = dense_kv(w, 0, h // 2, "v")[:n_vis].numpy()
            s = w.sm_scale * float(np.dot(w.q[i, h].double().numpy(), krow.double().numpy()))
            np.testing.assert_allclose(out[r], V.mean(axis=0), rtol=0, atol=1e-13)
            assert lse[r] == pytest.approx(s + math.log(n_vis), abs=1e-12)
            r += 1


# -------------------------------------------------- 3. causal invariants

def test_fresh_prefill_first_row_is_v0(oracle_mod):
    w = _decode_ws([33], [33])
    out, _ = oracle_mod.attention(w)
    for h in range(4):
        assert np.array_equal(out[h], dense_kv(w, 0, h // 2, "v")[0].numpy())


def test_future_keys_never_read(oracle_mod):
    w = _decode_ws([70], [20])
    out, lse = oracle_mod.attention(w)
    i = 5                                  # position 70-20+5 = 55
    p = 70 - 20 + i
    rows = np.arange(i * 4, i * 4 + 4, dtype=np.int64)
    npg = (70 + 15) // 16
    pages = w.block_table[0, :npg]
    for j in range(p + 1, 70):
        pg, sl = int(pages[j // 16]), j % 16
        w.k_cache[pg, sl] = float("nan")
        w.v_cache[pg, sl] = float("inf")
    o2, l2 = oracle_mod.attention(w, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


def test_dominant_logit_selects_its_value(oracle_mod):
    w = _decode_ws([90], [1], num_q_heads=2, num_kv_heads=1)
    w.sm_scale = 1.0
    w.k_cache.zero_()
    w.q.zero_()
    w.q[0, :, 0] = 8.0
    star = 41
    pg = int(w.block_table[0, star // 16])
    w.k_cache[pg, star % 16, 0, 0] = 8.0           # logit 64 vs 0 for every other key
    out, lse = oracle_mod.attention(w)
    v = dense_kv(w, 0, 0, "v")[star].numpy()
    for h in range(2):
        np.testing.assert_allclose(out[h], v, rtol=0, atol=100 * math.exp(-60))
        assert lse[h] == pytest.approx(64.0, abs=1e-20 + 100 * math.exp(-60))


# ------------------------------------------------- 4. split-K = unsplit

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_splitk_merge_equals_unsplit(oracle_mod, seed):
    w = W.decode_bf16(mtp=2, shrink=32)
    full_o, full_l = oracle_mod.attention(w)
    rng = np.random.default_rng(seed)
    max_ctx = int(w.context_lens.max())
    n_parts = int(rng.integers(1, 6))
    cuts = sorted(set(int(x) for x in rng.integers(1, max_ctx, size=n_parts - 1)))
    edges = [0] + cuts + [max_ctx + 1]
    parts = [oracle_mod.attention(w, key_lo=a, key_hi=b) for a, b in zip(edges[:-1], edges[1:])]
    for r in range(full_o.shape[0]):
        o, l = oracle_mod.combine(np.stack([p[0][r] for p in parts]),
                                  np.array([p[1][r] for p in parts]))
        np.testing.assert_allclose(o, full_o[r], rtol=0, atol=1e-12)
        assert l == pytest.approx(full_l[r], abs=1e-12)


def test_combine_closed_forms(oracle_mod):
    a = np.arange(8, dtype=np.float64)
    b = -np.arange(8, dtype=np.float64)
    o, l = oracle_mod.combine(a[None], np.array([0.7]))
    assert np.array_equal(o, a) and l == 0.7
    o, l = oracle_mod.combine(np.stack([a, b]), np.array([1.5, 1.5]))
    np.testing.assert_allclose(o, (a + b) / 2, atol=1e-15)
    assert l == pytest.approx(1.5 + math.log(2), abs=1e-15)
    o, l = oracle_mod.combine(np.stack([a, b]), np.array([-np.inf, 2.0]))
    assert np.array_equal(o, b) and l == 2.0
    o, l = oracle_mod.combine(np.stack([a, b]), np.array([-np.inf, -np.inf]))
    assert np.array_equal(o, np.zeros(8)) and l == -np.inf


# ----------------------------------------- 5. masked tiles contribute nothing

def test_masked_tiles_are_never_read(oracle_mod):
    w = W.prefill_bf16(sparse=True, shrink=32)
    out, lse = oracle_mod.attention(w)
    m = w.block_mask
    T = w.mask_tile
    # a key tile dropped by every q tile of the sequence is never read by anyone
    for b in range(w.num_seqs):
        for kt in range(m.shape[2]):
            if int(m[b, :, kt].max()) == 0:
                for j in range(kt * T, min((kt + 1) * T, int(w.context_lens[b]))):
                    pg = int(w.block_table[b, j // w.page_size])
                    w.k_cache[pg, j % w.page_size] = float("nan")
                    w.v_cache[pg, j % w.page_size] = float("nan")
    o2, l2 = oracle_mod.attention(w)
    assert np.array_equal(o2, out) and np.array_equal(l2, lse)
    # and dropping a tile really changes rows that could see it
    w2 = W.prefill_bf16(sparse=False, shrink=32)
    o3, _ = oracle_mod.attention(w2)
    assert not np.allclose(o3, out)


def test_empty_rows_zero_and_minus_inf(oracle_mod):
    w = W.prefill_bf16(sparse=True, shrink=32)
    w.block_mask.zero_()
    out, lse = oracle_mod.attention(w)
    assert np.array_equal(out, np.zeros_like(out)) and np.all(lse == -np.inf)


# ------------------------------------------ 6. layout / paging invariance

def test_nhd_hnd_and_page_permutation_invariance(oracle_mod):
    w = W.make_workload("lay", [70, 33, 129], [3, 1, 2], num_q_heads=8, num_kv_heads=2,
                        head_dim=64, page_size=16, layout=W.NHD, seed=11)
    out, lse = oracle_mod.attention(w)
    # same logical cache in HND
    w_h = W.make_workload("lay", [70, 33, 129], [3, 1, 2], num_q_heads=8, num_kv_heads=2,
                          head_dim=64, page_size=16, layout=W.NHD, seed=11)
    w_h.k_cache = w.k_cache.transpose(1, 2).contiguous()
    w_h.v_cache = w.v_cache.transpose(1, 2).contiguous()
    w_h.layout = W.HND
    o2, l2 = oracle_mod.attention(w_h)
    assert np.array_equal(o2, out) and np.array_equal(l2, lse)
    # move every page to a new physical index
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_pages)
    w_p = W.make_workload("lay", [70, 33, 129], [3, 1, 2], num_q_heads=8, num_kv_heads=2,
                          head_dim=64, page_size=16, layout=W.NHD, seed=11)
    w_p.k_cache = w.k_cache[inv]
    w_p.v_cache = w.v_cache[inv]
    bt = w.block_table.clone()
    bt[bt >= 0] = perm[bt[bt >= 0].long()].to(torch.int32)
    w_p.block_table = bt
    o3, l3 = oracle_mod.attention(w_p)
    assert np.array_equal(o3, out) and np.array_equal(l3, lse)


def test_gqa_head_mapping(oracle_mod):
    """q head h must read KV head h // G: make KV heads distinguishable."""
    w = W.make_workload("gqa", [20], [1], num_q_heads=6, num_kv_heads=3, head_dim=64,
                        page_size=16, seed=4)
    for hk in range(3):
        w.v_cache[:, :, hk, :] = float(hk + 1)
    out, _ = oracle_mod.attention(w)
    for h in range(6):
        np.testing.assert_allclose(out[h], float(h // 2 + 1), rtol=1e-14, atol=0)


def test_bad_page_is_reported(oracle_mod):
    w = _decode_ws([40], [1])
    w.block_table[0, 1] = w.num_pages + 3
    with pytest.raises(ValueError):
        oracle_mod.attention(w)


# -------------------------------------------------------- 7. FP8 decoding

def test_e4m3_all_256_codes_match_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = oracle_mod.e4m3_to_double(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), hex(c)


def test_e4m3_spec_points(oracle_mod):
    with open(os.path.join(GOLDEN, "e4m3fn_spec_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, val = line.split()
            got = oracle_mod.e4m3_to_double(int(code, 16))
            if val == "nan":
                assert math.isnan(got)
            else:
                assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_bf16_decoding_matches_torch(oracle_mod):
    g = torch.Generator().manual_seed(9)
    bits = torch.randint(0, 65536, (4096,), generator=g, dtype=torch.int32)
    ref = bits.to(torch.int16).view(torch.bfloat16).double().numpy()
    for b, r in zip(bits.tolist(), ref):
        got = oracle_mod.bf16_to_double(b)
        assert (math.isnan(got) and math.isnan(r)) or got == r


def test_fp8_scale_is_applied_per_page_and_head(oracle_mod):
    """Doubling one (page, head) scale doubles exactly that head's V contribution."""
    w = W.make_workload("fp8s", [16], [1], num_q_heads=2, num_kv_heads=2, head_dim=64,
                        page_size=16, kv_dtype=W.FP8_E4M3, layout=W.HND, seed=8)
    out, _ = oracle_mod.attention(w)
    pg = int(w.block_table[0, 0])
    w.v_scale[pg, 1] *= 2.0
    o2, _ = oracle_mod.attention(w)
    assert np.array_equal(o2[0], out[0])
    np.testing.assert_allclose(o2[1], 2 * out[1], rtol=1e-15, atol=0)


# ------------------------------------------------ generator properties

def test_block_mask_skip_ratio_matches_pages():
    """The block-sparse prefill workload skips ~74% of the off-diagonal causal
    tiles (the pages report 73.3%-74.6% tile skip for their sparse prefill)."""
    w = W.prefill_bf16(sparse=True)
    m = w.block_mask
    t = m.shape[1]
    off = torch.tril(torch.ones(t, t, dtype=torch.bool), diagonal=-1)
    kept = m.bool()[:, off].float().mean().item()
    assert 0.70 < 1.0 - kept < 0.78
    assert bool(m[:, torch.eye(t, dtype=torch.bool)].all())
    assert not bool(m[:, torch.triu(torch.ones(t, t, dtype=torch.bool), 1)].any())


# ------------------------------------------------ sliding window (local branch)
# "HiLS-Attention" page, 二.1 (the local sliding-window branch): query p sees
# the keys p - window < j <= p.  The bounds are our reading (the page gives
# none).

def _windowed(w, window):
    w.window = window
    return w


@pytest.mark.parametrize("which,window", [("decode", 100), ("prefill", 300), ("hybrid", 64),
                                          ("tiny", 7)])
def test_window_matches_torch_sdpa(oracle_mod, which, window):
    w = {"decode": lambda: W.decode_bf16(mtp=3, shrink=32),
         "prefill": lambda: W.prefill_bf16(sparse=False, shrink=32),
         "hybrid": lambda: W.hybrid_bf16(shrink=32),
         "tiny": W.tiny_mixed}[which]()
    _windowed(w, window)
    out, lse = oracle_mod.attention(w)
    ref_o, ref_l = library_reference(w)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_window_as_long_as_the_context_changes_nothing(oracle_mod):
    w = W.hybrid_bf16(shrink=32)
    out, lse = oracle_mod.attention(w)
    _windowed(w, int(w.context_lens.max()))
    o2, l2 = oracle_mod.attention(w)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_window_of_one_selects_the_own_key(oracle_mod):
    """Only key p is visible: O = v_p and LSE = sm_scale * q . k_p."""
    w = _windowed(_decode_ws([40, 9], [3, 9]), 1)
    out, lse = oracle_mod.attention(w)
    G = w.num_q_heads // w.num_kv_heads
    cu = 0
    for b in range(2):
        ctx, ql = int(w.context_lens[b]), int(w.q_lens[b])
        for hk in range(w.num_kv_heads):
            K, V = dense_kv(w, b, hk, "k"), dense_kv(w, b, hk, "v")
            for i in range(ql):
                p = ctx - ql + i
                for g in range(G):
                    h = hk * G + g
                    r = (cu + i) * w.num_q_heads + h
                    q = w.q[cu + i, h].double()
                    np.testing.assert_allclose(out[r], V[p].numpy(), rtol=0, atol=1e-12)
                    assert abs(lse[r] - float(w.sm_scale * (q @ K[p]))) <= 1e-12
        cu += ql


def test_keys_before_the_window_are_never_read(oracle_mod):
    """NaN in every key at or before p - window leaves a decode row unchanged."""
    w = _windowed(_decode_ws([70], [1]), 10)
    out, lse = oracle_mod.attention(w)
    p = 69
    pages = w.block_table[0, :(70 + 15) // 16]
    for j in range(0, p - 10 + 1):
        pg, sl = int(pages[j // 16]), j % 16
        w.k_cache[pg, sl] = float("nan")
        w.v_cache[pg, sl] = float("inf")
    o2, l2 = oracle_mod.attention(w)
    assert np.isfinite(o2).all()
    assert np.array_equal(o2, out) and np.array_equal(l2, lse)


# ------------------------------------------------- FP8 prefill quantisation
# "基于Triton-TLE优化Tencent HPC-Ops Attention", 二 (FP8 prefill over two
# quantisation types) and 三 (Q per-token per-head, K/V per-tensor).  Our
# reading of the other type: Q, K and V each with one scale.

def test_fp8_q_scale_is_a_per_row_logit_scale(oracle_mod):
    """Doubling the scale of one (token, q head) of an E4M3 Q doubles that
    row's logits, which is exactly doubling sm_scale for that row; every
    other row is bit-identical."""
    w = W.prefill_fp8(quant_type=1, shrink=64)
    row_tok, row_h = 37, 5
    rows = np.array([row_tok * w.num_q_heads + row_h, 3 * w.num_q_heads + 1], np.int64)
    base_o, base_l = oracle_mod.attention(w, rows=rows)
    w2 = W.prefill_fp8(quant_type=1, shrink=64)
    w2.q_scale = w2.q_scale.clone()
    w2.q_scale[row_tok, row_h] *= 2.0
    o2, l2 = oracle_mod.attention(w2, rows=rows)
    w3 = W.prefill_fp8(quant_type=1, shrink=64)
    w3.sm_scale = 2.0 * w3.sm_scale
    o3, l3 = oracle_mod.attention(w3, rows=rows[:1])
    assert np.array_equal(o2[0], o3[0]) and l2[0] == l3[0]
    assert np.array_equal(o2[1], base_o[1]) and l2[1] == base_l[1]
    assert not np.array_equal(o2[0], base_o[0])


def test_fp8_per_tensor_v_scale_scales_the_output(oracle_mod):
    """One V scale for the cache: doubling it doubles every output exactly
    and leaves every LSE unchanged."""
    w = W.prefill_fp8(quant_type=0, shrink=64)
    o1, l1 = oracle_mod.attention(w)
    w.v_scale = w.v_scale * 2.0
    o2, l2 = oracle_mod.attention(w)
    assert np.array_equal(o2, 2.0 * o1) and np.array_equal(l1, l2)


def test_fp8_quantised_inputs_are_e4m3_codes_times_scales():
    """The generator's Q bytes decode (torch float8_e4m3fn) to values whose
    largest magnitude per scale group is about 448 * scale."""
    w = W.prefill_fp8(quant_type=1, shrink=64)
    q = w.q.view(torch.float8_e4m3fn).float()
    amax = q.abs().amax(dim=2)
    assert torch.all((amax <= 448.0) & (amax >= 240.0))
    assert w.q_scale.shape == (w.total_q, w.num_q_heads)
    w0 = W.prefill_fp8(quant_type=0, shrink=64)
    assert w0.q_scale.numel() == 1 and w0.k_scale.numel() == 1 and w0.v_scale.numel() == 1
