"""Seeded synthetic inputs for paged-KV attention (shared by tests, bench, smoke).

This module only draws random numbers and lays them out; it contains none of
the attention, Assign or Combine arithmetic.  Both the CUDA path and the CPU
oracle consume the tensors it returns.

Workload shapes follow the five configurations the pages' workloads are
described by (HPC-Ops dynamic decode with MTP, FP8 decode with per-page-head
scales, block-sparse causal prefill, the chunked-prefill hybrid batch):

  tiny_mixed      bf16, Hq=4, Hkv=1, D=64, page 16, sm_scale 1/8: decode
                  sequences (ctx 37, ql 1), (ctx 100, ql 1) and one chunk of
                  32 new tokens over 48 cached (ctx 80, ql 32)
  decode_bf16     B=64, Hq=32, Hkv=8, D=128, page 64, NHD; ctx log-uniform in
                  [128, 32768]; q_len = 1 + MTP
  decode_fp8      B=128, Hq=64, Hkv=8, D=128, page 64, HND; E4M3 K/V with an
                  fp32 scale per (page, KV head); ctx uniform in [1024, 16384];
                  q_len 3 (MTP 2)
  prefill_bf16    B=4, ql=ctx=8192, Hq=64, Hkv=8, D=128, page 64, NHD; dense
                  causal, or block-sparse with a 128x128 tile mask keeping the
                  diagonal and each other causal tile with probability 0.26
  hybrid_bf16     one 1024-token chunk over 31744 cached tokens plus 255
                  decode sequences (ql 1, ctx uniform in [512, 8192]),
                  Hq=32, Hkv=8, D=128, page 16, NHD

Every call takes an explicit seed; the same seed gives the same bytes on any
machine.  Physical pages are a seeded random permutation of a pool that also
holds ~5% decoy pages.  Decoy pages and the slots past the end of each
sequence's last page are filled with NaN: a kernel that reads them, or lets
them leak into an output, is caught by the parity tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

NHD = 0
HND = 1
BF16 = 0
FP8_E4M3 = 1

BF16_NAN_BITS = 0x7FC0
E4M3_NAN_BYTE = 0x7F
E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    layout: int
    kv_dtype: int
    sm_scale: float
    q: torch.Tensor                       # bf16 [total_q, Hq, D]
    k_cache: torch.Tensor                 # bf16 / uint8, NHD or HND
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]       # fp32 [num_pages, Hkv] (FP8 only)
    v_scale: Optional[torch.Tensor]
    block_table: torch.Tensor             # int32 [B, max_pages_per_seq], -1 = unused
    context_lens: torch.Tensor            # int32 [B]
    q_lens: torch.Tensor                  # int32 [B]
    block_mask: Optional[torch.Tensor] = None   # uint8 [B, mask_q_tiles, mask_kv_tiles]
    mask_tile: int = 128
    mode: str = "decode"                  # which Assign mode the workload is run with
    window: int = 0                       # sliding window (0 = none): keys p - window < j <= p
    q_dtype: int = BF16                   # BF16, or FP8_E4M3 bytes times q_scale
    q_scale: Optional[torch.Tensor] = None    # fp32 [1] or [total_q, Hq] (E4M3 Q only)
    q_scale_mode: int = 0                 # 0: one Q scale; 1: one per (token, q head)
    kv_scale_mode: int = 0                # E4M3 K/V: 0 per (page, KV head); 1 one per cache
    meta: dict = field(default_factory=dict)

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def to(self, device) -> "Workload":
        """Copy of the workload with every tensor moved to ``device``."""
        kw = {k: getattr(self, k) for k in self.__dataclass_fields__}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        kw["meta"] = dict(self.meta)
        return Workload(**kw)


_RANDN_CHUNK = 1 << 24


def _randn_bf16(shape, g: torch.Generator, chunk: int = _RANDN_CHUNK) -> torch.Tensor:
    """N(0,1) rounded to bf16.  One 63-bit base seed is drawn from ``g``; chunk
    c of the flat tensor comes from its own generator seeded with
    base + c, so the chunks can be drawn on several host threads and the bytes
    depend only on (g's state, shape), not on the thread count."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16)
    base = int(torch.randint(0, 1 << 62, (1,), generator=g, dtype=torch.int64))
    starts = list(range(0, n, chunk))

    def fill(ci):
        s = starts[ci]
        e = min(n, s + chunk)
        gc = torch.Generator().manual_seed(base + ci)
        out[s:e] = torch.randn(e - s, generator=gc, dtype=torch.float32).to(torch.bfloat16)

    if len(starts) <= 1:
        for ci in range(len(starts)):
            fill(ci)
    else:
        import concurrent.futures as cf
        import os
        workers = max(1, min(len(starts), os.cpu_count() or 1, 32))
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(fill, range(len(starts))))
    return out.view(*shape)


def make_workload(name: str, context_lens: List[int], q_lens: List[int], *, num_q_heads: int,
                  num_kv_heads: int, head_dim: int, page_size: int, layout: int = NHD,
                  kv_dtype: int = BF16, sm_scale: Optional[float] = None, seed: int = 0,
                  block_mask: Optional[torch.Tensor] = None, mode: str = "decode",
                  max_pages_per_seq: Optional[int] = None, decoy_frac: float = 0.05,
                  nan_fill: bool = True, meta: Optional[dict] = None,
                  q_dtype: int = BF16, quant_type: int = 0) -> Workload:
    """Lay out a seeded paged KV cache for the given per-sequence lengths.

    q_dtype FP8_E4M3 (with E4M3 K/V): the FP8 prefill quantisation types --
    quant_type 0: Q, K and V each with one scale; quant_type 1: Q with one
    scale per (token, q head), K and V with one scale each.  Otherwise E4M3
    K/V carry one scale per (page, KV head)."""
    B = len(context_lens)
    assert len(q_lens) == B
    for c, q in zip(context_lens, q_lens):
        assert 0 <= q <= c, "q_len must not exceed context_len"
    assert num_q_heads % num_kv_heads == 0
    g = torch.Generator().manual_seed(int(seed))
    Hkv, D = num_kv_heads, head_dim
    pages_per_seq = [(c + page_size - 1) // page_size for c in context_lens]
    used = sum(pages_per_seq)
    n_decoy = max(1, int(math.ceil(decoy_frac * used)))
    num_pages = used + n_decoy
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    mpps = max_pages_per_seq or max(1, max(pages_per_seq) if B else 1)
    block_table = torch.full((B, mpps), -1, dtype=torch.int32)
    cur = 0
    for b, n in enumerate(pages_per_seq):
        assert n <= mpps
        block_table[b, :n] = perm[cur:cur + n]
        cur += n
    decoys = perm[cur:]

    total_q = sum(q_lens)
    q = _randn_bf16((total_q, num_q_heads, D), g)
    q_scale = None
    q_scale_mode = 0
    if q_dtype == FP8_E4M3:
        assert kv_dtype == FP8_E4M3, "E4M3 Q goes with E4M3 K/V"
        qf = q.float()
        if quant_type == 1:
            amax = qf.abs().amax(dim=2)                     # [total_q, Hq]
            q_scale_mode = 1
        else:
            amax = qf.abs().amax().reshape(1)
        sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).float()
        y = qf / (sc[:, :, None] if quant_type == 1 else sc)
        q = y.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
        q_scale = sc.contiguous()
    kv_scale_mode = 1 if q_dtype == FP8_E4M3 else 0
    if layout == NHD:
        shape = (num_pages, page_size, Hkv, D)
    else:
        shape = (num_pages, Hkv, page_size, D)

    k_scale = v_scale = None
    if kv_dtype == BF16:
        k_cache = _randn_bf16(shape, g)
        v_cache = _randn_bf16(shape, g)
    else:
        def quant_block(x: torch.Tensor):
            # per (page, kv head) scale: amax / 448, then round-to-nearest E4M3
            xf = x.float()
            if layout == NHD:
                amax = xf.abs().amax(dim=(1, 3))            # [pages, Hkv]
                sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
                y = xf / sc[:, None, :, None]
            else:
                amax = xf.abs().amax(dim=(2, 3))
                sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
                y = xf / sc[:, :, None, None]
            y = y.clamp(-E4M3_MAX, E4M3_MAX)
            return y.to(torch.float8_e4m3fn).view(torch.uint8), sc.float()

        def quant_tensor(x: torch.Tensor):
            # one scale for the whole cache: amax / 448, then round-to-nearest E4M3
            amax = torch.zeros((), dtype=torch.float32)
            for p0 in range(0, x.shape[0], 1024):
                amax = torch.maximum(amax, x[p0:p0 + 1024].float().abs().amax())
            sc = (amax / E4M3_MAX if float(amax) > 0 else torch.ones(())).reshape(1).float()
            q8 = torch.empty(x.shape, dtype=torch.uint8)
            for p0 in range(0, x.shape[0], 1024):
                y = (x[p0:p0 + 1024].float() / sc).clamp(-E4M3_MAX, E4M3_MAX)
                q8[p0:p0 + 1024] = y.to(torch.float8_e4m3fn).view(torch.uint8)
            return q8, sc.contiguous()

        def quant(x: torch.Tensor):
            if kv_scale_mode == 1:
                return quant_tensor(x)
            # pages are independent: quantise blocks of pages on host threads
            import concurrent.futures as cf
            import os
            q8 = torch.empty(x.shape, dtype=torch.uint8)
            sc = torch.empty((x.shape[0], Hkv), dtype=torch.float32)
            step = 256

            def one(p0):
                a, s_ = quant_block(x[p0:p0 + step])
                q8[p0:p0 + step] = a
                sc[p0:p0 + step] = s_

            starts = list(range(0, x.shape[0], step))
            with cf.ThreadPoolExecutor(max_workers=max(1, min(len(starts), os.cpu_count() or 1,
                                                               32))) as ex:
                list(ex.map(one, starts))
            return q8, sc.contiguous()

        k_cache, k_scale = quant(_randn_bf16(shape, g))
        v_cache, v_scale = quant(_randn_bf16(shape, g))

    if nan_fill:
        for cache in (k_cache, v_cache):
            if kv_dtype == BF16:
                raw, fill = cache.view(torch.int16), BF16_NAN_BITS
            else:
                raw, fill = cache, E4M3_NAN_BYTE
            if len(decoys):
                raw[decoys.long()] = fill
            for b, c in enumerate(context_lens):
                tail = c % page_size
                if tail == 0:
                    continue
                last = int(block_table[b, pages_per_seq[b] - 1])
                if layout == NHD:
                    raw[last, tail:] = fill
                else:
                    raw[last, :, tail:] = fill

    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    return Workload(
        name=name, num_seqs=B, num_q_heads=num_q_heads, num_kv_heads=Hkv, head_dim=D,
        page_size=page_size, num_pages=num_pages, layout=layout, kv_dtype=kv_dtype,
        sm_scale=float(sm_scale), q=q, k_cache=k_cache, v_cache=v_cache, k_scale=k_scale,
        v_scale=v_scale, block_table=block_table,
        context_lens=torch.tensor(context_lens, dtype=torch.int32),
        q_lens=torch.tensor(q_lens, dtype=torch.int32), block_mask=block_mask, mode=mode,
        q_dtype=q_dtype, q_scale=q_scale, q_scale_mode=q_scale_mode,
        kv_scale_mode=kv_scale_mode, meta=dict(meta or {}))


def _log_uniform_ints(n: int, lo: int, hi: int, g: torch.Generator) -> List[int]:
    u = torch.rand(n, generator=g, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [int(min(hi, max(lo, round(float(v))))) for v in x]


def _uniform_ints(n: int, lo: int, hi: int, g: torch.Generator) -> List[int]:
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=g)]


def causal_block_mask(num_seqs: int, q_tiles: int, kv_tiles: int, keep_prob: float,
                      g: torch.Generator, q_tile_offsets: Optional[List[int]] = None):
    """uint8 [B, q_tiles, kv_tiles]: the diagonal kept, each earlier tile kept
    with probability keep_prob, later tiles dropped.  q_tile_offsets[b] is the
    key-tile index of query tile 0 (for a chunk over cached history)."""
    m = torch.zeros((num_seqs, q_tiles, kv_tiles), dtype=torch.uint8)
    r = torch.rand((num_seqs, q_tiles, kv_tiles), generator=g, dtype=torch.float64)
    for b in range(num_seqs):
        off = 0 if q_tile_offsets is None else q_tile_offsets[b]
        for qt in range(q_tiles):
            diag = qt + off
            for kt in range(min(kv_tiles, diag + 1)):
                m[b, qt, kt] = 1 if (kt == diag or float(r[b, qt, kt]) < keep_prob) else 0
    return m


# --------------------------------------------------------------- the configs

def tiny_mixed(seed: int = 1001) -> Workload:
    return make_workload("tiny_mixed", [37, 100, 80], [1, 1, 32], num_q_heads=4,
                         num_kv_heads=1, head_dim=64, page_size=16, sm_scale=1.0 / 8.0,
                         seed=seed, mode="prefill")


def decode_bf16(mtp: int = 1, seed: int = 1002, shrink: int = 1) -> Workload:
    g = torch.Generator().manual_seed(seed * 7919 + mtp)
    B = max(2, 64 // shrink)
    ctx = _log_uniform_ints(B, max(8, 128 // shrink), 32768 // shrink, g)
    ql = [1 + mtp] * B
    ctx = [max(c, q) for c, q in zip(ctx, ql)]
    return make_workload(f"decode_bf16_mtp{mtp}" + (f"_s{shrink}" if shrink > 1 else ""), ctx,
                         ql, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64,
                         layout=NHD, kv_dtype=BF16, seed=seed + 17 * mtp, mode="decode",
                         max_pages_per_seq=(32768 // shrink + 63) // 64,
                         meta={"mtp": mtp, "shrink": shrink})


def decode_fp8(seed: int = 1003, shrink: int = 1, mtp: int = 2) -> Workload:
    g = torch.Generator().manual_seed(seed * 7919)
    B = max(2, 128 // shrink)
    ctx = _uniform_ints(B, 1024 // shrink, 16384 // shrink, g)
    ql = [1 + mtp] * B
    return make_workload("decode_fp8" + (f"_s{shrink}" if shrink > 1 else ""), ctx, ql,
                         num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                         layout=HND, kv_dtype=FP8_E4M3, seed=seed, mode="decode",
                         max_pages_per_seq=(16384 // shrink + 63) // 64,
                         meta={"mtp": mtp, "shrink": shrink})


def prefill_bf16(sparse: bool = False, seed: int = 1004, shrink: int = 1,
                 keep_prob: float = 0.26) -> Workload:
    B = 4 if shrink == 1 else 2
    L = 8192 // shrink
    mask = None
    if sparse:
        g = torch.Generator().manual_seed(seed * 7919 + 1)
        t = (L + 127) // 128
        mask = causal_block_mask(B, t, t, keep_prob, g)
    return make_workload("prefill_bf16" + ("_sparse" if sparse else "_dense") +
                         (f"_s{shrink}" if shrink > 1 else ""), [L] * B, [L] * B,
                         num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                         layout=NHD, kv_dtype=BF16, seed=seed, block_mask=mask, mode="prefill",
                         meta={"sparse": sparse, "shrink": shrink})


def prefill_fp8(quant_type: int = 1, sparse: bool = False, layout: int = NHD, seed: int = 1006,
                shrink: int = 1, keep_prob: float = 0.26) -> Workload:
    """The prefill workload's shape (B = 4 x 8192 causal, Hq=64, Hkv=8, D=128,
    64-token pages) with E4M3 Q, K and V: quant_type 0 (one scale each) or 1
    (Q per (token, q head), K and V one scale each); dense or block-sparse."""
    B = 4 if shrink == 1 else 2
    L = 8192 // shrink
    mask = None
    if sparse:
        g = torch.Generator().manual_seed(seed * 7919 + 1)
        t = (L + 127) // 128
        mask = causal_block_mask(B, t, t, keep_prob, g)
    return make_workload("prefill_fp8" + ("_sparse" if sparse else "_dense") + f"_q{quant_type}" +
                         ("_hnd" if layout == HND else "") + (f"_s{shrink}" if shrink > 1 else ""),
                         [L] * B, [L] * B, num_q_heads=64, num_kv_heads=8, head_dim=128,
                         page_size=64, layout=layout, kv_dtype=FP8_E4M3, seed=seed,
                         block_mask=mask, mode="prefill", q_dtype=FP8_E4M3,
                         quant_type=quant_type,
                         meta={"sparse": sparse, "shrink": shrink, "quant_type": quant_type})


def hybrid_bf16(seed: int = 1005, shrink: int = 1) -> Workload:
    g = torch.Generator().manual_seed(seed * 7919)
    n_dec = max(3, 255 // shrink)
    chunk, ctx_chunk = 1024 // shrink, 32768 // shrink
    dec_ctx = _uniform_ints(n_dec, max(2, 512 // shrink), 8192 // shrink, g)
    ctx = [ctx_chunk] + dec_ctx
    ql = [chunk] + [1] * n_dec
    return make_workload("hybrid_bf16" + (f"_s{shrink}" if shrink > 1 else ""), ctx, ql,
                         num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         layout=NHD, kv_dtype=BF16, seed=seed, mode="prefill",
                         meta={"shrink": shrink})


# ----------------------------------------------------------- work accounting

def decode_algorithmic_bytes(w: Workload) -> int:
    """Bytes a decode pass must move at minimum: every visible K and V element
    once, the FP8 scales of the pages touched, Q in, O out (bf16) and LSE out
    (fp32), and the block-table entries used."""
    ctx = [int(x) for x in w.context_lens]
    ql = [int(x) for x in w.q_lens]
    e = 2 if w.kv_dtype == BF16 else 1
    # first key any query of the sequence sees (a sliding window starts it late)
    lo = [max(0, c - q - w.window + 1) if w.window > 0 else 0 for c, q in zip(ctx, ql)]
    kv = sum(c - a for c, a in zip(ctx, lo)) * w.num_kv_heads * w.head_dim * 2 * e
    pages = sum((c + w.page_size - 1) // w.page_size - a // w.page_size for c, a in zip(ctx, lo))
    scales = pages * w.num_kv_heads * 2 * 4 if w.kv_dtype == FP8_E4M3 else 0
    rows = w.total_q * w.num_q_heads
    qo = rows * w.head_dim * 2 * 2 + rows * 4
    return kv + scales + qo + pages * 4


def visible_pairs(w: Workload) -> int:
    """Number of (query, key) pairs that are visible, per q head."""
    total = 0
    ctx = [int(x) for x in w.context_lens]
    ql = [int(x) for x in w.q_lens]
    if w.block_mask is None:
        for c, q in zip(ctx, ql):
            # query i sees keys 0 .. c-q+i
            total += q * (c - q) + q * (q + 1) // 2
        return total
    import numpy as np
    T = w.mask_tile
    m = w.block_mask.numpy().astype(np.int64)
    for b, (c, q) in enumerate(zip(ctx, ql)):
        i = np.arange(q, dtype=np.int64)
        p = c - q + i
        for kt in range(min(m.shape[2], c // T + 1)):
            lo = kt * T
            hi = np.minimum(p, lo + T - 1)
            cnt = np.clip(hi - lo + 1, 0, None)
            keep = m[b, np.minimum(i // T, m.shape[1] - 1), kt] * (i // T < m.shape[1])
            total += int((cnt * keep).sum())
    return total


def prefill_algorithmic_flops(w: Workload) -> int:
    """4 * D * Hq * (visible query-key pairs): QK^T and PV, 2 flops per MAC."""
    return 4 * w.head_dim * w.num_q_heads * visible_pairs(w)


def mixed_batch_parts(w: Workload):
    """A mixed batch without a block mask as the library runs it: the
    sequences with 1 <= G * q_len <= 16 rows go to the decode kernel, the
    others to the prefill kernel.  Returns (decode-part algorithmic bytes,
    prefill-part algorithmic FLOPs); the two parts' own bounds on the HBM and
    tensor rooflines add up to the batch's bound when they run one after the
    other."""
    import dataclasses
    ctx = w.context_lens.tolist()
    ql = w.q_lens.tolist()
    small = [1 <= w.gqa * q <= 16 and w.block_mask is None for q in ql]

    def part(keep):
        idx = [i for i, k in enumerate(keep) if k]
        c = [ctx[i] for i in idx]
        q = [ql[i] for i in idx]
        mask = w.block_mask[idx] if w.block_mask is not None else None
        return dataclasses.replace(w, context_lens=torch.tensor(c, dtype=torch.int32),
                                   q_lens=torch.tensor(q, dtype=torch.int32),
                                   num_seqs=len(c), block_mask=mask)

    dec = part(small)
    pre = part([not k for k in small])
    return (decode_algorithmic_bytes(dec) if dec.num_seqs else 0,
            prefill_algorithmic_flops(pre) if pre.num_seqs else 0)
