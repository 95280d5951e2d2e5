"""Host-side helpers: the counter fingerprint (comment edits keep measured
counters valid, code edits do not) and the bench's launch count per step."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from paged_attention_gb300 import build as build_mod  # noqa: E402
from paged_attention_gb300 import workloads as W  # noqa: E402


def test_code_only_strips_comments_not_strings():
    src = ('int a = 1; // one\n'
           '/* a block\n   comment */ const char* s = "// kept"; char c = \'/\';\n'
           '\n'
           '   x = "q\\"//still";   // tail\n')
    got = build_mod._code_only(src)
    assert "one" not in got and "block" not in got and "tail" not in got
    assert '"// kept"' in got and '"q\\"//still"' in got and "'/'" in got
    assert build_mod._code_only(src.replace("// one", "// two")) == got
    assert build_mod._code_only(src.replace("a = 1", "a = 2")) != got


def test_kernel_fingerprints_are_stable_and_distinct():
    a = build_mod.kernel_fingerprint("pa_prefill")
    b = build_mod.kernel_fingerprint("pa_decode_splitk")
    assert a == build_mod.kernel_fingerprint("pa_prefill")
    assert a != b and len(a) == 16


def test_launches_per_step():
    pytest.importorskip("torch")
    import bench
    from paged_attention_gb300 import binding as B
    # bf16 decode: Assign + the decode kernel (it finalizes its own split
    # units); E4M3 decode: and Combine
    assert bench.launches_per_step(W.decode_bf16(mtp=1, shrink=16), B.PA_MODE_DECODE) == 2
    assert bench.launches_per_step(W.decode_fp8(shrink=16), B.PA_MODE_DECODE) == 3
    # unmasked prefill-mode batch: 3 Assign + prefill + Combine, and the
    # decode part's Assign and kernel
    assert bench.launches_per_step(W.hybrid_bf16(shrink=16), B.PA_MODE_PREFILL) == 7
    assert bench.launches_per_step(W.prefill_bf16(sparse=True, shrink=32), B.PA_MODE_PREFILL) == 5


def test_windowed_algorithmic_bytes():
    """A window as long as every context changes nothing; a window of one
    reads exactly each sequence's q_len newest keys (the queries' own)."""
    w = W.decode_bf16(mtp=2, shrink=16)
    full = W.decode_algorithmic_bytes(w)
    w.window = int(w.context_lens.max()) + 5
    assert W.decode_algorithmic_bytes(w) == full
    w.window = 1
    ql = [int(x) for x in w.q_lens]
    ctx = [int(x) for x in w.context_lens]
    kv = sum(ql) * w.num_kv_heads * w.head_dim * 2 * 2
    pages = sum((c + w.page_size - 1) // w.page_size - (c - q) // w.page_size
                for c, q in zip(ctx, ql))
    rows = sum(ql) * w.num_q_heads
    assert W.decode_algorithmic_bytes(w) == kv + rows * w.head_dim * 4 + rows * 4 + pages * 4


@pytest.mark.parametrize("make", [
    lambda: W.prefill_bf16(sparse=True, shrink=16),
    lambda: W.prefill_bf16(sparse=False, shrink=16),
    lambda: W.hybrid_bf16(shrink=16),
])
def test_bench_per_row_visible_keys_sum_to_the_workload_pairs(make):
    """The bench's CPU-baseline accounting (visible keys per sampled row) adds
    up, over every row, to the FLOP accounting of the workload itself."""
    import bench
    w = make()
    total = 0
    for b in range(w.num_seqs):
        total += int(bench.visible_keys_per_row(w, b, range(int(w.q_lens[b]))).sum())
    assert total == W.visible_pairs(w)


def test_bench_windowed_visible_keys():
    import bench
    w = W.make_workload("win", [100, 37, 500], [3, 1, 2], num_q_heads=4, num_kv_heads=2,
                        head_dim=64, page_size=16, seed=3)
    w.window = 50
    got = [bench.visible_keys_per_row(w, b, range(int(w.q_lens[b]))).tolist()
           for b in range(w.num_seqs)]
    assert got == [[50, 50, 50], [37], [50, 50]]


def test_traffic_is_reported_only_for_the_kernel_it_was_taken_on(tmp_path, monkeypatch):
    """bench.py's roofline.traffic comes from profiles/traffic.json only while
    the entry's fingerprint matches the kernel sources (else null), and an
    entry without a q_len serves the workload's own q_len only."""
    import json
    import bench
    fp = build_mod.kernel_fingerprint("pa_prefill")
    fd = build_mod.kernel_fingerprint("pa_decode_splitk")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "pa_prefill:prefill_dense": {"source_hash": fp, "dram_bytes_per_launch": 123},
        "pa_prefill:prefill_sparse": {"source_hash": "0" * 16, "dram_bytes_per_launch": 456},
        "pa_decode_splitk:decode_fp8": {"source_hash": fd, "mtp": 2,
                                        "dram_bytes_per_launch": 789},
    }))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("pa_prefill", "prefill_dense") == 123
    assert bench.load_traffic("pa_prefill", "prefill_sparse") is None      # stale
    assert bench.load_traffic("pa_prefill", "hybrid") is None              # absent
    assert bench.load_traffic("pa_decode_splitk", "decode_fp8", 2) == 789
    assert bench.load_traffic("pa_decode_splitk", "decode_fp8", 3) is None  # other q_len


def test_mixed_batch_parts_split_the_work():
    """The hybrid batch's decode part holds the sequences with 1 <= G * q_len
    <= 16 (the library's split), the prefill part the others: bytes and FLOPs
    are additive over sequences, so the parts add up to the whole batch's; a
    masked batch has no decode part."""
    import dataclasses
    import torch
    w = W.hybrid_bf16(shrink=16)
    dec_bytes, pre_flops = W.mixed_batch_parts(w)
    small = [1 <= w.gqa * int(q) <= 16 for q in w.q_lens]
    assert 0 < sum(small) < len(small)

    def part(keep):
        c = [int(x) for x, k in zip(w.context_lens, keep) if k]
        q = [int(x) for x, k in zip(w.q_lens, keep) if k]
        return dataclasses.replace(w, context_lens=torch.tensor(c, dtype=torch.int32),
                                   q_lens=torch.tensor(q, dtype=torch.int32), num_seqs=len(c))

    big = [not k for k in small]
    assert dec_bytes == W.decode_algorithmic_bytes(part(small))
    assert pre_flops == W.prefill_algorithmic_flops(part(big))
    assert (W.decode_algorithmic_bytes(part(small)) + W.decode_algorithmic_bytes(part(big))
            == W.decode_algorithmic_bytes(w))
    assert (W.prefill_algorithmic_flops(part(small)) + pre_flops
            == W.prefill_algorithmic_flops(w))
    ws = W.prefill_bf16(sparse=True, shrink=32)
    assert W.mixed_batch_parts(ws) == (0, W.prefill_algorithmic_flops(ws))
