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
    assert bench.launches_per_step(W.decode_bf16(mtp=1, shrink=16), B.PA_MODE_DECODE) == 3
    # unmasked prefill-mode batch: 3 Assign + prefill + Combine, and the
    # decode part's Assign, kernel and Combine
    assert bench.launches_per_step(W.hybrid_bf16(shrink=16), B.PA_MODE_PREFILL) == 8
    assert bench.launches_per_step(W.prefill_bf16(sparse=True, shrink=32), B.PA_MODE_PREFILL) == 5
