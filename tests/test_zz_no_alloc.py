"""pa_decode_noalloc: the whole decode run out of the library's fixed scratch.

Some callers cannot hand the library device memory when they call it: a
serving engine that gave all free HBM to its KV-cache page pool up front, or a
plain C host with no device allocator.  pa_decode_noalloc serves them from a
file-scope device array inside the library.  Each case here calls it through
the C ABI and checks that it gives exactly what the caller-workspace path
(pa_assign + pa_decode_splitk + pa_combine) gives on the same device-resident
inputs -- the same kernels over the same task map, so bit for bit -- and,
directly, that it matches the fp64 oracle within the decode tolerances.  Calls
come in a row -- the same problem twice, then a different one, then the first
again -- so that every call after the first reuses a scratch that an earlier
call filled.  The file name sorts last, so the cases also run after every other
GPU test; they pass alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

import oracle
from gpu_util import compare

pytestmark = pytest.mark.gpu


def run_noalloc(w):
    p = B.problem_from(w)
    out = torch.full((w.total_q, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.total_q, w.num_q_heads), float("nan"), dtype=torch.float32,
                     device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.pa_decode_noalloc(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens, w.q_lens,
                        w.k_scale, w.v_scale, out, lse, err)
    torch.cuda.synchronize()
    return out, lse, int(err.item())


def run_reference_path(w):
    bufs = B.run_decode(w)
    torch.cuda.synchronize()
    return bufs.out.clone(), bufs.lse.clone()


def assert_same(got, want):
    """Bit equality with the caller-workspace path: the same kernels run the
    same task map, so any difference (a stale scratch word left by an earlier
    call, a partial read from the wrong slot) shows up here."""
    out, lse = got
    ref_out, ref_lse = want
    assert torch.isfinite(out.float()).all(), "non-finite output"
    assert torch.equal(out, ref_out), "out differs from the caller-workspace path"
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), fin), "LSE finiteness differs"
    assert torch.equal(lse[fin], ref_lse[fin]), "lse differs from the caller-workspace path"
    assert torch.equal(lse[~fin], ref_lse[~fin])


def check(w, w_cpu=None, rows=None):
    ref = run_reference_path(w)
    out, lse, err = run_noalloc(w)
    assert err == B.PA_DEV_OK
    assert_same((out, lse), ref)
    if w_cpu is not None:
        # and directly against the fp64 oracle, within the decode tolerances
        ref_o, ref_l = oracle.attention(w_cpu, rows=rows)
        compare(w_cpu, out, lse, ref_o, ref_l, rows=rows)


def test_noalloc_matches_caller_workspace_path_on_calls_in_a_row():
    a_cpu = W.decode_bf16(mtp=2, shrink=16)
    b_cpu = W.decode_fp8(shrink=16)
    a, b = a_cpu.to("cuda"), b_cpu.to("cuda")
    check(a, a_cpu)   # first call on this device: scratch address looked up here
    check(a)          # same problem again
    check(b, b_cpu)   # a different problem (FP8 KV, other shapes) in the same scratch
    check(a, a_cpu)   # and back


def test_noalloc_full_size_decode():
    w_cpu = W.decode_bf16(mtp=2)
    w = w_cpu.to("cuda")
    need = (-(-B.pa_assign_workspace_size(B.problem_from(w), B.PA_MODE_DECODE) // 256) * 256
            + B.pa_partial_workspace_size(B.problem_from(w), B.PA_MODE_DECODE))
    assert need <= B.PA_NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(w.total_q * w.num_q_heads, size=2048, replace=False))
    check(w, w_cpu, rows)
    check(w)


def test_noalloc_reports_a_device_check_through_device_error():
    """A length fault that only the device sees (q_lens > context_lens for one
    sequence): the call itself returns PA_OK, Assign flags the fault and
    builds an empty task map, and the flag reaches the caller's device_error
    word; the next valid call clears it."""
    w_cpu = W.decode_bf16(mtp=1, shrink=16)
    bad = W.decode_bf16(mtp=1, shrink=16)
    bad.context_lens[1] = 1            # q_len 2 > context length 1
    w, wb = w_cpu.to("cuda"), bad.to("cuda")
    out, lse, err = run_noalloc(wb)    # returns without raising: the host saw nothing wrong
    assert err & B.PA_DEV_BAD_LENGTHS
    check(w, w_cpu)                    # a valid call afterwards starts clean


def test_noalloc_refuses_problems_beyond_the_scratch():
    w = W.decode_bf16(mtp=1, shrink=16).to("cuda")
    p = B.problem_from(w)
    p.num_seqs = 4096          # partials far beyond the fixed scratch
    out = torch.empty((1, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PaError) as e:
        B.pa_decode_noalloc(p, w.q, w.k_cache, w.v_cache, w.block_table, w.context_lens,
                            w.q_lens, w.k_scale, w.v_scale, out, None)
    assert e.value.status == B.PA_ERR_WORKSPACE
    # the refused call launched nothing; the next valid call still works
    check(w)
