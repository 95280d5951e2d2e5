"""pa_decode_noalloc: the whole decode run out of the library's fixed scratch.

Each case calls the entry point through the C ABI and compares its out / lse
with the caller-workspace path (pa_assign + pa_decode_splitk + pa_combine) on
the same device-resident inputs, within the parity tolerance of the decode
tests.  Calls come in a row -- the same problem twice, then a different one,
then the first again -- so that every call after the first reuses a scratch
that an earlier call filled.  The file name sorts last, so the cases also run
after every other GPU test; they pass alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import LSE_ATOL, out_tol

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


def assert_close(w, got, want):
    out, lse = got
    ref_out, ref_lse = want
    o = out.float().cpu().numpy()
    ro = ref_out.float().cpu().numpy()
    assert np.isfinite(o).all(), "non-finite output"
    err_o = np.abs(o - ro).max()
    assert err_o <= out_tol(w), f"max |out - caller-workspace out| = {err_o}"
    l = lse.cpu().numpy()
    rl = ref_lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin), "LSE finiteness differs"
    assert np.all(l[~fin] == rl[~fin])
    if fin.any():
        err_l = np.abs(l[fin] - rl[fin]).max()
        assert err_l <= LSE_ATOL, f"max |lse - caller-workspace lse| = {err_l}"


def check(w):
    ref = run_reference_path(w)
    out, lse, err = run_noalloc(w)
    assert err == B.PA_DEV_OK
    assert_close(w, (out, lse), ref)


def test_noalloc_matches_caller_workspace_path_on_calls_in_a_row():
    a = W.decode_bf16(mtp=2, shrink=16).to("cuda")
    b = W.decode_fp8(shrink=16).to("cuda")
    check(a)          # first call on this device: scratch address looked up here
    check(a)          # same problem again
    check(b)          # a different problem (FP8 KV, other shapes) in the same scratch
    check(a)          # and back


def test_noalloc_full_size_decode():
    w = W.decode_bf16(mtp=2).to("cuda")
    need = (-(-B.pa_assign_workspace_size(B.problem_from(w), B.PA_MODE_DECODE) // 256) * 256
            + B.pa_partial_workspace_size(B.problem_from(w), B.PA_MODE_DECODE))
    assert need <= B.PA_NOALLOC_SCRATCH_BYTES
    check(w)
    check(w)


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
