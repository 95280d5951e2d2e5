"""Task trace (pa_set_task_trace): every task of a launch's Assign map gets its
start and end time and its CTA, one CTA's tasks in order, and tracing leaves
the results bit-identical.  The static path and the decode part of a mixed
batch are not traced."""
import numpy as np
import pytest
import torch

from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def traced(run, w, mode, bufs):
    tm0 = None
    cap = 4096
    trace = torch.full((cap, 3), -1, dtype=torch.int64, device="cuda")
    B.pa_set_task_trace(trace)
    try:
        run(w, bufs)
        torch.cuda.synchronize()
    finally:
        B.pa_set_task_trace(None)
    tm0 = B.pa_read_task_map(bufs.problem, mode, bufs.assign_ws)
    return trace.cpu().numpy(), tm0


def check_trace(tr, tm):
    T = tm["num_tasks"]
    assert T > 0
    cp = tm["cta_ptr"]
    rec = tr[:T]
    assert (rec[:, 0] > 0).all() and (rec[:, 1] >= rec[:, 0]).all()
    for c in range(len(cp) - 1):
        ks = np.arange(cp[c], cp[c + 1])
        assert (rec[ks, 2] == c).all()
        # one thread records a CTA's tasks, in map order
        assert (rec[ks[1:], 0] >= rec[ks[:-1], 1]).all()
    assert (tr[T:] == -1).all()


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_decode_trace(kind):
    w = (W.decode_bf16(mtp=1, shrink=8) if kind == "bf16" else W.decode_fp8(shrink=16)).to("cuda")
    ref = B.run_decode(w)
    o_ref, l_ref = ref.out.clone(), ref.lse.clone()
    bufs = B.make_buffers(w, B.PA_MODE_DECODE)
    tr, tm = traced(B.run_decode, w, B.PA_MODE_DECODE, bufs)
    check_trace(tr, tm)
    assert torch.equal(bufs.out, o_ref) and torch.equal(bufs.lse, l_ref)


def test_prefill_trace():
    w = W.prefill_bf16(sparse=True, shrink=16).to("cuda")
    bufs = B.make_buffers(w, B.PA_MODE_PREFILL)
    tr, tm = traced(B.run_prefill, w, B.PA_MODE_PREFILL, bufs)
    check_trace(tr, tm)


def test_mixed_batch_traces_the_prefill_map_only():
    w = W.hybrid_bf16(shrink=16).to("cuda")
    bufs = B.make_buffers(w, B.PA_MODE_PREFILL)
    tr, tm = traced(B.run_prefill, w, B.PA_MODE_PREFILL, bufs)
    check_trace(tr, tm)        # the prefill map's tasks, nothing beyond them


def test_static_path_not_traced():
    w = W.decode_bf16(mtp=1, shrink=16).to("cuda")
    bufs = B.StaticBuffers(w, 2)
    trace = torch.full((256, 3), -1, dtype=torch.int64, device="cuda")
    B.pa_set_task_trace(trace)
    try:
        B.run_decode_static(w, bufs)
        torch.cuda.synchronize()
    finally:
        B.pa_set_task_trace(None)
    assert (trace.cpu() == -1).all()
