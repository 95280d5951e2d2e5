"""The bounded pipeline waits: a wait that runs out is reported, every CTA
stops waiting, drains the tensor copies it issued and finishes, and the next
call is unaffected.  The timeout is made with the library's test hook: CTA 0's
producer leaves one K/V ring entry unfilled and the waits are limited to 20 ms,
so the consumer waiting for that entry gives up -- no fault, no trap, no
unbounded wait.  (Failure handling of a persistent split-K pipeline:
"基于Triton-TLE优化Tencent HPC-Ops Attention", 三.3, completion and
synchronisation of the compute CTAs.)"""
import ctypes
import time

import pytest
import torch

import oracle
from paged_attention_gb300 import binding as B
from paged_attention_gb300 import workloads as W

from gpu_util import compare

pytestmark = pytest.mark.gpu

PA_ERR_TIMEOUT = 6


def status_of_error_word(assign_ws):
    code = ctypes.c_int32(0)
    st = B.load().pa_last_device_error(ctypes.c_void_p(assign_ws.data_ptr()), ctypes.byref(code),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, code.value


CASES = {
    "decode_bf16": (lambda: W.decode_bf16(mtp=2, shrink=16), B.PA_MODE_DECODE),
    "decode_fp8": (lambda: W.decode_fp8(shrink=16), B.PA_MODE_DECODE),
    "prefill_sparse": (lambda: W.prefill_bf16(sparse=True, shrink=16), B.PA_MODE_PREFILL),
    "prefill_dense": (lambda: W.prefill_bf16(sparse=False, shrink=16), B.PA_MODE_PREFILL),
}


@pytest.mark.parametrize("which", list(CASES))
@pytest.mark.parametrize("skip", [0, 3])
def test_wait_timeout_is_reported_drained_and_the_next_call_is_clean(which, skip):
    make, mode = CASES[which]
    w = make()
    wd = w.to("cuda")
    bufs = B.make_buffers(wd, mode, num_ctas=8)
    run = B.run_decode if mode == B.PA_MODE_DECODE else B.run_prefill
    run(wd, bufs)                                  # warm: module loaded, clean state
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    B.pa_test_inject_wait_timeout(skip, 20_000_000)
    t0 = time.perf_counter()
    run(wd, bufs)
    torch.cuda.synchronize()                       # every CTA finished
    elapsed = time.perf_counter() - t0
    st, code = status_of_error_word(bufs.assign_ws)
    assert code == B.PA_DEV_WAIT_TIMEOUT and st == PA_ERR_TIMEOUT
    assert elapsed < 10.0
    # the hook disarmed itself: the next call is a normal one and matches the oracle
    bufs.out.zero_()
    run(wd, bufs)
    torch.cuda.synchronize()
    assert B.pa_last_device_error(bufs.assign_ws) == 0
    ref_o, ref_l = oracle.attention(w)
    compare(w, bufs.out, bufs.lse, ref_o, ref_l)


def test_hook_arguments_are_checked():
    with pytest.raises(B.PaError):
        B.pa_test_inject_wait_timeout(0, 10)       # below 1 ms
    B.pa_test_inject_wait_timeout(-1)              # disarm: always accepted
