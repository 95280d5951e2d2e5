"""Helpers shared by the GPU parity tests (comparison against the oracle)."""
import numpy as np
import torch

from paged_attention_gb300 import binding as B

BF16_OUT_ATOL = 2e-2     # max-abs error of bf16 outputs against the fp64 oracle
FP8_OUT_ATOL = 6e-2      # FP8-KV outputs
LSE_ATOL = 1e-3          # natural-log LSE


def out_tol(w):
    return FP8_OUT_ATOL if w.kv_dtype == 1 else BF16_OUT_ATOL


def compare(w, out, lse, ref_o, ref_l, rows=None):
    """Element-wise comparison of GPU out/lse with oracle rows."""
    o = out.float().reshape(-1, w.head_dim).cpu().numpy().astype(np.float64)
    l = lse.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.isfinite(o).all(), "non-finite output"
    err_o = np.abs(o - ref_o).max() if o.size else 0.0
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), "LSE finiteness differs"
    assert np.all(l[~fin] == ref_l[~fin])
    err_l = np.abs(l[fin] - ref_l[fin]).max() if fin.any() else 0.0
    assert err_o <= out_tol(w), f"max |out - oracle| = {err_o}"
    assert err_l <= LSE_ATOL, f"max |lse - oracle| = {err_l}"
    return err_o, err_l


def task_map_equal(gpu: dict, tm, with_active: bool):
    assert gpu["num_units"] == tm.num_units
    assert gpu["num_tasks"] == tm.num_tasks
    assert gpu["num_slots"] == tm.num_slots
    assert np.array_equal(gpu["cta_ptr"], tm.cta_ptr)
    assert np.array_equal(gpu["tasks"], tm.tasks)
    assert np.array_equal(gpu["units"], tm.units)
    assert np.array_equal(gpu["unit_ntiles"], tm.unit_ntiles)
    assert np.array_equal(gpu["unit_nsplit"], tm.unit_nsplit)
    assert np.array_equal(gpu["unit_slot0"], tm.unit_slot0)
    if with_active:
        for u, n in enumerate(tm.unit_ntiles):
            assert np.array_equal(gpu["active"][u, :n], tm.active[u, :n]), f"unit {u}"
