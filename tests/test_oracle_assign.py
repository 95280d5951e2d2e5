"""Pins for the oracle's Assign task map (CPU only).

Assign tiles every unit's KV and hands the tiles to N CTAs so each carries an
equal share of the work ("基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2
Assign step and 三.3 均分调度); prefill units list only the KV tiles the block
mask keeps (二.1 active-KV-tile list).  The exact procedure is this project's
reading and is written out in oracle/pa_oracle.c above oracle_assign().

Pinned by: hand-worked examples (tests/golden/assign_worked_examples.json),
structural invariants that hold for any input (every tile covered once, in
ascending contiguous runs; balanced per-CTA cost; slot numbering), and an
independent brute force written differently (bisect over CTA bounds,
itertools.groupby for runs).
"""
import bisect
import itertools
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_oracle(oracle_mod, ex):
    bm = None if ex["block_mask"] is None else np.array(ex["block_mask"], dtype=np.uint8)
    return oracle_mod.assign(ex["mode"], ex["num_seqs"], ex["num_q_heads"], ex["num_kv_heads"],
                             ex["num_ctas"], ex["kv_tile"], ex["balance_rows"],
                             np.array(ex["context_lens"], np.int32),
                             np.array(ex["q_lens"], np.int32), bm,
                             window=ex.get("window", 0))


def load_examples():
    with open(os.path.join(GOLDEN, "assign_worked_examples.json")) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("ex", load_examples(), ids=lambda e: e["name"])
def test_worked_examples(oracle_mod, ex):
    tm = run_oracle(oracle_mod, ex)
    e = ex["expect"]
    assert tm.units.tolist() == e["units"]
    assert tm.unit_ntiles.tolist() == e["unit_ntiles"]
    assert tm.cta_ptr.tolist() == e["cta_ptr"]
    assert tm.tasks.tolist() == e["tasks"]
    assert tm.unit_nsplit.tolist() == e["unit_nsplit"]
    assert tm.unit_slot0.tolist() == e["unit_slot0"]
    assert tm.num_slots == e["num_slots"]
    if "active" in e:
        assert [tm.active[u, :n].tolist() for u, n in enumerate(tm.unit_ntiles)] == e["active"]


# ------------------------------------------------------- brute force

def brute_force(mode, B, Hq, Hkv, N, T, rbal, ctx, ql, mask=None, mask_tile=128, window=0,
                unit_cost=0):
    G = Hq // Hkv
    units = []
    for b in range(B):
        if mode == 0:
            for hk in range(Hkv):
                units.append((b, hk, 0, ql[b], ctx[b] if ql[b] > 0 else 0))
        else:
            qtok = 128 if (mask is not None and G == 1) else 256 // G
            for hk in range(Hkv):
                for q0 in range(0, ql[b], qtok):
                    nq = min(qtok, ql[b] - q0)
                    units.append((b, hk, q0, nq, ctx[b] - ql[b] + q0 + nq))
    lists = []
    for (b, hk, q0, nq, L) in units:
        reach = list(range(-(-L // T)))
        if window > 0:
            # the unit's first query sits at ctx - ql + q0 and sees keys after
            # p - window: keep the tiles whose last key reaches that far
            first_key = ctx[b] - ql[b] + q0 - window + 1
            reach = [t for t in reach if (t + 1) * T - 1 >= first_key]
        if mask is not None:
            reach = [t for t in reach if t < mask.shape[2] and mask[b, q0 // mask_tile, t]]
        lists.append(reach)
    weights = [max(1, -(-(G * u[3]) // rbal)) for u in units]
    # a unit with tiles carries unit_cost ahead of its first tile
    fixed = [unit_cost if len(l) else 0 for l in lists]
    costs = list(itertools.accumulate([0] + [h + len(l) * w
                                             for h, l, w in zip(fixed, lists, weights)]))
    C = costs[-1]
    bounds = [c * C // N for c in range(N + 1)]
    owned = []                      # (cta, unit, position)
    for u, lst in enumerate(lists):
        for t in range(len(lst)):
            x = costs[u] + fixed[u] + t * weights[u]
            owned.append((bisect.bisect_right(bounds, x) - 1 if C else 0, u, t))
    owned = [(min(c, N - 1), u, t) for c, u, t in owned]
    tasks = []
    for (c, u), grp in itertools.groupby(owned, key=lambda z: (z[0], z[1])):
        grp = list(grp)
        tasks.append([c, u, grp[0][2], grp[-1][2] + 1])
    nsplit = [0] * len(units)
    for t in tasks:
        nsplit[t[1]] += 1
    slot0, s = [], 0
    for n in nsplit:
        slot0.append(s if n > 1 else -1)
        s += n if n > 1 else 0
    seen = [0] * len(units)
    out_tasks = []
    for c, u, t0, t1 in tasks:
        out_tasks.append([u, t0, t1, slot0[u] + seen[u] if nsplit[u] > 1 else -1])
        seen[u] += 1
    cta_ptr = [sum(1 for t in tasks if t[0] < c) for c in range(N + 1)]
    return dict(units=[list(u[:4]) for u in units], lists=lists, tasks=out_tasks,
                cta_ptr=cta_ptr, nsplit=nsplit, slot0=slot0, slots=s, weights=weights,
                C=C, task_cta=[t[0] for t in tasks])


def random_case(rng):
    mode = int(rng.integers(0, 2))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 7))
    N = int(rng.integers(1, 20))
    T = int(rng.choice([16, 64, 128])) if mode == 0 else 128
    rbal = int(rng.choice([16, 64, 128, 288]))
    ctx, ql = [], []
    for _ in range(B):
        c = int(rng.integers(0, 700))
        q = int(rng.integers(0, min(c, 300) + 1)) if mode == 1 else int(rng.integers(0, min(c, 4) + 1))
        ctx.append(c)
        ql.append(q)
    mask = None
    if mode == 1 and rng.random() < 0.5:
        mq = max(1, -(-max(ql) // 128)) if max(ql) > 0 else 1
        mk = max(1, -(-max(ctx) // 128)) if max(ctx) > 0 else 1
        mask = (rng.random((B, mq, mk)) < 0.5).astype(np.uint8)
    return mode, B, G * Hkv, Hkv, N, T, rbal, ctx, ql, mask


@pytest.mark.parametrize("seed", range(60))
def test_matches_brute_force_and_invariants(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    mode, B, Hq, Hkv, N, T, rbal, ctx, ql, mask = random_case(rng)
    tm = oracle_mod.assign(mode, B, Hq, Hkv, N, T, rbal, np.array(ctx, np.int32),
                           np.array(ql, np.int32), mask)
    bf = brute_force(mode, B, Hq, Hkv, N, T, rbal, ctx, ql, mask)
    assert tm.units.tolist() == bf["units"]
    assert [tm.active[u, :n].tolist() for u, n in enumerate(tm.unit_ntiles)] == bf["lists"]
    assert tm.tasks.tolist() == bf["tasks"]
    assert tm.cta_ptr.tolist() == bf["cta_ptr"]
    assert tm.unit_nsplit.tolist() == bf["nsplit"]
    assert tm.unit_slot0.tolist() == bf["slot0"]
    assert tm.num_slots == bf["slots"]

    # invariant: every unit's list covered exactly once, ascending contiguous runs
    for u, n in enumerate(tm.unit_ntiles):
        runs = [t for t in tm.tasks.tolist() if t[0] == u]
        pos = 0
        for _, t0, t1, _ in runs:
            assert t0 == pos and t1 > t0
            pos = t1
        assert pos == n
    # invariant: per-CTA cost within one max weight of C/N
    wmax = max(bf["weights"]) if bf["weights"] else 1
    for c in range(N):
        cost = 0
        for k in range(tm.cta_ptr[c], tm.cta_ptr[c + 1]):
            u, t0, t1, _ = tm.tasks[k]
            cost += (t1 - t0) * bf["weights"][u]
        assert abs(cost - bf["C"] / N) <= wmax + 1e-9
    # invariant: slots are 0..n_slots-1, each once, only for split units
    slots = [int(t[3]) for t in tm.tasks if t[3] >= 0]
    assert sorted(slots) == list(range(tm.num_slots))
    # invariant: task count never exceeds units + CTAs
    assert tm.num_tasks <= tm.num_units + N


def test_full_size_decode_map_is_balanced(oracle_mod):
    from paged_attention_gb300 import workloads as W
    g = torch.Generator().manual_seed(1)
    ctx = W._log_uniform_ints(64, 128, 32768, g)
    tm = oracle_mod.assign(0, 64, 32, 8, 152, 64, 128, np.array(ctx, np.int32),
                           np.array([2] * 64, np.int32))
    per_cta = []
    for c in range(152):
        per_cta.append(sum(int(t[2] - t[1]) for t in tm.tasks[tm.cta_ptr[c]:tm.cta_ptr[c + 1]]))
    assert max(per_cta) - min(per_cta) <= 1
    assert tm.num_tasks <= 512 + 152


@pytest.mark.parametrize("seed", range(24))
def test_prefill_split_covers_every_query_row_once(oracle_mod, seed):
    """Prefill-mode Assign without a block mask sends a sequence to the decode
    part iff 1 <= G * q_len <= 16.  Independently of how the two maps are
    built: together they hold every (sequence, KV head, query token) exactly
    once, each unit reaches exactly the keys its rows may see (decode part:
    all ctx keys in 64-token tiles; prefill part: up to its last query's
    position in 128-token tiles), and each part is balanced like any map."""
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hq = G * Hkv
    B = int(rng.integers(1, 9))
    N = int(rng.integers(1, 20))
    rbal = int(rng.choice([16, 128, 288]))
    ctx, ql = [], []
    for _ in range(B):
        c = int(rng.integers(0, 900))
        q = int(rng.integers(0, min(c, 4) + 1)) if rng.random() < 0.6 else \
            int(rng.integers(0, min(c, 300) + 1))
        ctx.append(c)
        ql.append(q)
    pre, dec = oracle_mod.assign_prefill(B, Hq, Hkv, N, rbal, np.array(ctx, np.int32),
                                         np.array(ql, np.int32))
    assert dec is not None
    small = [1 <= G * q <= 16 for q in ql]
    seen = {}
    for (b, hk, q0, nq), n in zip(pre.units.tolist(), pre.unit_ntiles.tolist()):
        assert not small[b] and nq >= 1
        assert n == -(-(ctx[b] - ql[b] + q0 + nq) // 128)
        for i in range(q0, q0 + nq):
            seen[(b, hk, i)] = seen.get((b, hk, i), 0) + 1
    assert dec.units.tolist() == [[b, hk, 0, ql[b] if small[b] else 0]
                                  for b in range(B) for hk in range(Hkv)]
    for (b, hk, q0, nq), n in zip(dec.units.tolist(), dec.unit_ntiles.tolist()):
        assert n == (-(-ctx[b] // 64) if nq > 0 else 0)
        for i in range(nq):
            seen[(b, hk, i)] = seen.get((b, hk, i), 0) + 1
    want = {(b, hk, i) for b in range(B) for hk in range(Hkv) for i in range(ql[b])}
    assert set(seen) == want and all(v == 1 for v in seen.values())
    for tm in (pre, dec):
        for u, n in enumerate(tm.unit_ntiles):
            runs = [t for t in tm.tasks.tolist() if t[0] == u]
            assert sum(t1 - t0 for _, t0, t1, _ in runs) == n
        assert tm.num_tasks <= tm.num_units + N


def test_prefill_split_absent_with_mask_or_wide_groups(oracle_mod):
    ctx = np.array([300, 40, 500], np.int32)
    ql = np.array([1, 40, 2], np.int32)
    mask = np.ones((3, 1, 4), np.uint8)
    pre, dec = oracle_mod.assign_prefill(3, 8, 2, 5, 128, ctx, ql, block_mask=mask)
    assert dec is None and sorted({int(u[0]) for u in pre.units}) == [0, 1, 2]
    pre, dec = oracle_mod.assign_prefill(3, 32, 1, 5, 128, ctx, ql)   # G = 32 > 16
    assert dec is None and sorted({int(u[0]) for u in pre.units}) == [0, 1, 2]


@pytest.mark.parametrize("seed", range(20))
def test_window_maps_match_brute_force(oracle_mod, seed):
    """Sliding window ("HiLS-Attention", 二.1 local branch; keys p - window < j
    <= p): a unit's tiles start at the first one its first query can see."""
    rng = np.random.default_rng(500 + seed)
    mode = int(rng.integers(0, 2))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 7))
    N = int(rng.integers(1, 20))
    T = 64 if mode == 0 else 128
    window = int(rng.choice([1, 17, 64, 100, 300, 5000]))
    ctx, ql = [], []
    for _ in range(B):
        c = int(rng.integers(0, 900))
        q = int(rng.integers(0, min(c, 4 if mode == 0 else 300) + 1))
        ctx.append(c)
        ql.append(q)
    tm = oracle_mod.assign(mode, B, G * Hkv, Hkv, N, T, 128, np.array(ctx, np.int32),
                           np.array(ql, np.int32), window=window)
    bf = brute_force(mode, B, G * Hkv, Hkv, N, T, 128, ctx, ql, window=window)
    assert tm.unit_ntiles.tolist() == [len(x) for x in bf["lists"]]
    assert tm.tasks.tolist() == bf["tasks"]
    assert tm.cta_ptr.tolist() == bf["cta_ptr"]
    assert tm.unit_slot0.tolist() == bf["slot0"]
    # a window as long as every context changes nothing
    full = oracle_mod.assign(mode, B, G * Hkv, Hkv, N, T, 128, np.array(ctx, np.int32),
                             np.array(ql, np.int32), window=max(ctx + [1]) + 1)
    plain = oracle_mod.assign(mode, B, G * Hkv, Hkv, N, T, 128, np.array(ctx, np.int32),
                              np.array(ql, np.int32))
    assert full.tasks.tolist() == plain.tasks.tolist()


def test_prefill_split_worked_example(oracle_mod):
    """The two maps of a small mixed batch, worked by hand
    (tests/golden/assign_prefill_split_example.json)."""
    with open(os.path.join(GOLDEN, "assign_prefill_split_example.json")) as f:
        ex = json.load(f)["example"]
    pre, dec = oracle_mod.assign_prefill(ex["num_seqs"], ex["num_q_heads"], ex["num_kv_heads"],
                                         ex["num_ctas"], ex["balance_rows"],
                                         np.array(ex["context_lens"], np.int32),
                                         np.array(ex["q_lens"], np.int32))
    for tm, e in ((pre, ex["expect_prefill"]), (dec, ex["expect_decode"])):
        assert tm.units.tolist() == e["units"]
        assert tm.unit_ntiles.tolist() == e["unit_ntiles"]
        assert tm.cta_ptr.tolist() == e["cta_ptr"]
        assert tm.tasks.tolist() == e["tasks"]
        assert tm.unit_nsplit.tolist() == e["unit_nsplit"]
        assert tm.unit_slot0.tolist() == e["unit_slot0"]
        assert tm.num_slots == e["num_slots"]


@pytest.mark.parametrize("seed", range(12))
def test_prefill_split_with_window(oracle_mod, seed):
    """Both prefill-mode maps take the sliding window ("HiLS-Attention", 二.1
    local branch: keys p - window < j <= p): a unit's tiles start at the tile
    holding its first query's first visible key, p0 - window + 1, and end
    where they would without a window; with a block mask the active list is
    the kept tiles of that range."""
    rng = np.random.default_rng(3000 + seed)
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 4, 8]))
    B = int(rng.integers(1, 7))
    N = int(rng.integers(1, 20))
    window = int(rng.choice([1, 50, 128, 300, 700]))
    ctx, ql = [], []
    for _ in range(B):
        c = int(rng.integers(1, 900))
        q = int(rng.integers(1, min(c, 4) + 1)) if rng.random() < 0.5 else \
            int(rng.integers(1, min(c, 300) + 1))
        ctx.append(c)
        ql.append(q)
    masked = seed % 3 == 0
    mask = None
    if masked:
        qt = -(-max(ql) // 128)
        kt = -(-max(ctx) // 128)
        mask = (rng.random((B, qt, kt)) < 0.6).astype(np.uint8)
    pre, dec = oracle_mod.assign_prefill(B, G * Hkv, Hkv, N, 128, np.array(ctx, np.int32),
                                         np.array(ql, np.int32), block_mask=mask,
                                         window=window)
    for u, ((b, hk, q0, nq), n) in enumerate(zip(pre.units.tolist(), pre.unit_ntiles.tolist())):
        first = max(0, ctx[b] - ql[b] + q0 - window + 1) // 128
        end = -(-(ctx[b] - ql[b] + q0 + nq) // 128)
        want = [t for t in range(first, end)
                if mask is None or (t < mask.shape[2] and mask[b, q0 // 128, t])]
        assert n == len(want)
        if mask is not None:
            assert pre.active[u, :n].tolist() == want
    if dec is not None:
        for (b, hk, q0, nq), n in zip(dec.units.tolist(), dec.unit_ntiles.tolist()):
            first = max(0, ctx[b] - ql[b] - window + 1) // 64
            assert n == ((-(-ctx[b] // 64) - first) if nq > 0 else 0)


@pytest.mark.parametrize("seed", range(40))
def test_unit_cost_matches_brute_force(oracle_mod, seed):
    """A fixed cost per unit with tiles (our reading of "equal work per CTA":
    a unit costs its CTA something besides its tiles), placed ahead of the
    unit's first tile: the oracle and the brute force agree, every tile is
    still covered once, and a CTA's tile work plus the fixed costs of the
    units it starts stays within one tile weight plus one fixed cost of C/N."""
    rng = np.random.default_rng(1000 + seed)
    mode, B, Hq, Hkv, N, T, rbal, ctx, ql, mask = random_case(rng)
    h = int(rng.choice([1, 2, 3, 7]))
    tm = oracle_mod.assign(mode, B, Hq, Hkv, N, T, rbal, np.array(ctx, np.int32),
                           np.array(ql, np.int32), mask, unit_cost=h)
    bf = brute_force(mode, B, Hq, Hkv, N, T, rbal, ctx, ql, mask, unit_cost=h)
    assert tm.units.tolist() == bf["units"]
    assert tm.tasks.tolist() == bf["tasks"]
    assert tm.cta_ptr.tolist() == bf["cta_ptr"]
    assert tm.unit_nsplit.tolist() == bf["nsplit"]
    assert tm.unit_slot0.tolist() == bf["slot0"]
    for u, n in enumerate(tm.unit_ntiles):
        runs = [t for t in tm.tasks.tolist() if t[0] == u]
        pos = 0
        for _, t0, t1, _ in runs:
            assert t0 == pos and t1 > t0
            pos = t1
        assert pos == n
    wmax = max(bf["weights"]) if bf["weights"] else 1
    for c in range(N):
        cost = 0
        for k in range(tm.cta_ptr[c], tm.cta_ptr[c + 1]):
            u, t0, t1, _ = tm.tasks[k]
            cost += (t1 - t0) * bf["weights"][u] + (h if t0 == 0 else 0)
        assert abs(cost - bf["C"] / N) <= wmax + h + 1e-9


def test_unit_cost_zero_is_the_plain_map(oracle_mod):
    """unit_cost = 0 leaves the map of the plain procedure unchanged."""
    rng = np.random.default_rng(7)
    mode, B, Hq, Hkv, N, T, rbal, ctx, ql, mask = random_case(rng)
    a = oracle_mod.assign(mode, B, Hq, Hkv, N, T, rbal, np.array(ctx, np.int32),
                          np.array(ql, np.int32), mask)
    b = oracle_mod.assign(mode, B, Hq, Hkv, N, T, rbal, np.array(ctx, np.int32),
                          np.array(ql, np.int32), mask, unit_cost=0)
    assert a.tasks.tolist() == b.tasks.tolist() and a.cta_ptr.tolist() == b.cta_ptr.tolist()
