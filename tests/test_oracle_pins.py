"""Pins of the float64 oracle against things other than itself.

Each pin is a hand-worked fixture (tests/golden/, derived from the Epoch
walk-through's definitions), a closed form, a brute-force search on tiny inputs,
or a special case that reduces to the plain dense MoE formula computed in a
different arrangement. The mutation tests at the end plant plausible mistakes
in the oracle and check that some pin catches each one.
"""
import dataclasses
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from oracle import epoch_moe as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ fixtures

def _floats(s):
    return np.array([float(v) for v in s.split(",")])


def _ints(s):
    return [] if s == "-" else [int(v) for v in s.split(",")]


def load_schedules():
    scheds, cur = [], None
    with open(os.path.join(GOLDEN, "fresh_schedules.txt"), encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "schedule":
                cur = dict(name=tok[1], R=None if tok[3] == "inf" else int(tok[3]), steps=[])
                scheds.append(cur)
            else:
                kv = dict(zip(tok[0::2], tok[1::2]))
                cur["steps"].append(dict(i=int(kv["i"]), decoded=[int(c) for c in kv["decoded"]],
                                         fresh=_ints(kv["fresh"]), fallback=int(kv["fallback"]),
                                         cats=[int(c) for c in kv["cats"].split("/")]))
    return scheds


def load_routing():
    cases = {"gate": [], "topk": [], "plan": []}
    with open(os.path.join(GOLDEN, "routing_cases.txt"), encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            kv = dict(zip(tok[1::2], tok[2::2]))
            cases[tok[0]].append(kv)
    return cases


def tiny_layer(E=6, H=5, I=4, k=2, tau=1.0, R=None, n_shared=0, seed=0, max_positions=16,
               residual=False):
    rng = np.random.default_rng(seed)
    wr = rng.normal(size=(E, H))
    b = rng.normal(size=E)
    experts = [(rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I)))
               for _ in range(E)]
    shared = [(rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I)))
              for _ in range(n_shared)]
    lay = oracle.LayerOracle(n_experts=E, top_k=k, tau=tau, refresh_R=R, w_router=wr, b_router=b,
                             expert=lambda e: experts[e], shared=shared, residual=residual,
                             max_positions=max_positions)
    return lay, wr, b, experts, shared


# ------------------------------------------------------------------ closed forms

def test_gate_golden():
    for c in load_routing()["gate"]:
        x = _floats(c["x"])[None, :]
        wr = np.array([[float(v) for v in r.split(",")] for r in c["wr"].split(";")])
        G = oracle.gate_logits(x, wr, _floats(c["b"]))
        np.testing.assert_allclose(G[0], _floats(c["G"]), rtol=0, atol=1e-15)


def test_silu_closed_forms():
    ln3 = math.log(3.0)
    assert oracle.silu(np.array(0.0)) == 0.0
    assert abs(oracle.silu(np.array(ln3)) - 0.75 * ln3) < 1e-15
    assert abs(oracle.silu(np.array(-ln3)) + 0.25 * ln3) < 1e-15
    z = np.linspace(-30, 30, 241)
    # silu(z) - silu(-z) = z because sigmoid(-z) = 1 - sigmoid(z)
    np.testing.assert_allclose(oracle.silu(z) - oracle.silu(-z), z, atol=1e-12)
    # silu(z) -> z for large z and -> 0 for very negative z
    assert abs(oracle.silu(np.array(40.0)) - 40.0) < 1e-12
    assert abs(oracle.silu(np.array(-40.0))) < 1e-15


def test_swiglu_golden():
    ln3 = math.log(3.0)
    x = np.array([[1.0, 0.0]])
    wg = np.array([[0, 0], [ln3, 0], [0, 0]], dtype=float)
    wu = np.array([[1, 0], [2, 0], [5, 7]], dtype=float)
    wd = np.array([[1, 1, 4], [0, 1, 9]], dtype=float)
    y = oracle.swiglu_expert(x, (wg, wu, wd))
    np.testing.assert_allclose(y[0], [1.5 * ln3, 1.5 * ln3], rtol=0, atol=1e-15)


def test_softmax_closed_form():
    w = oracle.renorm_softmax(np.array([2.0, 2.0, 0.5]))
    d = 2.0 + math.exp(-1.5)
    np.testing.assert_allclose(w, [1 / d, 1 / d, math.exp(-1.5) / d], rtol=1e-15)
    assert oracle.renorm_softmax(np.array([7.25]))[0] == 1.0
    # ratios are exp of logit differences, whatever the shift
    g = np.array([1000.0, 999.0, 997.5])
    w = oracle.renorm_softmax(g)
    np.testing.assert_allclose([w[0] / w[1], w[1] / w[2]], [math.e, math.exp(1.5)], rtol=1e-12)
    assert abs(w.sum() - 1.0) < 1e-15


# ------------------------------------------------------------------ routing

def test_topk_golden():
    for c in load_routing()["topk"]:
        elig = np.array([ch == "1" for ch in c["elig"]])
        sel = oracle.topk_select(_floats(c["g"]), elig, int(c["k"]))
        assert list(sel) == _ints(c["sel"]), c


def brute_topk(g, elig, k):
    """Max-sum k-subset of the eligible experts; among equal sums, the
    lexicographically smallest sorted id tuple (= ties to the lower id)."""
    ids = [e for e in range(len(g)) if elig[e]]
    best = None
    for comb in itertools.combinations(ids, k):
        key = (-sum(g[e] for e in comb), comb)
        if best is None or key < best:
            best = key
    return set(best[1])


def test_topk_bruteforce():
    rng = np.random.default_rng(11)
    for trial in range(400):
        E = int(rng.integers(2, 9))
        # few distinct values, so exact ties are common
        g = rng.integers(-3, 4, size=E).astype(float) * 0.5
        elig = rng.random(E) < 0.8
        if elig.sum() == 0:
            elig[rng.integers(E)] = True
        k = int(rng.integers(1, elig.sum() + 1))
        sel = oracle.topk_select(g, elig, k)
        assert set(sel.tolist()) == brute_topk(g, elig, k)
        # selection order: logit descending, lower id first among equal logits
        keys = [(-g[e], e) for e in sel]
        assert keys == sorted(keys)
        assert all(elig[e] for e in sel)


def test_hit_counts_bruteforce():
    rng = np.random.default_rng(12)
    for _ in range(30):
        N, E = int(rng.integers(1, 9)), int(rng.integers(2, 7))
        k = int(rng.integers(1, E + 1))
        G = rng.integers(-2, 3, size=(N, E)).astype(float)
        cnt = oracle.hit_counts(G, k)
        assert cnt.sum() == N * k
        ref = np.zeros(E, dtype=int)
        for t in range(N):
            for e in brute_topk(G[t], np.ones(E, bool), k):
                ref[e] += 1
        assert (cnt == ref).all()


def test_plan_golden():
    for c in load_routing()["plan"]:
        cnt = np.array(_ints(c["cnt"]))
        k, n, tau = int(c["k"]), int(c["n"]), float(c["tau"])
        assert oracle.coverage_threshold(tau, n, k) == int(c["T"])
        ranked, slen = oracle.plan_support(cnt, k, tau, n)
        assert list(ranked) == _ints(c["ranked"])
        assert slen == int(c["len"])


def test_plan_minimal_support_bruteforce():
    """|S| = max(k, fewest experts whose counts reach T), and S holds the largest
    counts, ties to the lower id: checked over every subset of up to 9 experts."""
    rng = np.random.default_rng(13)
    for _ in range(150):
        E = int(rng.integers(2, 10))
        k = int(rng.integers(1, min(E, 4) + 1))
        n = int(rng.integers(1, 7))
        # counts summing to n*k, each at most n (a position picks an expert once)
        cnt = np.zeros(E, dtype=int)
        for _t in range(n):
            cnt[rng.choice(E, size=k, replace=False)] += 1
        tau = float(rng.choice([0.3, 0.5, 0.75, 0.9, 0.95, 0.99, 1.0]))
        ranked, slen = oracle.plan_support(cnt, k, tau, n)
        if tau >= 1.0:
            assert slen == E
            continue
        T = math.ceil(tau * n * k)
        best = None
        for m in range(0, E + 1):
            for comb in itertools.combinations(range(E), m):
                if sum(cnt[e] for e in comb) >= T:
                    key = (m, -sum(cnt[e] for e in comb), comb)
                    if best is None or key < best:
                        best = key
        m_star = best[0]
        assert slen == min(max(m_star, k), E)
        S = set(ranked[:slen].tolist())
        if slen == m_star:
            assert S == set(best[2])
        # the support is closed upward in (count desc, id asc)
        for a in S:
            for b in set(range(E)) - S:
                assert (cnt[a], -a) > (cnt[b], -b)


def test_near_tie_detects_close_logits():
    g = np.array([1.0, 0.5, 0.5 + 5e-6, -1.0])
    assert oracle.near_tie(g, np.ones(4, bool), 2)
    assert not oracle.near_tie(np.array([3.0, 2.0, 1.0, 0.0]), np.ones(4, bool), 2)


# ------------------------------------------------------------------ liveness schedules

@pytest.mark.parametrize("sched", load_schedules(), ids=lambda s: s["name"])
def test_fresh_schedules_golden(sched):
    N = len(sched["steps"][0]["decoded"])
    lay, *_ = tiny_layer(E=5, H=4, I=3, k=2, tau=1.0, R=sched["R"], max_positions=N)
    rng = np.random.default_rng(5)
    x = rng.normal(size=(N, 4))
    lay.plan_block(x)
    for st in sched["steps"]:
        dec = np.array(st["decoded"], dtype=np.uint8)
        res = lay.iterate(x + 0.01 * st["i"], 1 - dec, dec, st["i"])
        assert list(res.fresh_pos) == st["fresh"], (sched["name"], st)
        assert int(res.fallback) == st["fallback"], (sched["name"], st)
        cl = res.classified
        assert [cl.n_live, cl.n_new, cl.n_miss, cl.n_stale, cl.n_forced, cl.n_reuse] == st["cats"], (sched["name"], st)


# ------------------------------------------------------------------ dense special case

def masked_dense(x, wr, b, experts, k, shared=(), eligible=None):
    """Every expert on every token, combined with a [N, E] weight matrix that is
    zero outside each token's brute-force top-k (over `eligible`, default all)."""
    G = x @ wr.T + b
    N, E = G.shape
    elig = np.ones(E, bool) if eligible is None else np.asarray(eligible, bool)
    Wt = np.zeros((N, E))
    for t in range(N):
        s = sorted(brute_topk(G[t], elig, k))
        ex = np.exp(G[t, s] - G[t, s].max())
        Wt[t, s] = ex / ex.sum()
    y = np.zeros_like(x)
    for e in range(E):
        wg, wu, wd = experts[e]
        h = x @ wg.T
        y += Wt[:, e:e + 1] * (((h / (1 + np.exp(-h))) * (x @ wu.T)) @ wd.T)
    for wg, wu, wd in shared:
        h = x @ wg.T
        y += ((h / (1 + np.exp(-h))) * (x @ wu.T)) @ wd.T
    return y


@pytest.mark.parametrize("n_shared", [0, 1])
def test_tau1_R1_equals_dense_moe(n_shared):
    """tau = 1 and refresh period 1: every position fresh, every expert eligible,
    so each iteration equals the dense MoE layer."""
    N, H, E, I, k = 12, 6, 7, 5, 3
    lay, wr, b, experts, shared = tiny_layer(E=E, H=H, I=I, k=k, tau=1.0, R=1,
                                             n_shared=n_shared, seed=3, max_positions=N)
    rng = np.random.default_rng(4)
    x = rng.normal(size=(N, H))
    lay.plan_block(x)
    dec = np.zeros(N, np.uint8)
    for i in range(6):
        dec[rng.choice(N, size=2, replace=False)] = 1
        xi = x + 0.05 * rng.normal(size=(N, H))
        res = lay.iterate(xi, 1 - dec, dec, i)
        assert res.fresh_pos.size == N
        np.testing.assert_allclose(res.y, masked_dense(xi, wr, b, experts, k, shared),
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(
            res.y, oracle.dense_moe(xi, wr, b, lambda e: experts[e], E, k, shared),
            rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ invariants

def run_random_block(E=8, H=6, I=5, k=2, tau=0.7, R=3, N=24, iters=10, seed=7, n_shared=1):
    lay, wr, b, experts, shared = tiny_layer(E=E, H=H, I=I, k=k, tau=tau, R=R, n_shared=n_shared,
                                             seed=seed, max_positions=N)
    rng = np.random.default_rng(seed + 100)
    x = rng.normal(size=(N, H))
    plan = lay.plan_block(x)
    dec = np.zeros(N, np.uint8)
    history = []
    for i in range(iters):
        res = lay.iterate(x, 1 - dec, dec, i)
        history.append((i, dec.copy(), x.copy(), res, lay.stamp.copy()))
        live = np.nonzero(dec == 0)[0]
        if live.size:
            dec[rng.choice(live, size=min(3, live.size), replace=False)] = 1
        x = x + 0.05 * rng.normal(size=(N, H))
    return lay, plan, history, (wr, b, experts, shared)


def test_iteration_invariants():
    k, R = 2, 3
    lay, plan, hist, (wr, b, experts, shared) = run_random_block(k=k, R=R)
    S = set(plan.support.tolist())
    prev_dec = np.zeros_like(hist[0][1])
    last_fresh = {}
    for i, dec, x, res, stamp in hist:
        fresh = set(res.fresh_pos.tolist())
        live = set(np.nonzero(dec == 0)[0].tolist())
        new = set(np.nonzero((dec == 1) & (prev_dec == 0))[0].tolist())
        assert live <= fresh                      # a live position never reads the cache
        assert new <= fresh                       # newly decoded rows are fresh once
        assert res.n_edges == k * len(fresh)      # worklist length = k |F|
        assert res.offsets[-1] == res.n_edges
        assert not res.fallback
        assert set(res.wl_expert.tolist()) <= S   # only support experts are eligible
        pairs = list(zip(res.wl_expert.tolist(), res.wl_pos.tolist()))
        assert all(a < b_ for a, b_ in zip(pairs, pairs[1:]))  # (expert, position) strictly ordered
        np.testing.assert_allclose(res.w.sum(axis=1), 1.0, rtol=1e-14)
        for t in range(len(dec)):
            if t in fresh:
                last_fresh[t] = (i, res.routed[t].copy())
            else:
                j, row = last_fresh[t]
                assert 1 <= i - j <= R - 1        # bounded age of reused rows
                assert np.array_equal(res.routed[t], row)  # the cached routed output, unchanged
        prev_dec = dec


def test_block_outputs_equal_restricted_moe_at_each_rows_last_refresh():
    """Every output of a block, reused rows included: y_i[t] is the restricted
    MoE of the support evaluated on x at the iteration t was last fresh, plus
    the shared expert on x_i ([W] "Liveness-Shard Parallelism", merge
    equations), with both sides written out independently of the oracle by
    masked_dense."""
    k, R = 2, 3
    lay, plan, hist, (wr, b, experts, shared) = run_random_block(k=k, R=R)
    elig = lay.support_mask  # the block's support (no hot update in this block)
    routed_at = {}
    n_reused = 0
    for i, dec, x, res, stamp in hist:
        routed_now = masked_dense(x, wr, b, experts, k, (), eligible=elig)
        shared_now = masked_dense(x, wr, b, experts, k, shared, eligible=elig) - routed_now
        fresh = set(res.fresh_pos.tolist())
        for t in range(x.shape[0]):
            if t in fresh:
                routed_at[t] = routed_now[t]
            else:
                n_reused += 1
            np.testing.assert_allclose(res.y[t], routed_at[t] + shared_now[t], rtol=1e-11, atol=1e-11)
    assert n_reused > 0


def test_support_equal_k_selects_whole_support():
    lay, wr, b, experts, shared = tiny_layer(E=9, H=5, I=4, k=3, tau=0.05, R=2, seed=21,
                                             max_positions=10)
    rng = np.random.default_rng(22)
    x = rng.normal(size=(10, 5))
    plan = lay.plan_block(x)
    assert plan.support_len == 3
    res = lay.iterate(x, np.ones(10, np.uint8), np.zeros(10, np.uint8), 0)
    for row in res.sel:
        assert set(row.tolist()) == set(plan.support.tolist())


def test_never_refresh_all_decoded_is_pure_cache():
    N = 8
    lay, wr, b, experts, shared = tiny_layer(E=6, H=5, I=4, k=2, tau=0.8, R=None, n_shared=1,
                                             seed=31, max_positions=N)
    rng = np.random.default_rng(32)
    x = rng.normal(size=(N, 5))
    lay.plan_block(x)
    dec = np.zeros(N, np.uint8)
    lay.iterate(x, 1 - dec, dec, 0)
    dec[:] = 1
    r1 = lay.iterate(x, 1 - dec, dec, 1)        # all newly decoded: fresh
    cached = r1.routed.copy()
    for i in range(2, 5):
        xi = x + 0.1 * i
        res = lay.iterate(xi, 1 - dec, dec, i)
        assert res.n_edges == 0
        sh = sum(oracle.swiglu_expert(xi, s) for s in shared)
        np.testing.assert_allclose(res.y, cached + sh, rtol=1e-13, atol=1e-13)


def test_residual_adds_input():
    N = 6
    a, *_ = tiny_layer(seed=41, max_positions=N, residual=False, n_shared=1)
    c, *_ = tiny_layer(seed=41, max_positions=N, residual=True, n_shared=1)
    x = np.random.default_rng(42).normal(size=(N, 5))
    a.plan_block(x)
    c.plan_block(x)
    live, dec = np.ones(N, np.uint8), np.zeros(N, np.uint8)
    np.testing.assert_allclose(c.iterate(x, live, dec, 0).y, a.iterate(x, live, dec, 0).y + x,
                               rtol=1e-14, atol=1e-14)


def test_no_plan_or_skip_is_full_fresh_with_all_experts():
    N = 10
    lay, *_ = tiny_layer(E=8, k=2, tau=0.3, R=4, seed=51, max_positions=N)
    rng = np.random.default_rng(52)
    x = rng.normal(size=(N, 5))
    dec = np.zeros(N, np.uint8)
    dec[:6] = 1
    res = lay.iterate(x, 1 - dec, dec, 0)       # no plan yet
    assert res.host_fallback and res.fresh_pos.size == N
    lay.plan_block(x)
    assert lay.plan.support_len < 8
    res = lay.iterate(x, 1 - dec, dec, 0)
    assert not res.fallback
    res = lay.iterate(x, 1 - dec, dec, 1)
    assert res.fresh_pos.size == N - 6
    res = lay.iterate(x, 1 - dec, dec, 5)       # skipped iterations
    assert res.host_fallback and res.fresh_pos.size == N
    # in a fallback every expert is eligible: the selection equals the dense top-k
    G = res.G
    for f, t in enumerate(res.fresh_pos):
        assert set(res.sel[f].tolist()) == brute_topk(G[t], np.ones(8, bool), 2)


def test_both_or_neither_flag_is_treated_live():
    N = 4
    lay, *_ = tiny_layer(E=5, k=2, tau=1.0, R=None, seed=61, max_positions=N)
    x = np.random.default_rng(62).normal(size=(N, 5))
    lay.plan_block(x)
    lay.iterate(x, np.ones(N, np.uint8), np.zeros(N, np.uint8), 0)
    dec = np.array([1, 1, 1, 1], np.uint8)
    lay.iterate(x, 1 - dec, dec, 1)
    live = np.array([1, 0, 0, 0], np.uint8)      # position 0 both flags -> live -> anomaly
    res = lay.iterate(x, live, dec, 2)
    assert res.classified.bad_flags == 1 and res.fallback
    live = np.array([0, 0, 0, 0], np.uint8)
    dec2 = np.array([1, 1, 0, 1], np.uint8)      # position 2 neither -> live
    res = lay.iterate(x, live, dec2, 3)
    assert res.classified.bad_flags == 1 and 2 in res.fresh_pos.tolist()


def test_refresh_path_recomputes_every_position_over_the_support():
    """A refresh-path iteration sends every position through the fresh routed
    path with the block's support: y equals the restricted MoE computed from
    scratch, every stamp becomes this iteration, and the following iteration
    reuses the refreshed rows."""
    N, E, k = 12, 8, 2
    lay, wr, b, experts, shared = tiny_layer(E=E, H=5, I=4, k=k, tau=0.6, R=None, n_shared=1,
                                             seed=71, max_positions=N)
    rng = np.random.default_rng(72)
    x = rng.normal(size=(N, 5))
    plan = lay.plan_block(x)
    assert plan.support_len < E
    dec = np.zeros(N, np.uint8)
    for i in range(4):
        lay.iterate(x + 0.05 * i, 1 - dec, dec, i)
        dec[rng.choice(np.nonzero(dec == 0)[0], size=3, replace=False)] = 1
    x4 = x + 0.3
    res = lay.iterate(x4, 1 - dec, dec, 4, refresh=True)
    assert res.fresh_pos.size == N and not res.fallback and res.n_edges == k * N
    assert res.classified.n_reuse == 0 and res.classified.n_forced == 0
    np.testing.assert_allclose(res.y, masked_dense(x4, wr, b, experts, k, shared, eligible=lay.support_mask),
                               rtol=1e-12, atol=1e-12)
    assert np.all(lay.stamp[:N] == 4)
    x5 = x + 0.4
    res5 = lay.iterate(x5, 1 - dec, dec, 5)     # no refresh: decoded rows come from the cache
    assert set(res5.fresh_pos.tolist()) == set(np.nonzero(dec == 0)[0].tolist())
    for t in np.nonzero(dec == 1)[0]:
        assert np.array_equal(res5.routed[t], res.routed[t])


def test_hot_update_rebuilds_the_support_from_current_logits():
    """A hot-update iteration rebuilds the support with the block-plan rule from
    its own input (the same support a new block plan on that input would give)
    and keeps every cached row, stamp and decoded flag."""
    N, E, k = 16, 10, 2
    lay, wr, b, experts, shared = tiny_layer(E=E, H=5, I=4, k=k, tau=0.5, R=None, n_shared=0,
                                             seed=81, max_positions=N)
    rng = np.random.default_rng(82)
    x = rng.normal(size=(N, 5))
    lay.plan_block(x)
    old = lay.support_mask.copy()
    dec = np.zeros(N, np.uint8)
    lay.iterate(x, 1 - dec, dec, 0)
    dec[:10] = 1
    r1 = lay.iterate(x, 1 - dec, dec, 1)
    stamps = lay.stamp.copy()
    x2 = rng.normal(size=(N, 5)) * 3.0          # routing moves elsewhere
    res = lay.iterate(x2, 1 - dec, dec, 2, hot_update=True)
    ref, *_ = tiny_layer(E=E, H=5, I=4, k=k, tau=0.5, R=None, n_shared=0, seed=81, max_positions=N)
    ref.plan_block(x2)
    assert np.array_equal(lay.support_mask, ref.support_mask)
    assert not np.array_equal(lay.support_mask, old)
    assert not res.fallback
    assert set(res.wl_expert.tolist()) <= set(np.nonzero(lay.support_mask)[0].tolist())
    for t in range(10):                          # stable decoded rows: the cache, untouched
        assert t not in res.fresh_pos.tolist()
        assert np.array_equal(res.routed[t], r1.routed[t])
        assert lay.stamp[t] == stamps[t]


# ------------------------------------------------------------------ group-limited sigmoid router

def test_grouped_router_with_one_group_is_plain_topk_of_biased_sigmoid():
    """One group: the rule reduces to the top-k of sigmoid(G) + b over the
    eligible experts (brute force), weights = their sigmoid scores normalised."""
    rng = np.random.default_rng(91)
    router = oracle.Router("sigmoid_group", 1, 1)
    for trial in range(300):
        E = int(rng.integers(3, 9))
        g = rng.normal(size=E)
        b = rng.integers(-2, 3, size=E) * 0.25
        elig = rng.random(E) < 0.8
        if elig.sum() < 2:
            elig[:2] = True
        k = int(rng.integers(1, elig.sum() + 1))
        sel, w = oracle.route_position(g, b, elig, k, router)
        c = 1.0 / (1.0 + np.exp(-g)) + b
        assert set(sel.tolist()) == brute_topk(c, elig, k)
        s = 1.0 / (1.0 + np.exp(-g[sel]))
        np.testing.assert_allclose(w, s / s.sum(), rtol=1e-15)
        assert all(c[a_] > c[b_] or (c[a_] == c[b_] and a_ < b_) for a_, b_ in zip(sel, sel[1:]))


def test_grouped_router_properties():
    """Several groups: the selection is the brute-force top-k over the chosen
    groups; a chosen group (among the first topk_group) never scores below an
    unchosen one that holds an eligible expert; the chosen groups hold at least
    k eligible experts; when every group holds two eligible experts, a common
    shift of the bias leaves the selection unchanged; the weights ignore the
    bias."""
    rng = np.random.default_rng(92)
    for trial in range(300):
        n_group = int(rng.choice([2, 4]))
        gs = int(rng.choice([2, 3]))
        E = n_group * gs
        topk_group = int(rng.integers(1, n_group + 1))
        router = oracle.Router("sigmoid_group", n_group, topk_group)
        g = rng.normal(size=E)
        b = rng.normal(size=E) * 0.5
        elig = rng.random(E) < 0.7
        if elig.sum() < 2:
            elig[rng.choice(E, 2, replace=False)] = True
        k = int(rng.integers(1, min(4, elig.sum()) + 1))
        sel, w = oracle.route_position(g, b, elig, k, router)
        c = 1.0 / (1.0 + np.exp(-g)) + b
        # group scores by sorting each group's eligible scores
        score = np.full(n_group, -np.inf)
        for q in range(n_group):
            v = np.sort(c[q * gs:(q + 1) * gs][elig[q * gs:(q + 1) * gs]])[::-1]
            if v.size:
                score[q] = v[:2].sum()
        groups = set(int(e) // gs for e in sel)
        in_groups = np.array([e // gs in groups for e in range(E)])
        n_in = int(np.sum(elig & in_groups))
        assert len(sel) == k and n_in >= k
        # every group holding a selected expert is among the best-scoring groups that hold one
        best = sorted([q for q in range(n_group) if elig[q * gs:(q + 1) * gs].any()],
                      key=lambda q: (-score[q], q))
        assert groups <= set(best[:max(topk_group, len(groups))])
        chosen = oracle.chosen_groups(score, np.array([elig[q * gs:(q + 1) * gs].sum() for q in range(n_group)]),
                                      topk_group, k)
        allowed = elig & np.repeat(chosen, gs)
        assert set(sel.tolist()) == brute_topk(c, allowed, k)
        if all(elig[q * gs:(q + 1) * gs].sum() >= 2 for q in range(n_group)):
            # every group score sums two entries: a common shift keeps every order
            sel2, w2 = oracle.route_position(g, b + 0.375, elig, k, router)
            assert np.array_equal(sel, sel2)
        s = 1.0 / (1.0 + np.exp(-g[sel]))
        np.testing.assert_allclose(w, s / s.sum(), rtol=1e-15)


def test_grouped_router_layer_counts_match_selection():
    """The block plan of a grouped-router layer counts each position's
    selection with every expert eligible, and its logits carry no bias."""
    N, E, k = 10, 8, 2
    rng = np.random.default_rng(93)
    wr = rng.normal(size=(E, 5))
    b = rng.normal(size=E)
    experts = [(rng.normal(size=(4, 5)), rng.normal(size=(4, 5)), rng.normal(size=(5, 4))) for _ in range(E)]
    router = oracle.Router("sigmoid_group", 4, 2)
    lay = oracle.LayerOracle(n_experts=E, top_k=k, tau=0.8, refresh_R=None, w_router=wr, b_router=b,
                             expert=lambda e: experts[e], max_positions=N, router=router)
    x = rng.normal(size=(N, 5))
    plan = lay.plan_block(x)
    np.testing.assert_allclose(plan.G, x @ wr.T, rtol=1e-15, atol=1e-15)
    cnt = np.zeros(E, dtype=np.int64)
    for t in range(N):
        for e in oracle.route_position(x[t] @ wr.T, b, np.ones(E, bool), k, router)[0]:
            cnt[e] += 1
    assert np.array_equal(plan.counts, cnt)
    res = lay.iterate(x, np.ones(N, np.uint8), np.zeros(N, np.uint8), 0)
    for f, t in enumerate(res.fresh_pos):
        sel, w = oracle.route_position(res.G[t], b, lay.support_mask, k, router)
        assert np.array_equal(res.sel[f], sel)


# ------------------------------------------------------------------ per-request supports

def test_per_request_supports_equal_independent_layers():
    """A batch of requests, each with its own support (its own diffusion block's
    plan), gives every position the same selections and outputs as running one
    layer per request on that request's positions alone."""
    E, H, I, k, rs, n_req = 10, 5, 4, 2, 8, 3
    N = rs * n_req
    rng = np.random.default_rng(111)
    wr = rng.normal(size=(E, H))
    b = rng.normal(size=E)
    experts = [(rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I))) for _ in range(E)]
    shared = [(rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I)))]

    def make(n, request_size=None):
        return oracle.LayerOracle(n_experts=E, top_k=k, tau=0.6, refresh_R=3, w_router=wr, b_router=b,
                                  expert=lambda e: experts[e], shared=shared, max_positions=n,
                                  request_size=request_size)
    batched = make(N, rs)
    singles = [make(rs) for _ in range(n_req)]
    # requests routed to different parts of the expert set
    x = np.concatenate([rng.normal(size=(rs, H)) + 2.0 * rng.normal(size=H) for _ in range(n_req)])
    batched.plan_block(x)
    for r in range(n_req):
        singles[r].plan_block(x[r * rs:(r + 1) * rs])
        assert np.array_equal(batched.request_masks[r], singles[r].support_mask)
    assert len({tuple(m) for m in batched.request_masks}) > 1   # the supports differ
    dec = np.zeros(N, np.uint8)
    for i in range(6):
        xi = x + 0.05 * i
        res = batched.iterate(xi, 1 - dec, dec, i)
        assert not res.fallback
        sel_b = {int(t): res.sel[f].tolist() for f, t in enumerate(res.fresh_pos)}
        for r in range(n_req):
            sl = slice(r * rs, (r + 1) * rs)
            rr = singles[r].iterate(xi[sl], 1 - dec[sl], dec[sl], i)
            np.testing.assert_allclose(res.y[sl], rr.y, rtol=1e-13, atol=1e-13)
            for f, t in enumerate(rr.fresh_pos):
                assert sel_b[r * rs + int(t)] == rr.sel[f].tolist()
        live = np.nonzero(dec == 0)[0]
        if live.size:
            dec[rng.choice(live, size=min(4, live.size), replace=False)] = 1


def test_one_request_is_the_single_support():
    lay, wr, b, experts, shared = tiny_layer(E=8, k=2, tau=0.7, R=2, seed=121, max_positions=12)
    one = oracle.LayerOracle(n_experts=8, top_k=2, tau=0.7, refresh_R=2, w_router=wr, b_router=b,
                             expert=lambda e: experts[e], max_positions=12, request_size=12)
    x = np.random.default_rng(122).normal(size=(12, 5))
    lay.plan_block(x)
    one.plan_block(x)
    assert np.array_equal(lay.support_mask, one.request_masks[0])
    live, dec = np.ones(12, np.uint8), np.zeros(12, np.uint8)
    np.testing.assert_allclose(lay.iterate(x, live, dec, 0).y, one.iterate(x, live, dec, 0).y, rtol=1e-14)


# ------------------------------------------------------------------ weights without renormalisation

def test_raw_weights_hand_worked():
    """Weights kept as the router's own scores (renormalize=False), worked by hand:
    softmax router, logits log(.5, .3, .15, .05), k = 2: the selection is
    experts 0, 1 with weights .5, .3 (renormalised: .625, .375); sigmoid router
    with no bias, one group, logits 0, ln 3, -ln 3, 0, k = 2: scores .5, .75,
    .25, .5, selection 1 then 0 (the tie with 3 goes to the lower id), weights
    .75, .5 (renormalised: .6, .4)."""
    g = np.log(np.array([.5, .3, .15, .05]))
    every = np.ones(4, dtype=bool)
    sel, w = oracle.route_position(g, np.zeros(4), every, 2, oracle.Router(renormalize=False))
    assert sel.tolist() == [0, 1]
    np.testing.assert_allclose(w, [.5, .3], rtol=1e-12)
    _, w = oracle.route_position(g, np.zeros(4), every, 2, oracle.Router())
    np.testing.assert_allclose(w, [.625, .375], rtol=1e-12)
    g = np.array([0.0, np.log(3.0), -np.log(3.0), 0.0])
    sel, w = oracle.route_position(g, np.zeros(4), every, 2, oracle.Router("sigmoid_group", 1, 1, False))
    assert sel.tolist() == [1, 0]
    np.testing.assert_allclose(w, [.75, .5], rtol=1e-12)
    _, w = oracle.route_position(g, np.zeros(4), every, 2, oracle.Router("sigmoid_group", 1, 1, True))
    np.testing.assert_allclose(w, [.6, .4], rtol=1e-12)


def test_raw_softmax_weights_are_the_topk_routing_mass():
    """Softmax router without renormalisation: the k weights add up to the k
    largest dense router probabilities (sorted independently here), all
    experts selected gives the renormalised weights, and a restricted
    selection keeps each expert's dense probability."""
    rng = np.random.default_rng(131)
    raw = oracle.Router(renormalize=False)
    for _ in range(50):
        E, k = int(rng.integers(2, 12)), 0
        k = int(rng.integers(1, E + 1))
        g = rng.normal(size=E) * 2
        every = np.ones(E, dtype=bool)
        p = np.exp(g) / np.sum(np.exp(g))
        _, w = oracle.route_position(g, np.zeros(E), every, k, raw)
        assert abs(np.sum(w) - np.sum(np.sort(p)[::-1][:k])) < 1e-12
        _, wk = oracle.route_position(g, np.zeros(E), every, E, raw)
        _, wn = oracle.route_position(g, np.zeros(E), every, E, oracle.Router())
        np.testing.assert_allclose(wk, wn, rtol=1e-12)
        mask = rng.random(E) < 0.6
        if mask.sum() >= k:
            sel, w = oracle.route_position(g, np.zeros(E), mask, k, raw)
            np.testing.assert_allclose(w, p[sel], rtol=1e-12)


# ------------------------------------------------------------------ support-coverage shortfall

def _coverage_layer(alpha, q, support, experts=4):
    """G = x (identity router, no bias), SwiGLU experts of a fixed seed, the
    support set by hand."""
    rng = np.random.default_rng(141)
    ex = [(rng.normal(size=(3, experts)), rng.normal(size=(3, experts)), rng.normal(size=(experts, 3)))
          for _ in range(experts)]
    lay = oracle.LayerOracle(n_experts=experts, top_k=1, tau=1.0, refresh_R=None, w_router=np.eye(experts),
                             b_router=np.zeros(experts), expert=lambda e: ex[e], max_positions=2,
                             coverage=(alpha, q))
    x = np.log(np.array([[.1, .2, .6, .1], [.7, .1, .1, .1]]))
    lay.plan_block(x)
    lay.adopt_support(np.array(support), len(support))
    return lay, x


def test_coverage_shortfall_hand_worked():
    """Support {0, 1}, top-1, two fresh positions with router probabilities
    (.1, .2, .6, .1) and (.7, .1, .1, .1): the first one's dense choice (expert
    2, mass .6) lies outside the support (covered 0 < alpha * .6), the second's
    inside. One of two under-covered: with q = .6 more than (1 - q) * 2 = .8
    positions are, so the support falls short and the next iteration is full
    fresh with every expert eligible (the first position then takes expert 2);
    with q = .4 the bound is 1.2 and nothing changes. Worked by hand from the
    definitions of the "Expert Atlas" and lifecycle sections."""
    live, dec = np.ones(2, np.uint8), np.zeros(2, np.uint8)
    lay, x = _coverage_layer(0.5, 0.6, [0, 1])
    r0 = lay.iterate(x, live, dec, 0)
    assert r0.n_under == 1 and lay.shortfall and not r0.fallback
    assert r0.sel[:, 0].tolist() == [1, 0]          # restricted to the support
    r1 = lay.iterate(x, live, dec, 1)
    assert r1.shortfall_prev and r1.fallback and not r1.host_fallback
    assert r1.sel[:, 0].tolist() == [2, 0]          # every expert eligible
    lay, x = _coverage_layer(0.5, 0.4, [0, 1])
    lay.iterate(x, live, dec, 0)
    assert not lay.shortfall
    assert not lay.iterate(x, live, dec, 1).fallback


def test_coverage_shortfall_special_cases():
    """alpha = 0 never falls short; a support of every expert covers every
    position; a new block plan clears a pending shortfall."""
    live, dec = np.ones(2, np.uint8), np.zeros(2, np.uint8)
    lay, x = _coverage_layer(0.0, 1.0, [0])
    lay.iterate(x, live, dec, 0)
    assert not lay.shortfall
    lay, x = _coverage_layer(1.0, 1.0, [0, 1, 2, 3])
    assert lay.iterate(x, live, dec, 0).n_under == 0 and not lay.shortfall
    lay, x = _coverage_layer(0.5, 1.0, [0])
    lay.iterate(x, live, dec, 0)
    assert lay.shortfall
    lay.plan_block(x)
    assert not lay.shortfall


# ------------------------------------------------------------------ Expert Atlas planner

def test_atlas_hand_worked_example():
    """Three tokens, four experts, k = 1, m = 1, B = 1, alpha = 1, q = 1, beta = 1,
    c = 1, logits = log of these router probabilities:
        t0 [.5 .3 .1 .1]  candidates e0 (.5), e1 (.3)  floor .5
        t1 [.1 .6 .2 .1]  candidates e1 (.6), e2 (.2)  floor .6
        t2 [.1 .1 .2 .6]  candidates e3 (.6), e2 (.2)  floor .6
    Popularity e0 .5, e1 .9, e2 .4, e3 .6 -> S = {e1}; covered t0 .3, t1 .6, t2 0,
    so U = {t0, t2}. Round 1: e0: G = min(.5, .2) = .2, H = 1 (.3 + .5 >= .5),
    score 1.2; e2: G = .2, H = 0, score .2; e3: G = .6, H = 1 (0 + .6 >= .6),
    score 1.6 -> e3 joins. U = {t0}. Round 2: e0 scores 1.2 -> joins; U empty.
    Worked by hand from the formulas of the "Expert Atlas" section."""
    P = np.array([[.5, .3, .1, .1], [.1, .6, .2, .1], [.1, .1, .2, .6]])
    res = oracle.atlas_support(np.log(P), k=1, m=1, B=1, alpha=1.0, q=1.0, beta=1.0, c=1)
    assert res.support.tolist() == [1, 3, 0]
    assert res.rounds == 2 and res.covered_ok and res.n_under == 0
    np.testing.assert_allclose(res.popularity, [.5, .9, .4, .6], rtol=1e-12)


def _atlas_under(G, k, m, alpha, support):
    """|U| for a support, recomputed with vectorised numpy."""
    E = G.shape[1]
    P = np.exp(G - G.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    order = np.lexsort((np.broadcast_to(np.arange(E), G.shape), -G), axis=1)[:, :k + m]
    W = np.take_along_axis(P, order, axis=1)
    inside = np.isin(order, support)
    return int(np.sum((W * inside).sum(axis=1) < alpha * W[:, :k].sum(axis=1)))


def test_atlas_special_cases_and_invariants():
    rng = np.random.default_rng(101)
    for trial in range(60):
        N, E = int(rng.integers(4, 40)), int(rng.integers(4, 20))
        k = int(rng.integers(1, min(4, E) + 1))
        m = int(rng.integers(0, 4))
        B = int(rng.integers(1, E + 1))
        alpha, q = float(rng.uniform(0.3, 1.0)), float(rng.uniform(0.5, 1.0))
        beta, c = float(rng.uniform(0.1, 2.0)), int(rng.integers(1, 4))
        G = rng.normal(size=(N, E)) * 2
        res = oracle.atlas_support(G, k, m, B, alpha, q, beta, c)
        sup = res.support.tolist()
        assert len(set(sup)) == len(sup) and len(sup) >= min(k, E)
        assert len(sup) <= min(max(B, k), E) + c * res.rounds
        n_under = _atlas_under(G, k, m, alpha, sup)
        assert n_under == res.n_under
        assert res.covered_ok == (n_under <= (1 - q) * N)
        # no floor: the B most popular experts, nothing repaired
        r0 = oracle.atlas_support(G, k, m, B, 0.0, q, beta, c)
        P = np.exp(G - G.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        order = np.lexsort((np.broadcast_to(np.arange(E), G.shape), -G), axis=1)[:, :min(k + m, E)]
        pop = np.zeros(E)
        np.add.at(pop, order.ravel(), np.take_along_axis(P, order, axis=1).ravel())
        top = sorted(range(E), key=lambda e: (-pop[e], e))[:max(B, k)]
        assert r0.rounds == 0 and set(r0.support.tolist()) == set(top)
        # every expert from the start: nothing under-covered
        rall = oracle.atlas_support(G, k, m, E, alpha, q, beta, c)
        assert rall.rounds == 0 and rall.n_under == 0 and len(rall.support) == E


# ------------------------------------------------------------------ mutations

def _pins_pass():
    """Run the pins that do not depend on fixtures' parametrisation."""
    checks = [test_gate_golden, test_silu_closed_forms, test_swiglu_golden, test_softmax_closed_form,
              test_topk_golden, test_topk_bruteforce, test_plan_golden,
              test_plan_minimal_support_bruteforce, test_iteration_invariants,
              lambda: test_tau1_R1_equals_dense_moe(1),
              lambda: [test_fresh_schedules_golden(s) for s in load_schedules()],
              test_grouped_router_with_one_group_is_plain_topk_of_biased_sigmoid,
              test_grouped_router_properties, test_grouped_router_layer_counts_match_selection,
              test_refresh_path_recomputes_every_position_over_the_support,
              test_hot_update_rebuilds_the_support_from_current_logits,
              test_atlas_hand_worked_example, test_atlas_special_cases_and_invariants,
              test_per_request_supports_equal_independent_layers, test_one_request_is_the_single_support,
              test_raw_weights_hand_worked, test_raw_softmax_weights_are_the_topk_routing_mass,
              test_coverage_shortfall_hand_worked, test_coverage_shortfall_special_cases]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


def _mut_rank_desc_ids(g_row, eligible):
    ids = np.nonzero(eligible)[0]
    return ids[np.lexsort((-ids, -g_row[ids]))]


def _mut_gate_no_bias(x, w, b):
    return x @ w.T


def _mut_silu_sign(z):
    return z / (1.0 + np.exp(z))


def _mut_swiglu_swapped(X, w):
    wg, wu, wd = w
    return (silu_orig(X @ wu.T) * (X @ wg.T)) @ wd.T


silu_orig = om.silu


def _mut_softmax_unnormalised(g):
    return np.exp(g - np.max(g))


def _mut_plan_off_by_one(cnt, k, tau, n_pos):
    ranked, slen = PLAN_ORIG(cnt, k, tau, n_pos)
    return ranked, min(slen + 1, len(cnt)) if tau < 1.0 else slen


PLAN_ORIG = om.plan_support


def _mut_stale_strict(live, decoded, prev, stamp, i, R, force):
    return CLASSIFY_ORIG(live, decoded, prev, stamp, i, None if R is None else R + 1, force)


CLASSIFY_ORIG = om.classify_positions


def _mut_forced_counted_as_reuse(live, decoded, prev, stamp, i, R, force):
    """Same fresh set, but positions a fallback made fresh are tallied as reused."""
    cl = CLASSIFY_ORIG(live, decoded, prev, stamp, i, R, force)
    return dataclasses.replace(cl, n_forced=0, n_reuse=cl.n_reuse + cl.n_forced)


def _mut_group_top1(c, eligible, n_group):
    E = c.shape[0]
    gs = E // n_group
    out = np.full(n_group, -np.inf)
    for g in range(n_group):
        vals = [c[e] for e in range(g * gs, (g + 1) * gs) if eligible[e]]
        if vals:
            out[g] = max(vals)
    return out


def _mut_groups_ignore_k(scores, n_elig, topk_group, k):
    return CHOSEN_ORIG(scores, n_elig, topk_group, 0)


CHOSEN_ORIG = om.chosen_groups


def _mut_weights_always_renormalised(g_row, sel, router):
    return SELW_ORIG(g_row, sel, oracle.Router(router.kind, router.n_group, router.topk_group, True))


SELW_ORIG = om.selection_weights


def _mut_raw_over_selection(g_row):
    return np.ones_like(g_row) / g_row.shape[0]


def _mut_shortfall_q_swapped(self, G, fresh_pos):
    alpha, q = self.coverage
    self.coverage = (alpha, 1.0 - q)
    try:
        return SHORT_ORIG(self, G, fresh_pos)
    finally:
        self.coverage = (alpha, q)


SHORT_ORIG = om.LayerOracle.coverage_shortfall


def _mut_sigmoid_neg(z):
    return 1.0 / (1.0 + np.exp(z))


@pytest.mark.parametrize("name,attr,mutant", [
    ("tie to higher id", "rank_eligible", _mut_rank_desc_ids),
    ("dropped router bias", "gate_logits", _mut_gate_no_bias),
    ("wrong sign in silu", "silu", _mut_silu_sign),
    ("gate/up swapped", "swiglu_expert", _mut_swiglu_swapped),
    ("weights not renormalised", "renorm_softmax", _mut_softmax_unnormalised),
    ("support one too long", "plan_support", _mut_plan_off_by_one),
    ("refresh one iteration late", "classify_positions", _mut_stale_strict),
    ("fallback positions tallied as reused", "classify_positions", _mut_forced_counted_as_reuse),
    ("group score from the best expert only", "group_scores", _mut_group_top1),
    ("groups not extended to k eligible experts", "chosen_groups", _mut_groups_ignore_k),
    ("sigmoid of -G", "sigmoid", _mut_sigmoid_neg),
    ("raw weights renormalised anyway", "selection_weights", _mut_weights_always_renormalised),
    ("dense probabilities replaced by a uniform", "dense_probabilities", _mut_raw_over_selection),
])
def test_planted_mistakes_are_caught(monkeypatch, name, attr, mutant):
    assert _pins_pass()
    monkeypatch.setattr(om, attr, mutant)
    monkeypatch.setattr(oracle, attr, mutant)
    assert not _pins_pass(), f"no pin caught: {name}"


def test_planted_shortfall_mistake_is_caught(monkeypatch):
    """The coverage bound taken as q |F| instead of (1 - q) |F|."""
    assert _pins_pass()
    monkeypatch.setattr(om.LayerOracle, "coverage_shortfall", _mut_shortfall_q_swapped)
    assert not _pins_pass(), "no pin caught: shortfall bound with q and 1 - q swapped"
