"""The parity checker itself, on the CPU: GPU-side records are fabricated from
a second run of the oracle, then changed the way a faulty kernel would change
them. A checker that let one of these through would let the same mistake in
the CUDA path through.

Inputs with exact ties: x = 0 makes every router logit its bias, and the bias
comes in groups of three equal values, so the top-2 of every position is a
pick of two out of three equal experts.
"""
import numpy as np

import synth
from parity_harness import GpuStep, Report, check_iteration, check_plan, oracle_layer

TIES = synth.WORKLOADS["tiny_fp32"].replace(name="checker_ties", bias_levels=3, tau=1.0, refresh_R=None)


def _inputs(wl, n_iters=3, zero=True):
    live, dec = synth.block_masks(wl, n_iters)
    if zero:
        xs = np.zeros((n_iters, wl.n_pos, wl.hidden), dtype=np.float32)
    else:
        xs = synth.hidden_states(wl, n_iters)
    return xs, live, dec


def _record(orc, wl, x, live, dec, i, force=None):
    """What a correct device would report for iteration i, except that the
    selections in `force` ({position: experts}) replace the rule's choice."""
    def adopt(t, s, g_row, eligible):
        return None if force is None or t not in force else np.asarray(force[t])
    res = orc.iterate(synth.to_f64(x, wl.dtype), live, dec, i, adopt=adopt)
    cl = res.classified
    stats = dict(n_live=cl.n_live, n_new=cl.n_new, n_miss=cl.n_miss, n_stale=cl.n_stale, n_forced=cl.n_forced,
                 n_reuse=cl.n_reuse, n_fresh=len(res.fresh_pos), n_edges=res.n_edges,
                 fallback=(1 if res.host_fallback else 0) | (2 if cl.anomaly else 0) | (4 if res.shortfall_prev else 0),
                 bad_flags=cl.bad_flags, n_under=res.n_under)
    dbg = dict(stats=stats, fresh_pos=res.fresh_pos.copy(), sel=res.sel.copy(), sel_w=res.w.astype(np.float32),
               offsets=res.offsets.copy(), wl_pos=res.wl_pos.copy(), slot=res.slot.copy())
    return GpuStep(x, res.y.copy(), dbg)


def _plan_record(orc, x0, counts=None):
    op = orc.plan_block(x0)
    return dict(support_len=op.support_len, support_ids=op.ranked.copy(),
                plan_counts=(op.counts if counts is None else counts).copy()), op


def _run(wl, steps, plan_rec=None):
    """Checks fabricated records against a fresh oracle; returns the report."""
    xs, live, dec = steps["xs"], steps["live"], steps["dec"]
    orc = oracle_layer(wl)
    rep = Report()
    gplan = plan_rec if plan_rec is not None else _plan_record(oracle_layer(wl), synth.to_f64(xs[0], wl.dtype))[0]
    check_plan(orc, gplan, synth.to_f64(xs[0], wl.dtype), wl, rep, "t")
    for i, step in enumerate(steps["records"]):
        check_iteration(orc, step, live[i], dec[i], i, wl, rep, "t")
    return rep


def _tied_triplet(wl):
    """The three experts of bias 0, in id order, and one expert of bias -1."""
    _, b = synth.router_payload(wl)
    top = sorted(int(e) for e in np.nonzero(b == 0)[0])
    below = sorted(int(e) for e in np.nonzero(b == -1)[0])
    assert len(top) == 3 and below
    return top, below[0]


def _steps(wl, xs, live, dec, force_at=None):
    dev = oracle_layer(wl)
    dev.plan_block(synth.to_f64(xs[0], wl.dtype))
    recs = [_record(dev, wl, xs[i], live[i], dec[i], i, force=(force_at or {}).get(i)) for i in range(len(xs))]
    return dict(xs=xs, live=live, dec=dec, records=recs)


def test_correct_records_pass_without_near_ties_logged():
    wl = synth.WORKLOADS["tiny_fp32"]
    xs, live, dec = _inputs(wl, 4, zero=False)
    rep = _run(wl, _steps(wl, xs, live, dec))
    assert not rep.mismatches and not rep.near_ties
    assert rep.iterations == 4


def test_in_tie_reordering_is_logged_not_failed():
    xs, live, dec = _inputs(TIES)
    (a, b, c), _ = _tied_triplet(TIES)
    rep = _run(TIES, _steps(TIES, xs, live, dec, force_at={1: {5: [c, a]}, 2: {7: [b, c]}}))
    assert not rep.mismatches, rep.mismatches
    assert len(rep.near_ties) == 2


def test_wrong_expert_at_a_near_tied_position_fails():
    xs, live, dec = _inputs(TIES)
    (a, b, c), d = _tied_triplet(TIES)
    rep = _run(TIES, _steps(TIES, xs, live, dec, force_at={1: {5: [a, d]}}))
    assert any("selection gpu" in m for m in rep.mismatches), rep.mismatches
    rep = _run(TIES, _steps(TIES, xs, live, dec, force_at={1: {5: [a, a]}}))  # duplicate
    assert rep.mismatches


def test_wrong_expert_without_a_tie_fails():
    wl = synth.WORKLOADS["tiny_fp32"]
    xs, live, dec = _inputs(wl, 3, zero=False)
    ref = _steps(wl, xs, live, dec)
    t = int(ref["records"][1].dbg["fresh_pos"][0])
    sel = [int(e) for e in ref["records"][1].dbg["sel"][0]]
    other = next(e for e in range(wl.n_experts) if e not in sel)
    rep = _run(wl, _steps(wl, xs, live, dec, force_at={1: {t: [sel[0], other]}}))
    assert any("selection gpu" in m for m in rep.mismatches), rep.mismatches


def test_swapped_worklist_slots_fail():
    wl = synth.WORKLOADS["tiny_fp32"]
    xs, live, dec = _inputs(wl, 3, zero=False)
    steps = _steps(wl, xs, live, dec)
    slot = steps["records"][2].dbg["slot"]
    slot[0, [0, 1]] = slot[0, [1, 0]]   # the worklist itself (positions, offsets) is unchanged
    rep = _run(wl, steps)
    assert any("slots differ" in m for m in rep.mismatches), rep.mismatches


def test_plan_counts_moved_along_a_tie_are_adopted():
    wl = TIES.replace(tau=0.9)
    xs, live, dec = _inputs(wl, 1)
    x0 = synth.to_f64(xs[0], wl.dtype)
    (a, b, c), d = _tied_triplet(wl)
    gplan, op = _plan_record(oracle_layer(wl), x0)
    cnt = op.counts.copy()
    cnt[b] -= 1
    cnt[c] += 1                          # one position took c instead of b: they tie
    import oracle
    ranked, slen = oracle.plan_support(cnt, wl.top_k, wl.tau, wl.n_pos)
    ok = dict(support_len=slen, support_ids=ranked, plan_counts=cnt)
    rep = Report()
    check_plan(oracle_layer(wl), ok, x0, wl, rep, "t")
    assert not rep.mismatches and len(rep.near_ties) == 1
    # an edge moved to an expert one bias level below: no tie explains it
    bad = op.counts.copy()
    bad[b] -= 1
    bad[d] += 1
    ranked, slen = oracle.plan_support(bad, wl.top_k, wl.tau, wl.n_pos)
    rep = Report()
    check_plan(oracle_layer(wl), dict(support_len=slen, support_ids=ranked, plan_counts=bad), x0, wl, rep, "t")
    assert rep.mismatches
    # counts that a tie explains, but a support that is not their prefix
    rep = Report()
    check_plan(oracle_layer(wl), dict(support_len=slen + 1, support_ids=ok["support_ids"], plan_counts=cnt),
               x0, wl, rep, "t")
    assert rep.mismatches
