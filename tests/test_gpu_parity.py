"""GPU parity: the sm_103a library against the float64 oracle, through the C ABI.

Every workload shape of the synthetic suite, full blocks where the oracle
finishes in seconds, plus edge cases: ragged position counts, an empty
worklist, every fallback path, malformed flags, determinism and the bounded
device wait.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_harness import (block_parity, device_weights, layer_for_workload, oracle_layer, payload_to_torch,
                            scenario_parity)

pytestmark = pytest.mark.gpu

TINY_BF16 = synth.WORKLOADS["tiny_fp32"].replace(
    name="tiny_bf16", wid=6, iid=6, dtype="bf16", n_shared=1, batch=3, iters=10, refresh_R=3,
    description="tiny bf16 layer with a shared expert: H256 E16 I128 top2, 3x32 positions")


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_layer_gate_gb300 import builder
    if builder.is_stale():
        builder.build()


def assert_clean(rep):
    assert not rep.mismatches, "\n".join(rep.mismatches[:20])
    if rep.near_ties:
        print(f"{len(rep.near_ties)} near-tie(s) logged: " + "; ".join(rep.near_ties[:5]))
    print(f"iterations {rep.iterations}, edges {rep.edges}, max rel err {rep.max_rel_err:.3g}")


def test_tiny_fp32_block():
    assert_clean(block_parity(synth.WORKLOADS["tiny_fp32"]))


def test_tiny_bf16_block_tcgen05():
    assert_clean(block_parity(TINY_BF16))


def test_llada_moe_7b_block():
    assert_clean(block_parity(synth.WORKLOADS["llada_moe_7b"]))


def test_llada2_mini_block():
    rep = block_parity(synth.WORKLOADS["llada2_mini"])
    assert_clean(rep)
    assert rep.iterations == 32


def test_llada2_flash_stack_of_four():
    """The whole block of all four layers: cold path, one commit per block per
    iteration, the R = 8 refreshes, and the late iterations where most
    positions reuse their cached rows."""
    rep = block_parity(synth.WORKLOADS["llada2_flash_x4"])
    assert_clean(rep)
    assert rep.iterations == 4 * 32


# The sweep on the LLaDA2.0-mini-shaped layer: at every batch, every tau and
# every R at least once, each over a whole 32-iteration block (the live
# fraction falls from 100% to 0%). The remaining points of the 4 x 4 x 3 grid
# run when EPOCH_FULL_SWEEP=1.
SWEEP_POINTS = [(1, 0.9, 1), (1, 0.95, 4), (1, 0.99, None), (1, 1.0, 1),
                (4, 0.9, 4), (4, 0.95, None), (4, 0.99, 1), (4, 1.0, 4),
                (16, 0.9, None), (16, 0.95, 1), (16, 0.99, 4), (16, 1.0, None),
                (64, 0.9, 1), (64, 0.95, 4), (64, 0.99, None), (64, 1.0, 1)]
SWEEP_REST = [(b, t, r) for b in (1, 4, 16, 64) for t in (0.9, 0.95, 0.99, 1.0) for r in (1, 4, None)
              if (b, t, r) not in SWEEP_POINTS]
_SWEEP_WEIGHTS = {}


def _sweep_parity(batch, tau, R):
    wl = synth.sweep_workload(batch, tau, R)
    if "w" not in _SWEEP_WEIGHTS:  # every point has the same layer weights
        _SWEEP_WEIGHTS["w"] = device_weights(wl)
    lay = layer_for_workload(wl, weights=_SWEEP_WEIGHTS["w"])
    rep = block_parity(wl, layers=[lay])
    lay.close()
    assert_clean(rep)
    assert rep.iterations == 32


@pytest.mark.parametrize("batch,tau,R", SWEEP_POINTS)
def test_sweep_points(batch, tau, R):
    _sweep_parity(batch, tau, R)


@pytest.mark.skipif(os.environ.get("EPOCH_FULL_SWEEP") != "1", reason="full grid: set EPOCH_FULL_SWEEP=1")
@pytest.mark.parametrize("batch,tau,R", SWEEP_REST)
def test_sweep_rest_of_grid(batch, tau, R):
    _sweep_parity(batch, tau, R)


def test_boundary_outputs_support_and_stats():
    """The support comes out of epoch_plan_block and the statistics out of
    epoch_moe_iter (device outputs, no host synchronisation inside the calls);
    both match the oracle."""
    wl = TINY_BF16
    lay = layer_for_workload(wl)
    orc = oracle_layer(wl)
    xs, live, dec = _steps_from(wl, 4)
    E = wl.n_experts
    ids = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    slen = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay.plan_block(payload_to_torch(xs[0], wl.dtype, lay.device), support_ids=ids, support_len=slen)
    from sparse_moe_layer_gate_gb300 import binding as B
    stats = [torch.full((len(B.STATS_FIELDS),), -7, dtype=torch.int32, device="cuda") for _ in range(4)]
    for i in range(4):
        lay.moe_iter(payload_to_torch(xs[i], wl.dtype, lay.device), torch.from_numpy(live[i]).cuda(),
                     torch.from_numpy(dec[i]).cuda(), i, stats=stats[i])
    torch.cuda.synchronize()
    op = orc.plan_block(synth.to_f64(xs[0], wl.dtype))
    n = int(slen.item())
    assert n == op.support_len
    assert ids.cpu().numpy().tolist() == op.ranked.tolist()
    for i in range(4):
        res = orc.iterate(synth.to_f64(xs[i], wl.dtype), live[i], dec[i], i)
        st = lay.stats_dict(stats[i])
        cl = res.classified
        want = dict(iteration=i, n_pos=wl.n_pos, n_live=cl.n_live, n_new=cl.n_new, n_miss=cl.n_miss,
                    n_stale=cl.n_stale, n_forced=cl.n_forced, n_reuse=cl.n_reuse, n_fresh=len(res.fresh_pos),
                    n_edges=res.n_edges, n_hit_experts=int(np.count_nonzero(np.diff(res.offsets))),
                    support_len=n, fallback=0, bad_flags=0)
        assert {k: st[k] for k in want} == want, (i, st, want)
    assert lay.stats() == lay.stats_dict(stats[3])  # the synchronising read agrees
    lay.close()


def test_every_expert_eligible_at_2048_positions():
    """tau = 1 keeps all 256 experts over 2048 positions: every expert is a
    candidate and each candidate's selection words span two 32-word blocks."""
    assert_clean(block_parity(synth.sweep_workload(64, 1.0, 4), n_iters=2))


def test_multi_wave_gate_uses_the_worklist_kernel():
    """4096 positions: the gate's clusters no longer fit in one wave, so the
    gate cannot build the worklist behind its grid barrier; the worklist
    kernel builds it (copying the rows for the tensor-core experts) on the
    normal iteration path."""
    wl = synth.sweep_workload(128, 0.95, 4).replace(name="mini_4096_positions", iters=3)
    lay = layer_for_workload(wl)
    lay.set_profiling(True)
    assert_clean(block_parity(wl, n_iters=3, layers=[lay]))
    prof = lay.read_profile()
    lay.set_profiling(False)
    assert prof.get("routing", {}).get("launches", 0) == 3, prof
    lay.close()


def test_wide_router_320_experts():
    """E = 320 > 256: the gate's wider per-lane top-k and larger partial-sum
    tiles (three 128-expert MMA blocks per tile)."""
    wl = TINY_BF16.replace(name="tiny_bf16_e320", wid=7, iid=7, n_experts=320, top_k=4, tau=0.8, iters=4,
                           description="tiny bf16 layer with 320 routed experts, top-4")
    assert_clean(block_parity(wl))


def test_exact_ties_break_to_lower_expert_id():
    """x = 0 makes every logit exactly its bias on both sides; a bias in groups
    of equal values then puts exact ties inside every top-k (plan and
    iterations), and each must go to the lower expert id, with no near-tie
    allowance. Covers one expert per lane (E = 16) and eight per lane
    (E = 256, ties within and across lanes)."""
    for wl in (TINY_BF16.replace(name="tiny_bf16_ties", top_k=4, tau=1.0, bias_levels=3, iters=3),
               TINY_BF16.replace(name="e256_ties", wid=8, n_experts=256, top_k=8, tau=1.0, bias_levels=5,
                                 iters=3)):
        live, dec = synth.block_masks(wl, 3)
        x = np.zeros((wl.n_pos, wl.hidden), dtype=np.uint16)  # bf16 zeros
        steps = [dict(op="plan", x=x)] + [dict(op="iter", x=x, live=live[i], dec=dec[i], i=i) for i in range(3)]
        rep = scenario_parity(wl, steps)
        assert_clean(rep)
        assert not rep.near_ties, rep.near_ties[:5]
        assert rep.iterations == 3


@pytest.mark.parametrize("name", ["tiny_bf16", "tiny_fp32"])
def test_hot_update_and_refresh_paths(name):
    """Lifecycle paths inside a block: hot-update iterations rebuild the support
    from their own logits (once with hidden states from another block, so that
    the support moves), refresh iterations send every position through the
    fresh path; both against the oracle, and counted."""
    wl = TINY_BF16 if name == "tiny_bf16" else synth.WORKLOADS["tiny_fp32"].replace(tau=0.6, refresh_R=None)
    n_it = 8
    xs, live, dec = _steps_from(wl, n_it)
    other = synth.hidden_states(wl, 1, block=1)[0]
    paths = {3: dict(hot_update=True), 5: dict(refresh=True), 6: dict(hot_update=True, refresh=True)}
    steps = [dict(op="plan", x=xs[0])]
    for i in range(n_it):
        st = dict(op="iter", x=other if i == 3 else xs[i], live=live[i], dec=dec[i], i=i)
        st.update(paths.get(i, {}))
        steps.append(st)
    lay = layer_for_workload(wl, 0)
    rep = scenario_parity(wl, steps, layer=lay)
    assert_clean(rep)
    assert rep.iterations == n_it
    assert lay.path_counters_ex() == (2, 2)
    lay.close()


@pytest.mark.parametrize("name", ["tiny_bf16_grouped", "e256_bf16_grouped", "tiny_fp32_grouped"])
def test_group_limited_sigmoid_router(name):
    """Group-limited sigmoid router: selection on sigmoid scores plus the bias
    within the best groups, weights from the selected sigmoid scores; block
    plan counts by the same rule."""
    wl = {
        "tiny_bf16_grouped": TINY_BF16.replace(name=name, wid=9, router="sigmoid_group", n_group=4, topk_group=2,
                                               iters=6),
        "e256_bf16_grouped": TINY_BF16.replace(name=name, wid=10, n_experts=256, top_k=8, tau=0.95,
                                               router="sigmoid_group", n_group=8, topk_group=4, iters=6),
        "tiny_fp32_grouped": synth.WORKLOADS["tiny_fp32"].replace(name=name, wid=11, router="sigmoid_group",
                                                                   n_group=4, topk_group=2, iters=6),
    }[name]
    rep = block_parity(wl)
    assert_clean(rep)
    assert rep.iterations == 6


@pytest.mark.parametrize("name", ["tiny_bf16_raw", "tiny_bf16_grouped_raw", "tiny_fp32_raw", "e256_bf16_raw"])
def test_weights_without_renormalisation(name):
    """Routing weights kept as the router's own scores: the dense router
    probabilities of the selected experts (softmax router) or their sigmoid
    scores (group-limited router), against the oracle."""
    wl = {
        "tiny_bf16_raw": TINY_BF16.replace(name=name, raw_weights=True, iters=6),
        "tiny_bf16_grouped_raw": TINY_BF16.replace(name=name, wid=9, router="sigmoid_group", n_group=4,
                                                   topk_group=2, raw_weights=True, iters=6),
        "tiny_fp32_raw": synth.WORKLOADS["tiny_fp32"].replace(name=name, raw_weights=True, iters=6),
        "e256_bf16_raw": TINY_BF16.replace(name=name, wid=10, n_experts=256, top_k=8, tau=0.95,
                                           raw_weights=True, iters=6),
    }[name]
    rep = block_parity(wl)
    assert_clean(rep)
    assert rep.iterations == 6


@pytest.mark.parametrize("name", ["tiny_bf16_cov", "tiny_fp32_cov", "e256_bf16_grouped_cov"])
def test_support_coverage_shortfall(name):
    """The per-iteration support-coverage check: a support planned small
    (tau 0.5) under-covers many fresh positions, so some iterations fall back
    to full fresh with every expert eligible; counts, fallbacks and outputs
    against the oracle."""
    wl = {
        "tiny_bf16_cov": TINY_BF16.replace(name=name, tau=0.5, coverage=(0.6, 0.7), iters=8),
        "tiny_fp32_cov": synth.WORKLOADS["tiny_fp32"].replace(name=name, tau=0.5, coverage=(0.6, 0.7)),
        "e256_bf16_grouped_cov": TINY_BF16.replace(name=name, wid=10, n_experts=256, top_k=8, tau=0.6,
                                                   router="sigmoid_group", n_group=8, topk_group=4,
                                                   coverage=(0.7, 0.6), iters=8),
    }[name]
    layers = [layer_for_workload(wl)]
    rep = block_parity(wl, layers=layers)
    assert_clean(rep)
    assert rep.iterations == wl.iters
    layers[0].close()


@pytest.mark.parametrize("name", ["tiny_bf16_req", "e256_bf16_req", "tiny_fp32_req", "req_grouped_hot"])
def test_per_request_supports(name):
    """One block plan per request (32 positions): each request's hit counts,
    threshold and support, their union as the worklist candidates, and every
    position selecting within its own request's support; with a hot update
    for the last case."""
    if name == "req_grouped_hot":
        wl = TINY_BF16.replace(name=name, wid=9, router="sigmoid_group", n_group=4, topk_group=2, tau=0.6,
                               request_size=32)
        xs, live, dec = _steps_from(wl, 6)
        steps = [dict(op="plan", x=xs[0])]
        steps += [dict(op="iter", x=xs[i], live=live[i], dec=dec[i], i=i, hot_update=(i == 3)) for i in range(6)]
        assert_clean(scenario_parity(wl, steps))
        return
    wl = {
        "tiny_bf16_req": TINY_BF16.replace(name=name, tau=0.6, request_size=32, iters=6),
        "e256_bf16_req": TINY_BF16.replace(name=name, wid=10, n_experts=256, top_k=8, tau=0.9, request_size=32,
                                           iters=6),
        "tiny_fp32_req": synth.WORKLOADS["tiny_fp32"].replace(name=name, batch=3, tau=0.6, request_size=32),
    }[name]
    rep = block_parity(wl)
    assert_clean(rep)


@pytest.mark.parametrize("name", ["tiny_bf16_atlas", "tiny_fp32_atlas", "e256_bf16_atlas", "mini_atlas_hot"])
def test_expert_atlas_planner(name):
    """The Expert Atlas planner on the GPU: candidates, popularity, greedy
    repair rounds; the support (in entry order), coverage outcome and rounds
    against the oracle, then iterations over that support; the last case
    plans the LLaDA2.0-mini-shaped layer and rebuilds its support with a hot
    update."""
    if name == "mini_atlas_hot":
        wl = synth.WORKLOADS["llada2_mini"].replace(name=name, atlas=(4, 16, 0.9, 0.95, 0.1, 4), iters=4)
        xs, live, dec = _steps_from(wl, 4)
        steps = [dict(op="plan", x=xs[0])]
        steps += [dict(op="iter", x=xs[i], live=live[i], dec=dec[i], i=i, hot_update=(i == 2)) for i in range(4)]
        assert_clean(scenario_parity(wl, steps))
        return
    wl = {
        "tiny_bf16_atlas": TINY_BF16.replace(name=name, atlas=(2, 3, 0.8, 0.9, 0.5, 2), iters=6),
        "tiny_fp32_atlas": synth.WORKLOADS["tiny_fp32"].replace(name=name, atlas=(2, 3, 0.8, 0.9, 0.5, 2)),
        "e256_bf16_atlas": TINY_BF16.replace(name=name, wid=10, n_experts=256, top_k=8, atlas=(4, 16, 0.9, 0.95,
                                                                                               0.1, 4), iters=6),
    }[name]
    rep = block_parity(wl)
    assert_clean(rep)


def test_tau1_R1_is_dense_moe():
    """tau = 1 and R = 1: every position fresh with every expert eligible, so the
    layer equals the dense MoE formula at every iteration."""
    wl = synth.sweep_workload(1, 1.0, 1)
    lay = layer_for_workload(wl)
    xs = synth.hidden_states(wl, 6)
    live, dec = synth.block_masks(wl, 6)
    wr, b = synth.router_payload(wl)
    orc = oracle_layer(wl)
    shared = orc.shared
    lay.plan_block(payload_to_torch(xs[0], wl.dtype, lay.device))
    for i in range(6):
        x = payload_to_torch(xs[i], wl.dtype, lay.device)
        y = lay.moe_iter(x, torch.from_numpy(live[i]).cuda(), torch.from_numpy(dec[i]).cuda(), i)
        st = lay.stats()
        assert st["n_fresh"] == wl.n_pos and st["support_len"] == wl.n_experts
        x64 = synth.to_f64(xs[i], wl.dtype)
        dense = oracle.dense_moe(x64, synth.to_f64(wr, wl.dtype), b.astype(np.float64), orc.expert,
                                 wl.n_experts, wl.top_k, shared)
        yg = y.float().cpu().numpy().astype(np.float64)
        assert np.max(np.abs(yg - dense)) <= 1e-2 * np.max(np.abs(dense))
    lay.close()


def _steps_from(wl, n_iters, n_pos=None, block=0):
    xs = synth.hidden_states(wl, n_iters, block)
    live, dec = synth.block_masks(wl, n_iters, block)
    n = n_pos or wl.n_pos
    return xs[:, :n], live[:, :n], dec[:, :n]


def test_ragged_position_count():
    """45 positions: a partial chunk of 32, partial MMA token tiles and a partial block."""
    wl = TINY_BF16
    xs, live, dec = _steps_from(wl, 6, n_pos=45)
    steps = [dict(op="plan", x=xs[0])] + [dict(op="iter", x=xs[i], live=live[i], dec=dec[i], i=i)
                                          for i in range(6)]
    assert_clean(scenario_parity(wl, steps, max_positions=64))


def test_single_position():
    wl = TINY_BF16
    xs, live, dec = _steps_from(wl, 3, n_pos=1)
    steps = [dict(op="plan", x=xs[0])] + [dict(op="iter", x=xs[i], live=live[i], dec=dec[i], i=i)
                                          for i in range(3)]
    assert_clean(scenario_parity(wl, steps, max_positions=96))


def test_empty_worklist_reuses_cache():
    """Never refresh, everything decoded and stable: L = 0, y = cached rows + shared."""
    wl = TINY_BF16.replace(refresh_R=None)
    xs, _, _ = _steps_from(wl, 5)
    N = wl.n_pos
    live0, dec0 = np.ones(N, np.uint8), np.zeros(N, np.uint8)
    live1, dec1 = np.zeros(N, np.uint8), np.ones(N, np.uint8)
    steps = [dict(op="plan", x=xs[0]), dict(op="iter", x=xs[0], live=live0, dec=dec0, i=0),
             dict(op="iter", x=xs[1], live=live1, dec=dec1, i=1)]
    steps += [dict(op="iter", x=xs[i], live=live1, dec=dec1, i=i) for i in range(2, 5)]
    lay = layer_for_workload(wl)
    rep = scenario_parity(wl, steps, layer=lay)
    assert_clean(rep)
    st = lay.stats()
    assert st["n_edges"] == 0 and st["n_fresh"] == 0 and st["n_reuse"] == N
    lay.close()


def test_fallback_paths():
    """No plan, a skipped iteration, a different position count, a decoded->live
    transition and malformed flags: each iteration is full fresh with every
    expert eligible (or, for the flags, treated live) and matches the oracle."""
    wl = TINY_BF16.replace(tau=0.5)
    xs, live, dec = _steps_from(wl, 8)
    N = wl.n_pos
    steps = [dict(op="iter", x=xs[0], live=live[0], dec=dec[0], i=0),        # no plan yet
             dict(op="plan", x=xs[0]),
             dict(op="iter", x=xs[0], live=live[0], dec=dec[0], i=0),
             dict(op="iter", x=xs[1], live=live[1], dec=dec[1], i=1),
             dict(op="iter", x=xs[3], live=live[3], dec=dec[3], i=3),        # skipped 2
             dict(op="iter", x=xs[4], live=live[4], dec=dec[4], i=4)]
    anomalous_live = live[5].copy()
    anomalous_dec = dec[5].copy()
    d_idx = np.nonzero(dec[4])[0]
    anomalous_live[d_idx[0]] = 1
    anomalous_dec[d_idx[0]] = 0                                              # decoded -> live
    steps += [dict(op="iter", x=xs[5], live=anomalous_live, dec=anomalous_dec, i=5)]
    both = live[6].copy()
    both[d_idx[1]] = 1                                                       # both flags set
    steps += [dict(op="iter", x=xs[6], live=both, dec=dec[6], i=6)]
    steps += [dict(op="iter", x=xs[7][:N - 5], live=live[7][:N - 5], dec=dec[7][:N - 5], i=7)]  # n_pos differs
    steps += [dict(op="end"), dict(op="iter", x=xs[7], live=live[7], dec=dec[7], i=8)]         # after block end
    lay = layer_for_workload(wl)
    rep = scenario_parity(wl, steps, layer=lay)
    assert_clean(rep)
    counters = lay.path_counters()
    assert counters["cold"] == 1
    assert counters["fallback"] == 4  # no plan, skip, n_pos mismatch, after block end
    code, word = lay.status()
    assert word & 1  # malformed flags were reported
    lay.clear_status()
    assert lay.status() == (0, 0)
    lay.close()


def test_determinism_bitwise():
    wl = synth.WORKLOADS["llada2_mini"]
    xs = synth.hidden_states(wl, 3)
    live, dec = synth.block_masks(wl, 3)
    outs = []
    for _ in range(2):
        lay = layer_for_workload(wl)
        x0 = payload_to_torch(xs[0], wl.dtype, lay.device)
        lay.plan_block(x0)
        ys, wls = [], []
        for i in range(3):
            x = payload_to_torch(xs[i], wl.dtype, lay.device)
            y = lay.moe_iter(x, torch.from_numpy(live[i]).cuda(), torch.from_numpy(dec[i]).cuda(), i)
            ys.append(y.view(torch.int16).cpu().numpy())
            wls.append(lay.debug(wl.n_pos)["wl_pos"])
        outs.append((ys, wls))
        lay.close()
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.array_equal(a, b)
    for a, b in zip(outs[0][1], outs[1][1]):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("n_iters,hot_at", [(4, None), (5, 2)])
def test_cuda_graph_replay_matches_eager(n_iters, hot_at):
    """A block (plan + iterations) captured into a CUDA graph and replayed
    three times gives, bit for bit, the outputs of the same block run eagerly;
    an eager block after the replays still does. An odd iteration count and a
    hot-update iteration (worklist kernel instead of the gate's tail) are
    included: no per-iteration state may depend on how many calls ran before."""
    wl = synth.WORKLOADS["llada2_mini"]
    xs = synth.hidden_states(wl, n_iters)
    live, dec = synth.block_masks(wl, n_iters)
    lay = layer_for_workload(wl)
    dev = lay.device
    X = [payload_to_torch(xs[i], wl.dtype, dev) for i in range(n_iters)]
    LV = [torch.from_numpy(live[i]).to(dev) for i in range(n_iters)]
    DC = [torch.from_numpy(dec[i]).to(dev) for i in range(n_iters)]
    Y = [torch.empty_like(X[0]) for _ in range(n_iters)]

    def block():
        lay.plan_block(X[0])
        for i in range(n_iters):
            lay.moe_iter(X[i], LV[i], DC[i], i, Y[i], hot_update=(i == hot_at))
        lay.block_end()

    def outputs():
        torch.cuda.synchronize()
        return [y.view(torch.int16).cpu().numpy() for y in Y]

    block()
    eager = outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        block()
    torch.cuda.current_stream().wait_stream(side)
    assert all(np.array_equal(a, b) for a, b in zip(eager, outputs()))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        block()
    for _ in range(3):
        for y in Y:
            y.zero_()
        graph.replay()
        got = outputs()
        for i, (a, b) in enumerate(zip(eager, got)):
            assert np.array_equal(a, b), f"iteration {i} differs after a replay"
    code, word = lay.status()
    assert code == 0, word
    block()
    assert all(np.array_equal(a, b) for a, b in zip(eager, outputs()))
    lay.close()


def test_bounded_wait_times_out_and_reports():
    lay = layer_for_workload(TINY_BF16)
    lay.test_wait_timeout(2_000_000)  # 2 ms on a barrier nothing completes
    code, word = lay.status()
    assert code == 4 and word & 2
    lay.clear_status()
    # the context is still usable
    assert_clean(block_parity(TINY_BF16, n_iters=2))
    lay.close()
