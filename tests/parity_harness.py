"""Lock-step driver comparing the CUDA layer with the float64 oracle.

The GPU runs first over the requested iterations (for a stack, layer by
layer, each fed the previous layer's output); every layer input, output and
the routing/worklist state is copied back. The oracle then replays each layer
on the GPU's own inputs (teacher forcing, so bf16 drift in one layer cannot
flip the next layer's routing) and each iteration is checked:

* fresh set, category counts, fallback flags, support, selections, worklist
  offsets and positions: bit-exact;
* worklist slots and the selection index of every worklist row: bit-exact;
* a selection that differs is accepted only when it is a reordering of the
  oracle's that rounding could produce (experts whose float64 scores lie within
  1e-5 of each other trade places; nothing else may change); the case is
  logged and the oracle adopts the GPU's selection so nothing cascades;
* a block-plan support that differs is accepted only when the GPU's hit counts
  differ from the oracle's by edges that near-tied positions could move, and
  the GPU's support is the prefix rule applied to the GPU's own counts;
* routing weights within 2e-5; y within max|dy| <= tol * max|y| (tol 1e-2 for
  bf16, 1e-5 for fp32).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

import oracle
import synth
from sparse_moe_layer_gate_gb300.layer import EpochLayer, payload_to_torch

NEAR_TIE = 1e-5


def device_weights(wl, layer_index: int = 0, device="cuda", threads: Optional[int] = None) -> dict:
    """The layer's weights drawn by synth and uploaded (CUDA tensors by name)."""
    wr, b = synth.router_payload(wl, layer_index)
    wg, wu, wd = synth.experts_payload(wl, layer_index, threads)
    weights = {
        "w_router": payload_to_torch(wr, wl.dtype, device),
        "b_router": torch.from_numpy(b).to(device),
        "w_gate": payload_to_torch(wg, wl.dtype, device),
        "w_up": payload_to_torch(wu, wl.dtype, device),
        "w_down": payload_to_torch(wd, wl.dtype, device),
    }
    del wg, wu, wd
    if wl.n_shared:
        sg, su, sd = synth.shared_experts_payload(wl, layer_index, threads)
        weights.update(ws_gate=payload_to_torch(sg, wl.dtype, device),
                       ws_up=payload_to_torch(su, wl.dtype, device),
                       ws_down=payload_to_torch(sd, wl.dtype, device))
    return weights


def layer_for_workload(wl, layer_index: int = 0, device="cuda", threads: Optional[int] = None,
                       max_positions: Optional[int] = None, weights: Optional[dict] = None) -> EpochLayer:
    """The device layer of a synth workload; `weights` reuses uploaded tensors
    (layers that differ only in tau, R or the position count share them)."""
    weights = weights if weights is not None else device_weights(wl, layer_index, device, threads)
    return EpochLayer(hidden=wl.hidden, n_experts=wl.n_experts, inter=wl.inter, top_k=wl.top_k,
                      max_positions=max_positions or wl.n_pos, dtype=wl.dtype, tau=wl.tau, refresh_R=wl.refresh_R,
                      weights=weights, n_shared=wl.n_shared, shared_inter=wl.shared_inter,
                      residual=wl.residual, router=wl.router, n_group=wl.n_group, topk_group=wl.topk_group,
                      raw_weights=wl.raw_weights, coverage=wl.coverage, request_size=wl.request_size,
                      atlas=atlas_dict(wl))


def atlas_dict(wl) -> Optional[dict]:
    """The workload's Expert Atlas parameters by name (None: the prefix rule)."""
    if wl.atlas is None:
        return None
    return dict(zip(("m", "B", "alpha", "q", "beta", "c"), wl.atlas))


def tol_for(dtype: str) -> float:
    return 1e-2 if dtype == "bf16" else 1e-5


def oracle_layer(wl, layer_index: int = 0, max_positions: Optional[int] = None) -> oracle.LayerOracle:
    wr, b = synth.router_payload(wl, layer_index)
    cache = {}

    def expert(e: int):
        if e not in cache:
            g, u, d = synth.expert_payload(wl, layer_index, e)
            cache[e] = (synth.to_f64(g, wl.dtype), synth.to_f64(u, wl.dtype), synth.to_f64(d, wl.dtype))
        return cache[e]

    shared = [tuple(synth.to_f64(p, wl.dtype) for p in synth.shared_payload(wl, layer_index, s))
              for s in range(wl.n_shared)]
    return oracle.LayerOracle(n_experts=wl.n_experts, top_k=wl.top_k, tau=wl.tau, refresh_R=wl.refresh_R,
                              w_router=synth.to_f64(wr, wl.dtype), b_router=b.astype(np.float64),
                              expert=expert, shared=shared, residual=wl.residual,
                              max_positions=max_positions or wl.n_pos,
                              router=oracle.Router(wl.router, wl.n_group, wl.topk_group, not wl.raw_weights),
                              coverage=wl.coverage, request_size=wl.request_size or None,
                              atlas=atlas_dict(wl))


def tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


@dataclasses.dataclass
class Report:
    near_ties: List[str] = dataclasses.field(default_factory=list)
    mismatches: List[str] = dataclasses.field(default_factory=list)
    max_rel_err: float = 0.0
    iterations: int = 0
    edges: int = 0


@dataclasses.dataclass
class GpuStep:
    x: np.ndarray        # layer input payload
    y: np.ndarray        # layer output (float64)
    dbg: dict


def run_gpu(wl, layers, xs_payload, live, dec, iters: List[int], plan: bool = True,
            stream=None) -> List[dict]:
    """Runs the GPU stack; returns, per layer, the plan debug and the per-iteration steps."""
    dev = layers[0].device
    rec = [dict(plan=None, steps=[]) for _ in layers]
    for ii, i in enumerate(iters):
        x = payload_to_torch(xs_payload[ii], wl.dtype, dev)
        lv = torch.from_numpy(live[ii]).to(dev)
        dc = torch.from_numpy(dec[ii]).to(dev)
        for l, lay in enumerate(layers):
            if plan and ii == 0:
                lay.plan_block(x)
                rec[l]["plan"] = lay.debug(x.shape[0], parts=("plan",))
            x_in = x.detach().clone()
            y = lay.moe_iter(x, lv, dc, i)
            dbg = lay.debug(x.shape[0], parts=("iter",))
            rec[l]["steps"].append(GpuStep(x_in.float().cpu().numpy() if wl.dtype == "f32"
                                           else x_in.view(torch.int16).cpu().numpy().view(np.uint16),
                                           tensor_to_f64(y), dbg))
            x = y
    torch.cuda.synchronize()
    return rec


# ------------------------------------------------------------------ near-tie rules
#
# A GPU result that differs from the oracle's is accepted only when the
# difference is a reordering that rounding could produce: experts whose
# float64 scores lie within NEAR_TIE of each other may trade places, nothing
# else may. Accepted cases are logged and the oracle adopts the GPU's choice so
# that nothing downstream cascades.

def selection_scores(orc, g_row: np.ndarray, eligible: np.ndarray):
    """(scores the selection ranks, experts that may be selected, whether the
    group choice itself is near-tied) for one position: the logits over the
    eligible experts (softmax router), or the selection scores
    c = sigmoid(G) + b over the eligible experts of the groups that can be
    chosen (group-limited router: a group whose score is within NEAR_TIE of the
    last chosen group's may replace it)."""
    if orc.router.kind == "softmax":
        return g_row, eligible.copy(), False
    c = oracle.sigmoid(g_row) + orc.b_router
    E, ng = g_row.shape[0], orc.router.n_group
    gs = E // ng
    scores = oracle.group_scores(c, eligible, ng)
    n_elig = np.array([int(np.sum(eligible[g * gs:(g + 1) * gs])) for g in range(ng)])
    chosen = oracle.chosen_groups(scores, n_elig, orc.router.topk_group, orc.k)
    low = np.min(scores[chosen]) if chosen.any() else np.inf
    possible = chosen | (np.isfinite(scores) & (scores >= low - NEAR_TIE))
    return c, eligible & np.repeat(possible, gs), bool(np.any(possible & ~chosen))


def valid_reordering(scores: np.ndarray, allowed: np.ndarray, mine, k: int) -> bool:
    """True when `mine` (k experts in selection order) is what an exact top-k
    of scores perturbed by at most NEAR_TIE / 2 per entry could return over the
    allowed experts: distinct, allowed, and each entry within NEAR_TIE of the
    best allowed expert not selected before it."""
    mine = [int(e) for e in mine]
    if len(mine) != k or len(set(mine)) != k:
        return False
    if any(e < 0 or e >= scores.shape[0] or not allowed[e] for e in mine):
        return False
    rest = allowed.copy()
    for e in mine:
        best = np.max(scores[rest])
        if scores[e] + NEAR_TIE < best:
            return False
        rest[e] = False
    return True


def flexible_edges(orc, G: np.ndarray):
    """Per position of a block plan (every expert eligible): the experts that
    a rounding-level change could drop from its selection and those that could
    join it. Empty for positions without a near-tie at the selection's edge;
    with a near-tied group choice every selected expert may leave and every
    expert of the possible groups may join."""
    E = G.shape[1]
    everyone = np.ones(E, dtype=bool)
    out = []
    for t in range(G.shape[0]):
        sel, _ = orc.select(G[t], everyone)
        scores, allowed, group_flip = selection_scores(orc, G[t], everyone)
        inside = np.zeros(E, dtype=bool)
        inside[sel] = True
        outside = allowed & ~inside
        if not outside.any():
            out.append((set(), set()))
            continue
        if group_flip:
            out.append(({int(e) for e in sel}, {int(e) for e in np.nonzero(outside)[0]}))
            continue
        kth = np.min(scores[sel])
        best_out = np.max(scores[outside])
        leave = {int(e) for e in sel if scores[e] <= best_out + NEAR_TIE}
        enter = {int(e) for e in np.nonzero(outside)[0] if scores[e] >= kth - NEAR_TIE}
        out.append((leave, enter) if leave and enter else (set(), set()))
    return out


def counts_explained(orc, G: np.ndarray, oracle_counts: np.ndarray, gpu_counts: np.ndarray) -> bool:
    """True when the GPU's block-plan hit counts differ from the oracle's only
    by experts leaving and joining selections at near-tied positions: every
    expert's surplus (deficit) is at most the number of positions where it
    could join (leave), and the total number of moved edges fits the
    positions' freedom."""
    D = np.asarray(gpu_counts, dtype=np.int64) - np.asarray(oracle_counts, dtype=np.int64)
    if not D.any():
        return True
    if D.sum() != 0:
        return False
    flex = flexible_edges(orc, G)
    can_join = np.zeros(D.shape[0], dtype=np.int64)
    can_leave = np.zeros(D.shape[0], dtype=np.int64)
    moves = 0
    for leave, enter in flex:
        for e in leave:
            can_leave[e] += 1
        for e in enter:
            can_join[e] += 1
        moves += min(len(leave), len(enter))
    if np.any(np.maximum(D, 0) > can_join) or np.any(np.maximum(-D, 0) > can_leave):
        return False
    return int(np.maximum(D, 0).sum()) <= moves


def _check_support(orc, op, gplan: dict, n_pos: int, rep: Report, what: str, adopt=None) -> None:
    glen = int(gplan["support_len"])
    gids = np.asarray(gplan["support_ids"])
    gcnt = np.asarray(gplan["plan_counts"])
    if glen == op.support_len and np.array_equal(gids[:glen], op.ranked[:glen]) and \
            np.array_equal(gcnt, op.counts):
        return
    if not counts_explained(orc, op.G, op.counts, gcnt):
        rep.mismatches.append(f"{what}: hit counts differ beyond near-tied edges "
                              f"(gpu len {glen}, oracle len {op.support_len})")
        return
    ranked, slen = oracle.plan_support(gcnt, orc.k, orc.tau, n_pos)
    if glen != slen or not np.array_equal(gids[:glen], ranked[:slen]):
        rep.mismatches.append(f"{what}: GPU support is not the prefix rule applied to the GPU's own counts")
        return
    moved = int(np.abs(gcnt - op.counts).sum()) // 2
    rep.near_ties.append(f"{what}: {moved} edge(s) moved at near-tied positions; adopting GPU support")
    (adopt or orc.adopt_support)(gids, glen)


def _check_atlas(orc, gplan: dict, rep: Report, what: str) -> None:
    """The Expert Atlas support: the same experts in the same entry order, and
    the same coverage outcome; a difference is accepted only when the oracle's
    run took a decision within NEAR_TIE (its smallest decision margin), and the
    GPU's support is then adopted."""
    res = orc.atlas_result
    glen = int(gplan["support_len"])
    gids = np.asarray(gplan["support_ids"])[:glen]
    ga = gplan["atlas"]
    same = (np.array_equal(gids, res.support) and ga["covered_ok"] == res.covered_ok and
            ga["n_under"] == res.n_under and ga["rounds"] == res.rounds)
    if same:
        return
    if res.min_margin <= NEAR_TIE:
        rep.near_ties.append(f"{what}: Atlas support differs at a decision margin of {res.min_margin:.2g}; "
                             "adopting GPU support")
        orc.adopt_support(gids, glen)
        return
    rep.mismatches.append(f"{what}: Atlas support gpu {gids.tolist()} oracle {res.support.tolist()} "
                          f"(covered {ga['covered_ok']}/{res.covered_ok}, under {ga['n_under']}/{res.n_under}, "
                          f"rounds {ga['rounds']}/{res.rounds})")


def _check_supports(orc, op, gplan: dict, n_pos: int, rep: Report, what: str) -> None:
    """The block's support, or with per-request supports each request's (its
    own counts, threshold and prefix) and their union, ascending."""
    if orc.atlas is not None:
        _check_atlas(orc, gplan, rep, what)
        return
    if not orc.request_size:
        _check_support(orc, op, gplan, n_pos, rep, what)
        return
    rs = orc.request_size
    for r, rp in enumerate(orc.request_plans):
        def adopt(ids, ln, r=r):
            orc.request_masks[r] = False
            orc.request_masks[r, np.asarray(ids[:ln], dtype=np.int64)] = True
        g = dict(support_len=gplan["request_len"][r], support_ids=gplan["request_ids"][r],
                 plan_counts=gplan["plan_counts"][r])
        _check_support(orc, rp, g, min(rs, n_pos - r * rs), rep, f"{what} request {r}", adopt)
        want_mask = orc.request_masks[r]
        if not np.array_equal(np.asarray(gplan["support_masks"][r], dtype=bool), want_mask):
            rep.mismatches.append(f"{what} request {r}: support mask differs")
    orc.support_mask = orc.request_masks.any(axis=0)
    union = np.nonzero(orc.support_mask)[0]
    glen = int(gplan["support_len"])
    if glen != union.size or not np.array_equal(np.asarray(gplan["support_ids"])[:glen], union):
        rep.mismatches.append(f"{what}: union of the request supports differs")


def check_plan(orc: oracle.LayerOracle, gplan: dict, x0: np.ndarray, wl, rep: Report, tag: str):
    op = orc.plan_block(x0)
    _check_supports(orc, op, gplan, x0.shape[0], rep, f"{tag} plan")
    return op


def check_hot_update(orc: oracle.LayerOracle, gplan: dict, x0: np.ndarray, wl, rep: Report, tag: str):
    """The support a hot-update iteration rebuilt (oracle.hot_update on the same
    input; near-ties as for the block plan)."""
    op = orc.hot_update(x0)
    _check_supports(orc, op, gplan, x0.shape[0], rep, f"{tag} hot update")
    return op


def check_iteration(orc, step: GpuStep, live, dec, i: int, wl, rep: Report, tag: str, refresh: bool = False):
    g = step.dbg
    gsel = {int(t): g["sel"][f] for f, t in enumerate(g["fresh_pos"])}

    def adopt(t, s, g_row, eligible):
        mine = gsel.get(t)
        if mine is None or np.array_equal(mine, s):
            return None
        scores, allowed, _ = selection_scores(orc, g_row, eligible)
        if valid_reordering(scores, allowed, mine, orc.k):
            rep.near_ties.append(f"{tag} i={i} t={t}: gpu {list(mine)} oracle {list(s)} (in-tie reordering)")
            return mine
        rep.mismatches.append(f"{tag} i={i} t={t}: selection gpu {list(mine)} oracle {list(s)}")
        return None

    x64 = synth.to_f64(step.x, wl.dtype)
    res = orc.iterate(x64, live, dec, i, adopt=adopt, refresh=refresh)
    st = g["stats"]
    cl = res.classified
    exp = dict(n_live=cl.n_live, n_new=cl.n_new, n_miss=cl.n_miss, n_stale=cl.n_stale, n_forced=cl.n_forced,
               n_reuse=cl.n_reuse, n_fresh=len(res.fresh_pos), n_edges=res.n_edges,
               fallback=(1 if res.host_fallback else 0) | (2 if cl.anomaly else 0) | (4 if res.shortfall_prev else 0),
               bad_flags=cl.bad_flags, n_under=res.n_under)
    for key, v in exp.items():
        if st[key] != v:
            rep.mismatches.append(f"{tag} i={i}: stats {key} gpu {st[key]} oracle {v}")
    if not np.array_equal(g["fresh_pos"], res.fresh_pos):
        rep.mismatches.append(f"{tag} i={i}: fresh sets differ")
        return res
    if not np.array_equal(g["sel"], res.sel):
        rep.mismatches.append(f"{tag} i={i}: selections differ after adoption")
    if not np.array_equal(g["offsets"], res.offsets):
        rep.mismatches.append(f"{tag} i={i}: worklist offsets differ")
    if not np.array_equal(g["wl_pos"], res.wl_pos):
        rep.mismatches.append(f"{tag} i={i}: worklist positions differ")
    gslot = np.asarray(g["slot"])
    if not np.array_equal(gslot, res.slot):
        rep.mismatches.append(f"{tag} i={i}: worklist slots differ")
    elif res.n_edges:
        # which of its position's k selections each worklist row is
        gj = np.full(res.n_edges, -1, dtype=np.int64)
        gj[gslot.reshape(-1)] = np.tile(np.arange(orc.k), gslot.shape[0])
        if not np.array_equal(gj, res.wl_j):
            rep.mismatches.append(f"{tag} i={i}: worklist selection indices differ")
    if res.sel.size:
        werr = float(np.max(np.abs(g["sel_w"] - res.w)))
        if werr > 2e-5:
            rep.mismatches.append(f"{tag} i={i}: routing weights differ by {werr:.3g}")
    scale = float(np.max(np.abs(res.y)))
    err = float(np.max(np.abs(step.y - res.y)))
    rel = err / scale if scale > 0 else err
    rep.max_rel_err = max(rep.max_rel_err, rel)
    if rel > tol_for(wl.dtype):
        rep.mismatches.append(f"{tag} i={i}: max|dy| = {err:.4g} = {rel:.3g} max|y| > {tol_for(wl.dtype)}")
    rep.iterations += 1
    rep.edges += res.n_edges
    return res


def block_parity(wl, n_iters: Optional[int] = None, iters: Optional[List[int]] = None,
                 layers: Optional[list] = None) -> Report:
    """Full lock-step parity of one block of workload wl (all layers)."""
    n_iters = wl.iters if n_iters is None else n_iters
    iters = list(range(n_iters)) if iters is None else iters
    n_gen = max(iters) + 1
    xs = synth.hidden_states(wl, n_gen)[iters]
    live, dec = synth.block_masks(wl, n_gen)
    live, dec = live[iters], dec[iters]
    own = layers is None
    if own:
        layers = [layer_for_workload(wl, l) for l in range(wl.layers)]
    rec = run_gpu(wl, layers, xs, live, dec, iters)
    if own:
        for lay in layers:
            lay.close()
        del layers
        torch.cuda.empty_cache()
    rep = Report()
    for l in range(wl.layers):
        orc = oracle_layer(wl, l)
        tag = f"{wl.name} layer {l}"
        check_plan(orc, rec[l]["plan"], synth.to_f64(rec[l]["steps"][0].x, wl.dtype), wl, rep, tag)
        for ii, i in enumerate(iters):
            check_iteration(orc, rec[l]["steps"][ii], live[ii], dec[ii], i, wl, rep, tag)
        del orc
    return rep


def scenario_parity(wl, steps, max_positions: Optional[int] = None, layer=None) -> Report:
    """Interleaved GPU/oracle run of an explicit call sequence on one layer.

    steps: dicts with "op" in {"plan", "iter", "end"}; "plan" takes "x" (payload
    [n, H]); "iter" takes "x", "live", "dec" (uint8 [n]) and "i", and optionally
    "hot_update" / "refresh" (the lifecycle path of the iteration).
    """
    maxp = max_positions or wl.n_pos
    lay = layer or layer_for_workload(wl, 0, max_positions=maxp)
    orc = oracle_layer(wl, 0, max_positions=maxp)
    dev = lay.device
    rep = Report()
    for n, st in enumerate(steps):
        tag = f"{wl.name} step {n}"
        if st["op"] == "plan":
            x = payload_to_torch(st["x"], wl.dtype, dev)
            lay.plan_block(x)
            gplan = lay.debug(x.shape[0], parts=("plan",))
            check_plan(orc, gplan, synth.to_f64(st["x"], wl.dtype), wl, rep, tag)
        elif st["op"] == "end":
            lay.block_end()
            orc.block_end()
        else:
            x = payload_to_torch(st["x"], wl.dtype, dev)
            lv = torch.from_numpy(np.ascontiguousarray(st["live"], dtype=np.uint8)).to(dev)
            dc = torch.from_numpy(np.ascontiguousarray(st["dec"], dtype=np.uint8)).to(dev)
            hu, rf = bool(st.get("hot_update")), bool(st.get("refresh"))
            y = lay.moe_iter(x, lv, dc, st["i"], hot_update=hu, refresh=rf)
            dbg = lay.debug(x.shape[0], parts=("plan", "iter") if hu else ("iter",))
            step = GpuStep(st["x"], tensor_to_f64(y), dbg)
            if hu:
                check_hot_update(orc, dbg, synth.to_f64(st["x"], wl.dtype), wl, rep, tag)
            check_iteration(orc, step, st["live"], st["dec"], st["i"], wl, rep, tag, refresh=rf)
    if layer is None:
        lay.close()
    return rep
