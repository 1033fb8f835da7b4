"""Lock-step driver comparing the CUDA layer with the float64 oracle.

The GPU runs first over the requested iterations (for a stack, layer by
layer, each fed the previous layer's output); every layer input, output and
the routing/worklist state is copied back. The oracle then replays each layer
on the GPU's own inputs (teacher forcing, so bf16 drift in one layer cannot
flip the next layer's routing) and each iteration is checked:

* fresh set, category counts, fallback flags, support, selections, worklist
  offsets and positions: bit-exact;
* a selection that differs is accepted only when the oracle's float64 logits
  hold a near-tie (two of the k+1 best eligible logits within 1e-5); the case
  is logged and the oracle adopts the GPU's selection so nothing cascades;
  the planner's support likewise;
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
from sparse_moe_layer_gate_gb300.layer import layer_for_workload, payload_to_torch

NEAR_TIE = 1e-5


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
                              router=oracle.Router(wl.router, wl.n_group, wl.topk_group))


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


def check_plan(orc: oracle.LayerOracle, gplan: dict, x0: np.ndarray, wl, rep: Report, tag: str):
    op = orc.plan_block(x0)
    glen = gplan["support_len"]
    gids = gplan["support_ids"]
    same = glen == op.support_len and np.array_equal(gids[:glen], op.ranked[:glen])
    counts_same = np.array_equal(gplan["plan_counts"], op.counts)
    if not (same and counts_same):
        everyone = np.ones(wl.n_experts, dtype=bool)
        ties = [t for t in range(x0.shape[0]) if orc.near_tie(op.G[t], everyone, NEAR_TIE)]
        if ties:
            rep.near_ties.append(f"{tag} plan: near-tie at positions {ties[:8]}; adopting GPU support")
            orc.adopt_support(gids, glen)
        else:
            rep.mismatches.append(f"{tag} plan: support/counts differ without a near-tie "
                                  f"(gpu len {glen}, oracle len {op.support_len})")
    return op


def check_hot_update(orc: oracle.LayerOracle, gplan: dict, x0: np.ndarray, wl, rep: Report, tag: str):
    """The support a hot-update iteration rebuilt (oracle.hot_update on the same
    input; near-ties as for the block plan)."""
    op = orc.hot_update(x0)
    glen = gplan["support_len"]
    gids = gplan["support_ids"]
    same = glen == op.support_len and np.array_equal(gids[:glen], op.ranked[:glen])
    if not (same and np.array_equal(gplan["plan_counts"], op.counts)):
        everyone = np.ones(wl.n_experts, dtype=bool)
        ties = [t for t in range(x0.shape[0]) if orc.near_tie(op.G[t], everyone, NEAR_TIE)]
        if ties:
            rep.near_ties.append(f"{tag} hot update: near-tie at positions {ties[:8]}; adopting GPU support")
            orc.adopt_support(gids, glen)
        else:
            rep.mismatches.append(f"{tag} hot update: support/counts differ without a near-tie "
                                  f"(gpu len {glen}, oracle len {op.support_len})")
    return op


def check_iteration(orc, step: GpuStep, live, dec, i: int, wl, rep: Report, tag: str, refresh: bool = False):
    g = step.dbg
    gsel = {int(t): g["sel"][f] for f, t in enumerate(g["fresh_pos"])}

    def adopt(t, s, g_row, eligible):
        mine = gsel.get(t)
        if mine is None or np.array_equal(mine, s):
            return None
        if orc.near_tie(g_row, eligible, NEAR_TIE):
            rep.near_ties.append(f"{tag} i={i} t={t}: gpu {list(mine)} oracle {list(s)} (near-tie)")
            return mine
        rep.mismatches.append(f"{tag} i={i} t={t}: selection gpu {list(mine)} oracle {list(s)}")
        return None

    x64 = synth.to_f64(step.x, wl.dtype)
    res = orc.iterate(x64, live, dec, i, adopt=adopt, refresh=refresh)
    st = g["stats"]
    cl = res.classified
    exp = dict(n_live=cl.n_live, n_new=cl.n_new, n_miss=cl.n_miss, n_stale=cl.n_stale, n_forced=cl.n_forced,
               n_reuse=cl.n_reuse, n_fresh=len(res.fresh_pos), n_edges=res.n_edges,
               fallback=(1 if res.host_fallback else 0) | (2 if cl.anomaly else 0), bad_flags=cl.bad_flags)
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
