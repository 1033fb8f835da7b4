"""Float64 oracle of one Epoch MoE-layer refinement iteration (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline/reference legs
may import this module. It shares no code with the CUDA library.

Source pages (cited by title and section; the walk-through is the method source):
  [W] "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元" (pinghaoyang.com.cn walk-through)
  [A] "Epoch: Compiling Diffusion Blocks for Sparse MoE Serving" (abstract page)

What one iteration computes, in the pages' notation:
  * MoE layer:  y_t = sum_{e in TopK(g(x_t))} w_{t,e} E_e(x_t)
        [W] section "MoE 路径为什么成为瓶颈" (why the MoE path is the bottleneck), layer equation.
  * Router logits G in R^{N x E} for every position, recomputed every iteration
        [W] section "Expert Atlas", definition of G; [A] abstract ("recomputing gate logits every iteration").
  * Top-k restricted to the block's active expert support S_l (a mask over
    experts; ids, order and weights of a token's selection may change each
    iteration)
        [W] section "Expert Atlas", third step (hot path reuses the support mask), Figure 7.
  * Fresh set: with D_i the decoded set, Z_i = D_i ∩ D_{i-1} (stable),
    N_i = D_i \\ D_{i-1} (newly decoded); F_i = all positions on a cache miss or
    refresh, otherwise the complement of Z_i; a newly decoded position is fresh once
        [W] section "Liveness-Shard Parallelism", equations for Z_i, N_i and F_i.
  * B_i = Compact(H, F_i); Y_F = SparseMoE(B_i, S_l); Y[F_i] = Y_F; Y[not F_i] = C_l[not F_i]
    where C_l caches the routed-expert output (not the layer output, not hidden)
        [W] section "Liveness-Shard Parallelism", the four merge equations.
  * Cached rows have bounded age; refresh period 1 makes the decoded branch exact
        [W] section "decoded-cache 的刷新周期为什么默认取 5" (refresh period), age bound.
  * Any cache miss, version/shape mismatch or liveness-transition anomaly falls
    back to the full fresh path
        [W] sections "Two Clocks" and "cold、hot-update、hot-skip" (lifecycle).
  * The worklist of (token, expert) pairs is grouped by expert and each expert
    runs once over its rows ("light-traffic expert kernel"); the combine returns
    rows by compact offset and the scatter/merge restores the dense shard
        [W] section "FreshLane Dispatch", steps 1-6.
  * The shared expert is untouched by the liveness split and runs on all positions
        [W] section "Liveness-Shard Parallelism" (closing paragraph).

Readings taken where the pages are silent:
  * support: experts ranked by block-start dense top-k hit count (count desc,
    id asc); the support is the smallest prefix whose counts reach
    T = ceil(tau * N * k), at least k experts; tau >= 1 means every expert;
  * selection uses raw logits (bias included); ties go to the lower expert id;
    weights are a softmax over the k selected logits (they sum to 1), or, with
    renormalisation off, the dense router probabilities of the selected experts
    (the sigmoid router: the selected sigmoid scores);
  * refresh: a decoded position is stale when i - stamp >= R (R = None: never);
    a refresh-path iteration makes every cached row stale (R = 0 for that
    iteration) and keeps the support;
  * hot-update: the support is rebuilt with the block-plan rule from the
    current iteration's logits; cache, stamps and decoded flags are kept;
  * per-request supports (optional): every request_size consecutive positions
    form one request with its own plan (its own counts and threshold), and a
    position selects within its request's support;
  * support-coverage check (optional, alpha and q): a fresh position is
    under-covered when the support holds less than alpha of the raw score mass
    of its dense selection; when more than (1 - q) of the fresh positions are,
    the support falls short and the next iteration runs full fresh with every
    expert eligible (a host fallback resets the check);
  * the expert is SwiGLU: E(x) = W_down (silu(W_gate x) * (W_up x)), silu(z) = z / (1 + e^-z);
  * a position flagged both live and decoded, or neither, is treated as live;
    a decoded -> live transition is an anomaly that makes the whole iteration
    full-fresh with every expert eligible;
  * optional residual: y = x + routed + shared (used to chain a layer stack).

Parity pins (tests/test_oracle_pins.py): brute-force top-k over all k-subsets,
minimal-cardinality support by brute force over expert subsets, hand-worked
fresh-set schedules (tests/golden/), closed-form silu values, the dense-MoE
special case (tau = 1, R = 1) against an all-experts masked formulation, the
cache/staleness invariants, and the hot-update and refresh paths (the rebuilt
support equals a block plan on the same input; a refresh iteration equals a
from-scratch restricted MoE on every position), the group-limited sigmoid
router (its one-group reduction to a brute-force top-k, group properties), and
the Expert Atlas planner (a hand-worked example, its no-floor and all-experts
special cases, and |U| recomputed independently), and per-request supports (a
batch of requests equals one independent layer per request). Outputs after many iterations with reused rows are
pinned only through those invariants.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

ExpertWeights = Tuple[np.ndarray, np.ndarray, np.ndarray]   # (W_gate [I,H], W_up [I,H], W_down [H,I])


# ------------------------------------------------------------------ expert math

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def swiglu_expert(X: np.ndarray, w: ExpertWeights) -> np.ndarray:
    """E(x) = W_down (silu(W_gate x) * (W_up x)) for every row x of X."""
    wg, wu, wd = w
    return (silu(X @ wg.T) * (X @ wu.T)) @ wd.T


# ------------------------------------------------------------------ routing

def gate_logits(x: np.ndarray, w_router: np.ndarray, b_router: np.ndarray) -> np.ndarray:
    """G = x W_r^T + b, one row per position ([W] "Expert Atlas", G in R^{N x E})."""
    return x @ w_router.T + b_router[None, :]


def rank_eligible(g_row: np.ndarray, eligible: np.ndarray) -> np.ndarray:
    """Eligible expert ids ordered by logit descending, lower id first on equal logits."""
    ids = np.nonzero(eligible)[0]
    order = np.lexsort((ids, -g_row[ids]))
    return ids[order]


def topk_select(g_row: np.ndarray, eligible: np.ndarray, k: int) -> np.ndarray:
    """The k experts a token selects among the eligible ones, in selection order."""
    return rank_eligible(g_row, eligible)[:k]


def renorm_softmax(g_sel: np.ndarray) -> np.ndarray:
    """w_j = exp(g_j) / sum_m exp(g_m) over the selected logits only."""
    m = np.max(g_sel)
    ex = np.exp(g_sel - m)
    return ex / np.sum(ex)


def near_tie(g_row: np.ndarray, eligible: np.ndarray, k: int, eps: float = 1e-5) -> bool:
    """True when two of the k+1 best eligible logits are within eps of each other,
    so that a rounding difference could change the selection or its order."""
    ranked = rank_eligible(g_row, eligible)[: k + 1]
    vals = g_row[ranked]
    return bool(np.any(np.abs(np.diff(vals)) <= eps))


# ------------------------------------------------------------------ router variants

@dataclasses.dataclass(frozen=True)
class Router:
    """How a position's router logits become a selection and its weights.

    "softmax" (default): G = x W_r^T + b; top-k of G over the eligible experts;
    weights = softmax over the k selected logits.

    "sigmoid_group" (the group-limited rule of routers in the LLaDA2.0 /
    DeepSeek-V3 family, which [W] "Expert Atlas" step three names as "the
    model's group-limited top-k rule", applied to the support): G = x W_r^T
    (no bias); scores s = sigmoid(G); selection scores c = s + b (the bias only
    steers the selection); the experts form n_group groups of consecutive ids;
    a group's score is the sum of the two largest c among its eligible experts
    (one eligible: that c; none: never chosen); the topk_group best groups
    (score desc, lower group id first) are chosen, and further groups in that
    order while the chosen ones hold fewer than k eligible experts; the
    selection is the top-k of c over the eligible experts of the chosen groups
    (c desc, lower id first); weights = s of the selected experts divided by
    their sum.

    renormalize=False keeps the router's own scores as the weights instead of
    dividing them by the selection's sum: for "softmax" the dense router
    probability of each selected expert (softmax of G over all E experts, so the
    weights add up to the selection's share of the routing mass), for
    "sigmoid_group" the selected sigmoid scores s."""
    kind: str = "softmax"
    n_group: int = 1
    topk_group: int = 1
    renormalize: bool = True


def sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def group_scores(c: np.ndarray, eligible: np.ndarray, n_group: int) -> np.ndarray:
    """Per group of consecutive experts: sum of its two largest eligible c
    (one eligible: that value; none: -inf)."""
    E = c.shape[0]
    gs = E // n_group
    out = np.full(n_group, -np.inf)
    for g in range(n_group):
        vals = sorted((c[e] for e in range(g * gs, (g + 1) * gs) if eligible[e]), reverse=True)
        if vals:
            out[g] = sum(vals[:2])
    return out


def chosen_groups(scores: np.ndarray, n_elig: np.ndarray, topk_group: int, k: int) -> np.ndarray:
    """Groups with an eligible expert, ranked by score desc (lower id first):
    the first topk_group, then more in rank order while the chosen ones hold
    fewer than k eligible experts."""
    n_group = scores.shape[0]
    order = sorted(range(n_group), key=lambda g: (-scores[g], g))
    chosen = np.zeros(n_group, dtype=bool)
    n_chosen = held = 0
    for g in order:
        if n_elig[g] == 0:
            continue
        if n_chosen >= topk_group and held >= k:
            break
        chosen[g] = True
        n_chosen += 1
        held += int(n_elig[g])
    return chosen


def dense_probabilities(g_row: np.ndarray) -> np.ndarray:
    """Softmax of one position's router logits over all experts."""
    ex = np.exp(g_row - np.max(g_row))
    return ex / np.sum(ex)


def selection_weights(g_row: np.ndarray, sel: np.ndarray, router: Router) -> np.ndarray:
    """Weights of the selected experts (see Router)."""
    if router.kind == "softmax":
        return renorm_softmax(g_row[sel]) if router.renormalize else dense_probabilities(g_row)[sel]
    s = sigmoid(g_row[sel])
    return s / np.sum(s) if router.renormalize else s


def route_position(g_row: np.ndarray, b_router: np.ndarray, eligible: np.ndarray, k: int,
                   router: Router) -> Tuple[np.ndarray, np.ndarray]:
    """(selected experts in selection order, their weights) of one position
    whose router logits are g_row (bias already included for "softmax")."""
    if router.kind == "softmax":
        sel = topk_select(g_row, eligible, k)
        return sel, selection_weights(g_row, sel, router)
    s = sigmoid(g_row)
    c = s + b_router
    E = g_row.shape[0]
    gs = E // router.n_group
    n_elig = np.array([int(np.sum(eligible[g * gs:(g + 1) * gs])) for g in range(router.n_group)])
    groups = chosen_groups(group_scores(c, eligible, router.n_group), n_elig, router.topk_group, k)
    in_groups = np.repeat(groups, gs)
    sel = topk_select(c, eligible & in_groups, k)
    return sel, selection_weights(g_row, sel, router)


def route_near_tie(g_row: np.ndarray, b_router: np.ndarray, eligible: np.ndarray, k: int,
                   router: Router, eps: float = 1e-5) -> bool:
    """near_tie for either router: for "sigmoid_group" the selection scores c
    and the group scores are both checked."""
    if router.kind == "softmax":
        return near_tie(g_row, eligible, k, eps)
    c = sigmoid(g_row) + b_router
    if near_tie(c, eligible, k, eps):
        return True
    sc = np.sort(group_scores(c, eligible, router.n_group))[::-1]
    sc = sc[np.isfinite(sc)][: router.topk_group + 1]
    return bool(np.any(np.abs(np.diff(sc)) <= eps))


# ------------------------------------------------------------------ block plan

def hit_counts(G: np.ndarray, k: int) -> np.ndarray:
    """cnt[e] = number of positions whose dense top-k (all experts eligible) contains e."""
    N, E = G.shape
    everyone = np.ones(E, dtype=bool)
    cnt = np.zeros(E, dtype=np.int64)
    for t in range(N):
        for e in topk_select(G[t], everyone, k):
            cnt[e] += 1
    return cnt


def coverage_threshold(tau: float, n_pos: int, k: int) -> int:
    """T = ceil(tau * N * k) edges, evaluated in float64."""
    return int(math.ceil(tau * float(n_pos * k)))


def plan_support(cnt: np.ndarray, k: int, tau: float, n_pos: int) -> Tuple[np.ndarray, int]:
    """Experts ranked by (count desc, id asc) and the support length |S|.

    |S| is the smallest prefix length whose counts reach T = ceil(tau N k),
    raised to at least k (so every token can still pick k experts); tau >= 1
    keeps every expert, zero-count ones included.
    """
    E = cnt.shape[0]
    ranked = np.array(sorted(range(E), key=lambda e: (-int(cnt[e]), e)), dtype=np.int64)
    if tau >= 1.0:
        return ranked, E
    T = coverage_threshold(tau, n_pos, k)
    covered, j = 0, 0
    while j < E and covered < T:
        covered += int(cnt[ranked[j]])
        j += 1
    return ranked, min(max(j, k), E)


# ------------------------------------------------------------------ Expert Atlas planner

@dataclasses.dataclass
class AtlasResult:
    support: np.ndarray      # expert ids in the order they entered the support
    covered_ok: bool         # |U| <= (1 - q) N at the end
    n_under: int             # |U|, tokens below their coverage floor
    rounds: int              # repair rounds run
    popularity: np.ndarray   # p_e
    # the smallest gap at any decision of the run (popularity at the cut of
    # the initial support, |C_t - r_t| of every coverage test, the score at the
    # cut of every repair round and its distance from zero): a GPU run in
    # float32 may decide differently only where this is tiny
    min_margin: float = float("inf")


def softmax_rows(G: np.ndarray) -> np.ndarray:
    """Dense router probabilities of every position over all experts."""
    m = np.max(G, axis=1, keepdims=True)
    ex = np.exp(G - m)
    return ex / np.sum(ex, axis=1, keepdims=True)


def atlas_support(G: np.ndarray, k: int, m: int, B: int, alpha: float, q: float, beta: float,
                  c: int) -> AtlasResult:
    """The Expert Atlas planner ([W] section "Expert Atlas"), for the softmax router.

    Extended candidates: each token's top K_ext = k + m experts by logit (lower
    id first on ties), with weights W[t, j] = the dense router probability of
    candidate j. Coverage floor r_t = alpha * (mass of the token's top-k
    candidates); covered mass C_t(S) = sum of W[t, j] over candidates in S;
    under-covered tokens U = {t : C_t < r_t}. Step one: the B experts of
    largest popularity p_e = sum of W over the candidate edges to e (lower id
    first on ties), or the k most popular when B < k (every token must still
    be able to select k experts). Step two, while |U| > (1 - q) N: for every
    expert e not in S, G_e = sum over t in U and candidates j of t pointing to
    e of min(W[t, j], r_t - C_t), and H_e = number of t in U with C_t + (t's
    candidate mass on e) >= r_t; the at most c experts of largest positive
    score H_e + beta G_e (lower id first on ties) join S; the loop ends when no
    score is positive."""
    N, E = G.shape
    K = min(k + m, E)
    P = softmax_rows(G)
    cand = np.zeros((N, K), dtype=np.int64)
    W = np.zeros((N, K))
    for t in range(N):
        cand[t] = rank_eligible(G[t], np.ones(E, dtype=bool))[:K]
        W[t] = P[t, cand[t]]
    r = alpha * W[:, :k].sum(axis=1)
    pop = np.zeros(E)
    for t in range(N):
        for j in range(K):
            pop[cand[t, j]] += W[t, j]
    by_pop = sorted(range(E), key=lambda e: (-pop[e], e))
    n_init = min(max(B, k), E)
    support = list(by_pop[:n_init])
    margin = [abs(pop[by_pop[n_init - 1]] - pop[by_pop[n_init]])] if n_init < E else []
    in_s = np.zeros(E, dtype=bool)
    in_s[support] = True

    def coverage():
        return np.array([sum(W[t, j] for j in range(K) if in_s[cand[t, j]]) for t in range(N)])

    rounds = 0
    C = coverage()
    margin.append(float(np.min(np.abs(C - r))))
    under = [t for t in range(N) if C[t] < r[t]]
    while len(under) > (1.0 - q) * N:
        Gs = np.zeros(E)
        Hs = np.zeros(E)
        for t in under:
            mass = {}
            for j in range(K):
                e = int(cand[t, j])
                if in_s[e]:
                    continue
                Gs[e] += min(W[t, j], r[t] - C[t])
                mass[e] = mass.get(e, 0.0) + W[t, j]
            for e, w in mass.items():
                margin.append(abs(C[t] + w - r[t]))
                if C[t] + w >= r[t]:
                    Hs[e] += 1
        score = Hs + beta * Gs
        pos = [e for e in range(E) if not in_s[e] and score[e] > 0]
        if not pos:
            break
        ranked = sorted(pos, key=lambda e: (-score[e], e))
        add = ranked[:c]
        margin.append(min(score[e] for e in pos))
        if len(ranked) > c:
            margin.append(score[ranked[c - 1]] - score[ranked[c]])
        for e in add:
            in_s[e] = True
            support.append(e)
        rounds += 1
        C = coverage()
        margin.append(float(np.min(np.abs(C - r))))
        under = [t for t in range(N) if C[t] < r[t]]
    return AtlasResult(np.array(support, dtype=np.int64), len(under) <= (1.0 - q) * N, len(under), rounds, pop,
                       float(min(margin)) if margin else float("inf"))


# ------------------------------------------------------------------ liveness

@dataclasses.dataclass
class Classified:
    fresh: np.ndarray        # bool [N]
    is_live: np.ndarray      # bool [N] (both/neither flags count as live)
    anomaly: bool            # a decoded -> live transition was seen
    bad_flags: int           # positions flagged both live and decoded, or neither
    n_live: int
    n_new: int
    n_miss: int
    n_stale: int
    n_forced: int            # would have been reused, made fresh by a fallback
    n_reuse: int


def classify_positions(live: np.ndarray, decoded: np.ndarray, prev_decoded: np.ndarray,
                       stamp: np.ndarray, i: int, refresh_R: Optional[int],
                       force_all: bool) -> Classified:
    """Fresh set of iteration i ([W] "Liveness-Shard Parallelism", F_i).

    live: still Mask; new: in D_i but not D_{i-1}; miss: decoded without a cached
    row; stale: cached row at least R iterations old. Every other decoded
    position is in Z_i and reuses its cached row, unless the iteration falls back
    to full fresh (a host-side mismatch, or a decoded -> live transition).
    """
    N = live.shape[0]
    lv = np.asarray(live, dtype=bool)
    dc = np.asarray(decoded, dtype=bool)
    is_live = lv | ~dc
    bad = int(np.sum(lv == dc))
    anomaly = bool(np.any(prev_decoded[:N].astype(bool) & is_live))
    force = force_all or anomaly
    fresh = np.zeros(N, dtype=bool)
    n = dict(live=0, new=0, miss=0, stale=0, forced=0, reuse=0)
    for t in range(N):
        if is_live[t]:
            cat = "live"
        elif not prev_decoded[t]:
            cat = "new"
        elif stamp[t] < 0:
            cat = "miss"
        elif refresh_R is not None and i - int(stamp[t]) >= refresh_R:
            cat = "stale"
        else:
            cat = "forced" if force else "reuse"
        n[cat] += 1
        fresh[t] = cat != "reuse"
    return Classified(fresh, is_live, anomaly, bad, n["live"], n["new"], n["miss"],
                      n["stale"], n["forced"], n["reuse"])


# ------------------------------------------------------------------ results

@dataclasses.dataclass
class PlanResult:
    G: np.ndarray
    counts: np.ndarray
    ranked: np.ndarray
    support_len: int
    threshold: int

    @property
    def support(self) -> np.ndarray:
        return self.ranked[: self.support_len]


@dataclasses.dataclass
class IterResult:
    y: np.ndarray                 # [N, H]
    G: np.ndarray                 # [N, E]
    fresh_pos: np.ndarray         # ascending positions in F_i
    sel: np.ndarray               # [|F|, k] selected experts, selection order
    w: np.ndarray                 # [|F|, k] weights
    wl_expert: np.ndarray         # worklist edges sorted by (expert, position)
    wl_pos: np.ndarray
    wl_j: np.ndarray              # which of the token's k selections the edge is
    offsets: np.ndarray           # [E+1] edge offsets per expert
    routed: np.ndarray            # [N, H] routed-expert output (fresh or cached)
    fallback: bool
    host_fallback: bool
    classified: Classified
    slot: np.ndarray              # [|F|, k] worklist row of selection (f, j)
    shortfall_prev: bool = False  # full fresh because the previous iteration's support coverage fell short
    n_under: int = 0              # fresh positions under the coverage floor (coverage check on)

    @property
    def n_edges(self) -> int:
        return int(self.wl_pos.shape[0])


# ------------------------------------------------------------------ the layer

class LayerOracle:
    """One MoE layer with its block plan, per-position cache and stamps.

    ``expert(e)`` returns routed expert e's float64 weights; ``shared`` lists the
    always-on shared experts. State arrays are sized ``max_positions``.
    """

    def __init__(self, *, n_experts: int, top_k: int, tau: float, refresh_R: Optional[int],
                 w_router: np.ndarray, b_router: np.ndarray,
                 expert: Callable[[int], ExpertWeights],
                 shared: Sequence[ExpertWeights] = (), residual: bool = False,
                 max_positions: int, router: Router = Router(), request_size: Optional[int] = None,
                 coverage: Optional[Tuple[float, float]] = None, atlas: Optional[dict] = None):
        self.E = n_experts
        self.k = top_k
        self.tau = tau
        self.R = refresh_R
        self.w_router = w_router
        self.b_router = b_router
        self.expert = expert
        self.shared = list(shared)
        self.residual = residual
        self.H = w_router.shape[1]
        self.max_positions = max_positions
        self.stamp = -np.ones(max_positions, dtype=np.int64)
        self.prev_decoded = np.zeros(max_positions, dtype=bool)
        self.cache = np.zeros((max_positions, self.H))
        self.planned = False
        self.n_pos = 0
        self.last_iter = -1
        self.support_mask = np.ones(self.E, dtype=bool)
        self.plan: Optional[PlanResult] = None
        self.router = router
        # per-request supports: every request_size consecutive positions are one
        # request (one diffusion block) with its own plan; None = one support
        self.request_size = request_size
        self.request_masks: Optional[np.ndarray] = None
        self.request_plans: List[PlanResult] = []
        # support-coverage check (alpha, q) or None: see coverage_shortfall
        self.coverage = coverage
        self.shortfall = False
        # Expert Atlas planner instead of the hit-count prefix: dict of m, B,
        # alpha, q, beta, c (atlas_support), or None
        self.atlas = atlas
        self.atlas_result: Optional[AtlasResult] = None
        if atlas is not None and (request_size is not None or router.kind != "softmax"):
            raise ValueError("the Expert Atlas planner is built for one support per call and the softmax router")

    def logits(self, x: np.ndarray) -> np.ndarray:
        """Router logits G (the bias is part of G only for the softmax router)."""
        if self.router.kind == "softmax":
            return gate_logits(x, self.w_router, self.b_router)
        return gate_logits(x, self.w_router, np.zeros_like(self.b_router))

    def select(self, g_row: np.ndarray, eligible: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        return route_position(g_row, self.b_router, eligible, self.k, self.router)

    def weights(self, g_row: np.ndarray, sel: np.ndarray) -> np.ndarray:
        return selection_weights(g_row, sel, self.router)

    def near_tie(self, g_row: np.ndarray, eligible: np.ndarray, eps: float = 1e-5) -> bool:
        return route_near_tie(g_row, self.b_router, eligible, self.k, self.router, eps)

    def counts(self, G: np.ndarray) -> np.ndarray:
        """Block-plan hit counts: each position's selection with every expert eligible."""
        if self.router.kind == "softmax":
            return hit_counts(G, self.k)
        everyone = np.ones(self.E, dtype=bool)
        cnt = np.zeros(self.E, dtype=np.int64)
        for t in range(G.shape[0]):
            for e in self.select(G[t], everyone)[0]:
                cnt[e] += 1
        return cnt

    # cold path ([W] "cold、hot-update、hot-skip": clear the per-block cache,
    # initialise the live set, build the support of each layer)
    def _supports(self, G: np.ndarray) -> PlanResult:
        """The plan rule on G: one support, or one per request (each request's
        own positions, counts and threshold); support_mask is then their union."""
        N = G.shape[0]
        if self.atlas is not None:
            res = atlas_support(G, self.k, **self.atlas)
            self.atlas_result = res
            self.support_mask = np.zeros(self.E, dtype=bool)
            self.support_mask[res.support] = True
            return PlanResult(G, res.popularity, res.support, int(res.support.size), 0)
        cnt = self.counts(G)
        if self.request_size is None:
            ranked, slen = plan_support(cnt, self.k, self.tau, N)
            self.support_mask = np.zeros(self.E, dtype=bool)
            self.support_mask[ranked[:slen]] = True
            return PlanResult(G, cnt, ranked, slen, coverage_threshold(self.tau, N, self.k))
        rs = self.request_size
        n_req = (N + rs - 1) // rs
        self.request_masks = np.zeros((n_req, self.E), dtype=bool)
        self.request_plans = []
        for r in range(n_req):
            Gr = G[r * rs:min(N, (r + 1) * rs)]
            cr = self.counts(Gr)
            ranked, slen = plan_support(cr, self.k, self.tau, Gr.shape[0])
            self.request_masks[r, ranked[:slen]] = True
            self.request_plans.append(PlanResult(Gr, cr, ranked, slen,
                                                 coverage_threshold(self.tau, Gr.shape[0], self.k)))
        self.support_mask = self.request_masks.any(axis=0)
        union = np.nonzero(self.support_mask)[0]
        return PlanResult(G, cnt, union, int(union.size), coverage_threshold(self.tau, rs, self.k))

    def eligible_for(self, t: int) -> np.ndarray:
        """Experts position t may select (outside a fallback)."""
        if self.request_size is None:
            return self.support_mask
        return self.request_masks[t // self.request_size]

    def plan_block(self, x: np.ndarray) -> PlanResult:
        N = x.shape[0]
        G = self.logits(x)
        self.plan = self._supports(G)
        self.stamp[:] = -1
        self.prev_decoded[:] = False
        self.cache[:] = 0.0
        self.planned = True
        self.n_pos = N
        self.last_iter = -1
        self.shortfall = False
        return self.plan

    # hot-update path ([W] "cold、hot-update、hot-skip": inside a block, the
    # support is rebuilt from the current router logits, e.g. when an update
    # counter expires). Same rule as the block plan, on this iteration's x; the
    # per-position cache, stamps and decoded flags are kept.
    def hot_update(self, x: np.ndarray) -> PlanResult:
        return self._supports(self.logits(x))

    def adopt_support(self, ranked: np.ndarray, slen: int) -> None:
        """Replace the plan's support (used after a logged near-tie at plan time)."""
        self.support_mask = np.zeros(self.E, dtype=bool)
        self.support_mask[np.asarray(ranked[:slen], dtype=np.int64)] = True

    def block_end(self) -> None:
        self.planned = False

    def coverage_shortfall(self, G: np.ndarray, fresh_pos: np.ndarray) -> Tuple[int, bool]:
        """Support coverage of an iteration's fresh positions ([W] "cold、
        hot-update、hot-skip": a support that no longer covers the routing sends
        the layer back to the full fresh path; [W] "Expert Atlas" defines the
        coverage). For fresh position t: the dense selection D_t (the router's
        rule with every expert eligible), R_t = the sum of its raw scores (dense
        probabilities, or sigmoid scores), C_t = the part of that sum whose
        experts are in t's support. t is under-covered when C_t < alpha R_t; the
        support falls short when more than (1 - q) |F| fresh positions are.
        Returns (under-covered count, shortfall)."""
        alpha, q = self.coverage
        everyone = np.ones(self.E, dtype=bool)
        raw = Router(self.router.kind, self.router.n_group, self.router.topk_group, False)
        n_under = 0
        for t in fresh_pos:
            sel, w = route_position(G[t], self.b_router, everyone, self.k, raw)
            inside = self.eligible_for(int(t))[sel]
            if np.sum(w[inside]) < alpha * np.sum(w):
                n_under += 1
        return n_under, n_under > (1.0 - q) * len(fresh_pos)

    def iterate(self, x: np.ndarray, live: np.ndarray, decoded: np.ndarray, i: int,
                adopt: Optional[Callable[[int, np.ndarray, np.ndarray, np.ndarray],
                                         Optional[np.ndarray]]] = None,
                hot_update: bool = False, refresh: bool = False) -> IterResult:
        """One refinement iteration. ``adopt(t, sel, g_row, eligible)`` may return a
        replacement selection for position t (the parity harness uses it after a
        logged near-tie).

        hot_update: rebuild the support from this iteration's logits first (see
        ``hot_update``). refresh: the refresh path ([W] "cold、hot-update、
        hot-skip") -- every position goes through the fresh routed path, which
        resets the age of every cached row; read here as a refresh period of 0
        for this iteration (each cached row counts as stale), so the selection
        stays restricted to the support and nothing else changes."""
        N = x.shape[0]
        host_fallback = (not self.planned) or (i != self.last_iter + 1) or (N != self.n_pos)
        short_prev = self.shortfall and not host_fallback
        if hot_update:
            self.hot_update(x)
        G = self.logits(x)
        R = 0 if refresh else self.R
        cl = classify_positions(live, decoded, self.prev_decoded, self.stamp, i, R, host_fallback or short_prev)
        fallback = host_fallback or short_prev or cl.anomaly
        everyone = np.ones(self.E, dtype=bool)

        fresh_pos = np.nonzero(cl.fresh)[0]
        F = fresh_pos.shape[0]
        sel = np.zeros((F, self.k), dtype=np.int64)
        w = np.zeros((F, self.k))
        for f, t in enumerate(fresh_pos):
            eligible = everyone if fallback else self.eligible_for(int(t))
            s, wt = self.select(G[t], eligible)
            if adopt is not None:
                repl = adopt(int(t), s, G[t], eligible)
                if repl is not None:
                    s = np.asarray(repl, dtype=np.int64)
                    wt = self.weights(G[t], s)
            sel[f] = s
            w[f] = wt

        # worklist: every (position, selection) edge, grouped by expert, positions ascending
        edges = sorted(((int(sel[f, j]), int(fresh_pos[f]), j, f)
                        for f in range(F) for j in range(self.k)))
        wl_expert = np.array([e for e, _, _, _ in edges], dtype=np.int64)
        wl_pos = np.array([t for _, t, _, _ in edges], dtype=np.int64)
        wl_j = np.array([j for _, _, j, _ in edges], dtype=np.int64)
        wl_f = np.array([f for _, _, _, f in edges], dtype=np.int64)
        offsets = np.zeros(self.E + 1, dtype=np.int64)
        for e in wl_expert:
            offsets[e + 1] += 1
        offsets = np.cumsum(offsets)

        # each expert runs once over its rows
        out = np.zeros((len(edges), self.H))
        for e in range(self.E):
            lo, hi = offsets[e], offsets[e + 1]
            if hi > lo:
                out[lo:hi] = swiglu_expert(x[wl_pos[lo:hi]], self.expert(e))
        slot = np.zeros((F, self.k), dtype=np.int64)
        slot[wl_f, wl_j] = np.arange(len(edges))

        # combine (selection order) + cache fill for fresh rows; cached rows elsewhere
        routed = np.zeros((N, self.H))
        for f, t in enumerate(fresh_pos):
            acc = np.zeros(self.H)
            for j in range(self.k):
                acc = acc + w[f, j] * out[slot[f, j]]
            routed[t] = acc
            self.cache[t] = acc
            self.stamp[t] = i
        reuse = ~cl.fresh
        routed[reuse] = self.cache[:N][reuse]

        y = routed.copy()
        for sw in self.shared:
            y = y + swiglu_expert(x, sw)
        if self.residual:
            y = y + x

        n_under = 0
        if self.coverage is not None:
            n_under, self.shortfall = self.coverage_shortfall(G, fresh_pos)
        else:
            self.shortfall = False
        self.prev_decoded[:N] = ~cl.is_live
        self.last_iter = i
        return IterResult(y, G, fresh_pos, sel, w, wl_expert, wl_pos, wl_j, offsets, routed,
                          fallback, host_fallback, cl, slot, short_prev, n_under)


def dense_moe(x: np.ndarray, w_router: np.ndarray, b_router: np.ndarray,
              expert: Callable[[int], ExpertWeights], n_experts: int, k: int,
              shared: Sequence[ExpertWeights] = ()) -> np.ndarray:
    """y_t = sum over the dense top-k of g(x_t) of w_{t,e} E_e(x_t), plus shared experts
    ([W] "MoE 路径为什么成为瓶颈", layer equation), one position at a time."""
    G = gate_logits(x, w_router, b_router)
    everyone = np.ones(n_experts, dtype=bool)
    y = np.zeros_like(x)
    for t in range(x.shape[0]):
        s = topk_select(G[t], everyone, k)
        wt = renorm_softmax(G[t, s])
        for j, e in enumerate(s):
            y[t] += wt[j] * swiglu_expert(x[t:t + 1], expert(int(e)))[0]
    for sw in shared:
        y = y + swiglu_expert(x, sw)
    return y
