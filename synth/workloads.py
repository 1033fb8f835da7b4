"""Workload shapes and seeded generators.

Shapes follow the models named on the Epoch pages (walk-through page
"Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元", section "实验设置" (setup):
LLaDA-MoE, LLaDA2.0-mini, LLaDA2.0-Flash, block size 32). The pages give no
weights and no datasets, so every tensor is drawn here from a seeded
distribution:

* hidden states: x_0 ~ N(0, 1); x_{i+1} = x_i + 0.05 * N(0, 1) per iteration;
* router weight W_r ~ N(0, std = 1/sqrt(H)); router bias b_e = log of a
  Zipf(s) probability at a seeded rank permutation of the experts (or, for
  tie tests, minus the rank's group index, groups of `bias_levels` ranks;
  for the group-limited sigmoid router, 0.05 x the centred log-probability);
* expert weights W_gate, W_up ~ N(0, 1/sqrt(H)), W_down ~ N(0, 1/sqrt(I));
* commit schedules: per block of 32 positions, a number of still-live
  positions is committed after each iteration, chosen by a seeded U(0, 1)
  confidence (highest first).

Every value is drawn in float32 and rounded once (round-to-nearest-even) to
the storage dtype. bf16 payloads are numpy uint16 arrays holding the bf16 bit
patterns; fp32 payloads are float32 arrays.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Optional

import numpy as np

BLOCK = 32

# stream tags for SeedSequence, so that every tensor has its own stream
_T_ROUTER, _T_BIAS_PERM, _T_EXPERT, _T_SHARED, _T_X0, _T_DRIFT, _T_CONF, _T_NCOMMIT = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int               # seeds the weights (router, experts)
    iid: int               # seeds the inputs (hidden states, commits)
    hidden: int
    n_experts: int
    inter: int
    top_k: int
    n_shared: int
    batch: int
    iters: int
    tau: float
    refresh_R: Optional[int]   # None = never refresh
    zipf_s: float
    dtype: str             # "f32" or "bf16"
    commit: str            # "top4" | "one" | "rand1to4" | "linear_live"
    layers: int = 1
    residual: bool = False  # y = x + routed + shared (used to chain a stack)
    bias_levels: Optional[int] = None  # router bias in groups of this many equal values (exact ties)
    router: str = "softmax"  # or "sigmoid_group" (group-limited sigmoid router)
    n_group: int = 1
    topk_group: int = 1
    raw_weights: bool = False  # weights not renormalised over the selection
    coverage: Optional[tuple] = None  # (alpha, q) of the per-iteration support-coverage check
    request_size: int = 0  # > 0: positions per request, each request with its own block plan
    atlas: Optional[tuple] = None  # Expert Atlas planner (m, B, alpha, q, beta, c) instead of the prefix rule
    description: str = ""

    @property
    def n_pos(self) -> int:
        return self.batch * BLOCK

    @property
    def shared_inter(self) -> int:
        return self.inter

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", wid=1, iid=1, hidden=256, n_experts=16, inter=128, top_k=2,
        n_shared=0, batch=1, iters=8, tau=0.9, refresh_R=2, zipf_s=1.1,
        dtype="f32", commit="top4",
        description="tiny fp32 layer: H256 E16 I128 top2, 1x32 positions, 8 iters"),
    "llada_moe_7b": Workload(
        "llada_moe_7b", wid=2, iid=2, hidden=2048, n_experts=64, inter=1024, top_k=8,
        n_shared=0, batch=8, iters=32, tau=0.95, refresh_R=4, zipf_s=1.1,
        dtype="bf16", commit="one",
        description="LLaDA-MoE-7B-shaped layer: H2048 E64 I1024 top8, 8x32 positions"),
    "llada2_mini": Workload(
        "llada2_mini", wid=3, iid=3, hidden=2048, n_experts=256, inter=512, top_k=8,
        n_shared=1, batch=32, iters=32, tau=0.95, refresh_R=4, zipf_s=1.1,
        dtype="bf16", commit="rand1to4",
        description="LLaDA2.0-mini-shaped layer: H2048 E256 I512 top8 + 1 shared, 32x32 positions"),
    "llada2_flash_x4": Workload(
        "llada2_flash_x4", wid=4, iid=4, hidden=4096, n_experts=256, inter=1024, top_k=8,
        n_shared=1, batch=16, iters=32, tau=0.97, refresh_R=8, zipf_s=1.3,
        dtype="bf16", commit="one", layers=4, residual=True,
        description="LLaDA2.0-flash-shaped stack of 4 layers: H4096 E256 I1024 top8 + 1 shared, 16x32"),
}


def sweep_workload(batch: int, tau: float, refresh_R: Optional[int]) -> Workload:
    """The LLaDA2.0-mini-shaped layer (same weights) under a linear live-fraction schedule."""
    base = WORKLOADS["llada2_mini"]
    r_tag = 0 if refresh_R is None else refresh_R
    return base.replace(
        name=f"sweep_b{batch}_tau{tau}_R{'inf' if refresh_R is None else refresh_R}",
        iid=5000 + 10 * batch,  # inputs depend on the batch only, so tau/R points share them
        batch=batch, tau=tau, refresh_R=refresh_R, commit="linear_live",
        description=f"LLaDA2.0-mini layer sweep point: batch {batch}, tau {tau}, R {r_tag or 'inf'}")


# ---------------------------------------------------------------- rounding

def round_payload(a32: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float32 array once to the storage dtype (bf16: RNE on the bit pattern)."""
    a32 = np.ascontiguousarray(a32, dtype=np.float32)
    if dtype == "f32":
        return a32
    if dtype != "bf16":
        raise ValueError(dtype)
    u = a32.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_f64(payload: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of a payload to float64."""
    if dtype == "f32":
        return np.asarray(payload, dtype=np.float32).astype(np.float64)
    return bf16_bits_to_f64(payload)


def _rng(*tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(t) for t in tags])))


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    rng.standard_normal(out=out, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


# ---------------------------------------------------------------- weights

def router_payload(wl: Workload, layer: int = 0):
    """(W_r [E, H] payload, b [E] float32): b_e = log(Zipf_s pmf at rank r_e)."""
    E, H = wl.n_experts, wl.hidden
    w = round_payload(_normal(_rng(wl.wid, layer, _T_ROUTER), (E, H), 1.0 / np.sqrt(H)), wl.dtype)
    ranks = _rng(wl.wid, layer, _T_BIAS_PERM).permutation(E) + 1
    harmonic = np.sum(np.arange(1, E + 1, dtype=np.float64) ** (-wl.zipf_s))
    bias = (-wl.zipf_s * np.log(ranks.astype(np.float64)) - np.log(harmonic)).astype(np.float32)
    if wl.bias_levels:
        # experts of ranks [1, levels] share bias 0, the next `levels` ranks -1, ...
        bias = (-np.floor((ranks - 1) / wl.bias_levels)).astype(np.float32)
    elif wl.router == "sigmoid_group":
        # a selection bias on sigmoid scores in (0, 1): the same Zipf ranks,
        # centred and scaled to a spread of a few tenths
        lp = -wl.zipf_s * np.log(ranks.astype(np.float64))
        bias = (0.05 * (lp - lp.mean())).astype(np.float32)
    return w, bias


def _expert_from(rng: np.random.Generator, wl: Workload, inter: int):
    H = wl.hidden
    wg = _normal(rng, (inter, H), 1.0 / np.sqrt(H))
    wu = _normal(rng, (inter, H), 1.0 / np.sqrt(H))
    wd = _normal(rng, (H, inter), 1.0 / np.sqrt(inter))
    return (round_payload(wg, wl.dtype), round_payload(wu, wl.dtype), round_payload(wd, wl.dtype))


def expert_payload(wl: Workload, layer: int, e: int):
    """(W_gate [I, H], W_up [I, H], W_down [H, I]) payloads of routed expert e."""
    return _expert_from(_rng(wl.wid, layer, _T_EXPERT, e), wl, wl.inter)


def shared_payload(wl: Workload, layer: int, s: int):
    """Same as expert_payload for always-on shared expert s."""
    return _expert_from(_rng(wl.wid, layer, _T_SHARED, s), wl, wl.shared_inter)


def _stack(wl: Workload, layer: int, count: int, one, threads: Optional[int]):
    H, I = wl.hidden, (wl.inter if one is expert_payload else wl.shared_inter)
    pdt = np.float32 if wl.dtype == "f32" else np.uint16
    wg = np.empty((count, I, H), pdt)
    wu = np.empty((count, I, H), pdt)
    wd = np.empty((count, H, I), pdt)

    def fill(e):
        g, u, d = one(wl, layer, e)
        wg[e], wu[e], wd[e] = g, u, d

    nthreads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(fill, range(count)))
    return wg, wu, wd


def experts_payload(wl: Workload, layer: int = 0, threads: Optional[int] = None):
    """All routed experts stacked: W_gate/W_up [E, I, H], W_down [E, H, I]."""
    return _stack(wl, layer, wl.n_experts, expert_payload, threads)


def shared_experts_payload(wl: Workload, layer: int = 0, threads: Optional[int] = None):
    return _stack(wl, layer, wl.n_shared, shared_payload, threads)


# ---------------------------------------------------------------- inputs

def hidden_states(wl: Workload, n_iters: Optional[int] = None, block: int = 0) -> np.ndarray:
    """x_i for i < n_iters as payloads [n_iters, N, H]; x_{i+1} = x_i + 0.05 N(0,1)."""
    n_iters = wl.iters if n_iters is None else n_iters
    N, H = wl.n_pos, wl.hidden
    x = _normal(_rng(wl.iid, block, _T_X0), (N, H), 1.0)
    drift = _rng(wl.iid, block, _T_DRIFT)
    pdt = np.float32 if wl.dtype == "f32" else np.uint16
    out = np.empty((n_iters, N, H), pdt)
    for i in range(n_iters):
        out[i] = round_payload(x, wl.dtype)
        if i + 1 < n_iters:
            x = x + _normal(drift, (N, H), 0.05)
    return out


def _commit_count(wl: Workload, i: int, n_live: int, rng: np.random.Generator) -> int:
    if wl.commit == "top4":
        c = 4
    elif wl.commit == "one":
        c = 1
    elif wl.commit == "rand1to4":
        c = int(rng.integers(1, 5))
    elif wl.commit == "linear_live":
        # live count at iteration j is round(32 (31 - j) / 31): 100% at j=0, 0% at j=31
        target = int(np.floor(BLOCK * (31 - (i + 1)) / 31.0 + 0.5)) if i + 1 <= 31 else 0
        c = n_live - max(target, 0)
    else:
        raise ValueError(wl.commit)
    return max(0, min(c, n_live))


def block_masks(wl: Workload, n_iters: Optional[int] = None, block: int = 0):
    """(live, decoded) uint8 masks [n_iters, N] seen by iteration i.

    Iteration 0 sees every position live (still Mask). After iteration i, each
    block of 32 commits the live positions with the highest seeded confidence;
    iteration i+1 sees them decoded. A finished block stays all-decoded.
    """
    n_iters = wl.iters if n_iters is None else n_iters
    N = wl.n_pos
    decoded = np.zeros(N, dtype=bool)
    live_out = np.empty((n_iters, N), np.uint8)
    dec_out = np.empty((n_iters, N), np.uint8)
    conf_rng = _rng(wl.iid, block, _T_CONF)
    cnt_rng = _rng(wl.iid, block, _T_NCOMMIT)
    for i in range(n_iters):
        live_out[i] = (~decoded).astype(np.uint8)
        dec_out[i] = decoded.astype(np.uint8)
        conf = conf_rng.random(N)
        for b in range(wl.batch):
            lo = b * BLOCK
            live_idx = np.nonzero(~decoded[lo:lo + BLOCK])[0]
            c = _commit_count(wl, i, live_idx.size, cnt_rng)
            if c:
                order = live_idx[np.argsort(-conf[lo + live_idx], kind="stable")]
                decoded[lo + order[:c]] = True
    return live_out, dec_out
