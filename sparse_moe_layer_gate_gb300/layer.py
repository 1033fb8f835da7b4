"""Torch-facing wrapper of one Epoch MoE layer (marshalling only).

PyTorch provides device memory and streams; every step of the layer runs in
the sm_103a library through the C ABI in ``binding``.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

import numpy as np
import torch

from . import binding as B

_TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
_ABI_DT = {"bf16": B.EPOCH_BF16, "f32": B.EPOCH_F32}
_ROUTER = {"softmax": 0, "sigmoid_group": 1}  # EPOCH_ROUTER_SOFTMAX, EPOCH_ROUTER_SIGMOID_GROUP


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class EpochLayer:
    """One routed-expert MoE layer with its block plan and routed-output cache.

    coverage: (alpha, q) turns on the per-iteration support-coverage check
    (see epoch_layer_config); None leaves it off. atlas: dict of m, B, alpha,
    q, beta, c selects the Expert Atlas planner; None the hit-count prefix.

    weights: dict of CUDA tensors -- w_router [E,H], b_router [E] float32,
    w_gate/w_up [E,I,H], w_down [E,H,I], and when n_shared > 0 ws_gate/ws_up
    [n_sh,I_s,H], ws_down [n_sh,H,I_s]; all contiguous, in the layer dtype.
    """

    def __init__(self, *, hidden: int, n_experts: int, inter: int, top_k: int, max_positions: int,
                 dtype: str, tau: float, refresh_R: Optional[int], weights: Dict[str, torch.Tensor],
                 n_shared: int = 0, shared_inter: Optional[int] = None, residual: bool = False,
                 router: str = "softmax", n_group: int = 1, topk_group: int = 1, raw_weights: bool = False,
                 coverage: Optional[tuple] = None, request_size: int = 0, atlas: Optional[dict] = None):
        self.dtype = dtype
        self.hidden, self.n_experts, self.inter, self.top_k = hidden, n_experts, inter, top_k
        self.n_shared = n_shared
        self.max_positions = max_positions
        self.request_size = int(request_size)
        self.cfg = B.epoch_layer_config(
            hidden=hidden, n_experts=n_experts, inter=inter, top_k=top_k, n_shared=n_shared,
            shared_inter=(shared_inter or inter) if n_shared else 0, max_positions=max_positions,
            dtype=_ABI_DT[dtype], tau=float(tau),
            refresh_R=B.EPOCH_REFRESH_NEVER if refresh_R is None else int(refresh_R),
            residual=1 if residual else 0, router=_ROUTER[router], n_group=int(n_group),
            topk_group=int(topk_group), raw_weights=1 if raw_weights else 0,
            coverage_check=1 if coverage else 0, coverage_alpha=float(coverage[0]) if coverage else 0.0,
            coverage_q=float(coverage[1]) if coverage else 0.0, request_size=int(request_size),
            planner=1 if atlas else 0, atlas_m=int(atlas["m"]) if atlas else 0,
            atlas_B=int(atlas["B"]) if atlas else 0, atlas_c=int(atlas["c"]) if atlas else 0,
            atlas_alpha=float(atlas["alpha"]) if atlas else 0.0, atlas_q=float(atlas["q"]) if atlas else 0.0,
            atlas_beta=float(atlas["beta"]) if atlas else 0.0)
        tdt = _TORCH_DT[dtype]
        for name, t in weights.items():
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError(f"weight {name} must be a contiguous CUDA tensor")
            want = torch.float32 if name == "b_router" else tdt
            if t.dtype != want:
                raise ValueError(f"weight {name} has dtype {t.dtype}, expected {want}")
        self._weights = weights  # keep alive: the library holds raw pointers
        self.wstruct = B.epoch_layer_weights(
            w_router=_ptr(weights["w_router"]), b_router=_ptr(weights["b_router"]),
            w_gate=_ptr(weights["w_gate"]), w_up=_ptr(weights["w_up"]), w_down=_ptr(weights["w_down"]),
            ws_gate=_ptr(weights.get("ws_gate")), ws_up=_ptr(weights.get("ws_up")),
            ws_down=_ptr(weights.get("ws_down")))
        self.workspace_bytes = B.epoch_workspace_bytes(self.cfg)
        if self.workspace_bytes == 0:
            raise ValueError("invalid layer configuration")
        dev = weights["w_router"].device
        self._ws = torch.empty(self.workspace_bytes + 256, dtype=torch.uint8, device=dev)
        base = self._ws.data_ptr()
        self._ws_ptr = (base + 255) // 256 * 256
        self.handle = B.epoch_layer_create(self.cfg, self.wstruct, self._ws_ptr, self.workspace_bytes)
        self.device = dev

    # ------------------------------------------------------------------ entry points
    def plan_block(self, x: torch.Tensor, stream=None, support_ids: Optional[torch.Tensor] = None,
                   support_len: Optional[torch.Tensor] = None) -> None:
        """Cold path of a block. support_ids (int32 [E]) and support_len (int32
        [1]), CUDA tensors, receive the ranked experts and |S| in stream order."""
        self._check_x(x)
        for t, n in ((support_ids, self.n_experts), (support_len, 1)):
            if t is not None and not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()
                                      and t.numel() >= n):
                raise ValueError("support outputs must be contiguous int32 CUDA tensors")
        B.check(B.epoch_plan_block(self.handle, x.data_ptr(), x.shape[0], _stream(stream), _ptr(support_ids),
                                   _ptr(support_len)), "epoch_plan_block")

    def moe_iter(self, x: torch.Tensor, live: torch.Tensor, decoded: torch.Tensor, iteration: int,
                 y: Optional[torch.Tensor] = None, stream=None, hot_update: bool = False,
                 refresh: bool = False, stats: Optional[torch.Tensor] = None) -> torch.Tensor:
        """One iteration; hot_update / refresh select the lifecycle path
        (epoch_moe_iter_path), the default being the hot-skip path. stats, an
        int32 CUDA tensor of len(binding.STATS_FIELDS) entries, receives the
        iteration's statistics in stream order (see stats_dict)."""
        self._check_x(x)
        n = x.shape[0]
        for m in (live, decoded):
            if not (m.is_cuda and m.dtype == torch.uint8 and m.is_contiguous() and m.numel() >= n):
                raise ValueError("live/decoded must be contiguous uint8 CUDA tensors of n_pos flags")
        if y is None:
            y = torch.empty_like(x)
        if stats is not None and not (stats.is_cuda and stats.dtype == torch.int32 and stats.is_contiguous()
                                       and stats.numel() >= len(B.STATS_FIELDS)):
            raise ValueError("stats must be a contiguous int32 CUDA tensor of len(STATS_FIELDS) entries")
        path = (B.PATH_HOT_UPDATE if hot_update else 0) | (B.PATH_REFRESH if refresh else 0)
        if path:
            B.check(B.epoch_moe_iter_path(self.handle, x.data_ptr(), live.data_ptr(), decoded.data_ptr(), n,
                                          int(iteration), path, y.data_ptr(), _stream(stream), _ptr(stats)),
                    "epoch_moe_iter_path")
        else:
            B.check(B.epoch_moe_iter(self.handle, x.data_ptr(), live.data_ptr(), decoded.data_ptr(), n,
                                     int(iteration), y.data_ptr(), _stream(stream), _ptr(stats)), "epoch_moe_iter")
        return y

    @staticmethod
    def stats_dict(stats: torch.Tensor) -> dict:
        """Host view of a stats tensor that moe_iter filled."""
        vals = stats.cpu().tolist()
        return {n: int(vals[i]) for i, n in enumerate(B.STATS_FIELDS)}

    def block_end(self) -> None:
        B.check(B.epoch_block_end(self.handle), "epoch_block_end")

    # ------------------------------------------------------------------ inspection
    def stats(self, stream=None) -> dict:
        st = B.epoch_iter_stats()
        B.check(B.lib().epoch_read_stats(self.handle, C.byref(st), _stream(stream)), "epoch_read_stats")
        return st.as_dict()

    def status(self, stream=None):
        word = C.c_uint32(0)
        code = B.lib().epoch_get_status(self.handle, _stream(stream), C.byref(word))
        return code, word.value

    def clear_status(self, stream=None) -> None:
        B.check(B.lib().epoch_clear_status(self.handle, _stream(stream)), "epoch_clear_status")

    def path_counters_ex(self):
        """(hot-update iterations, refresh iterations)."""
        hu, rf = C.c_int64(0), C.c_int64(0)
        B.check(B.lib().epoch_path_counters_ex(self.handle, C.byref(hu), C.byref(rf)), "epoch_path_counters_ex")
        return hu.value, rf.value

    def path_counters(self):
        c, h, f = C.c_int64(), C.c_int64(), C.c_int64()
        B.check(B.lib().epoch_path_counters(self.handle, C.byref(c), C.byref(h), C.byref(f)),
                "epoch_path_counters")
        return {"cold": c.value, "hot": h.value, "fallback": f.value}

    def set_wait_timeout(self, ns: int) -> None:
        B.check(B.lib().epoch_set_wait_timeout(self.handle, int(ns)), "epoch_set_wait_timeout")

    def test_wait_timeout(self, ns: int, stream=None) -> None:
        B.check(B.lib().epoch_test_wait_timeout(self.handle, int(ns), _stream(stream)),
                "epoch_test_wait_timeout")

    def set_tracing(self, on: bool) -> None:
        B.check(B.lib().epoch_set_tracing(self.handle, 1 if on else 0), "epoch_set_tracing")

    def read_trace(self, stream=None) -> np.ndarray:
        """[9, 1024, 8] int64 per-CTA trace rows (see epoch_debug_view.trace):
        gate, experts, expert epilogue, the gate's worklist tail (CTA 0), gate
        epilogue steps, unused, expert waits, combine, the gate tail's end per
        CTA."""
        v = B.epoch_debug_view()
        B.check(B.lib().epoch_debug_pointers(self.handle, C.byref(v)), "epoch_debug_pointers")
        return self._copy(v.trace, 9 * 1024 * 8, np.int64, stream).reshape(9, 1024, 8)

    def read_timeline(self, stream=None) -> dict:
        """{kernel: (first entry ns, last exit ns)} of the last traced iteration."""
        v = B.epoch_debug_view()
        B.check(B.lib().epoch_debug_pointers(self.handle, C.byref(v)), "epoch_debug_pointers")
        p = B.epoch_profile()
        B.check(B.lib().epoch_read_profile(self.handle, C.byref(p)), "epoch_read_profile")
        nk = sum(1 for i in range(B.EPOCH_PROF_KINDS) if p.name[i])
        raw = self._copy(v.timeline, 2 * nk, np.uint64, stream).reshape(2, nk)
        return {p.name[i].decode(): (int(raw[0, i]), int(raw[1, i])) for i in range(nk) if raw[1, i] > 0}

    def set_profiling(self, on: bool) -> None:
        B.check(B.lib().epoch_set_profiling(self.handle, 1 if on else 0), "epoch_set_profiling")

    def read_profile(self) -> dict:
        p = B.epoch_profile()
        B.check(B.lib().epoch_read_profile(self.handle, C.byref(p)), "epoch_read_profile")
        out = {}
        for i in range(B.EPOCH_PROF_KINDS):
            name = p.name[i].decode() if p.name[i] else ""
            if name and p.launches[i]:
                out[name] = {"launches": int(p.launches[i]), "total_ms": float(p.total_ms[i])}
        out["_kernels_launched"] = int(p.kernels_launched)
        return out

    def reset_profile(self) -> None:
        B.check(B.lib().epoch_reset_profile(self.handle), "epoch_reset_profile")

    def _copy(self, ptr: int, count: int, dtype, stream=None) -> np.ndarray:
        out = np.empty(count, dtype=dtype)
        if count:
            B.check(B.lib().epoch_debug_copy(out.ctypes.data, ptr, out.nbytes, _stream(stream)),
                    "epoch_debug_copy")
        return out

    def debug(self, n_pos: int, parts=("plan", "iter"), stream=None) -> dict:
        """Host copies of internal arrays. parts: "plan" (support, hit counts),
        "iter" (fresh list, selections, weights, worklist, stamps), "logits"
        (G of the last iteration), "cache" (routed-output cache rows)."""
        v = B.epoch_debug_view()
        B.check(B.lib().epoch_debug_pointers(self.handle, C.byref(v)), "epoch_debug_pointers")
        st = self.stats(stream)
        E, k, N = self.n_experts, self.top_k, self.max_positions
        nf, ne = st["n_fresh"], st["n_edges"]
        d = dict(stats=st)
        d["error_word"] = int(self._copy(v.error_word, 1, np.uint32, stream)[0])
        if "plan" in parts:
            d["support_len"] = int(self._copy(v.support_len, 1, np.int32, stream)[0])
            d["support_ids"] = self._copy(v.support_ids, E, np.int32, stream)
            if self.request_size > 0:
                R = (n_pos + self.request_size - 1) // self.request_size
                d["plan_counts"] = self._copy(v.plan_counts, R * E, np.int32, stream).reshape(R, E)
                d["request_ids"] = self._copy(v.request_ids, R * E, np.int32, stream).reshape(R, E)
                d["request_len"] = self._copy(v.request_len, R, np.int32, stream)
                d["support_masks"] = self._copy(v.support_masks, R * E, np.uint8, stream).reshape(R, E)
            else:
                d["plan_counts"] = self._copy(v.plan_counts, E, np.int32, stream)
            if self.cfg.planner == 1:
                res = self._copy(v.atlas_result, 3, np.int32, stream)
                d["atlas"] = dict(covered_ok=bool(res[0]), n_under=int(res[1]), rounds=int(res[2]))
        if "iter" in parts:
            # selections, weights and slots are stored per position; rows of the
            # fresh positions, in fresh-list order
            fp = self._copy(v.fresh_pos, nf, np.int32, stream)
            d["fresh_pos"] = fp
            d["sel"] = self._copy(v.sel, n_pos * k, np.int32, stream).reshape(n_pos, k)[fp]
            d["sel_w"] = self._copy(v.sel_w, n_pos * k, np.float32, stream).reshape(n_pos, k)[fp]
            d["offsets"] = self._copy(v.offsets, E + 1, np.int32, stream)
            d["wl_pos"] = self._copy(v.wl_pos, ne, np.int32, stream)
            d["slot"] = self._copy(v.slot, n_pos * k, np.int32, stream).reshape(n_pos, k)[fp]
            d["stamp"] = self._copy(v.stamp, n_pos, np.int32, stream)
        if "logits" in parts:
            d["logits"] = self._copy(v.logits, N * E, np.float32, stream).reshape(N, E)[:n_pos]
        if "cache" in parts:
            cdt = np.uint16 if self.dtype == "bf16" else np.float32
            d["cache"] = self._copy(v.cache, n_pos * self.hidden, cdt, stream).reshape(n_pos, self.hidden)
        return d

    def _check_x(self, x: torch.Tensor) -> None:
        if not (x.is_cuda and x.is_contiguous() and x.dtype == _TORCH_DT[self.dtype] and x.dim() == 2
                and x.shape[1] == self.hidden):
            raise ValueError(f"x must be a contiguous CUDA {self.dtype} tensor [n_pos, {self.hidden}]")

    def close(self) -> None:
        if getattr(self, "handle", None):
            B.epoch_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def payload_to_torch(payload: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Uploads a synth payload (bf16 bit patterns as uint16, or float32) as a CUDA tensor."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(payload).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(payload, dtype=np.float32))
    return t.to(device)
