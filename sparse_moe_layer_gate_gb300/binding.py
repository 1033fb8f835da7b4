"""ctypes binding of the Epoch MoE-layer C ABI (include/epoch.h).

Argument marshalling only: every step of the layer runs in the sm_103a
library. Loading fails loudly when the library has not been built; there is no
other implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libepoch.so")

EPOCH_OK, EPOCH_EINVAL, EPOCH_ESTATE, EPOCH_ECUDA, EPOCH_ETIMEOUT, EPOCH_EDEVICE = range(6)
EPOCH_F32, EPOCH_BF16 = 0, 1
EPOCH_REFRESH_NEVER = 2**31 - 1
EPOCH_DEVERR_FLAGS, EPOCH_DEVERR_TIMEOUT, EPOCH_DEVERR_BOUNDS = 1, 2, 4
EPOCH_PROF_KINDS = 12


class epoch_layer_config(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_experts", C.c_int32), ("inter", C.c_int32),
                ("top_k", C.c_int32), ("n_shared", C.c_int32), ("shared_inter", C.c_int32),
                ("max_positions", C.c_int32), ("dtype", C.c_int32), ("tau", C.c_double),
                ("refresh_R", C.c_int32), ("residual", C.c_int32), ("router", C.c_int32),
                ("n_group", C.c_int32), ("topk_group", C.c_int32), ("raw_weights", C.c_int32),
                ("coverage_check", C.c_int32), ("coverage_alpha", C.c_double), ("coverage_q", C.c_double),
                ("request_size", C.c_int32), ("planner", C.c_int32), ("atlas_m", C.c_int32),
                ("atlas_B", C.c_int32), ("atlas_c", C.c_int32), ("atlas_alpha", C.c_double),
                ("atlas_q", C.c_double), ("atlas_beta", C.c_double)]


class epoch_layer_weights(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("b_router", C.c_void_p), ("w_gate", C.c_void_p),
                ("w_up", C.c_void_p), ("w_down", C.c_void_p), ("ws_gate", C.c_void_p),
                ("ws_up", C.c_void_p), ("ws_down", C.c_void_p)]


STATS_FIELDS = ("iteration", "n_pos", "n_live", "n_new", "n_miss", "n_stale", "n_forced", "n_reuse",
                "n_fresh", "n_edges", "n_hit_experts", "support_len", "fallback", "bad_flags",
                "tiles_up", "tiles_down", "n_under")


class epoch_iter_stats(C.Structure):
    _fields_ = [(n, C.c_int32) for n in STATS_FIELDS]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class epoch_debug_view(C.Structure):
    _fields_ = [("support_ids", C.c_void_p), ("support_len", C.c_void_p), ("plan_counts", C.c_void_p),
                ("logits", C.c_void_p),
                ("fresh_pos", C.c_void_p),
                ("sel", C.c_void_p), ("sel_w", C.c_void_p), ("offsets", C.c_void_p),
                ("wl_pos", C.c_void_p), ("slot", C.c_void_p), ("stamp", C.c_void_p),
                ("cache", C.c_void_p), ("stats", C.c_void_p), ("error_word", C.c_void_p),
                ("trace", C.c_void_p), ("timeline", C.c_void_p), ("support_masks", C.c_void_p),
                ("request_ids", C.c_void_p), ("request_len", C.c_void_p), ("atlas_result", C.c_void_p)]


class epoch_profile(C.Structure):
    _fields_ = [("name", C.c_char_p * EPOCH_PROF_KINDS), ("launches", C.c_int64 * EPOCH_PROF_KINDS),
                ("total_ms", C.c_double * EPOCH_PROF_KINDS), ("kernels_launched", C.c_int64)]


_lib: Optional[C.CDLL] = None

_SIGS = {
    "epoch_workspace_bytes": (C.c_size_t, [C.POINTER(epoch_layer_config)]),
    "epoch_layer_create": (C.c_int, [C.POINTER(epoch_layer_config), C.POINTER(epoch_layer_weights),
                                     C.c_void_p, C.c_size_t, C.POINTER(C.c_void_p)]),
    "epoch_plan_block": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "epoch_moe_iter": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                 C.c_void_p, C.c_void_p, C.c_void_p]),
    "epoch_moe_iter_path": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                      C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "epoch_block_end": (C.c_int, [C.c_void_p]),
    "epoch_get_status": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(C.c_uint32)]),
    "epoch_clear_status": (C.c_int, [C.c_void_p, C.c_void_p]),
    "epoch_read_stats": (C.c_int, [C.c_void_p, C.POINTER(epoch_iter_stats), C.c_void_p]),
    "epoch_debug_pointers": (C.c_int, [C.c_void_p, C.POINTER(epoch_debug_view)]),
    "epoch_debug_copy": (C.c_int, [C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "epoch_path_counters": (C.c_int, [C.c_void_p, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                      C.POINTER(C.c_int64)]),
    "epoch_path_counters_ex": (C.c_int, [C.c_void_p, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "epoch_set_wait_timeout": (C.c_int, [C.c_void_p, C.c_int64]),
    "epoch_set_tracing": (C.c_int, [C.c_void_p, C.c_int32]),
    "epoch_set_profiling": (C.c_int, [C.c_void_p, C.c_int32]),
    "epoch_read_profile": (C.c_int, [C.c_void_p, C.POINTER(epoch_profile)]),
    "epoch_reset_profile": (C.c_int, [C.c_void_p]),
    "epoch_test_wait_timeout": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p]),
    "epoch_plan_support_noalloc": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_double,
                                             C.c_int32, C.c_void_p, C.c_int32, C.c_int32,
                                             C.c_void_p, C.c_void_p, C.c_void_p]),
    "epoch_layer_destroy": (None, [C.c_void_p]),
    "epoch_status_str": (C.c_char_p, [C.c_int]),
}


def exported_names():
    return list(_SIGS)


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"Epoch CUDA library not built ({LIB_PATH} missing); "
                               "run __graft_entry__.build() or sparse_moe_layer_gate_gb300/builder.py")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


class EpochError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib().epoch_status_str(status).decode()} ({status})")


def check(status: int, what: str) -> None:
    if status != EPOCH_OK:
        raise EpochError(status, what)


# Same-named entry points (thin wrappers over the C functions).
def epoch_workspace_bytes(cfg: epoch_layer_config) -> int:
    return int(lib().epoch_workspace_bytes(C.byref(cfg)))


def epoch_layer_create(cfg, weights, workspace_ptr: int, nbytes: int) -> int:
    out = C.c_void_p()
    check(lib().epoch_layer_create(C.byref(cfg), C.byref(weights), C.c_void_p(workspace_ptr), nbytes,
                                   C.byref(out)), "epoch_layer_create")
    return out.value


def epoch_plan_block(layer: int, x_ptr: int, n_pos: int, stream: int = 0, support_ids_ptr: Optional[int] = None,
                     support_len_ptr: Optional[int] = None) -> int:
    return lib().epoch_plan_block(layer, x_ptr, n_pos, stream, support_ids_ptr, support_len_ptr)


def epoch_moe_iter(layer: int, x_ptr: int, live_ptr: int, decoded_ptr: int, n_pos: int, iteration: int,
                   y_ptr: int, stream: int = 0, stats_ptr: Optional[int] = None) -> int:
    return lib().epoch_moe_iter(layer, x_ptr, live_ptr, decoded_ptr, n_pos, iteration, y_ptr, stream, stats_ptr)


PATH_HOT_UPDATE = 1  # epoch_path values
PATH_REFRESH = 2


def epoch_moe_iter_path(layer: int, x_ptr: int, live_ptr: int, decoded_ptr: int, n_pos: int, iteration: int,
                        path: int, y_ptr: int, stream: int = 0, stats_ptr: Optional[int] = None) -> int:
    return lib().epoch_moe_iter_path(layer, x_ptr, live_ptr, decoded_ptr, n_pos, iteration, path, y_ptr, stream,
                                     stats_ptr)


def epoch_block_end(layer: int) -> int:
    return lib().epoch_block_end(layer)


def epoch_layer_destroy(layer: int) -> None:
    lib().epoch_layer_destroy(layer)
