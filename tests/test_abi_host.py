"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every entry point include/epoch.h declares, and rejects invalid arguments
before touching the device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_moe_layer_gate_gb300 import binding, builder
    if builder.is_stale():
        builder.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "epoch.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(epoch_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "epoch_moe_iter" in names and "epoch_plan_block" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/epoch.h but not exported"


def test_binding_covers_every_declared_symbol():
    from sparse_moe_layer_gate_gb300 import binding
    assert sorted(binding.exported_names()) == declared_functions()


def good_cfg(**kw):
    from sparse_moe_layer_gate_gb300 import binding as B
    c = dict(hidden=2048, n_experts=256, inter=512, top_k=8, n_shared=1, shared_inter=512,
             max_positions=1024, dtype=B.EPOCH_BF16, tau=0.95, refresh_R=4, residual=0)
    c.update(kw)
    return B.epoch_layer_config(**c)


def test_workspace_size_and_config_validation(lib):
    from sparse_moe_layer_gate_gb300 import binding as B
    n = B.epoch_workspace_bytes(good_cfg())
    assert n > 0 and n % 256 == 0
    # the routed output cache, compact buffers and split-K logits all fit
    assert n >= 1024 * 2048 * 2 + 8 * 1024 * 2048 * (2 + 4)
    bad = [dict(hidden=2000), dict(inter=100), dict(top_k=0), dict(top_k=17), dict(n_experts=4, top_k=8),
           dict(n_experts=2000), dict(tau=0.0), dict(tau=1.5), dict(tau=float("nan")), dict(refresh_R=0),
           dict(max_positions=0), dict(max_positions=100000), dict(dtype=7), dict(n_shared=1, shared_inter=0),
           dict(n_shared=-1)]
    for b in bad:
        assert B.epoch_workspace_bytes(good_cfg(**b)) == 0, b
    # fp32 layers only need multiples of 4
    assert B.epoch_workspace_bytes(good_cfg(dtype=B.EPOCH_F32, hidden=256, inter=132, shared_inter=132)) > 0
    # router variants: the group-limited sigmoid router needs a valid group shape
    assert B.epoch_workspace_bytes(good_cfg(router=1, n_group=8, topk_group=4)) > 0
    assert B.epoch_workspace_bytes(good_cfg(router=0, n_group=0, topk_group=0)) > 0  # ignored
    for b in [dict(router=2), dict(router=-1), dict(router=1, n_group=0, topk_group=1),
              dict(router=1, n_group=33, topk_group=1), dict(router=1, n_group=3, topk_group=1),
              dict(router=1, n_group=8, topk_group=0), dict(router=1, n_group=8, topk_group=9)]:
        assert B.epoch_workspace_bytes(good_cfg(**b)) == 0, b


def test_invalid_arguments_return_einval(lib):
    from sparse_moe_layer_gate_gb300 import binding as B
    cfg = good_cfg()
    w = B.epoch_layer_weights()
    out = C.c_void_p()
    assert lib.epoch_layer_create(C.byref(cfg), C.byref(w), None, 0, C.byref(out)) == B.EPOCH_EINVAL
    assert lib.epoch_layer_create(C.byref(cfg), C.byref(w), C.c_void_p(4096), 1 << 40,
                                  C.byref(out)) == B.EPOCH_EINVAL  # null weights
    w2 = B.epoch_layer_weights(w_router=4097, b_router=4096, w_gate=4096, w_up=4096, w_down=4096,
                               ws_gate=4096, ws_up=4096, ws_down=4096)
    assert lib.epoch_layer_create(C.byref(cfg), C.byref(w2), C.c_void_p(4096), 1 << 40,
                                  C.byref(out)) == B.EPOCH_EINVAL  # misaligned router
    assert lib.epoch_layer_create(C.byref(cfg), C.byref(w), C.c_void_p(4096), 16,
                                  C.byref(out)) == B.EPOCH_EINVAL  # workspace too small
    assert lib.epoch_plan_block(None, C.c_void_p(4096), 32, None, None, None) == B.EPOCH_EINVAL
    assert lib.epoch_moe_iter(None, 4096, 4096, 4096, 32, 0, 4096, None, None) == B.EPOCH_EINVAL
    assert lib.epoch_moe_iter_path(None, 4096, 4096, 4096, 32, 0, 1, 4096, None, None) == B.EPOCH_EINVAL
    # the allocation-free planner checks its sizes and router before any CUDA call
    noalloc = lib.epoch_plan_support_noalloc
    assert noalloc(None, 32, 16, 2, 0.9, 0, None, 1, 1, 4096, 4096, None) == B.EPOCH_EINVAL       # no logits
    assert noalloc(4096, 32, 1025, 2, 0.9, 0, None, 1, 1, 4096, 4096, None) == B.EPOCH_EINVAL     # E > 1024
    assert noalloc(4096, (1 << 26) + 1, 16, 2, 0.9, 0, None, 1, 1, 4096, 4096, None) == B.EPOCH_EINVAL
    assert noalloc(4096, 32, 16, 2, 0.9, 1, None, 4, 2, 4096, 4096, None) == B.EPOCH_EINVAL       # no bias
    assert noalloc(4096, 32, 16, 2, 0.9, 1, 4096, 3, 2, 4096, 4096, None) == B.EPOCH_EINVAL       # 16 % 3
    assert noalloc(4096, 32, 16, 2, 0.9, 2, None, 1, 1, 4096, 4096, None) == B.EPOCH_EINVAL       # router
    assert lib.epoch_path_counters_ex(None, None, None) == B.EPOCH_EINVAL
    assert lib.epoch_block_end(None) == B.EPOCH_EINVAL
    assert lib.epoch_get_status(None, None, None) == B.EPOCH_EINVAL
    assert lib.epoch_read_stats(None, None, None) == B.EPOCH_EINVAL
    assert lib.epoch_debug_copy(None, None, 4, None) == B.EPOCH_EINVAL
    lib.epoch_layer_destroy(None)  # ignored
    assert lib.epoch_status_str(B.EPOCH_ETIMEOUT) == b"device wait timed out"
    assert lib.epoch_status_str(99) == b"unknown status"
