"""The allocation-free block planner (epoch_plan_support_noalloc) against the
layer's own cold path (epoch_plan_block), through the C ABI, on two calls in a
row (the second reuses the shared scratch array the first one filled).

Callers that cannot allocate device memory -- code captured into a graph with
a fixed memory pool, runtimes that only hand out buffers of a pre-planned
arena, serving loops that forbid cudaMalloc between requests -- plan with this
entry point; its scratch lives in a fixed device array, so it must agree with
the regular planner exactly (integer output: bit-exact).
"""
import ctypes as C

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_layer_gate_gb300 import builder
    if builder.is_stale():
        builder.build()


GROUPED = synth.WORKLOADS["tiny_fp32"].replace(
    name="noalloc_grouped", wid=9, iid=6, dtype="bf16", n_shared=1, batch=3, iters=3, refresh_R=3,
    router="sigmoid_group", n_group=4, topk_group=2)


@pytest.mark.parametrize("name", ["llada2_mini", "noalloc_grouped"])
def test_noalloc_planner_matches_plan_block_twice(name):
    """Softmax router (bias inside the logits) and group-limited sigmoid router
    (logits without the bias, bias passed separately): the support equals the
    one epoch_plan_block returns for the same x, on two calls in a row."""
    from sparse_moe_layer_gate_gb300 import binding as B
    from sparse_moe_layer_gate_gb300.layer import payload_to_torch
    from parity_harness import layer_for_workload
    wl = synth.WORKLOADS[name] if name in synth.WORKLOADS else GROUPED
    router = 0 if wl.router == "softmax" else 1
    lay = layer_for_workload(wl)
    xs = synth.hidden_states(wl, 3)
    live, dec = synth.block_masks(wl, 1)
    n, E = wl.n_pos, wl.n_experts
    stream = torch.cuda.current_stream()
    ids = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    slen = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_ids = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    ref_len = torch.zeros(1, dtype=torch.int32, device="cuda")
    bias = lay._weights["b_router"]
    for call, block in enumerate((0, 2)):
        x = payload_to_torch(xs[block], wl.dtype, lay.device)
        lay.plan_block(x, support_ids=ref_ids, support_len=ref_len)
        # the layer's router logits of the same x, left in its workspace
        lay.moe_iter(x, torch.from_numpy(live[0]).cuda(), torch.from_numpy(dec[0]).cuda(), 0)
        v = B.epoch_debug_view()
        assert B.lib().epoch_debug_pointers(lay.handle, C.byref(v)) == B.EPOCH_OK
        rc = B.lib().epoch_plan_support_noalloc(v.logits, n, E, wl.top_k, wl.tau, router,
                                                 bias.data_ptr() if router else None, wl.n_group, wl.topk_group,
                                                 ids.data_ptr(), slen.data_ptr(), stream.cuda_stream)
        assert rc == B.EPOCH_OK, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        got_len, want_len = int(slen.item()), int(ref_len.item())
        assert got_len == want_len, f"call {call}"
        assert torch.equal(ids[:got_len].cpu(), ref_ids[:got_len].cpu()), f"call {call}"
        lay.block_end()
    # sizes beyond the fixed scratch are refused before anything is enqueued
    assert B.lib().epoch_plan_support_noalloc(v.logits, n, 1025, 8, 0.95, 0, None, 1, 1, ids.data_ptr(),
                                              slen.data_ptr(), stream.cuda_stream) == B.EPOCH_EINVAL
    lay.close()
