"""The benchmark's roofline arithmetic (host code, no GPU): the work one
iteration must do and the expert kernel's algorithmic bytes, checked against
figures computed by hand for the LLaDA2.0-mini-shaped layer."""
import types

import pytest

import bench

MINI = types.SimpleNamespace(hidden=2048, n_experts=256, inter=512, shared_inter=512, n_pos=1024,
                             n_shared=1, dtype="bf16")


def test_iteration_zero_work_of_the_mini_layer():
    # every position fresh, 35 routed experts hit plus the shared expert, k = 8
    st = {"n_edges": 1024 * 8, "n_hit_experts": 35, "n_fresh": 1024, "n_reuse": 0}
    flops, nbytes = bench.iteration_work(MINI, st)
    gate = 2 * 1024 * 2048 * 256                 # G = x W_r^T over every position
    routed = 6 * 2048 * 512 * 8192               # three projections per edge
    shared = 6 * 2048 * 512 * 1024               # the shared expert on every position
    assert flops == gate + routed + shared
    assert abs(flops / 1e9 - 59.1) < 0.1
    weights = (35 + 1) * 3 * 2048 * 512 * 2      # hit routed experts and the shared one, bf16
    router = 256 * 2048 * 2 + 4 * 256
    acts = 2 * 1024 * 2048 * 2 + 1024 * 2048 * 2 + 2 * 1024  # x in, y out, cache rows written, masks
    assert nbytes == weights + router + acts
    assert abs(nbytes / 1e6 - 240.1) < 0.1


def test_reused_rows_are_read_not_written():
    st_fresh = {"n_edges": 800, "n_hit_experts": 34, "n_fresh": 100, "n_reuse": 924}
    st_all = {"n_edges": 800, "n_hit_experts": 34, "n_fresh": 1024, "n_reuse": 0}
    _, b1 = bench.iteration_work(MINI, st_fresh)
    _, b2 = bench.iteration_work(MINI, st_all)
    assert b1 == b2  # a cache row is either written (fresh) or read (reused): same bytes


def test_expert_kernel_algorithmic_bytes():
    st = {"n_hit_experts": 34}
    assert bench.experts_kernel_bytes(MINI, st) == 220_200_960  # (34 + 1) x 3 x 2048 x 512 x 2


@pytest.mark.parametrize("hit", [0, 1, 256])
def test_expert_bytes_grow_with_hit_experts(hit):
    st = {"n_hit_experts": hit}
    assert bench.experts_kernel_bytes(MINI, st) == 3 * 2048 * 2 * 512 * (hit + 1)
