"""The benchmark's bookkeeping on CPU: the algorithmic bytes and FLOPs each kernel is
charged with (closed forms written out here from the layer's definition), and the key of
the committed ncu traffic, which must not depend on where the repository is checked out."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import gen  # noqa: E402


def test_algorithmic_work_expert_major():
    cfg = gen.CONFIGS["mixtral_ll_em"]
    T, k, H, I, E = cfg.tokens, cfg.k, cfg.H, cfg.I, cfg.E
    R = T * k
    w = bench.algorithmic_work(cfg, {"R": R, "active_experts": E, "n_recv": 0})
    # x read once, each kept pick's row written once
    assert w["dispatch_copy"]["bytes"] == T * H * 2 + R * H * 2
    # GEMM1: every active expert's gate/up weights once, the rows, the bf16 activation
    assert w["gemm1_swiglu"]["bytes"] == E * 2 * I * H * 2 + R * H * 2 + R * I * 2
    assert w["gemm1_swiglu"]["flops"] == 2 * R * H * (2 * I)
    # GEMM2: down weights, the activation, float32 expert_out rows
    assert w["gemm2"]["bytes"] == E * H * I * 2 + R * I * 2 + R * H * 4
    assert w["gemm2"]["flops"] == 2 * R * I * H
    assert "reduce_ranks" not in w
    assert w["combine"]["bytes"] == R * H * 4 + T * k * 8 + T * H * 2


def test_algorithmic_work_flat_counts_pick_rows_in_dispatch():
    cfg = gen.CONFIGS["dsv3_ht_flat"]
    T, k, H = cfg.tokens, cfg.k, cfg.H
    R, n_recv = T * k, 173743
    w = bench.algorithmic_work(cfg, {"R": R, "active_experts": cfg.E, "n_recv": n_recv})
    # the row scatter writes every received row and every kept pick's row
    assert w["dispatch_copy"]["bytes"] == T * H * 2 + (n_recv + R) * H * 2
    assert "gather_picks" not in w
    assert w["reduce_ranks"]["bytes"] == R * H * 4 + n_recv * H * 4 + R * 8
    assert w["combine"]["bytes"] == n_recv * H * 4 + T * H * 2


def test_traffic_key_does_not_depend_on_the_checkout_path(monkeypatch):
    import importlib
    B = importlib.import_module("combine_topk_ids_gb300.build")
    h0 = bench.src_hash("bf16")
    monkeypatch.setattr(B, "ROOT", "/some/other/checkout")
    assert bench.src_hash("bf16") == h0
    assert bench.src_hash("fp8") != h0


@pytest.mark.parametrize("tokens,steps,world,secs,want", [(1024, 20, 1, 0.5, 40960.0), (1024, 20, 2, 0.5, 81920.0)])
def test_job_tokens_per_s(tokens, steps, world, secs, want):
    assert bench.job_tokens_per_s(tokens, steps, world, secs) == pytest.approx(want)
