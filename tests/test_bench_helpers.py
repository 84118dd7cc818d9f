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
    # the bf16-pair activation (the default) issues two MMAs per product
    assert w["gemm2"]["mma_flops"] == 2 * w["gemm2"]["flops"]
    assert "mma_flops" not in bench.algorithmic_work(cfg.with_(act="bf16"), {"R": R, "active_experts": E,
                                                                         "n_recv": 0})["gemm2"]
    assert "reduce_ranks" not in w
    # combine: the expert_out rows, the routing weights, the bf16 output
    assert w["combine"]["bytes"] == R * H * 4 + T * k * 4 + T * H * 2


@pytest.mark.parametrize("layout", ["RM", "FLAT"])
def test_algorithmic_work_rank_layouts(layout):
    """RANK_MAJOR / FLAT: dispatch writes each received row once, the FFN's output is one row
    per received row (N_recv), combine reads those; the pick-ordered rows, the per-pick GEMM2
    rows and the local-pick reduction are this design's, not the layer's, and count nothing."""
    cfg = gen.CONFIGS["dsv3_ht_flat"].with_(layout=layout)
    T, k, H, I, E = cfg.tokens, cfg.k, cfg.H, cfg.I, cfg.E
    R, n_recv = T * k, 173743
    w = bench.algorithmic_work(cfg, {"R": R, "active_experts": E, "n_recv": n_recv})
    assert w["dispatch_copy"]["bytes"] == T * H * 2 + n_recv * H * 2
    assert "gather_picks" not in w
    assert w["gemm1_swiglu"]["bytes"] == E * 2 * I * H * 2 + R * H * 2 + R * I * 2
    assert w["gemm2"]["bytes"] == E * H * I * 2 + R * I * 2 + n_recv * H * 4
    assert w["reduce_ranks"]["bytes"] == 0 and w["reduce_ranks"]["flops"] == 0
    assert w["combine"]["bytes"] == n_recv * H * 4 + T * H * 2
    layer = sum(v["bytes"] for v in w.values()) - w["routing"]["bytes"]
    # dispatch + FFN + combine as one closed form: x in, received rows out, weights once,
    # rows into the FFN, the activation out and back in, expert_out out and back in, output
    assert layer == (T * H * 2 + n_recv * H * 2 + E * 3 * I * H * 2 + R * H * 2 + 2 * R * I * 2 +
                     2 * n_recv * H * 4 + T * H * 2)
    extra = bench.moved_beyond_algorithmic(cfg, {"R": R, "n_recv": n_recv})
    assert extra["dispatch_copy"] == R * H * 2
    assert extra["gemm1_swiglu"] == R * I * 2      # the low half of the bf16-pair activation
    assert extra["gemm2"] == R * I * 2 + (R - n_recv) * H * 4


def test_kernel_roofline_picks_the_bound_and_the_peak():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    mem = bench.kernel_roofline({"bytes": 6e9, "flops": 1e9}, 2e-3, peaks)
    assert mem["bound"] == "hbm" and mem["frac"] == pytest.approx(0.5)
    assert mem["frac_of_nominal"] == pytest.approx(3000.0 / bench.NOMINAL_PEAKS["hbm_gbs"])
    tc = bench.kernel_roofline({"bytes": 1e9, "flops": 1.6e13}, 10e-3, peaks, sustained=True)
    assert tc["bound"] == "tensor" and tc["peak_kind"] == "sustained" and tc["frac"] == pytest.approx(1.0)
    assert bench.kernel_roofline({"bytes": 1e9, "flops": 1.6e13}, 10e-3, peaks)["frac"] == pytest.approx(0.8)
    pair = bench.kernel_roofline({"bytes": 1e9, "flops": 0.8e13, "mma_flops": 1.6e13}, 10e-3, peaks)
    assert pair["frac"] == pytest.approx(0.4) and pair["issued_mma_frac"] == pytest.approx(0.8)


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


def test_traffic_key_follows_code_not_comments():
    src = "int f(int a) {  // add one\n    return a + 1; /* the result */\n}\n"
    same = "int f(int a) {\n  return a + 1;\n}  // reformatted, comments changed\n"
    other = "int f(int a) { return a + 2; }"
    assert bench.strip_comments(src) == bench.strip_comments(same)
    assert bench.strip_comments(src) != bench.strip_comments(other)
