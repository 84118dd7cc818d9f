"""The EP layer against the same kernels run without expert parallelism (one logical rank).

The FlashInfer MoE-EP page checks its EP layer against the same computation run non-EP on
the same tokens and weights ("MoE-EP implementation & usage", section 4 "Usage
walkthrough").  Here the logical world size W only partitions one batch, so the method
fixes exact identities:
- EXPERT_MAJOR: an expert's rows are packed in ascending (token, pick) order whatever W is,
  and each output is the same fmaf chain over the token's picks, so the output for W = 1,
  2 and 4 is the same bit for bit;
- FLAT with W = 1: every pick is local to the one destination, whose received row holds
  the fmaf chain over the token's picks in ascending order, the same operations as the
  EXPERT_MAJOR combine, so FLAT (W = 1) equals EXPERT_MAJOR bit for bit;
- FLAT and RANK_MAJOR with W > 1 sum per destination first, a different association of
  the same fp32 terms, so they agree with EXPERT_MAJOR to one bf16 step of the result, or
  a few fp32 steps of the terms where those cancel.
"""
import numpy as np
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
from gen.device import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


def _out(cfg, case, W, layout):
    """Run the layer on the case's tokens, weights and routing with W logical ranks."""
    T = cfg.tokens
    Tr = -(-T // W)
    layer = moe.MoELayer1GPU(W, Tr, T, cfg.H, cfg.E, cfg.k, cfg.I, layout, cfg.algo)
    layer.set_weights(case.w1, case.w2)
    layer.forward(case.x, case.ids, case.w)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return layer.out.clone()


@pytest.mark.parametrize("name", ["small_em", "pair_em", "tall_em"])
def test_expert_major_output_does_not_depend_on_world(name):
    base = gen.SMALL[name].with_(W=4, mask_frac=0.1, seed=41)
    case = make_case(base, "cuda")
    outs = [_out(base, case, W, "EM") for W in (1, 2, 4)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("name", ["small_em", "pair_em", "tall_em"])
def test_flat_single_rank_equals_expert_major(name):
    base = gen.SMALL[name].with_(W=4, mask_frac=0.1, seed=42)
    case = make_case(base, "cuda")
    em = _out(base, case, 4, "EM")
    flat1 = _out(base, case, 1, "FLAT")
    assert torch.equal(flat1.view(torch.int16), em.view(torch.int16))


@pytest.mark.parametrize("layout", ["RM", "FLAT"])
def test_rank_layouts_agree_with_expert_major(layout):
    base = gen.SMALL["small_em"].with_(W=4, seed=43)
    case = make_case(base, "cuda")
    em = _out(base, case, 4, "EM").float().cpu().numpy().astype(np.float64)
    other = _out(base, case, 4, layout).float().cpu().numpy().astype(np.float64)
    # the fp32 sums differ only in association: by at most a few fp32 steps of the terms
    # (|w * y| below 8 here, so 1e-6 covers them), which after the rounding to bf16 is one
    # bf16 step of the result, or that absolute amount where the terms cancel
    step = np.ldexp(1.0, np.frexp(np.maximum(np.abs(em), np.abs(other)))[1] - 8)
    d = np.abs(em - other)
    print("%s vs EXPERT_MAJOR: %.4f of outputs equal, largest difference %.3g" % (layout, np.mean(d == 0), d.max()))
    assert np.all(d <= step + 1e-6)
    assert np.mean(d == 0) > 0.95
