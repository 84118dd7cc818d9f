"""The layer's accuracy at the shapes of the FlashInfer MoE-EP page's own accuracy check
("MoE-EP implementation & usage", section 4 "Usage walkthrough" for the configuration:
16 experts, top-8, 128 tokens per rank, hidden 8192, intermediate 2048, world 8; section 5
"Correctness status" for the figures): the page's EP layer matches a dense MoE to a
relative error of about 0.0045 on both LL layouts (EXPERT_MAJOR, RANK_MAJOR) and about
0.007 on HT FLAT at 4096 tokens per rank.

The page defines neither its relative error nor its comparator's precision.  Reading:
rel-err = ||out - ref||_F / ||ref||_F over the tokens compared, with ref the dense MoE
evaluated exactly (float64, no intermediate rounding: ref[t] = sum over j of
w[t, j] * W2[e] (silu(g) * u), [g; u] = W1[e] x[t]).  Every rounding this layer takes (the
bf16 activation, float32 accumulation, the bf16 output) counts against it, and its
figure must not exceed the page's.  On the same sampled tokens the output also meets the
element-wise bound against the oracle (which rounds where the layer does)."""
import numpy as np
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from gen.device import make_case
from parity_util import bf16_tensor_to_f64, check_out, geom_dict, run_layer

pytestmark = pytest.mark.gpu

# the page's reported relative errors, by layout
PAGE_REL_ERR = {"EM": 0.0045, "RM": 0.0045, "FLAT": 0.007}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


def exact_dense_moe(case, tokens):
    """ref[t] = sum_j w[t, j] * FFN_e(x[t]) in float64 with the activation unrounded (the
    oracle's expert with act="pair" keeps it unrounded), summed in ascending j."""
    cfg = case.cfg
    g = dict(geom_dict(cfg), act="pair")
    rt = oracle.route(g, case.ids_np, case.w_np)
    k = cfg.k
    picks = [int(t) * k + j for t in tokens for j in range(k) if rt["pick_pos"][t, j] >= 0]
    ys = oracle.pick_outputs(g, rt, case.x_bits, case.w1_host, case.w2_host, picks=picks)
    w = case.w_np.astype(np.float64)
    ref = np.zeros((len(tokens), cfg.H))
    for n, t in enumerate(tokens):
        for j in range(k):
            if rt["pick_pos"][t, j] >= 0:
                ref[n] += w[t, j] * ys[int(t) * k + j]
    return ref


@pytest.mark.parametrize("name", list(gen.ACCURACY))
def test_rel_err_within_the_pages_figure(name):
    cfg = gen.ACCURACY[name]
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    assert layer.status() == 0
    rng = np.random.default_rng(5)
    ntok = 16 if cfg.layout != "FLAT" else 8
    toks = np.array(sorted(set(rng.choice(cfg.tokens, size=ntok, replace=False).tolist()) | {cfg.tokens - 1}))
    check_out(layer, case, tokens=toks)
    got = bf16_tensor_to_f64(layer.out[torch.as_tensor(toks)])
    ref = exact_dense_moe(case, toks)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    print("%s: rel-err against the exact dense MoE %.5f (page: %.4f)" % (name, rel, PAGE_REL_ERR[cfg.layout]))
    assert rel <= PAGE_REL_ERR[cfg.layout], (name, rel)
    del layer, case
    torch.cuda.empty_cache()
