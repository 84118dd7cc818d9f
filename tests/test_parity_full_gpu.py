"""The five workloads at full size, in the launch configuration bench.py times:
routing and every permuted row bit-exact against the oracle, expert_out and the combined
output on sampled rows / tokens that the oracle evaluates one by one."""
import numpy as np
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from gen.device import make_case
from parity_util import check_dispatch_rows, check_expert_out, check_out, check_routing, geom_dict, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


def _sample(n_total, n, seed):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(n_total, size=min(n, n_total), replace=False).tolist())
    pick |= {0, n_total - 1}
    return np.array(sorted(pick))


@pytest.mark.parametrize("name", list(gen.CONFIGS))
def test_full_size(name):
    cfg = gen.CONFIGS[name]
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    assert layer.status() == 0
    g = geom_dict(cfg)
    rt = oracle.route(g, case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    ntok = 64 if cfg.E * cfg.H * cfg.I <= (1 << 30) else 6
    toks = _sample(cfg.tokens, ntok, 1)
    if cfg.layout == "EM":
        picks = np.array([t * cfg.k + j for t in toks for j in range(cfg.k) if rt["pick_pos"][t, j] >= 0])
        check_expert_out(layer, rt, case, picks_or_rows=picks)
    else:
        rows = [(d, int(rt["recv_row"][t, d])) for t in toks for d in range(cfg.W) if rt["recv_row"][t, d] >= 0]
        check_expert_out(layer, rt, case, picks_or_rows=rows)
    check_out(layer, case, tokens=toks)
    del layer, case
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["mixtral_ll_em_eo16", "dsv3_ll_rm_eo16", "ragged_em_eo16"])
def test_full_size_bf16_expert_out(name):
    """The bf16 expert_out option at full size: on sampled tokens, the fraction of outputs
    outside the output bound (|d| <= 2e-2*|ref| + 1e-3) against the full-precision (float32 expert_out) oracle."""
    cfg = gen.ALL[name]
    case = make_case(cfg, "cuda")
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout,
                             cfg.algo, expert_out="bf16")
    layer.set_weights(case.w1, case.w2)
    layer.forward(case.x, case.ids, case.w)
    torch.cuda.synchronize()
    assert layer.status() == 0
    toks = _sample(cfg.tokens, 16 if cfg.E * cfg.H * cfg.I <= (1 << 30) else 4, 2)
    _, ref = oracle.layer(geom_dict(cfg), case.x_bits, case.ids_np, case.w_np, case.w1_host,
                          case.w2_host, tokens=toks)
    got = oracle.bf16_bits_to_f64(layer.out[torch.as_tensor(toks)].contiguous().view(torch.int16)
                                  .cpu().numpy().view(np.uint16))
    fail = float((np.abs(got - ref) > 2e-2 * np.abs(ref) + 1e-3).mean())
    print("%s: fraction outside the output bound vs the float32 expert_out oracle: %.2e"
          % (name, fail))
    assert fail < 2e-2
    del layer, case
    torch.cuda.empty_cache()
