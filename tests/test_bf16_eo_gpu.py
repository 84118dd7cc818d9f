"""bf16 expert_out option (MOE_EXPERT_OUT_BFLOAT16) against the oracle with the same rounding
points (oracle.layer(..., eo_bf16=True)).

The GPU rounds its fp32 GEMM results to bf16 where the oracle rounds exact values, so a
rounding can land on the other side of a bf16 tie: each held bf16 value may differ by one
bf16 ulp beyond the plain tolerance.  The checks: routing bit-exact; expert_out rows within
|d| <= 2e-2 |ref| + 1e-3 + the ulps of the roundings that produced the row; out within the
same bound carried through the routing weights.  The fraction of outputs that fall outside
the plain output bound (|d| <= 2e-2*|ref| + 1e-3) against the full-precision (float32 expert_out) oracle is the
cost of the option; it is checked to stay small and printed."""
import numpy as np
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from gen.device import make_case
from parity_util import ATOL, RTOL, act_flip_allowance, bf16_tensor_to_f64, check_routing, geom_dict

pytestmark = pytest.mark.gpu

CASES = {
    "eo16_small_em": gen.SMALL["small_em"],
    "eo16_small_rm": gen.SMALL["small_rm"],
    "eo16_small_flat": gen.SMALL["small_flat"],
    "eo16_pair_flat": gen.SMALL["pair_flat"],
    "eo16_tall_rm_h384": gen.SMALL["tall_rm"],
    "eo16_small_flat_k1": gen.SMALL["small_flat"].with_(k=1, seed=20),
    "eo16_world64_flat": gen.MoeConfig("eo16_world64_flat", W=64, Tr=4, H=256, E=128, k=4, I=128,
                                       layout="FLAT", algo="HT", routing="uniform", T=256),
    "eo16_small_em_h384": gen.SMALL["small_em"].with_(H=384, seed=6),
    "eo16_blocks_rm": gen.SMALL["blocks_rm"],
}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


def _ulp(v):
    """One bf16 ulp at |v| (8 significant bits)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    return np.where(v > 0, np.ldexp(1.0, np.frexp(v)[1] - 8), 0.0)


@pytest.mark.parametrize("name", list(CASES))
def test_bf16_expert_out_parity(name):
    cfg = CASES[name]
    case = make_case(cfg, "cuda")
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout,
                             cfg.algo, expert_out="bf16", act=cfg.act)
    assert layer.expert_out.dtype == torch.bfloat16
    layer.set_weights(case.w1, case.w2)
    layer.forward(case.x, case.ids, case.w)
    torch.cuda.synchronize()
    assert layer.status() == 0
    g = geom_dict(cfg)
    rt = oracle.route(g, case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    k, H, cap = cfg.k, cfg.H, cfg.W * cfg.Tr
    picks = [i for i in range(cfg.tokens * k) if rt["pick_pos"].reshape(-1)[i] >= 0]
    ys = oracle.pick_outputs(g, rt, case.x_bits, case.w1_host, case.w2_host, picks=picks)
    wv = case.w_np.astype(np.float64).reshape(-1)
    aflip = act_flip_allowance(layer, rt, case, picks)
    eo = bf16_tensor_to_f64(layer.expert_out.view(-1, H))
    # expert_out rows
    if cfg.layout == "EM":
        ref = oracle.round_bf16(np.array([ys[i] for i in picks]))
        got = eo[rt["slot"].reshape(-1)[picks]]
        extra = _ulp(ref) + np.array([aflip[i] * np.ones(H) for i in picks])
    else:
        rows = [(d, r) for d in range(cfg.W) for r in range(cap) if rt["recv_src"][d, r] >= 0]
        ref = oracle.ffn_ranks(g, rt, case.w_np, ys.__getitem__, rows, eo_bf16=True)
        got = eo[[d * cap + r for d, r in rows]]
        extra = _ulp(ref)
        for n, (d, r) in enumerate(rows):
            t = int(rt["recv_src"][d, r])
            for j in range(k):
                if rt["recv_topk_idx"][d, r, j] >= 0:
                    extra[n] += abs(float(rt["recv_topk_w"][d, r, j])) * (_ulp(ys[t * k + j])
                                                                          + aflip[t * k + j])
    bad = ~(np.abs(got - ref) <= RTOL * np.abs(ref) + ATOL + extra)
    assert not bad.any(), "expert_out: %d/%d outside tolerance" % (bad.sum(), bad.size)
    # combined output against the same rounding points
    _, out_ref = oracle.layer(g, case.x_bits, case.ids_np, case.w_np, case.w1_host, case.w2_host,
                              eo_bf16=True)
    allow = np.zeros((cfg.tokens, H))
    for i in picks:
        allow[i // k] += abs(wv[i]) * (2 * _ulp(ys[i]) + aflip[i])   # the pick's value, its row sum
    got_out = bf16_tensor_to_f64(layer.out)
    bad = ~(np.abs(got_out - out_ref) <= RTOL * np.abs(out_ref) + ATOL + allow)
    assert not bad.any(), "out: %d/%d outside tolerance" % (bad.sum(), bad.size)
    # the option's cost against the full-precision expert_out oracle
    _, out_full = oracle.layer(g, case.x_bits, case.ids_np, case.w_np, case.w1_host, case.w2_host)
    fail = float((np.abs(got_out - out_full) > RTOL * np.abs(out_full) + ATOL + allow).mean())
    print("%s: fraction of outputs outside the output bound vs the float32 expert_out "
          "oracle: %.2e" % (name, fail))
    assert fail < 2e-2

