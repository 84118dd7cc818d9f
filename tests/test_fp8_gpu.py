"""FP8 variant (FP8 dispatch + FP8 grouped SwiGLU FFN) against the FP8 oracle through the C ABI.

Bit-exact: the weight quantisation (codes and block scales, in the interleaved W1 order),
the FP8-dispatched receive rows and their scales, routing.  The SwiGLU activation codes are
a rounding decision taken on tensor-core sums: each GPU code must be the oracle's or, where
the oracle's quotient lies within its accumulation band of a rounding midpoint, the other
neighbour (oracle.fp8.valid_act_codes).  expert_out and the combined output then match the
oracle within |d| <= 2e-2 |ref| + 1e-3 plus, per output, the effect of the activation codes
that legitimately differ (oracle.fp8.flip_allowance, carried through the routing weights)."""
import numpy as np
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from oracle import fp8
from gen.device import make_case
from parity_util import RTOL, ATOL, bf16_tensor_to_f64, check_routing, geom_dict

pytestmark = pytest.mark.gpu

CASES = {
    "f8_small_em": gen.SMALL["small_em"].with_(quant="fp8"),
    "f8_small_rm": gen.SMALL["small_rm"].with_(quant="fp8"),
    "f8_small_flat": gen.SMALL["small_flat"].with_(quant="fp8"),
    "f8_small_em_h384": gen.SMALL["small_em"].with_(quant="fp8", H=384, seed=6),   # 128-wide GEMM2 tiles
    "f8_pair_em": gen.SMALL["pair_em"].with_(quant="fp8"),                         # several m-blocks
    "f8_pair_flat_masked": gen.SMALL["pair_flat"].with_(quant="fp8", mask_frac=0.2, seed=9),
    "f8_tiny": gen.CONFIGS["tiny_ll_em"].with_(quant="fp8"),
    # second GEMM with fewer than three k-blocks per tile (direct row stores) and with
    # 128-column tiles; many routing blocks
    "f8_blocks_flat": gen.SMALL["blocks_flat"].with_(quant="fp8"),
    "f8_pair_rm": gen.SMALL["pair_rm"].with_(quant="fp8"),
    # limits: top_k 32 and world 64 (the row scatter writes up to 64 + 32 destinations)
    "f8_topk32_flat": gen.MoeConfig("f8_topk32_flat", W=4, Tr=16, H=256, E=64, k=32, I=128,
                                    layout="FLAT", algo="HT", routing="uniform", T=64, quant="fp8"),
    "f8_world64_rm": gen.MoeConfig("f8_world64_rm", W=64, Tr=4, H=256, E=64, k=4, I=128,
                                   layout="RM", algo="LL", routing="zipf", T=250, quant="fp8"),
    # 2048 experts (the limit), most with 0-4 rows, one Zipf-hot expert with a few hundred
    "f8_emax_em": gen.MoeConfig("f8_emax_em", W=8, Tr=64, H=256, E=2048, k=8, I=128,
                                layout="EM", algo="LL", routing="zipf", T=500, quant="fp8"),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


def _layer(cfg):
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout,
                             cfg.algo, quant="fp8")
    return layer


def _interleave_rows(a, I):
    """Prepared W1 row order: blocks of 128 gate rows and the matching 128 up rows alternate."""
    nb = I // 128
    blocks = [a[128 * b:128 * (b + 1)] for b in range(2 * nb)]
    out = []
    for j in range(nb):
        out += [blocks[j], blocks[nb + j]]
    return np.concatenate(out)


def test_weight_quantization_bit_exact():
    cfg = CASES["f8_small_em"]
    case = make_case(cfg, "cuda")
    layer = _layer(cfg)
    layer.set_weights(case.w1, case.w2)
    torch.cuda.synchronize()
    w1q, w1s = layer.w1p.cpu().numpy(), layer.w1s.cpu().numpy()
    w2q, w2s = layer.w2.cpu().numpy(), layer.w2s.cpu().numpy()
    for e in range(cfg.E):
        q1, s1 = fp8.quantize_blocks(oracle.bf16_bits_to_f64(case.w1_host[e]))
        q2, s2 = fp8.quantize_blocks(oracle.bf16_bits_to_f64(case.w2_host[e]))
        np.testing.assert_array_equal(w1q[e], _interleave_rows(q1, cfg.I))
        np.testing.assert_array_equal(w1s[e], _interleave_rows(np.repeat(s1, 128, 0), cfg.I)[::128])
        np.testing.assert_array_equal(w2q[e], q2)
        np.testing.assert_array_equal(w2s[e], s2)


def test_prepare_weights_fp8_interleaves_given_codes():
    cfg = CASES["f8_small_em"].with_(seed=21)
    case = make_case(cfg, "cuda")
    q = [fp8.quantize_blocks(oracle.bf16_bits_to_f64(case.w1_host[e])) for e in range(cfg.E)]
    w1q = torch.from_numpy(np.stack([a for a, _ in q])).cuda()
    w1s = torch.from_numpy(np.stack([b for _, b in q])).cuda()
    pq, ps = torch.empty_like(w1q), torch.empty_like(w1s)
    g = moe.make_geom(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo, "fp8")
    moe.moe_prepare_weights_fp8(g, w1q, w1s, pq, ps)
    torch.cuda.synchronize()
    for e in range(cfg.E):
        np.testing.assert_array_equal(pq[e].cpu().numpy(), _interleave_rows(q[e][0], cfg.I))
        np.testing.assert_array_equal(ps[e].cpu().numpy(),
                                      _interleave_rows(np.repeat(q[e][1], 128, 0), cfg.I)[::128])


@pytest.mark.parametrize("name", ["f8_small_em", "f8_small_rm", "f8_small_flat"])
def test_fp8_dispatch_bit_exact(name):
    cfg = CASES[name]
    case = make_case(cfg, "cuda")
    layer = _layer(cfg)
    layer.dispatch(case.x, case.ids, case.w)
    torch.cuda.synchronize()
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    rows, toks = oracle.dispatch_rows(geom_dict(cfg), rt)
    nrecv = (cfg.E if cfg.layout == "EM" else cfg.W) * cfg.W * cfg.Tr
    recv = layer.view("recv_x", (nrecv, cfg.H), torch.uint8).cpu().numpy()
    scales = layer.view("recv_scales", (cfg.H // 128, nrecv), torch.float32).cpu().numpy()
    codes, sc, _ = fp8.quantize_rows(oracle.bf16_bits_to_f64(case.x_bits))
    np.testing.assert_array_equal(recv[rows], codes[toks])
    np.testing.assert_array_equal(scales[:, rows].T, sc[toks])
    if cfg.layout != "EM":
        # the kept picks' rows in pick-list order (the first GEMM's operand), codes and scales
        R, P = rt["R"], cfg.tokens * cfg.k
        src = rt["pick_src"].astype(np.int64) // cfg.k
        prow = layer.view("pick_rows", (R, cfg.H), torch.uint8).cpu().numpy()
        psc = layer.view("pick_row_scales", (cfg.H // 128, P), torch.float32).cpu().numpy()
        np.testing.assert_array_equal(prow, codes[src])
        np.testing.assert_array_equal(psc[:, :R].T, sc[src])


def _check_layer(cfg, active=None, tokens=None, layer=None, case=None):
    """The FP8 layer against the FP8 oracle: every activation code of the checked picks valid,
    expert_out rows and out within the tolerance plus the flip allowance.  tokens: check only
    these tokens (their picks, received rows and outputs; full-size workloads)."""
    if layer is None:
        case = make_case(cfg, "cuda")
        layer = _layer(cfg)
        layer.set_weights(case.w1, case.w2)
        act_t = None if active is None else torch.as_tensor(active, dtype=torch.int32, device="cuda")
        layer.forward(case.x, case.ids, case.w, act_t)
        torch.cuda.synchronize()
    assert layer.status() == (0 if active is None else moe.STATUS_INACTIVE_RANK)
    g = geom_dict(cfg)
    rt, out_ref, res, w2d = fp8.layer_fp8(g, case.x_bits, case.ids_np, case.w_np, case.w1_host,
                                          case.w2_host, tokens=tokens, active=active)
    check_routing(layer, rt, cfg)
    toks = np.arange(cfg.tokens) if tokens is None else np.asarray(tokens)
    k, H, I, P = cfg.k, cfg.H, cfg.I, cfg.tokens * cfg.k
    R = rt["R"]
    picks = sorted(res)
    pos = torch.as_tensor([int(rt["pick_pos"].reshape(-1)[i]) for i in picks], dtype=torch.int64, device="cuda")
    act = layer.view("ffn_act", (max(R, 1), I), torch.uint8)[pos].cpu().numpy()
    act_s = layer.view("ffn_act_scales", (I // 128, P), torch.float32)[:, pos].cpu().numpy()
    ids = rt["ids"].reshape(-1)
    allow = {}
    n_flip = 0
    for n, i in enumerate(picks):
        r = res[i]
        gc, gs = act[n], act_s[:, n]
        ok = fp8.valid_act_codes(gc[None], r["act_quo"][None], r["act_band"][None])
        assert ok.all(), "pick %d: %d activation codes outside the oracle's band" % (i, (~ok).sum())
        np.testing.assert_allclose(gs, r["act_scales"], rtol=fp8.TC_REL * 4, atol=0)
        n_flip += int((gc != r["act_codes"]).sum())
        allow[i] = fp8.flip_allowance(gc[None], gs[None], r["act_codes"][None], r["act_scales"][None],
                                      w2d[int(ids[i])])[0]
    # expert_out
    eo = layer.expert_out.view(-1, H)
    cap = cfg.W * cfg.Tr
    wabs = np.abs(case.w_np.astype(np.float64)).reshape(-1)
    if cfg.layout == "EM":
        idx = torch.as_tensor(rt["slot"].reshape(-1)[picks], dtype=torch.int64, device="cuda")
        got = eo[idx].cpu().numpy().astype(np.float64)
        ref = np.array([res[i]["y"] for i in picks])
        extra = np.array([allow[i] for i in picks])
    else:
        rows = sorted({(d, int(rt["recv_row"][t, d])) for t in toks for d in range(cfg.W)
                       if rt["recv_row"][t, d] >= 0})
        ref = oracle.ffn_ranks(g, rt, case.w_np, lambda i: res[i]["y"], rows)
        idx = torch.as_tensor([d * cap + r for d, r in rows], dtype=torch.int64, device="cuda")
        got = eo[idx].cpu().numpy().astype(np.float64)
        extra = []
        for d, r in rows:
            t = int(rt["recv_src"][d, r])
            a = np.zeros(H)
            for j in range(k):
                if rt["recv_topk_idx"][d, r, j] >= 0:
                    a += abs(float(rt["recv_topk_w"][d, r, j])) * allow[t * k + j]
            extra.append(a)
        extra = np.array(extra)
    tol = RTOL * np.abs(ref) + ATOL
    bad = ~(np.abs(got - ref) <= tol + extra)
    assert not bad.any(), "expert_out: %d/%d outside tolerance" % (bad.sum(), bad.size)
    plain_fail = float((np.abs(got - ref) > tol).mean())
    # combined output: the allowance of every pick of the token, times |w|
    out_extra = np.zeros((len(toks), H))
    row_of = {int(t): n for n, t in enumerate(toks)}
    for i, a in allow.items():
        out_extra[row_of[i // k]] += wabs[i] * a
    got_out = bf16_tensor_to_f64(layer.out[torch.as_tensor(toks, dtype=torch.int64, device="cuda")])
    bad = ~(np.abs(got_out - out_ref) <= RTOL * np.abs(out_ref) + ATOL + out_extra)
    assert not bad.any(), "out: %d/%d outside tolerance" % (bad.sum(), bad.size)
    return n_flip, len(res) * I, plain_fail


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_layer_parity(name):
    n_flip, n_act, plain_fail = _check_layer(CASES[name])
    # flips are the rare exception; most outputs meet the plain tolerance with no allowance
    assert n_flip <= max(8, n_act // 500), (n_flip, n_act)
    assert plain_fail < 1e-2, plain_fail


def test_fp8_inactive_rank():
    cfg = CASES["f8_small_rm"].with_(seed=31)
    active = np.ones(cfg.W, np.int32)
    active[2] = 0
    _check_layer(cfg, active=active)


def test_fp8_handle_rejects_bf16_ffn():
    cfg = CASES["f8_tiny"]
    case = make_case(cfg, "cuda")
    layer = _layer(cfg)
    layer.set_weights(case.w1, case.w2)
    layer.dispatch(case.x, case.ids, case.w)
    with pytest.raises(moe.MoeError):
        moe.moe_expert_ffn(layer.handle, layer.w1p, layer.w2, layer.expert_out)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", list(gen.FP8))
def test_fp8_full_size(name):
    """The FP8 workloads at full size, in the launch configuration bench.py times: routing
    bit-exact; activation codes, expert_out and out on the picks of a few sampled tokens."""
    cfg = gen.FP8[name]
    case = make_case(cfg, "cuda")
    layer = _layer(cfg)
    layer.set_weights(case.w1, case.w2)
    layer.forward(case.x, case.ids, case.w)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    ntok = 4 if cfg.E * cfg.H * cfg.I <= (1 << 30) else 2
    toks = np.unique(np.concatenate([[0, cfg.tokens - 1], rng.choice(cfg.tokens, ntok, replace=False)]))
    n_flip, n_act, plain_fail = _check_layer(cfg, tokens=toks, layer=layer, case=case)
    assert n_flip <= max(8, n_act // 500), (n_flip, n_act)
    del layer, case
    torch.cuda.empty_cache()
