"""GPU layer vs the CPU oracle through the C ABI: routing and permuted rows bit-exact,
expert_out and the combined output within |d| <= 2e-2*|ref| + 1e-3."""
import numpy as np
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from gen.device import make_case
from parity_util import (assert_close, bf16_tensor_to_f64, check_dispatch_rows, check_expert_out,
                         check_out, check_routing, geom_dict, run_layer)

pytestmark = pytest.mark.gpu

SMALL_CASES = {
    "tiny_ll_em": gen.CONFIGS["tiny_ll_em"],
    "small_em": gen.SMALL["small_em"],
    "small_rm": gen.SMALL["small_rm"],
    "small_flat": gen.SMALL["small_flat"],
    "small_em_masked_i32": gen.SMALL["small_em"].with_(mask_frac=0.3, ids_dtype="int32", seed=3),
    "small_rm_masked": gen.SMALL["small_rm"].with_(mask_frac=0.3, seed=4),
    "small_flat_i32": gen.SMALL["small_flat"].with_(ids_dtype="int32", seed=5),
    "small_em_h384": gen.SMALL["small_em"].with_(H=384, seed=6),          # 128-wide GEMM2 tiles
    "small_flat_w1": gen.SMALL["small_flat"].with_(W=1, Tr=350, seed=7),  # one logical rank
    "small_rm_w8": gen.SMALL["small_rm"].with_(W=8, Tr=48, T=380, E=16, seed=8),
    # top-1: every received row has one local pick, so the second GEMM writes every
    # expert_out row itself and the local-pick reduction has nothing left to add
    "small_flat_k1": gen.SMALL["small_flat"].with_(k=1, seed=18),
    "small_rm_k1_masked": gen.SMALL["small_rm"].with_(k=1, mask_frac=0.2, seed=19),
    # two-SM GEMM tiles (many rows per expert)
    "pair_em": gen.SMALL["pair_em"],
    "pair_rm_h384": gen.SMALL["pair_rm"],
    "pair_flat": gen.SMALL["pair_flat"],
    "pair_em_masked_i32": gen.SMALL["pair_em"].with_(mask_frac=0.2, ids_dtype="int32", seed=9),
    # one-CTA 256-row GEMM tiles (long K loops, many rows per expert)
    "tall_em": gen.SMALL["tall_em"],
    "tall_rm_h384": gen.SMALL["tall_rm"],
    "tall_flat": gen.SMALL["tall_flat"],
    "tall_flat_h4096": gen.SMALL["tall_flat"].with_(H=4096, I=512, seed=17),
    "tall_em_masked_i32": gen.SMALL["tall_em"].with_(mask_frac=0.2, ids_dtype="int32", seed=16),
    # the 256-row tiles in dynamic order with fewer tiles than CTAs (one expert, 600 rows:
    # three row blocks, the last a short 88-row tail, one n-block)
    "tall_few_tiles": gen.MoeConfig("tall_few_tiles", W=1, Tr=600, H=4096, E=1, k=1, I=128,
                                    layout="EM", algo="LL", routing="uniform", T=600),
    # multi-block routing (more than 3072 picks; these hold more than 16384)
    "blocks_em": gen.SMALL["blocks_em"],
    "blocks_rm": gen.SMALL["blocks_rm"],
    "blocks_flat": gen.SMALL["blocks_flat"],
    # limits: top_k = 32 (every lane of the warp-level routing busy), world = 64 (64-bit
    # destination masks, ranks lane and lane + 32 in the scans), one local expert per rank
    "topk32_em": gen.MoeConfig("topk32_em", W=2, Tr=32, H=256, E=64, k=32, I=128,
                               layout="EM", algo="LL", routing="uniform", T=64),
    "topk32_flat": gen.MoeConfig("topk32_flat", W=4, Tr=16, H=256, E=64, k=32, I=128,
                                 layout="FLAT", algo="HT", routing="uniform", T=64),
    "world64_rm": gen.MoeConfig("world64_rm", W=64, Tr=4, H=256, E=64, k=4, I=128,
                                layout="RM", algo="LL", routing="zipf", T=250),
    "world64_flat": gen.MoeConfig("world64_flat", W=64, Tr=4, H=256, E=128, k=4, I=128,
                                  layout="FLAT", algo="HT", routing="uniform", T=256),
    # the most experts the library accepts (MOE_MAX_EXPERTS = 2048): 2048-entry count and
    # offset scans over the routing chunks, tile enumeration over mostly empty experts
    # (0-4 rows each); FLAT also at world 64 (32 local experts per rank)
    "emax_em": gen.MoeConfig("emax_em", W=8, Tr=64, H=256, E=2048, k=8, I=128,
                             layout="EM", algo="LL", routing="zipf", T=500),
    "emax_flat": gen.MoeConfig("emax_flat", W=64, Tr=8, H=256, E=2048, k=8, I=128,
                               layout="FLAT", algo="HT", routing="dirichlet", T=512),
    # the widest hidden the library accepts (MOE_MAX_HIDDEN = 65536): a 65536-long K loop
    # in the first GEMM (1024 k-blocks), 256 n-tiles in the second, 64 copy chunks per row
    "hmax_em": gen.MoeConfig("hmax_em", W=2, Tr=8, H=65536, E=4, k=2, I=128,
                             layout="EM", algo="LL", routing="uniform", T=13),
    "hmax_flat": gen.MoeConfig("hmax_flat", W=2, Tr=8, H=65536, E=4, k=2, I=128,
                               layout="FLAT", algo="HT", routing="uniform", T=13),
    # the single-bf16 activation option (one bf16 operand of the second GEMM; its codes are
    # rounding decisions checked against the oracle's band, and the outputs get the
    # allowance of the codes that differ); the tall cases take the one-CTA 256-row tiles
    # in the second GEMM too, which only this option uses
    "act16_em": gen.SMALL["small_em"].with_(act="bf16", seed=13),
    "act16_rm_h384": gen.SMALL["small_rm"].with_(act="bf16", H=384, seed=14),
    "act16_twosm_flat": gen.SMALL["pair_flat"].with_(act="bf16", seed=15),
    "act16_tall_em": gen.SMALL["tall_em"].with_(act="bf16"),
    "act16_tall_rm_h384": gen.SMALL["tall_rm"].with_(act="bf16"),
    "act16_tall_flat": gen.SMALL["tall_flat"].with_(act="bf16"),
    "act16_hmax_flat": gen.MoeConfig("act16_hmax_flat", W=2, Tr=8, H=65536, E=4, k=2, I=128,
                                     layout="FLAT", algo="HT", routing="uniform", T=13, act="bf16"),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_layer_parity_small(name):
    cfg = SMALL_CASES[name]
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    n_eo = check_expert_out(layer, rt, case)
    n_out = check_out(layer, case)
    if cfg.act == "pair":
        # the default activation meets the plain bound with no allowance at all
        assert n_eo == 0 and n_out == 0


@pytest.mark.parametrize("name", ["small_em", "small_rm", "small_flat", "pair_em", "pair_flat"])
def test_deterministic(name):
    cfg = SMALL_CASES[name]
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    out1, eo1 = layer.out.clone(), layer.expert_out.clone()
    run_layer(case, layer)
    assert torch.equal(layer.out.view(torch.int16), out1.view(torch.int16))
    # expert_out rows that hold data (padding rows are unspecified)
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    H, cap = cfg.H, cfg.W * cfg.Tr
    if cfg.layout == "EM":
        rows = rt["slot"].reshape(-1)
        rows = rows[rows >= 0]
    else:
        d, r = np.nonzero(rt["recv_src"] >= 0)
        rows = d * cap + r
    idx = torch.from_numpy(np.asarray(rows, np.int64)).cuda()
    assert torch.equal(layer.expert_out.view(-1, H)[idx], eo1.view(-1, H)[idx])


@pytest.mark.parametrize("layout", ["EM", "RM", "FLAT"])
def test_combine_alone_on_seeded_expert_out(layout):
    """combine on an expert_out drawn by the generator (not produced by the GPU path)."""
    cfg = SMALL_CASES["small_" + layout.lower()].with_(seed=11)
    case = make_case(cfg, "cuda")
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo)
    layer.dispatch(case.x, case.ids, case.w)
    rng = np.random.default_rng(123)
    eo_np = rng.standard_normal(layer.expert_out.numel()).astype(np.float32)
    layer.expert_out.copy_(torch.from_numpy(eo_np))
    out = torch.empty((cfg.tokens, cfg.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(layer.handle, layer.expert_out, case.w, out)
    torch.cuda.synchronize()
    g = geom_dict(cfg)
    rt = oracle.route(g, case.ids_np, case.w_np)
    eo = eo_np.reshape(-1, cfg.H).astype(np.float64)
    cap = cfg.W * cfg.Tr
    toks = np.arange(cfg.tokens)
    if layout == "EM":
        ref = oracle.combine_em(g, rt, case.w_np, lambda i: eo[rt["slot"].reshape(-1)[i]], toks)
    else:
        ref = oracle.combine_ranks(g, rt, lambda d, r: eo[d * cap + r], toks)
    got = bf16_tensor_to_f64(out)
    # fp32 sum vs float64 sum, both rounded once to bf16: at most one bf16 step apart
    np.testing.assert_allclose(got, ref, rtol=2 ** -7, atol=1e-30)


def test_identity_expert_via_recv_buffer():
    """expert_out := fp32(recv): EM combine equals bf16(x * sum of kept weights)."""
    cfg = SMALL_CASES["small_em"].with_(mask_frac=0.2, seed=12)
    case = make_case(cfg, "cuda")
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo)
    layer.dispatch(case.x, case.ids, case.w)
    nrows = cfg.E * cfg.W * cfg.Tr
    recv = layer.view("recv_x", (nrows, cfg.H), torch.bfloat16)
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    rows = torch.from_numpy(np.asarray(oracle.dispatch_rows(geom_dict(cfg), rt)[0], np.int64)).cuda()
    eo = layer.expert_out.view(nrows, cfg.H)
    eo[rows] = recv[rows].float()
    layer.combine(case.w)
    torch.cuda.synchronize()
    ws = np.where(case.ids_np >= 0, case.w_np.astype(np.float64), 0.0).sum(axis=1)
    ref = oracle.round_bf16(oracle.bf16_bits_to_f64(case.x_bits) * ws[:, None])
    np.testing.assert_allclose(bf16_tensor_to_f64(layer.out), ref, rtol=2 ** -7, atol=1e-30)


@pytest.mark.parametrize("name", ["small_em", "tall_em", "tall_flat", "tall_few_tiles"])
def test_ffn_twice_on_one_dispatch(name):
    """moe_expert_ffn run twice on the same dispatch gives the same expert_out bit for bit:
    the first GEMM's dynamic tile order (256-row tiles) leaves its tile counter at zero for
    the next launch, which here is not preceded by a dispatch that would zero it."""
    cfg = SMALL_CASES[name]
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    H, cap = cfg.H, cfg.W * cfg.Tr
    if cfg.layout == "EM":
        rows = rt["slot"].reshape(-1)
        rows = rows[rows >= 0]
    else:
        d, r = np.nonzero(rt["recv_src"] >= 0)
        rows = d * cap + r
    idx = torch.from_numpy(np.asarray(rows, np.int64)).cuda()
    first = layer.expert_out.view(-1, H)[idx].clone()
    out1 = layer.out.clone()
    for _ in range(2):
        layer.expert_out.zero_()
        layer.expert_ffn()
        layer.combine(case.w)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(layer.expert_out.view(-1, H)[idx], first)
        assert torch.equal(layer.out.view(torch.int16), out1.view(torch.int16))


M64_CASES = {
    # 128-row tiles (under 192 rows per expert on average): last blocks of 64 / 65 rows,
    # a second block of 64 / 65, one row, 63 and 127 rows, an empty expert
    "m64_rows128_em": (dict(W=2, Tr=400, H=256, E=8, k=1, I=256, layout="EM", algo="LL"),
                       [64, 65, 192, 193, 1, 0, 63, 127]),
    "m64_rows128_flat": (dict(W=2, Tr=400, H=256, E=8, k=1, I=256, layout="FLAT", algo="HT"),
                         [64, 65, 192, 193, 1, 0, 63, 127]),
    # one-CTA 256-row tiles in the first GEMM (K 4096, >= 512 rows per expert on average):
    # last blocks of 64 and 65 rows (M = 64 or 128 on the first half) and of 192 and 193
    # rows (M = 64 or 128 on the second half); the second GEMM's 128-row tiles see 64/65 too
    "m64_tall_em": (dict(W=2, Tr=1100, H=4096, E=4, k=1, I=256, layout="EM", algo="LL"),
                    [576, 577, 448, 449]),
}


@pytest.mark.parametrize("name", list(M64_CASES))
def test_m64_block_boundaries(name):
    """Blocks of 64 rows or fewer take M = 64 MMAs (accumulator rows 16 per lane quarter):
    every boundary of that rule, against the oracle at the plain bound."""
    geo, counts = M64_CASES[name]
    T = sum(counts)
    cfg = gen.MoeConfig(name, routing="uniform", T=T, seed=63, **geo)
    ids = np.repeat(np.arange(len(counts)), counts)
    ids = np.random.default_rng(63).permutation(ids).reshape(T, 1).astype(np.int64)
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    assert list(rt["counts"]) == counts
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    n_eo = check_expert_out(layer, rt, case)
    n_out = check_out(layer, case)
    assert n_eo == 0 and n_out == 0


@pytest.mark.parametrize("name", ["tall_em", "tall_flat", "pair_em", "pair_flat", "small_flat"])
def test_repeated_calls_alternating_batches(name):
    """Forty forwards on one layer alternating between two batches of different routing:
    each output equals the first output of its batch bit for bit and the status stays
    clear, so nothing a call leaves behind (the 256-row tiles' tile counter and ring, the
    two-SM clusters' hand-offs, the routing state in the workspace) changes a later call."""
    cfg = SMALL_CASES[name]
    cases = [make_case(cfg.with_(seed=70 + i, routing=r), "cuda")
             for i, r in enumerate(["zipf", "uniform"])]
    layer = run_layer(cases[0])
    first = [layer.out.clone(), None]
    run_layer(cases[1], layer)
    first[1] = layer.out.clone()
    assert not torch.equal(first[0].view(torch.int16), first[1].view(torch.int16))
    outs = []
    for i in range(40):   # back to back on the stream; each output copied on the stream too
        c = i % 2
        layer.forward(cases[c].x, cases[c].ids, cases[c].w)
        outs.append(layer.out.clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), first[i % 2].view(torch.int16)), i


# ----------------------------------------------------------------------- edge cases
def test_empty_batch():
    cfg = SMALL_CASES["small_rm"].with_(T=0)
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    assert layer.status() == 0
    assert layer.view("counts", (cfg.E,), torch.int32).sum().item() == 0
    assert layer.out.numel() == 0


@pytest.mark.parametrize("layout", ["EM", "FLAT"])
def test_all_picks_masked(layout):
    cfg = SMALL_CASES["small_" + layout.lower()]
    ids = np.full((cfg.tokens, cfg.k), -1, np.int64)
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == 0
    assert torch.count_nonzero(layer.out.float()).item() == 0


def test_bad_ids_are_flagged_and_dropped():
    cfg = SMALL_CASES["small_rm"].with_(seed=13)
    ids, _ = gen.gen_routing(cfg)
    ids[5, 1] = cfg.E + 3
    ids[17, 0] = -7
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == moe.STATUS_BAD_EXPERT_ID
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    assert rt["n_bad"] == 2
    check_routing(layer, rt, cfg)
    check_out(layer, case)


@pytest.mark.parametrize("name", ["small_em", "small_rm", "small_flat", "blocks_rm", "pair_flat"])
def test_inactive_ranks_are_masked(name):
    """EP rank-health mask: picks on a failed rank and tokens owned by it are dropped."""
    cfg = SMALL_CASES[name].with_(seed=31)
    active = np.ones(cfg.W, np.int32)
    active[1] = 0
    case = make_case(cfg, "cuda")
    layer = run_layer(case, active=active)
    assert layer.status() == moe.STATUS_INACTIVE_RANK
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np, active)
    assert rt["n_inactive"] > 0
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    check_out(layer, case, active=active)


@pytest.mark.parametrize("name", ["small_em", "small_rm", "small_flat", "pair_flat"])
def test_duplicate_experts_in_a_token(name):
    """Ids drawn with replacement (-1 included): a token may name one expert twice or more
    (reading 7: separate picks in (t, j) order).  On RANK_MAJOR / FLAT such picks share one
    received row and are summed there in ascending j; the rest is the usual path."""
    cfg = SMALL_CASES[name].with_(seed=57)
    rng = np.random.default_rng(57)
    ids = rng.integers(-1, cfg.E, size=(cfg.tokens, cfg.k)).astype(np.int64)
    dup = sum(len(r[r >= 0]) - len(set(r[r >= 0].tolist())) for r in ids)
    assert dup > 0
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    n_eo = check_expert_out(layer, rt, case)
    n_out = check_out(layer, case)
    assert n_eo == 0 and n_out == 0


def test_expert_major_region_overflow():
    """A token naming one expert twice can overflow the W*Tr-row EM region: the extra picks
    are dropped and flagged, the rest matches the oracle."""
    cfg = gen.MoeConfig("ovf", W=1, Tr=6, H=256, E=2, k=3, I=128, layout="EM", algo="LL",
                        routing="uniform")
    ids = np.array([[0, 0, 1], [0, 1, 0], [1, 1, 1], [0, 0, 0], [1, 0, -1], [0, 1, 1]])
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == moe.STATUS_EM_OVERFLOW
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    assert rt["n_over"] > 0
    check_routing(layer, rt, cfg)
    check_out(layer, case)


@pytest.mark.parametrize("layout,T", [("EM", 350), ("EM", 256), ("FLAT", 350)])
def test_every_pick_on_one_expert(layout, T):
    """All tokens pick expert 2 (top-1): one expert holds every row (several full 128-row
    blocks, or an exact multiple of 128), the others none, so most experts issue no tiles."""
    cfg = gen.MoeConfig("onehot", W=2, Tr=200, H=512, E=4, k=1, I=384, layout=layout,
                        algo="LL", routing="uniform", T=T)
    ids = np.full((T, 1), 2, np.int64)
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    n_eo = check_expert_out(layer, rt, case)
    n_out = check_out(layer, case)
    if cfg.act == "pair":
        # the default activation meets the plain bound with no allowance at all
        assert n_eo == 0 and n_out == 0


@pytest.mark.parametrize("layout,act", [("EM", "pair"), ("RM", "pair"), ("FLAT", "pair"), ("EM", "bf16")])
def test_two_sm_block_boundaries(layout, act):
    """Experts with 256, 384, 385, 128, 129, 0, 1 and 317 rows (top-1, 1600 picks over 8
    experts: two-SM 256-row tiles in both GEMMs): a last block that is full, holds exactly
    128 or 129 rows (the second CTA's half empty or holding one row), a single row, or
    nothing, and an empty expert."""
    counts = [256, 384, 385, 128, 129, 0, 1, 317]
    T = sum(counts)
    cfg = gen.MoeConfig("tails", W=2, Tr=800, H=256, E=8, k=1, I=256, layout=layout,
                        algo="HT" if layout == "FLAT" else "LL", routing="uniform", T=T,
                        seed=61, act=act)
    ids = np.repeat(np.arange(8), counts)
    ids = np.random.default_rng(61).permutation(ids).reshape(T, 1).astype(np.int64)
    case = make_case(cfg, "cuda", ids_override=ids)
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    assert list(rt["counts"]) == counts
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    n_eo = check_expert_out(layer, rt, case)
    n_out = check_out(layer, case)
    if act == "pair":
        assert n_eo == 0 and n_out == 0
