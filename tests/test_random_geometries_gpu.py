"""GPU layer against the CPU oracle on seeded random geometries.

Each case draws the logical world, experts, top-k, hidden and intermediate sizes, batch
size (ragged, sometimes empty), layout, routing skew, masked-pick fraction, id dtype and
activation precision, so that the sweep crosses the thresholds at which the library picks
its tile paths (128-row, two-SM, one-CTA 256-row tiles; 128- or 256-column second-GEMM
tiles) and its routing paths (one fused CTA or three kernels).  Routing and dispatched
rows bit for bit; expert_out and the output within |d| <= 2e-2*|ref| + 1e-3 (plus, for the
single-bf16 activation option, the allowance of the activation codes that differ)."""
import numpy as np
import pytest
import torch

import gen
import oracle
from gen.device import make_case
from parity_util import check_dispatch_rows, check_expert_out, check_out, check_routing, geom_dict, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_ids_gb300 as moe
    moe.build()


def random_config(seed):
    rng = np.random.default_rng(1000 + seed)
    W = int(rng.choice([1, 2, 4, 8]))
    long_k = rng.random() < 0.3           # a 4096-long first GEMM, one local expert per rank
    E = W if long_k else W * int(rng.integers(1, max(2, 64 // W) + 1))
    k = int(rng.integers(1, min(8, E) + 1))
    H = 4096 if long_k else 128 * int(rng.integers(1, 9))
    I = 128 * int(rng.integers(1, 5 if long_k else 7))
    Tr = int(rng.integers(300, 700)) if long_k else int(rng.integers(1, 600))
    T = int(rng.integers(0, W * Tr + 1)) if rng.random() < 0.9 else W * Tr
    layout = str(rng.choice(["EM", "RM", "FLAT"]))
    routing = str(rng.choice(["uniform", "zipf", "dirichlet"]))
    return gen.MoeConfig("rand%d" % seed, W=W, Tr=Tr, H=H, E=E, k=k, I=I, layout=layout,
                         algo="HT" if layout == "FLAT" else "LL", routing=routing, T=T,
                         seed=seed, ids_dtype=str(rng.choice(["int64", "int32"])),
                         mask_frac=float(rng.choice([0.0, 0.0, 0.15])),
                         act="bf16" if rng.random() < 0.2 else "pair")


@pytest.mark.parametrize("seed", range(24))
def test_random_geometry_parity(seed):
    cfg = random_config(seed)
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    check_dispatch_rows(layer, rt, case)
    if rt["R"] == 0:
        assert torch.count_nonzero(layer.out.float()).item() == 0
        return
    n_eo = check_expert_out(layer, rt, case)
    n_out = check_out(layer, case)
    if cfg.act == "pair":
        assert n_eo == 0 and n_out == 0
