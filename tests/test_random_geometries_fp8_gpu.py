"""FP8 layer against the FP8 oracle on seeded random geometries (the generator of the bf16
sweep, test_random_geometries_gpu.py, on its own seeds, with quant="fp8").

Each case draws world, experts, top-k, hidden and intermediate sizes, batch size (ragged,
sometimes empty), layout, routing skew, masked-pick fraction and id dtype, so the sweep
crosses the FP8 GEMMs' 128- and 256-column second-GEMM tiles, 1 to 64 k-blocks, both routing
paths and all three layouts.  Routing bit for bit; on 64 sampled tokens (all of them when
the batch is smaller) every activation code is the oracle's or its legitimate neighbour, and
expert_out and the output are within |d| <= 2e-2*|ref| + 1e-3 plus the allowance of the
codes that differ (test_fp8_gpu._check_layer)."""
import numpy as np
import pytest
import torch

from test_fp8_gpu import _check_layer
from test_random_geometries_gpu import random_config

pytestmark = pytest.mark.gpu

SEEDS = range(100, 112)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_ids_gb300 as moe
    moe.build()


def fp8_config(seed):
    return random_config(seed).with_(quant="fp8", act="pair")


@pytest.mark.parametrize("seed", SEEDS)
def test_random_geometry_fp8_parity(seed):
    cfg = fp8_config(seed)
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(cfg.tokens, size=min(64, cfg.tokens), replace=False))
    n_flip, n_act, plain_fail = _check_layer(cfg, tokens=toks)
    assert n_flip <= max(8, n_act // 500), (n_flip, n_act)
    assert plain_fail < 1e-2, plain_fail
