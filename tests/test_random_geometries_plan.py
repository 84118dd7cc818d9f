"""The seeded random geometries of the GPU sweep (test_random_geometries_gpu.py) reach every
GEMM tile path and both routing paths: checked on the host against the library's selection
rules, restated here (two-SM tiles: at least 192 rows per expert on average with K and N at
most 2048; one-CTA 256-row tiles: at least 512 rows per expert and K at least 4096; routing
in one CTA up to 3072 picks and 64 experts)."""
import numpy as np

import gen
from test_random_geometries_gpu import random_config

SEEDS = range(24)


def test_random_configs_cover_the_tile_paths():
    paths = set()
    for seed in SEEDS:
        c = random_config(seed)
        P = c.tokens * c.k
        for K, N in ((c.H, 2 * c.I), (c.I, c.H)):
            if P >= 192 * c.E and K <= 2048 and N <= 2048:
                paths.add("two-sm")
                # an expert's last 256-row block: its second CTA's half empty, or holding rows
                ids = gen.gen_routing(c)[0]
                rem = np.bincount(ids[ids >= 0], minlength=c.E) % 256
                if np.any((rem > 0) & (rem <= 128)):
                    paths.add("two-sm short last block")
                if np.any(rem > 128):
                    paths.add("two-sm long last block")
            elif P >= 512 * c.E and K >= 4096:
                paths.add("tall")
            else:
                paths.add("128-row")
        paths.add("fused-routing" if P <= 3072 and c.E <= 64 and c.E * c.W <= 4096 else "three-kernel-routing")
        paths.add("128-col" if c.H % 256 else "256-col")
        paths.add(c.layout)
        paths.add(c.act)
    assert {"two-sm", "two-sm short last block", "two-sm long last block", "tall", "128-row", "fused-routing", "three-kernel-routing", "128-col", "256-col",
            "EM", "RM", "FLAT", "pair", "bf16"} <= paths, paths


def test_fp8_random_configs_cover_the_paths():
    """The FP8 sweep (test_random_geometries_fp8_gpu.py) reaches all three layouts, both
    second-GEMM tile widths, a second GEMM of a single k-block, both routing paths and
    masked picks."""
    from test_random_geometries_fp8_gpu import SEEDS as F8_SEEDS, fp8_config
    paths = set()
    for seed in F8_SEEDS:
        c = fp8_config(seed)
        assert c.quant == "fp8"
        P = c.tokens * c.k
        paths.add(c.layout)
        paths.add("128-col" if c.H % 256 else "256-col")
        if c.I // 128 == 1:
            paths.add("one-k-block GEMM2")
        paths.add("fused-routing" if P <= 3072 and c.E <= 64 and c.E * c.W <= 4096 else "three-kernel-routing")
        if c.mask_frac > 0:
            paths.add("masked")
    assert {"EM", "RM", "FLAT", "128-col", "256-col", "one-k-block GEMM2", "fused-routing",
            "three-kernel-routing", "masked"} <= paths, paths
