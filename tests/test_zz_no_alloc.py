"""moe_route_noalloc (routing with no workspace and no allocation) against moe_dispatch.

Callers such as plugin hosts that own all device memory can pass only inputs and
outputs; this entry point serves them with a fixed scratch array inside the library.
Its outputs must equal the routing outputs of the regular dispatch, bit for bit, on
consecutive calls that share (and overwrite) that scratch array.  This file is collected
last so that a failure here cannot hide the rest of the suite.
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
    import os
    if not os.path.exists(moe.LIB_PATH):
        moe.build()


def _reference(cfg, case):
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo)
    layer.dispatch(case.x, case.ids, case.w)
    T, k, E, W = cfg.tokens, cfg.k, cfg.E, cfg.W
    i32 = torch.int32
    out = {"counts": layer.view("counts", (E,), i32), "offsets": layer.view("offsets", (E + 1,), i32),
           "pick_pos": layer.view("pick_pos", (T * k,), i32), "slot": layer.view("slot", (T * k,), i32),
           "layout_range": layout_view(layer, E, W), "pick_src": layer.view("pick_src", (T * k,), i32)}
    torch.cuda.synchronize()
    assert layer.status() == 0
    return {n: v.clone() for n, v in out.items()}


def layout_view(layer, E, W):
    return layer.view("layout_range", (E * W * 2,), torch.int32)


def _noalloc(cfg, case):
    T, k, E, W = cfg.tokens, cfg.k, cfg.E, cfg.W
    z = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")  # noqa: E731
    bufs = {"counts": z(E), "offsets": z(E + 1), "pick_pos": z(T * k), "pick_src": z(T * k),
            "slot": z(T * k), "layout_range": z(E * W * 2)}
    status = z(1)
    g = moe.make_geom(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo)
    moe.moe_route_noalloc(g, case.ids, bufs["counts"], bufs["offsets"], bufs["pick_pos"], bufs["pick_src"],
                          bufs["slot"], bufs["layout_range"], status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return bufs


@pytest.mark.parametrize("ids_dtype", ["int64", "int32"])
@pytest.mark.parametrize("name", ["small_em", "ragged_em"])
def test_noalloc_routing_matches_dispatch_on_consecutive_calls(name, ids_dtype):
    base = gen.ALL[name]
    cfgs = [base.with_(seed=seed, mask_frac=0.1, ids_dtype=ids_dtype) for seed in (21, 22)]
    cases = [make_case(c, "cuda") for c in cfgs]
    for c in cases:
        assert c.ids.dtype == getattr(torch, ids_dtype)
    refs = [_reference(c, cs) for c, cs in zip(cfgs, cases)]
    # two calls in a row on different batches: the second reuses the scratch the first left
    gots = [_noalloc(c, cs) for c, cs in zip(cfgs, cases)]
    for ref, got in zip(refs, gots):
        R = int(ref["offsets"][-1].item())
        for n in ("counts", "offsets", "pick_pos", "slot", "layout_range"):
            assert torch.equal(got[n], ref[n]), n
        assert torch.equal(got["pick_src"][:R], ref["pick_src"][:R])


def test_noalloc_rejects_geometries_beyond_its_scratch():
    # 2048 experts x 256 routing chunks need about 4 MiB of scratch, beyond the 1 MiB array
    g = moe.make_geom(8, 16384, 8, 128, 2048, 1, 128, "EM", "LL")
    ids = torch.zeros((8, 1), dtype=torch.int64, device="cuda")
    b = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_noalloc(g, ids, b, b, b, b, b, b, b)
    assert ei.value.code == -13
