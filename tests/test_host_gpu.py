"""moe_forward_host (the layer from host buffers) against the device-buffer calls.

With page-locked host tensors the kernels read the inputs from host memory and the
combine writes the output there directly; with pageable tensors the call stages copies
through the device buffers.  Both must give the device path's output bit for bit (the same
kernels on the same values), on two calls in a row."""
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


CASES = {n: gen.ALL[n] for n in ("small_em", "small_rm", "small_flat", "tiny_ll_em", "pair_flat", "blocks_flat")}
CASES["small_flat_eo16"] = gen.ALL["small_flat"].with_(expert_out="bf16", seed=31)
CASES["small_rm_eo16"] = gen.ALL["small_rm"].with_(expert_out="bf16", seed=32)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_matches_device_path(name, pinned):
    """For RANK_MAJOR / FLAT the host call folds the rank reduction into the combine; its
    expert_out is scratch, filled with NaN before each call here, so that reading a row it
    leaves unwritten would show in the output."""
    cfg = CASES[name]
    case = make_case(cfg, "cuda")
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo,
                             expert_out=cfg.expert_out)
    layer.set_weights(case.w1, case.w2)
    layer.forward(case.x, case.ids, case.w)
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = layer.out.cpu().view(torch.int16).clone()

    host = (lambda t: t.cpu().pin_memory()) if pinned else (lambda t: t.cpu())
    x_h, ids_h, w_h = host(case.x), host(case.ids), host(case.w)
    out_h = torch.full((cfg.tokens, cfg.H), float("nan"), dtype=torch.bfloat16)
    if pinned:
        out_h = out_h.pin_memory()
        stage = (None, None, None, None)   # not used with page-locked buffers
    else:
        stage = (torch.empty_like(case.x), torch.empty_like(case.ids), torch.empty_like(case.w),
                 torch.empty_like(layer.out))
    h = moe.MoeHandle()
    for _ in range(2):
        out_h.fill_(float("nan"))
        layer.expert_out.fill_(float("nan"))
        moe.moe_forward_host(layer.geom, x_h, ids_h, w_h, out_h, *stage, layer.w1p, layer.w2,
                             layer.expert_out, layer.workspace, h)
        torch.cuda.synchronize()
        assert moe.moe_get_status(h) == 0
        assert torch.equal(out_h.view(torch.int16), ref)
