"""The Python layer object checks every tensor it hands to the C ABI (dtype, shape,
contiguity, device) and raises before any library call; the C ABI takes bare pointers.
CPU only: the layer's buffers live in host memory here, so a call that passes the checks
reaches the library, which then refuses to launch without a GB300."""
import pytest
import torch

import combine_topk_ids_gb300 as moe

W, Tr, T, H, E, k, I = 2, 8, 12, 256, 4, 2, 128


@pytest.fixture(scope="module")
def layer():
    try:
        moe.lib()
    except RuntimeError:
        moe.build()
    return moe.MoELayer1GPU(W, Tr, T, H, E, k, I, "EM", "LL", device="cpu")


def good():
    return (torch.zeros((T, H), dtype=torch.bfloat16), torch.zeros((T, k), dtype=torch.int64),
            torch.zeros((T, k), dtype=torch.float32))


@pytest.mark.parametrize("which,bad,err", [
    (0, lambda: torch.zeros((T, H), dtype=torch.float32), TypeError),           # x not bf16
    (0, lambda: torch.zeros((T, H + 128), dtype=torch.bfloat16), ValueError),   # x of another width
    (0, lambda: torch.zeros((H, T), dtype=torch.bfloat16).t(), ValueError),     # x not contiguous
    (1, lambda: torch.zeros((T, k), dtype=torch.int16), TypeError),             # ids int16
    (1, lambda: torch.zeros((T, k + 1), dtype=torch.int64), ValueError),        # ids of another top_k
    (2, lambda: torch.zeros((T, k), dtype=torch.float64), TypeError),           # weights float64
    (2, lambda: [[0.5] * k] * T, TypeError),                                    # not a tensor
])
def test_forward_rejects_bad_inputs(layer, which, bad, err):
    args = list(good())
    args[which] = bad()
    with pytest.raises(err):
        layer.forward(*args)


def test_active_ranks_checked(layer):
    with pytest.raises(ValueError):
        layer.dispatch(*good(), active_ranks=torch.ones(W + 1, dtype=torch.int32))
    with pytest.raises(TypeError):
        layer.dispatch(*good(), active_ranks=torch.ones(W, dtype=torch.int64))


def test_set_weights_checks_shapes_and_dtypes(layer):
    w1 = torch.zeros((E, 2 * I, H), dtype=torch.bfloat16)
    w2 = torch.zeros((E, H, I), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        layer.set_weights(w1, torch.zeros((E, I, H), dtype=torch.bfloat16))   # w2 transposed
    with pytest.raises(TypeError):
        layer.set_weights(w1.float(), w2)
    with pytest.raises(ValueError):
        layer.set_weights(torch.zeros((E, 2 * I, H), dtype=torch.bfloat16)[:, ::2], w2)


def test_combine_checks_weights(layer):
    with pytest.raises(ValueError):
        layer.combine(torch.zeros((T + 1, k), dtype=torch.float32))


def test_expert_ffn_requires_weights():
    fresh = moe.MoELayer1GPU(W, Tr, T, H, E, k, I, "EM", "LL", device="cpu")
    with pytest.raises(RuntimeError, match="set_weights"):
        fresh.expert_ffn()


def test_valid_inputs_pass_the_checks(layer):
    # the checks pass; what stops the call here is the missing GPU (no CUDA stream on this
    # host, or the library's MoeError on a host without a GB300), not a TypeError/ValueError
    with pytest.raises(RuntimeError):
        layer.dispatch(*good())


def test_forward_host_checks_host_and_staging_tensors(layer):
    x, ids, w = good()
    out = torch.zeros((T, H), dtype=torch.bfloat16)
    rest = (layer.w1p, layer.w2, layer.expert_out, layer.workspace, moe.MoeHandle())
    with pytest.raises(TypeError):   # float32 rows
        moe.moe_forward_host(layer.geom, x.float(), ids, w, out, None, None, None, None, *rest)
    with pytest.raises(ValueError):  # output of another width
        moe.moe_forward_host(layer.geom, x, ids, w, out[:, :128], None, None, None, None, *rest)
    with pytest.raises(ValueError):  # a staging tensor of the wrong shape
        moe.moe_forward_host(layer.geom, x, ids, w, out, torch.zeros((T + 1, H), dtype=torch.bfloat16),
                             None, None, None, *rest)
    with pytest.raises(TypeError):   # ids missing
        moe.moe_forward_host(layer.geom, x, None, w, out, None, None, None, None, *rest)


def _cases():
    import gen
    names = list(gen.SMALL) + ["tiny_ll_em"]
    cfgs = [gen.ALL[n] for n in names]
    cfgs += [gen.SMALL["small_em"].with_(quant="fp8"), gen.SMALL["small_flat"].with_(expert_out="bf16"),
             gen.SMALL["small_rm"].with_(act="bf16"), gen.SMALL["small_em"].with_(ids_dtype="int32", mask_frac=0.3)]
    return cfgs


@pytest.mark.parametrize("cfg", _cases(), ids=lambda c: "%s-%s-%s-%s" % (c.name, c.quant, c.expert_out, c.act))
def test_checks_accept_what_the_gpu_tests_pass(cfg):
    """The inputs the GPU tests build for each geometry (gen.device.make_case) pass every
    check: the only error left on this GPU-less host is the missing device."""
    from gen.device import make_case
    case = make_case(cfg, "cpu")
    layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo,
                             device="cpu", quant=cfg.quant, expert_out=cfg.expert_out, act=cfg.act)
    for call in (lambda: layer.set_weights(case.w1, case.w2),
                 lambda: layer.dispatch(case.x, case.ids, case.w,
                                        torch.ones(cfg.W, dtype=torch.int32)),
                 lambda: layer.combine(case.w)):
        with pytest.raises(RuntimeError):
            call()
