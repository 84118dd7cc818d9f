"""The seeded input generator follows its stated recipe (gen/inputs.py): bf16 rounding of
normal draws, k distinct experts per token, the Zipf / Dirichlet skews, softmax routing
weights, masked picks, determinism; and the seed-0 Mixtral-like counts that the design
notes quote (three experts a few rows over 256: tail blocks of 2, 6 and 33 rows)."""
import numpy as np
import pytest
import torch

import gen
from gen.inputs import bf16_bits_to_f32, expert_weights_numpy, f32_to_bf16_bits


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        # exact ties between two bf16 values: round to the even one
                        (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    ours = f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_x_is_standard_normal_in_bf16():
    cfg = gen.CONFIGS["mixtral_ll_em"]
    x = bf16_bits_to_f32(gen.gen_x(cfg)).astype(np.float64)
    assert x.shape == (cfg.tokens, cfg.H)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_weights_are_bf16_normal_002():
    cfg = gen.SMALL["small_em"]
    w1, w2 = expert_weights_numpy(cfg, 3)
    assert w1.shape == (2 * cfg.I, cfg.H) and w2.shape == (cfg.H, cfg.I)
    v = bf16_bits_to_f32(np.concatenate([w1.ravel(), w2.ravel()])).astype(np.float64)
    assert abs(v.std() - 0.02) < 0.0005 and abs(v.mean()) < 0.0005
    # another expert draws from its own stream
    assert not np.array_equal(w1, expert_weights_numpy(cfg, 4)[0])


@pytest.mark.parametrize("name", ["mixtral_ll_em", "dsv3_ll_rm", "dsv3_ht_flat", "ragged_em", "tiny_ll_em"])
def test_routing_picks_distinct_experts_with_softmax_weights(name):
    cfg = gen.CONFIGS[name]
    ids, w = gen.gen_routing(cfg)
    assert ids.shape == (cfg.tokens, cfg.k) and ids.dtype == np.int64
    assert ids.min() >= 0 and ids.max() < cfg.E
    s = np.sort(ids, axis=1)
    assert (np.diff(s, axis=1) > 0).all()   # k distinct experts per token
    assert w.dtype == np.float32 and (w > 0).all()
    np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)


def test_routing_skews():
    counts = lambda cfg: np.bincount(gen.gen_routing(cfg)[0].ravel(), minlength=cfg.E)  # noqa: E731
    uni = counts(gen.CONFIGS["dsv3_ht_flat"])          # uniform: 1024 per expert on average
    assert uni.max() < 1.15 * uni.mean() and uni.min() > 0.85 * uni.mean()
    zipf = counts(gen.CONFIGS["dsv3_ll_rm"])           # Zipf(1.1), expert 0 hottest
    assert zipf.argmax() == 0
    assert zipf[:8].sum() > zipf[-128:].sum()
    diri = counts(gen.CONFIGS["ragged_em"])            # Dirichlet(0.1): many experts empty
    assert (diri == 0).sum() > 32 and diri.max() > 10 * diri.mean()


def test_seed0_mixtral_counts_quoted_in_the_design_notes():
    cfg = gen.CONFIGS["mixtral_ll_em"]
    c = np.bincount(gen.gen_routing(cfg)[0].ravel(), minlength=cfg.E)
    assert c.tolist() == [253, 243, 262, 258, 289, 253, 250, 240]
    tails = sorted(int(n % 128) for n in c if n > 256)
    assert tails == [2, 6, 33]


def test_masked_picks_and_int32_ids():
    cfg = gen.SMALL["blocks_flat"]                     # mask_frac 0.1
    ids, _ = gen.gen_routing(cfg)
    frac = (ids == -1).mean()
    assert 0.08 < frac < 0.12
    ids32, _ = gen.gen_routing(cfg.with_(ids_dtype="int32"))
    assert ids32.dtype == np.int32
    np.testing.assert_array_equal(ids32, ids)


def test_determinism_and_seed():
    cfg = gen.SMALL["small_rm"]
    a, b = gen.gen_routing(cfg), gen.gen_routing(cfg)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(gen.gen_x(cfg), gen.gen_x(cfg))
    c = gen.gen_routing(cfg.with_(seed=1))
    assert not np.array_equal(a[0], c[0])
