"""Pins of the FP8 oracle (oracle/fp8.py) against things other than itself (CPU only).

- the e4m3 code table against closed forms of the format and a hand-worked example
  (tests/golden/fp8_hand_example.json);
- round-to-nearest-even to e4m3 against torch's float8_e4m3fn conversion on every code,
  every rounding midpoint and its float32 neighbours, and random values;
- the row and block quantisers against the same steps done with torch float32 ops and
  torch's float8 cast, plus their invariants (largest code 448, reconstruction within
  half an e4m3 step);
- the FP8 expert against torch float64 matmuls of the dequantised operands, and against
  the full-precision bf16 oracle within the FP8 error;
- the activation band against a real float32 evaluation of the expert;
- planted mistakes are caught.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F8 = torch.float8_e4m3fn


def torch_e4m3(v32):
    """Codes of torch's float32 -> float8_e4m3fn cast (valid below 464 in magnitude)."""
    return torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(F8).view(torch.uint8).numpy()


# ------------------------------------------------------------------------ code table
def test_e4m3_table_closed_forms():
    v = fp8.e4m3_values()
    assert v[0x00] == 0.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    assert v[0x01] == 2.0 ** -9           # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9       # largest subnormal
    assert v[0x08] == 2.0 ** -6           # smallest normal
    assert v[0x38] == 1.0                 # exponent field 7 = bias
    assert v[0x7E] == 448.0               # largest finite: 1.75 * 2**8
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.all(np.diff(v[:127]) > 0)   # codes increase with value
    np.testing.assert_array_equal(v[0x80:0xFF], -v[0x00:0x7F])
    # the table agrees with torch's float8 decode
    t = torch.arange(256, dtype=torch.uint8).view(F8).float().numpy().astype(np.float64)
    fin = ~np.isnan(v)
    np.testing.assert_array_equal(v[fin], t[fin])


def test_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "fp8_hand_example.json")))
    x = np.array(g["row"], dtype=np.float64)[None, :]
    codes, scales, _ = fp8.quantize_rows(x)
    assert scales[0, 0] == np.float32(g["scale"])
    np.testing.assert_array_equal(codes[0, :len(g["codes"])], np.array(g["codes"], np.uint8))


# --------------------------------------------------------------------------- rounding
def _probe_values():
    v = fp8.e4m3_values()[:127]
    mids = 0.5 * (v[:-1] + v[1:])
    pts = np.concatenate([v, mids]).astype(np.float32)
    nb = np.concatenate([pts, np.nextafter(pts, np.float32(np.inf)), np.nextafter(pts, np.float32(0))])
    rng = np.random.default_rng(5)
    rnd = np.concatenate([rng.uniform(-463, 463, 20000), rng.uniform(-0.02, 0.02, 20000),
                          rng.standard_normal(20000) * 10]).astype(np.float32)
    allv = np.concatenate([nb, -nb, rnd])
    return allv[np.abs(allv) < 464]


def test_round_e4m3_matches_torch():
    v = _probe_values()
    np.testing.assert_array_equal(fp8.round_e4m3(v.astype(np.float64)), torch_e4m3(v))


def test_round_e4m3_saturates_and_round_trips():
    big = np.array([464.0, 480.0, 1e6, 3.4e38], np.float32)
    assert np.all(fp8.round_e4m3(big.astype(np.float64)) == 0x7E)
    assert np.all(fp8.round_e4m3(-big.astype(np.float64)) == 0xFE)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(fp8.round_e4m3(fp8.decode_e4m3(codes)), codes)
    # ties go to the even code: 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39)
    assert fp8.round_e4m3(np.array([1.0625]))[0] == 0x38
    assert fp8.round_e4m3(np.array([1.1875]))[0] == 0x3A


# ------------------------------------------------------------------------ quantisers
def _torch_rows(x):
    t = torch.from_numpy(np.asarray(x, np.float32))
    n, C = t.shape
    b = t.view(n, C // 128, 128)
    amax = b.abs().amax(dim=2).clamp_min(2.0 ** -100)
    scale = amax / 448.0
    inv = torch.full_like(amax, 448.0) / amax    # tensor / tensor: IEEE division
    q = (b * inv[:, :, None]).clamp(-448.0, 448.0).to(F8).view(torch.uint8)
    return q.reshape(n, C).numpy(), scale.numpy()


def _torch_blocks(w):
    t = torch.from_numpy(np.asarray(w, np.float32))
    R, C = t.shape
    b = t.view(R // 128, 128, C // 128, 128)
    amax = b.abs().amax(dim=(1, 3)).clamp_min(2.0 ** -100)
    inv = torch.full_like(amax, 448.0) / amax
    q = (b * inv[:, None, :, None]).clamp(-448.0, 448.0).to(F8).view(torch.uint8)
    return q.reshape(R, C).numpy(), (amax / 448.0).numpy()


@pytest.mark.parametrize("seed", range(4))
def test_quantize_rows_matches_torch_steps(seed):
    rng = np.random.default_rng(seed)
    x = oracle.round_bf16(rng.standard_normal((37, 512)) * (10.0 ** rng.uniform(-3, 3, (37, 1))))
    x[3, 128:256] = 0.0                   # an all-zero block
    x[4, :128] *= 1e-36                   # a block below the scale floor
    codes, scales, _ = fp8.quantize_rows(x)
    tq, ts = _torch_rows(x)
    np.testing.assert_array_equal(codes, tq)
    np.testing.assert_array_equal(scales, ts)


def test_quantize_rows_invariants():
    rng = np.random.default_rng(9)
    x = oracle.round_bf16(rng.standard_normal((50, 1024)) * 3)
    codes, scales, _ = fp8.quantize_rows(x)
    v = np.abs(fp8.decode_e4m3(codes)).reshape(50, 8, 128)
    assert np.all(v.max(axis=2) == 448.0)          # each block's largest element maps to 448
    xd = fp8.dequantize_rows(codes, scales)
    s = np.repeat(scales.astype(np.float64), 128, axis=1)
    # half an e4m3 step: 2**-4 relative for normals, 2**-10 * scale in the subnormal range,
    # plus the float32 roundings of inv and of the product
    assert np.all(np.abs(x - xd) <= 2.0 ** -4 * np.abs(x) * (1 + 2.0 ** -20) + 2.0 ** -10 * s)


def test_quantize_blocks_matches_torch_steps():
    rng = np.random.default_rng(2)
    w = oracle.round_bf16(rng.standard_normal((384, 256)) * 0.02)
    w[128:256, 0:128] *= 100.0            # blocks of different magnitude
    codes, scales = fp8.quantize_blocks(w)
    tq, ts = _torch_blocks(w)
    np.testing.assert_array_equal(codes, tq)
    np.testing.assert_array_equal(scales, ts)
    assert scales.shape == (3, 2)
    wd = fp8.dequantize_blocks(codes, scales)
    assert np.all(np.abs(w - wd) <= 2.0 ** -4 * np.abs(w) * (1 + 2.0 ** -20) +
                  2.0 ** -10 * np.repeat(np.repeat(scales.astype(np.float64), 128, 0), 128, 1))


# ----------------------------------------------------------------------------- expert
def _expert_inputs(seed, n=24, H=256, I=384):
    rng = np.random.default_rng(seed)
    x = oracle.round_bf16(rng.standard_normal((n, H)))
    w1 = oracle.round_bf16(rng.standard_normal((2 * I, H)) * 0.05)
    w2 = oracle.round_bf16(rng.standard_normal((H, I)) * 0.05)
    return x, w1, w2


def test_expert_fp8_vs_torch_on_dequantised_operands():
    x, w1, w2 = _expert_inputs(0)
    w1q, w1s = fp8.quantize_blocks(w1)
    w2q, w2s = fp8.quantize_blocks(w2)
    r = fp8.expert_fp8(x, w1q, w1s, w2q, w2s)
    xq, xs = _torch_rows(x)
    f = lambda q, s, blocks: torch.from_numpy(  # noqa: E731
        fp8.dequantize_blocks(q, s) if blocks else fp8.dequantize_rows(q, s))
    xt, w1t, w2t = f(xq, xs, False), f(w1q, w1s, True), f(w2q, w2s, True)
    I = w2.shape[1]
    h = xt @ w1t.T
    act = torch.nn.functional.silu(h[:, :I]) * h[:, I:]
    aq, as_ = _torch_rows(act.numpy().astype(np.float32))
    np.testing.assert_array_equal(r["act_codes"], aq)
    np.testing.assert_array_equal(r["act_scales"], as_)
    y = f(aq, as_, False) @ w2t.T
    np.testing.assert_allclose(r["y"], y.numpy(), rtol=1e-12, atol=1e-12)


def test_expert_fp8_close_to_full_precision_expert():
    x, w1, w2 = _expert_inputs(1)
    w1q, w1s = fp8.quantize_blocks(w1)
    w2q, w2s = fp8.quantize_blocks(w2)
    y8 = fp8.expert_fp8(x, w1q, w1s, w2q, w2s)["y"]
    y = oracle.swiglu_expert(x, w1, w2)
    rel = np.linalg.norm(y8 - y) / np.linalg.norm(y)
    # four e4m3 quantisations (x, W1, act, W2) of relative rms error about 2**-4/sqrt(3)
    # each: about 4e-2 together; not exact (the quantisation does something) and not
    # far off (no scale or layout mistake)
    assert 5e-3 < rel < 8e-2, rel


def test_act_band_covers_a_float32_evaluation():
    x, w1, w2 = _expert_inputs(3, n=64, H=1024, I=512)
    w1q, w1s = fp8.quantize_blocks(w1)
    w2q, w2s = fp8.quantize_blocks(w2)
    r = fp8.expert_fp8(x, w1q, w1s, w2q, w2s)
    # float32 evaluation: per-128 partial sums in float32, promoted with float32 FMAs
    xq, xs, _ = fp8.quantize_rows(x)
    xd = fp8.dequantize_rows(xq, xs).astype(np.float32)
    w1d = fp8.dequantize_blocks(w1q, w1s).astype(np.float32)
    h = np.zeros((x.shape[0], w1.shape[0]), np.float32)
    for kb in range(0, x.shape[1], 128):
        h = (h + xd[:, kb:kb + 128] @ w1d[:, kb:kb + 128].T).astype(np.float32)
    I = w2.shape[1]
    g, u = h[:, :I], h[:, I:]
    act32 = (g / (np.float32(1) + np.exp(-g)) * u).astype(np.float32)
    codes, scales, _ = fp8.quantize_rows(act32)
    ok = fp8.valid_act_codes(codes, r["act_quo"], r["act_band"])
    assert ok.all()
    differ = (codes != r["act_codes"]).mean()
    assert differ < 1e-2          # flips are rare; all lie inside the band
    allow = fp8.flip_allowance(codes, scales, r["act_codes"], r["act_scales"], r["w2"])
    ad = fp8.dequantize_rows(codes, scales)
    y32 = ad @ r["w2"].T
    # besides the flips, the block scales differ by the relative shift of each block's
    # largest magnitude (within the band's rel term)
    assert np.all(np.abs(y32 - r["y"]) <= allow + fp8.TC_REL * (np.abs(ad) @ np.abs(r["w2"]).T))


def test_valid_act_codes_rejects_far_codes():
    x, w1, w2 = _expert_inputs(4)
    w1q, w1s = fp8.quantize_blocks(w1)
    w2q, w2s = fp8.quantize_blocks(w2)
    r = fp8.expert_fp8(x, w1q, w1s, w2q, w2s)
    bad = r["act_codes"].copy()
    bad[0, 5] ^= 0x02                     # two steps away
    bad[1, 7] ^= 0x80                     # sign flip
    ok = fp8.valid_act_codes(bad, r["act_quo"], r["act_band"])
    assert not ok[0, 5] and not ok[1, 7]
    assert ok.sum() == ok.size - 2


def test_planted_mistakes_are_caught(monkeypatch):
    v = _probe_values()
    good = fp8.round_e4m3
    ref = torch_e4m3(v)
    ties_away = lambda a: good(np.where(np.isin(np.abs(a), 0.5 * (fp8._POS[:-1] + fp8._POS[1:])),  # noqa: E731
                                        np.nextafter(a, np.where(a < 0, -np.inf, np.inf)), a))
    truncate = lambda a: good(np.sign(a) * fp8._POS[np.maximum(  # noqa: E731
        np.searchsorted(fp8._POS, np.minimum(np.abs(a), 448), side="right") - 1, 0)])
    for f in (ties_away, truncate):
        assert not np.array_equal(f(v.astype(np.float64)), ref)
    # a wrong scale constant or a transposed block-scale grid breaks the torch pins
    x = oracle.round_bf16(np.random.default_rng(0).standard_normal((8, 256)))
    tq, ts = _torch_rows(x)
    monkeypatch.setattr(fp8, "E4M3_MAX", 240.0)
    assert not np.array_equal(fp8.quantize_rows(x)[0], tq)
    monkeypatch.setattr(fp8, "E4M3_MAX", 448.0)
    w = oracle.round_bf16(np.random.default_rng(1).standard_normal((256, 384)))
    q, s = fp8.quantize_blocks(w)
    tq, ts = _torch_blocks(w)
    assert not np.array_equal(fp8.dequantize_blocks(q, s.T.copy().reshape(s.shape)), fp8.dequantize_blocks(tq, ts))
