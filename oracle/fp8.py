"""CPU oracle of the FP8 variant of the layer: FP8 dispatch (rows sent as e4m3 data plus
scales) feeding an FP8 grouped SwiGLU FFN.

TEST INFRASTRUCTURE ONLY (same rule as the rest of this package: only tests/, the smoke
check and the benchmark's CPU legs may import it).

Sources (page title, section):
  * Mooncake EP guide, "Buffer.dispatch(...)": with use_fp8 the dispatch returns the
    received rows as a (packed FP8 data, packed scales) pair instead of bf16 rows.
  * FlashInfer "MoE-EP implementation & usage", section 2 "Call stack" and section 4
    step 1: the grouped expert GEMMs over w1 [E, 2I, H] and w2 [E, H, I].
Readings where the pages are silent (each listed in the design notes):
  * FP8 format: OCP e4m3 "fn" (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
    subnormals, largest finite 448, no infinities; code 0x7F / 0xFF is NaN).
  * Scale granularity: one float32 scale per 128 consecutive columns of a row (rows of
    token activations and of the SwiGLU activation), one per 128 x 128 block of a weight
    matrix.  The hidden size is a multiple of 128 (the pages' input assertion).
  * Quantisation of a block with largest magnitude amax (float32):
        a     = max(amax, 2**-100)            (keeps 448 / a finite)
        scale = float32(a / 448)               stored; dequantised value = code * scale
        inv   = float32(448 / a)
        code  = e4m3_rne_satfinite(float32(v * inv))
    Both divisions and the product are single IEEE float32 operations, round to nearest
    even; the e4m3 rounding is round-to-nearest-even with saturation to +-448.
  * The FFN evaluates h = x^ W1^^T and act = silu(g) * u in full precision (float64) from
    the DEQUANTISED rows and weights, rounds act to float32, quantises it per 128
    columns as above (the operand of the second FP8 GEMM), and y = act^ W2^^T in float64.

Functions (none of their values is printed by the pages: "parity unpinned" by the pages,
pinned in tests by torch's float8_e4m3fn conversion, closed forms, round trips, error
bounds and the bf16 oracle):
  e4m3_values, round_e4m3, quantize_rows, dequantize_rows, quantize_blocks,
  dequantize_blocks, expert_fp8, act_band, valid_act_codes, flip_allowance, pick_results,
  layer_fp8.
"""
import numpy as np

E4M3_MAX = 448.0
SCALE_FLOOR = 2.0 ** -100
BLOCK = 128


def e4m3_values():
    """float64 value of each of the 256 e4m3fn codes (NaN for 0x7F and 0xFF), from the
    bit layout: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0; exponent 0
    is subnormal (m/8 * 2**-6)."""
    v = np.empty(256)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            v[c] = np.nan
        elif e == 0:
            v[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            v[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


_VALS = e4m3_values()
_POS = _VALS[:127]          # codes 0..126: the non-negative finite values, increasing


def round_e4m3(v):
    """e4m3fn code (uint8) nearest to each value of v (float64 holding float32 values):
    round to nearest, ties to the even code, magnitudes above 448 saturate to 448, the
    sign (also of zero) is kept."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    hi = np.searchsorted(_POS, np.minimum(a, E4M3_MAX), side="left")   # _POS[hi] >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS[hi] - a
    d_lo = a - _POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(a >= E4M3_MAX, 126, np.where(pick_hi, hi, lo))
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def decode_e4m3(codes):
    return _VALS[np.asarray(codes, dtype=np.uint8)]


def _scale_inv(amax32):
    a = np.maximum(amax32, np.float32(SCALE_FLOOR)).astype(np.float32)
    scale = (a / np.float32(E4M3_MAX)).astype(np.float32)
    inv = (np.float32(E4M3_MAX) / a).astype(np.float32)
    return scale, inv


def quantize_rows(v):
    """Per-row, per-128-column quantisation of v [n, C] (values rounded to float32 first).
    Returns (codes uint8 [n, C], scales float32 [n, C/128], quotients float64 [n, C]) where
    quotients are the float32 products v * inv that were rounded to e4m3."""
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    n, C = v32.shape
    b = v32.reshape(n, C // BLOCK, BLOCK)
    amax = np.abs(b).max(axis=2) if n else np.zeros((0, C // BLOCK), np.float32)
    scale, inv = _scale_inv(amax)
    quo = (b * inv[:, :, None]).astype(np.float32)
    codes = round_e4m3(quo.astype(np.float64)).reshape(n, C)
    return codes, scale, quo.astype(np.float64).reshape(n, C)


def dequantize_rows(codes, scales):
    n, C = codes.shape
    return (decode_e4m3(codes).reshape(n, C // BLOCK, BLOCK) *
            scales.astype(np.float64)[:, :, None]).reshape(n, C)


def quantize_blocks(w):
    """Per-128x128-block quantisation of a weight matrix w [R, C] (float32 values).
    Returns (codes uint8 [R, C], scales float32 [R/128, C/128])."""
    w32 = np.asarray(w, dtype=np.float64).astype(np.float32)
    R, C = w32.shape
    b = w32.reshape(R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    amax = np.abs(b).max(axis=(1, 3))
    scale, inv = _scale_inv(amax)
    quo = (b * inv[:, None, :, None]).astype(np.float32)
    return round_e4m3(quo.astype(np.float64)).reshape(R, C), scale


def dequantize_blocks(codes, scales):
    R, C = codes.shape
    return (decode_e4m3(codes).reshape(R // BLOCK, BLOCK, C // BLOCK, BLOCK) *
            scales.astype(np.float64)[:, None, :, None]).reshape(R, C)


def expert_fp8(xrows, w1q, w1s, w2q, w2s):
    """One expert's FP8 FFN on token rows xrows [n, H] (float64 values of the bf16 rows).
    w1q/w1s: codes [2I, H] and block scales of W1 (gate rows [0, I), up rows [I, 2I));
    w2q/w2s: codes [H, I] and block scales of W2.
    Returns a dict: y [n, H] float64; act_codes uint8 [n, I] and act_scales float32
    [n, I/128] (the second GEMM's operand); act_quo (the float32 quotients rounded to
    e4m3) and act_band (act_band below) float64 [n, I]; w2 (dequantised W2, float64)."""
    xq, xs, _ = quantize_rows(xrows)
    x = dequantize_rows(xq, xs)
    w1 = dequantize_blocks(w1q, w1s)
    w2 = dequantize_blocks(w2q, w2s)
    I = w2.shape[1]
    h = x @ w1.T
    g, u = h[:, :I], h[:, I:]
    with np.errstate(over="ignore"):
        silu = g / (1.0 + np.exp(-g))
    act = silu * u
    aq, as_, quo = quantize_rows(act)
    y = dequantize_rows(aq, as_) @ w2.T
    habs = np.abs(x) @ np.abs(w1).T
    band = act_band(act, silu, u, habs[:, :I], habs[:, I:], quo)
    return dict(y=y, act_codes=aq, act_scales=as_, act_quo=quo, act_band=band, w2=w2)


# Relative error allowed for a tensor-core sum of products against the exact sum, as a
# fraction of sum |x_k w_k|.  The float32 sum of 128 exact FP8 products per k-block,
# then a float32 fused multiply-add per k-block, stays far inside it; the tensor core's
# internal accumulator may keep fewer than 24 bits, hence the margin.
TC_REL = 2.0 ** -16


def act_band(act, silu, u, gabs, uabs, quo, rel=TC_REL):
    """Half-width (in quotient units) of the band around each activation quotient inside
    which a GPU that accumulates h in float32 may legitimately land.

    h has error at most rel * sum_k |x_k w_k| (gabs, uabs: those sums for the gate and up
    columns); act = silu(g) * u then moves by at most 1.1 |u| dg + |silu(g)| du (|silu'| <=
    1.1) plus 2**-18 |act| for the float32 evaluation of silu and the product; the quotient
    act * inv moves by that times inv, plus rel * |quotient| for the shift of the block's
    largest magnitude (and so of inv)."""
    n, I = act.shape
    a32 = np.abs(act.astype(np.float32)).reshape(n, I // BLOCK, BLOCK).max(axis=2)
    inv = (np.float32(E4M3_MAX) / np.maximum(a32, np.float32(SCALE_FLOOR))).astype(np.float64)
    dact = 1.1 * np.abs(u) * rel * gabs + np.abs(silu) * rel * uabs + 2.0 ** -18 * np.abs(act)
    return dact * np.repeat(inv, BLOCK, axis=1) + rel * np.abs(quo)


def valid_act_codes(gpu_codes, quo, band):
    """True where a GPU activation code is a correct result: the code of some quotient
    within [quo - band, quo + band] (the code of quo itself, or a neighbour when a rounding
    boundary lies inside the band)."""
    lo = round_e4m3(quo - band)
    hi = round_e4m3(quo + band)
    v = decode_e4m3(gpu_codes)
    vlo, vhi = decode_e4m3(lo), decode_e4m3(hi)
    return (v >= np.minimum(vlo, vhi)) & (v <= np.maximum(vlo, vhi))


def flip_allowance(gpu_codes, gpu_scales, act_codes, act_scales, w2):
    """Per output column n: sum over activation columns c whose GPU code differs from the
    oracle's of |W2[n, c]| * |value difference| (the GPU codes must first pass
    valid_act_codes).  The rest of y must match to the plain tolerance."""
    n, I = act_codes.shape
    dv = np.abs(dequantize_rows(gpu_codes, gpu_scales) - dequantize_rows(act_codes, act_scales))
    dv = np.where(gpu_codes != act_codes, dv, 0.0)
    return dv @ np.abs(w2).T


def weight_codes(w1, w2, e, cache):
    """Block-quantised weights of expert e from the bf16 bit arrays (or per-expert
    callables) w1 [E, 2I, H] / w2 [E, H, I]: (w1q, w1s, w2q, w2s)."""
    if e not in cache:
        from . import bf16_bits_to_f64
        a = w1(e) if callable(w1) else w1[e]
        b = w2(e) if callable(w2) else w2[e]
        cache[e] = quantize_blocks(bf16_bits_to_f64(a)) + quantize_blocks(bf16_bits_to_f64(b))
    return cache[e]


def pick_results(geom, rt, x_bits, w1, w2, picks, cache=None):
    """FP8 expert stage of the given valid picks (t*k + j): each pick's token row, as the
    FP8 dispatch delivers it, through expert_fp8 of its expert.  Returns
    ({pick: dict(y, act_codes, act_scales, act_quo, act_band)}, {expert: dequantised W2})."""
    from . import bf16_bits_to_f64
    cache = {} if cache is None else cache
    k = geom["k"]
    ids = rt["ids"].reshape(-1)
    by_e = {}
    for i in picks:
        by_e.setdefault(int(ids[i]), []).append(int(i))
    out, w2d = {}, {}
    for e, lst in sorted(by_e.items()):
        w1q, w1s, w2q, w2s = weight_codes(w1, w2, e, cache)
        r = expert_fp8(bf16_bits_to_f64(x_bits[np.array(lst) // k]), w1q, w1s, w2q, w2s)
        for n, i in enumerate(lst):
            out[i] = {key: r[key][n] for key in ("y", "act_codes", "act_scales", "act_quo", "act_band")}
        w2d[e] = r["w2"]
    return out, w2d


def layer_fp8(geom, x_bits, ids, topk_w, w1, w2, tokens=None, active=None, cache=None):
    """The FP8 layer for `tokens` (default all): route -> FP8 dispatch -> FP8 expert FFN ->
    combine (as in the bf16 oracle, float64 sums, one rounding to bf16).  Returns
    (route metadata, out [len(tokens), H], pick results of pick_results, W2 per expert).
    cache: optional dict of already quantised expert weights (see weight_codes)."""
    from . import combine_em, combine_ranks, ffn_ranks, route
    T, k = geom["T"], geom["k"]
    rt = route(geom, ids, topk_w, active)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    picks = [t * k + j for t in tokens for j in range(k) if rt["pick_pos"][t, j] >= 0]
    res, w2d = pick_results(geom, rt, x_bits, w1, w2, picks, cache)
    y = lambda i: res[i]["y"]  # noqa: E731
    if geom["layout"] == "EM":
        return rt, combine_em(geom, rt, topk_w, y, tokens), res, w2d
    rows = sorted({(d, int(rt["recv_row"][t, d])) for t in tokens for d in range(geom["W"])
                   if rt["recv_row"][t, d] >= 0})
    eo = dict(zip(rows, ffn_ranks(geom, rt, topk_w, y, rows)))
    return rt, combine_ranks(geom, rt, lambda d, r: eo[(d, r)], tokens), res, w2d
