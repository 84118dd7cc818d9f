"""CPU oracle of the MoE expert-parallel layer: dispatch -> per-expert SwiGLU FFN -> combine.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the benchmark's
CPU-baseline leg (bench.py --impl reference / cpu_baseline) may import this package.
The product library never calls it and shares no code with it.

Plain and slow on purpose: routing is the literal (t, j)-ordered loop in moe_oracle.c;
the FFN and combine are numpy in float64, one expert at a time; the only rounding is the
final output's to bf16 (plus, for the library's options, the SwiGLU activation's to bf16
and expert_out's to bf16 where those options round).

Sources (page title, section):
  * FlashInfer "MoE-EP implementation & usage", section 2 "Call stack": dispatch ->
    EP->compute bridge -> per-expert grouped GEMM (no routing) -> combine ->
    [num_tokens, hidden] bf16.
  * same page, section 3 "Algorithm / layout contracts": EXPERT_MAJOR computes top_k=1
    per dispatched row and reweights per token on combine; RANK_MAJOR / HT FLAT compute
    the real top_k over the received routing with non-local picks masked to weight 0,
    and combine is an unweighted sum across ranks.
  * same page, section 4 step 1: w1 [E, 2*I, H], w2 [E, H, I].
  * Mooncake EP guide, "Buffer.combine(...)": expert outputs are returned by routing
    weight and reduced to the token's owner.
Readings where the pages are silent (each listed in the design notes):
  * with the bf16 expert_out option the expert stage's outputs are rounded to bf16 where
    the GPU rounds them (each pick's y; for RANK_MAJOR / FLAT also the per-row sum);
  * gate = rows [0, I) of w1[e], up = rows [I, 2I); SwiGLU act = silu(gate) * up with
    silu(g) = g / (1 + exp(-g))  (parity unpinned by the pages: a fixed convention);
  * the expert FFN is evaluated in full precision (float64) from the bf16 weights and
    inputs, the SwiGLU activation unrounded (FlashInfer page, section 4 step 6: the EP
    layer is checked against a dense MoE evaluated in fp32); only with geom["act"] ==
    "bf16" (the library's single-bf16 activation option) is the activation, the operand
    of the second bf16 GEMM, rounded to bf16 (round to nearest even) first; expert_out is
    not rounded (float64 here); the final combined output is rounded to bf16
    (round-to-nearest-even);
  * RANK_MAJOR / FLAT apply topk_weights in the FFN stage's reduction over the local
    picks of a received row (ascending j), and combine sums over destinations without
    weights (ascending d).

Functions whose values the pages never print ("parity unpinned" by the pages; pinned in
tests by brute force, closed forms, a library special case and exact invariants):
route, pick_outputs, ffn_ranks, combine_em, combine_ranks, layer (swiglu_act_band and bf16_act_allowance
are the tolerance helpers of the single-bf16 activation option).
"""
import ctypes
import os

import numpy as np

from .build import build as _build_c, LIB_PATH

_lib = None


def _c():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            _build_c()
        _lib = ctypes.CDLL(LIB_PATH)
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        ci = ctypes.c_int
        _lib.oracle_route_experts.argtypes = [ci, ci, ci, ci, ci, ctypes.c_int64, i64p, ctypes.c_void_p,
                                              i32p, i32p, i32p, i32p, i32p, i32p, i32p]
        _lib.oracle_route_experts.restype = ci
        _lib.oracle_route_ranks.argtypes = [ci, ci, ci, ci, ci, ci, i64p, ctypes.c_void_p, f32p,
                                            i32p, i32p, i32p, i32p, i32p, f32p]
        _lib.oracle_route_ranks.restype = None
    return _lib


LAYOUT = {"EM": 0, "RM": 1, "FLAT": 2}


def round_bf16(a):
    """Nearest bf16 value (8 significant bits, ties to even) of float64 values, as float64.

    Single rounding from float64.  Values below 2**-126 keep 8 significant bits (bf16
    subnormals are not modelled; no tested quantity lands there).
    """
    a = np.asarray(a, dtype=np.float64)
    m, ex = np.frexp(a)
    return np.ldexp(np.rint(m * 256.0), ex - 8)


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def route(geom, ids, topk_w, active=None):
    """All routing metadata of one dispatch (Mooncake EP "Buffer.dispatch" outputs and the
    FlashInfer layout contracts).  geom: dict with W, Tr, T, E, k, layout ("EM"|"RM"|"FLAT").
    active: optional EP rank-health mask [W] (0 = failed rank): picks whose expert or whose
    token's source rank is inactive are dropped.

    Returns a dict of int32 arrays: counts, offsets, pick_pos, pick_src (first R entries),
    layout_range [E, W, 2], slot (EM recv row per pick or -1), and for RM/FLAT recv_row
    [T, W], recv_count [W, W], num_recv [W], recv_src, recv_topk_idx, recv_topk_w
    (the last three as [W, cap(, k)] with cap = W*Tr; rows >= count are unspecified and
    left at -1 / 0 here), plus n_bad (ids outside [-1, E)) and n_over (EXPERT_MAJOR picks
    dropped because their expert's region of W*Tr rows was full, which only a token that
    names one expert twice can cause).
    """
    W, Tr, T, E, k = geom["W"], geom["Tr"], geom["T"], geom["E"], geom["k"]
    lay = LAYOUT[geom["layout"]]
    ids64 = np.ascontiguousarray(np.asarray(ids).reshape(T, k), dtype=np.int64)
    w32 = np.ascontiguousarray(np.asarray(topk_w).reshape(T, k), dtype=np.float32)
    lib = _c()
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    pick_pos = np.full(T * k, -1, np.int32)
    pick_src = np.full(max(T * k, 1), -1, np.int32)
    lrange = np.zeros(E * W * 2, np.int32)
    n_over = np.zeros(1, np.int32)
    n_inact = np.zeros(1, np.int32)
    cap = W * Tr
    act = None if active is None else np.ascontiguousarray(np.asarray(active), dtype=np.int32)
    act_p = None if act is None else act.ctypes.data_as(ctypes.c_void_p)
    # only the EXPERT_MAJOR region has a per-expert row capacity (W*Tr rows)
    n_bad = lib.oracle_route_experts(T, k, E, W, Tr, cap if lay == 0 else -1, ids64, act_p, counts,
                                     offsets, pick_pos, pick_src, lrange, n_over, n_inact)
    R = int(offsets[E])
    out = dict(ids=ids64, counts=counts, offsets=offsets, pick_pos=pick_pos.reshape(T, k),
               pick_src=pick_src[:R], layout_range=lrange.reshape(E, W, 2), n_bad=n_bad,
               n_over=int(n_over[0]), n_inactive=int(n_inact[0]), R=R, active=act)
    # EXPERT_MAJOR receive row: expert e's region starts at e*cap, packed from its row 0.
    slot = np.full(T * k, -1, np.int64)
    valid = (pick_pos >= 0) & (lay == 0)
    e_of = ids64.reshape(-1)
    slot[valid] = e_of[valid] * cap + (pick_pos[valid] - offsets[e_of[valid]])
    out["slot"] = slot.reshape(T, k)
    if lay != 0:
        recv_row = np.full(T * W, -1, np.int32)
        recv_count = np.zeros(W * W, np.int32)
        num_recv = np.zeros(W, np.int32)
        recv_src = np.full(W * cap, -1, np.int32)
        rti = np.full(W * cap * k, -1, np.int32)
        rtw = np.zeros(W * cap * k, np.float32)
        lib.oracle_route_ranks(T, k, E, W, Tr, lay, ids64, act_p, w32, recv_row, recv_count,
                               num_recv, recv_src, rti, rtw)
        out.update(recv_row=recv_row.reshape(T, W), recv_count=recv_count.reshape(W, W),
                   num_recv=num_recv, recv_src=recv_src.reshape(W, cap),
                   recv_topk_idx=rti.reshape(W, cap, k), recv_topk_w=rtw.reshape(W, cap, k))
    return out


def dispatch_rows(geom, rt):
    """Where each token row lands: arrays (recv_row_index, token) for every received row.

    EXPERT_MAJOR: one row per valid pick, recv index e*cap + position in e's region.
    RANK_MAJOR / FLAT: one row per (token, destination) pair, recv index d*cap + row.
    The expected content of recv row `r` is x[token]: dispatch is a bit copy.
    """
    W, Tr = geom["W"], geom["Tr"]
    cap = W * Tr
    if geom["layout"] == "EM":
        T, k = rt["slot"].shape
        s = rt["slot"].reshape(-1)
        tok = np.repeat(np.arange(T), k)
        m = s >= 0
        return s[m], tok[m]
    rr = rt["recv_row"]
    t_idx, d_idx = np.nonzero(rr >= 0)
    return d_idx.astype(np.int64) * cap + rr[t_idx, d_idx], t_idx


def swiglu_act(xrows, w1e):
    """SwiGLU activation of the rows xrows [n, H] (float64 values of bf16 inputs):
    h = x W1e^T, act = silu(h[:, :I]) * h[:, I:], float64, unrounded."""
    I = w1e.shape[0] // 2
    h = xrows @ w1e.T
    g, u = h[:, :I], h[:, I:]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def swiglu_act_band(xrows, w1e, rel=2.0 ** -14):
    """Half-width (absolute, in activation units) of the band around each exact activation
    inside which a GPU that accumulates h = x W1e^T in float32 on tensor cores may land:
    h moves by at most rel * sum_k |x_k w_k|, act = silu(g) * u by 1.1 |u| dg + |silu(g)| du
    (|silu'| <= 1.1) plus 2**-18 |act| for the float32 evaluation of silu and the product.
    A bf16 activation code of the GPU is then a correct result if it is the rounding of some
    value inside [act - band, act + band]."""
    I = w1e.shape[0] // 2
    h = xrows @ w1e.T
    habs = np.abs(xrows) @ np.abs(w1e).T
    g, u = h[:, :I], h[:, I:]
    with np.errstate(over="ignore"):
        silu = g / (1.0 + np.exp(-g))
    act = silu * u
    return act, 1.1 * np.abs(u) * rel * habs[:, :I] + np.abs(silu) * rel * habs[:, I:] + 2.0 ** -18 * np.abs(act)


def bf16_act_allowance(geom, rt, x_bits, w1, w2, picks, gpu_act):
    """For the single-bf16 activation option: which of a GPU's activation codes are correct
    results, and what their differences from the oracle's codes may do to y.

    gpu_act: float64 [len(picks), I], the GPU's bf16 activation of each pick.  A code is
    correct if it is the bf16 rounding of some value within swiglu_act_band of the exact
    activation.  Returns (allowance {pick: [H]} = sum over columns c whose GPU code differs
    from round_bf16(act) of |W2[:, c]| * |difference|, number of incorrect codes, number of
    differing codes)."""
    k = geom["k"]
    ids = rt["ids"].reshape(-1)
    row_of = {int(i): n for n, i in enumerate(picks)}
    by_e = {}
    for i in picks:
        by_e.setdefault(int(ids[i]), []).append(int(i))
    out, n_bad, n_flip = {}, 0, 0
    for e, lst in sorted(by_e.items()):
        w1e, w2e = _expert_weights(w1, w2, e)
        act, band = swiglu_act_band(bf16_bits_to_f64(x_bits[np.array(lst) // k]), w1e)
        ref = round_bf16(act)
        lo, hi = round_bf16(act - band), round_bf16(act + band)
        v = np.asarray(gpu_act, dtype=np.float64)[[row_of[i] for i in lst]]
        n_bad += int((~((v >= np.minimum(lo, hi)) & (v <= np.maximum(lo, hi)))).sum())
        dv = np.abs(v - ref)
        n_flip += int((dv != 0).sum())
        allow = dv @ np.abs(w2e).T
        for n, i in enumerate(lst):
            out[i] = allow[n]
    return out, n_bad, n_flip


def swiglu_expert(xrows, w1e, w2e, act_bf16=False, return_act=False):
    """One expert's FFN on the rows xrows [n, H]: y = act W2e^T in float64, act from
    swiglu_act; act_bf16: the activation is the second GEMM's bf16 operand, rounded to
    nearest even first (the library's default activation precision).  return_act: also
    return the unrounded activation."""
    act = swiglu_act(xrows, w1e)
    y = (round_bf16(act) if act_bf16 else act) @ w2e.T
    return (y, act) if return_act else y


def _expert_weights(w1, w2, e):
    """float64 values of expert e's weights; w1/w2 are uint16 bf16 bit arrays or callables
    returning them for one expert (large weight sets are fetched one expert at a time)."""
    a = w1(e) if callable(w1) else w1[e]
    b = w2(e) if callable(w2) else w2[e]
    return bf16_bits_to_f64(a), bf16_bits_to_f64(b)


def pick_outputs(geom, rt, x_bits, w1, w2, picks=None, expert_fn=None, acts=None):
    """Expert output y(t, j) = FFN_e(x[t]) of each valid pick, e = topk_ids[t, j].

    This is EXPERT_MAJOR's expert stage (top_k = 1 per dispatched row) and the per-pick
    term of the RANK_MAJOR / FLAT stage.  Returns {pick index t*k+j: float64 [H]} for
    `picks` (default: all valid picks).  expert_fn(e, xrows) replaces the SwiGLU expert
    (the identity-expert pin uses it).  The activation is unrounded (the FFN in full
    precision) unless geom["act"] == "bf16", the library's single-bf16 activation option,
    whose second GEMM takes the activation as one bf16 operand (FlashInfer "MoE-EP
    implementation & usage" section 4 step 3: the expert GEMMs take bf16 operands).
    acts: optional dict that receives each pick's unrounded activation (float64 [I]).
    """
    act_bf16 = geom.get("act", "pair") == "bf16"
    k = geom["k"]
    pp = rt["pick_pos"].reshape(-1)
    ids = rt["ids"].reshape(-1)
    want = np.nonzero(pp >= 0)[0] if picks is None else np.asarray(picks)
    out = {}
    by_e = {}
    for i in want:
        e = int(ids[i])
        by_e.setdefault(e, []).append(int(i))
    for e, lst in sorted(by_e.items()):
        xr = bf16_bits_to_f64(x_bits[np.array(lst) // k])
        if expert_fn is not None:
            y = expert_fn(e, xr)
        else:
            a, b = _expert_weights(w1, w2, e)
            y, act = swiglu_expert(xr, a, b, act_bf16=act_bf16, return_act=True)
            if acts is not None and act is not None:
                for n, i in enumerate(lst):
                    acts[i] = act[n]
        for n, i in enumerate(lst):
            out[i] = y[n]
    return out


def combine_em(geom, rt, topk_w, y_of_pick, tokens, eo_bf16=False):
    """EXPERT_MAJOR combine: out[t] = bf16( sum_j w[t, j] * expert_out[slot[t, j]] ),
    masked picks contribute nothing; float64 sum in ascending j.  eo_bf16: expert_out
    holds bf16(y) (the bf16 expert_out option)."""
    k = geom["k"]
    pp = rt["pick_pos"]
    w = np.asarray(topk_w, dtype=np.float64).reshape(-1, k)
    res = []
    for t in tokens:
        acc = None
        for j in range(k):
            if pp[t, j] < 0:
                continue
            y = y_of_pick(t * k + j)
            term = w[t, j] * (round_bf16(y) if eo_bf16 else y)
            acc = term if acc is None else acc + term
        res.append(np.zeros(geom["H"]) if acc is None else acc)
    return round_bf16(np.array(res))


def ffn_ranks(geom, rt, topk_w, y_of_pick, dest_rows, eo_bf16=False):
    """RANK_MAJOR / FLAT expert stage on received rows: for destination d and row r with
    token t, expert_out[d, r] = sum over j ascending of recv_topk_w[d, r, j] * y(t, j),
    non-local picks (recv_topk_idx == -1) masked to weight 0 (skipped).
    dest_rows: iterable of (d, r).  Returns float64 [len, H].  eo_bf16 (the bf16
    expert_out option): each y(t, j) is held as bf16 and the sum is rounded to bf16."""
    k = geom["k"]
    res = []
    for d, r in dest_rows:
        t = int(rt["recv_src"][d, r])
        acc = np.zeros(geom["H"])
        for j in range(k):
            if rt["recv_topk_idx"][d, r, j] < 0:
                continue
            y = y_of_pick(t * k + j)
            acc = acc + float(rt["recv_topk_w"][d, r, j]) * (round_bf16(y) if eo_bf16 else y)
        res.append(round_bf16(acc) if eo_bf16 else acc)
    return np.array(res)


def combine_ranks(geom, rt, expert_out_of, tokens):
    """RANK_MAJOR / FLAT combine: out[t] = bf16( sum over destinations d ascending that
    received t of expert_out[d, recv_row[t, d]] ), unweighted."""
    res = []
    for t in tokens:
        acc = np.zeros(geom["H"])
        for d in range(geom["W"]):
            r = int(rt["recv_row"][t, d])
            if r >= 0:
                acc = acc + expert_out_of(d, r)
        res.append(acc)
    return round_bf16(np.array(res))


def layer(geom, x_bits, ids, topk_w, w1, w2, tokens=None, expert_fn=None, active=None,
          eo_bf16=False):
    """The whole layer for `tokens` (default all): route -> dispatch -> expert FFN ->
    combine, returning (route metadata, out [len(tokens), H] float64 holding bf16 values).
    Only the picks of the requested tokens are evaluated.  active: EP rank-health mask.
    eo_bf16: expert_out (and the RANK_MAJOR / FLAT per-pick rows) held as bf16."""
    T, k = geom["T"], geom["k"]
    rt = route(geom, ids, topk_w, active)
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    picks = [t * k + j for t in tokens for j in range(k) if rt["pick_pos"][t, j] >= 0]
    ys = pick_outputs(geom, rt, x_bits, w1, w2, picks=picks, expert_fn=expert_fn)
    if geom["layout"] == "EM":
        return rt, combine_em(geom, rt, topk_w, ys.__getitem__, tokens, eo_bf16)
    rows = sorted({(d, int(rt["recv_row"][t, d])) for t in tokens for d in range(geom["W"])
                   if rt["recv_row"][t, d] >= 0})
    eo = dict(zip(rows, ffn_ranks(geom, rt, topk_w, ys.__getitem__, rows, eo_bf16)))
    return rt, combine_ranks(geom, rt, lambda d, r: eo[(d, r)], tokens)


def geom_of(cfg):
    """Geometry dict of a gen.configs.MoeConfig."""
    return dict(W=cfg.W, Tr=cfg.Tr, T=cfg.tokens, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I,
                layout=cfg.layout, act=getattr(cfg, "act", "pair"))
