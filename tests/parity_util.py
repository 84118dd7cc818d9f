"""Shared checks of the GPU layer against the CPU oracle (used by the -m gpu tests)."""
import numpy as np
import torch

import combine_topk_ids_gb300 as moe
import oracle

# output tolerance on floating outputs: |d| <= 2e-2 * |ref| + 1e-3, elementwise
RTOL, ATOL = 2e-2, 1e-3


def assert_close(got, ref, what, extra=0.0):
    """|got - ref| <= RTOL |ref| + ATOL (+ extra: a per-element allowance for rounding
    decisions that legitimately differ).  Returns the number of elements outside the plain
    bound (without `extra`), i.e. those that pass only through the allowance, and prints
    it whenever an allowance was given."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = np.abs(got - ref)
    bound = RTOL * np.abs(ref) + ATOL
    bad = ~(d <= bound + extra)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d/%d elements outside tolerance; first at %s: got %r ref %r"
                             % (what, bad.sum(), bad.size, tuple(i), got[tuple(i)], ref[tuple(i)]))
    n_plain = int((~(d <= bound)).sum())
    if np.any(np.asarray(extra) != 0):
        print("%s: %d of %d elements outside the plain bound (pass only through the allowance)"
              % (what, n_plain, d.size))
    return n_plain


def bf16_tensor_to_f64(t):
    return oracle.bf16_bits_to_f64(t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def geom_dict(cfg):
    return oracle.geom_of(cfg)


def run_layer(case, layer=None, active=None):
    cfg = case.cfg
    if layer is None:
        layer = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I,
                                 cfg.layout, cfg.algo, act=cfg.act)
        layer.set_weights(case.w1, case.w2)
    act = None if active is None else torch.as_tensor(active, dtype=torch.int32, device=case.x.device)
    layer.forward(case.x, case.ids, case.w, act)
    torch.cuda.synchronize()
    return layer


def check_routing(layer, rt, cfg):
    """Bit-exact comparison of every routing output the handle exposes."""
    T, k, E, W, cap = cfg.tokens, cfg.k, cfg.E, cfg.W, cfg.W * cfg.Tr
    v = lambda f, shape, dt=torch.int32: layer.view(f, shape, dt).cpu().numpy()  # noqa: E731
    np.testing.assert_array_equal(v("counts", (E,)), rt["counts"])
    np.testing.assert_array_equal(v("offsets", (E + 1,)), rt["offsets"])
    np.testing.assert_array_equal(v("pick_pos", (T, k)), rt["pick_pos"])
    R = rt["R"]
    np.testing.assert_array_equal(v("pick_src", (T * k,))[:R], rt["pick_src"])
    if cfg.layout == "EM":
        np.testing.assert_array_equal(v("slot", (T, k)), rt["slot"])
        np.testing.assert_array_equal(v("layout_range", (E, W, 2)), rt["layout_range"])
    else:
        np.testing.assert_array_equal(v("recv_row", (T, W)), rt["recv_row"])
        np.testing.assert_array_equal(v("recv_count", (W, W)), rt["recv_count"])
        np.testing.assert_array_equal(v("num_recv", (W,)), rt["num_recv"])
        used = rt["recv_src"] >= 0             # rows that hold a token
        np.testing.assert_array_equal(v("recv_src", (W, cap))[used], rt["recv_src"][used])
        np.testing.assert_array_equal(v("recv_topk_idx", (W, cap, k))[used], rt["recv_topk_idx"][used])
        np.testing.assert_array_equal(v("recv_topk_weights", (W, cap, k), torch.float32)[used],
                                      rt["recv_topk_w"][used])


def check_dispatch_rows(layer, rt, case):
    """Every received row equals its token's x row, bit for bit (checked on the device)."""
    cfg = case.cfg
    rows, toks = oracle.dispatch_rows(geom_dict(cfg), rt)
    nrows = (cfg.E if cfg.layout == "EM" else cfg.W) * cfg.W * cfg.Tr
    recv = layer.view("recv_x", (nrows, cfg.H), torch.int16)
    x = case.x.view(torch.int16)
    dev = case.x.device
    r_t = torch.from_numpy(np.asarray(rows, np.int64)).to(dev)
    t_t = torch.from_numpy(np.asarray(toks, np.int64)).to(dev)
    for s in range(0, len(rows), 1 << 16):
        assert torch.equal(recv[r_t[s:s + (1 << 16)]], x[t_t[s:s + (1 << 16)]]), "dispatch rows differ"
    if cfg.layout != "EM" and getattr(cfg, "quant", "bf16") == "bf16" and rt["R"] > 0:
        # RANK_MAJOR / FLAT: the kept picks' rows in pick-list order (the first GEMM's
        # operand) hold x[token of pick_src[p]], bit for bit
        pr = layer.view("pick_rows", (rt["R"], cfg.H), torch.int16)
        src = torch.from_numpy(rt["pick_src"].astype(np.int64) // cfg.k).to(dev)
        for s in range(0, rt["R"], 1 << 16):
            assert torch.equal(pr[s:s + (1 << 16)], x[src[s:s + (1 << 16)]]), "pick-ordered rows differ"


def act_flip_allowance(layer, rt, case, picks):
    """The single-bf16 activation option is a rounding decision taken on tensor-core sums: a GPU
    code may be the neighbour of the oracle's where the exact activation lies within the
    accumulation band of a bf16 midpoint.  Checks every GPU activation code of `picks` is
    a correct result (oracle.bf16_act_allowance) and returns {pick: [H] allowance}; zero
    for the default bf16-pair activation."""
    cfg = case.cfg
    picks = [int(i) for i in picks]
    if getattr(cfg, "act", "pair") != "bf16" or not picks:
        return {i: 0.0 for i in picks}
    pp = rt["pick_pos"].reshape(-1)
    pos = torch.as_tensor([int(pp[i]) for i in picks], dtype=torch.int64, device=layer.out.device)
    gpu = bf16_tensor_to_f64(layer.view("ffn_act", (max(rt["R"], 1), cfg.I), torch.bfloat16)[pos])
    allow, n_bad, n_flip = oracle.bf16_act_allowance(geom_dict(cfg), rt, case.x_bits, case.w1_host,
                                                     case.w2_host, picks, gpu)
    assert n_bad == 0, "%d activation codes outside the oracle's band" % n_bad
    # a guard on how many codes may sit on the other side of a midpoint: the tensor-core
    # sum's distance from the exact sum grows with the number of terms it accumulates, and
    # the measured rate is about 0.11% of the codes per 1024 terms of the first GEMM's K
    # (0.05% at K 512, 0.41% at 4096, 0.72% at 7168, 7.0% at 65536); allow twice that
    # rate plus 0.1%
    cap = 0.001 + 0.0022 * cfg.H / 1024.0
    n_codes = len(picks) * cfg.I
    print("%s: %d of %d activation codes on the other side of a midpoint (%.3g%%)"
          % (cfg.name, n_flip, n_codes, 100.0 * n_flip / max(n_codes, 1)))
    assert n_flip <= cap * n_codes, "%d of %d activation codes differ" % (n_flip, n_codes)
    return allow


def check_expert_out(layer, rt, case, picks_or_rows=None, max_rows=None):
    """expert_out against the oracle: per pick (EM) or per received row (RM/FLAT)."""
    cfg = case.cfg
    g = geom_dict(cfg)
    k, H, cap = cfg.k, cfg.H, cfg.W * cfg.Tr
    eo = layer.expert_out.view(-1, H)
    if cfg.layout == "EM":
        picks = np.nonzero(rt["pick_pos"].reshape(-1) >= 0)[0] if picks_or_rows is None else picks_or_rows
        if max_rows is not None:
            picks = picks[:max_rows]
        ys = oracle.pick_outputs(g, rt, case.x_bits, case.w1_host, case.w2_host, picks=picks)
        allow = act_flip_allowance(layer, rt, case, picks)
        slots = rt["slot"].reshape(-1)[picks]
        got = eo[torch.from_numpy(slots).to(eo.device)].cpu().numpy()
        extra = np.array([allow[int(i)] * np.ones(H) for i in picks])
        return assert_close(got, np.array([ys[i] for i in picks]), "expert_out (EM)", extra=extra)
    else:
        rows = picks_or_rows
        if rows is None:
            rows = [(d, r) for d in range(cfg.W) for r in range(cap) if rt["recv_src"][d, r] >= 0]
        if max_rows is not None:
            rows = rows[:max_rows]
        need = sorted({int(rt["recv_src"][d, r]) * k + j for d, r in rows for j in range(k)
                       if rt["recv_topk_idx"][d, r, j] >= 0})
        ys = oracle.pick_outputs(g, rt, case.x_bits, case.w1_host, case.w2_host, picks=need)
        allow = act_flip_allowance(layer, rt, case, need)
        ref = oracle.ffn_ranks(g, rt, case.w_np, ys.__getitem__, rows)
        extra = np.zeros_like(ref)
        for n, (d, r) in enumerate(rows):
            t = int(rt["recv_src"][d, r])
            for j in range(k):
                if rt["recv_topk_idx"][d, r, j] >= 0:
                    extra[n] += abs(float(rt["recv_topk_w"][d, r, j])) * allow[t * k + j]
        idx = torch.tensor([d * cap + r for d, r in rows], dtype=torch.int64, device=eo.device)
        return assert_close(eo[idx].cpu().numpy(), ref, "expert_out (%s)" % cfg.layout, extra=extra)


def targeted_tokens(cfg, rt, n_random=0, seed=0):
    """Tokens whose picks reach the GEMM tile paths a random sample can miss at full size:
    for every expert with rows, the token of its last row (the expert's tail row block, a
    partial tile) and, when it has more than 128 rows, one row in 128..255 (the second
    accumulator of a one-CTA 256-row tile, or the second CTA of a two-SM tile); for the
    most loaded expert (the Zipf-hot one under skewed routing) also its first and middle
    rows; plus token 0, the last token and n_random tokens drawn with `seed`.  Row r of
    expert e is pick-list entry offsets[e] + r, whose token is pick_src // k."""
    counts, offsets, src = rt["counts"], rt["offsets"], rt["pick_src"]
    rows = []
    for e in np.nonzero(counts > 0)[0]:
        n = int(counts[e])
        rows.append(int(offsets[e]) + n - 1)
        if n > 128:
            rows.append(int(offsets[e]) + 128 + (int(e) * 37) % min(128, n - 128))
    hot = int(np.argmax(counts))
    if counts[hot] > 0:
        rows += [int(offsets[hot]), int(offsets[hot]) + int(counts[hot]) // 2]
    toks = {int(src[r]) // cfg.k for r in rows} | {0, cfg.tokens - 1}
    if n_random:
        rng = np.random.default_rng(seed)
        toks |= set(rng.choice(cfg.tokens, size=min(n_random, cfg.tokens), replace=False).tolist())
    return np.array(sorted(toks))


def check_layer_tokens(layer, rt, case, toks):
    """expert_out (per pick for EM, per received row for RM/FLAT) and the combined output
    of `toks` against the oracle, evaluating each pick's expert output once for both.
    Returns the counts of elements outside the plain bound (expert_out, out)."""
    cfg = case.cfg
    g = geom_dict(cfg)
    k = cfg.k
    picks = [int(t) * k + j for t in toks for j in range(k) if rt["pick_pos"][t, j] >= 0]
    ys = oracle.pick_outputs(g, rt, case.x_bits, case.w1_host, case.w2_host, picks=picks)
    allow = act_flip_allowance(layer, rt, case, picks)
    H, cap = cfg.H, cfg.W * cfg.Tr
    eo = layer.expert_out.view(-1, H)
    if cfg.layout == "EM":
        slots = rt["slot"].reshape(-1)[picks]
        got = eo[torch.from_numpy(slots).to(eo.device)].cpu().numpy()
        extra = np.array([allow[i] * np.ones(H) for i in picks])
        n_eo = assert_close(got, np.array([ys[i] for i in picks]), "expert_out (EM)", extra=extra)
        ref = oracle.combine_em(g, rt, case.w_np, ys.__getitem__, toks)
    else:
        drows = sorted({(d, int(rt["recv_row"][t, d])) for t in toks for d in range(cfg.W)
                        if rt["recv_row"][t, d] >= 0})
        ref_rows = oracle.ffn_ranks(g, rt, case.w_np, ys.__getitem__, drows)
        extra = np.zeros_like(ref_rows)
        for n, (d, r) in enumerate(drows):
            t = int(rt["recv_src"][d, r])
            for j in range(k):
                if rt["recv_topk_idx"][d, r, j] >= 0:
                    extra[n] += abs(float(rt["recv_topk_w"][d, r, j])) * allow[t * k + j]
        idx = torch.tensor([d * cap + r for d, r in drows], dtype=torch.int64, device=eo.device)
        n_eo = assert_close(eo[idx].cpu().numpy(), ref_rows, "expert_out (%s)" % cfg.layout, extra=extra)
        by_row = dict(zip(drows, ref_rows))
        ref = oracle.combine_ranks(g, rt, lambda d, r: by_row[(d, r)], toks)
    wv = np.abs(case.w_np.astype(np.float64)).reshape(-1)
    extra = np.zeros((len(toks), H))
    row_of = {int(t): n for n, t in enumerate(toks)}
    for i in picks:
        extra[row_of[i // k]] += wv[i] * allow[i]
    got = bf16_tensor_to_f64(layer.out[torch.as_tensor(np.asarray(toks), device=layer.out.device)])
    n_out = assert_close(got, ref, "out (%s)" % cfg.name, extra=extra)
    return n_eo, n_out


def check_out(layer, case, tokens=None, active=None):
    """The combined output against the oracle, plus the activation flip allowance of every
    pick of each token (carried through |topk weight|)."""
    cfg = case.cfg
    rt, ref = oracle.layer(geom_dict(cfg), case.x_bits, case.ids_np, case.w_np, case.w1_host,
                           case.w2_host, tokens=tokens, active=active)
    toks = np.arange(cfg.tokens) if tokens is None else np.asarray(tokens)
    k = cfg.k
    picks = [int(t) * k + j for t in toks for j in range(k) if rt["pick_pos"][t, j] >= 0]
    allow = act_flip_allowance(layer, rt, case, picks)
    wv = np.abs(case.w_np.astype(np.float64)).reshape(-1)
    extra = np.zeros((len(toks), cfg.H))
    row_of = {int(t): n for n, t in enumerate(toks)}
    for i in picks:
        extra[row_of[i // k]] += wv[i] * allow[i]
    got = bf16_tensor_to_f64(layer.out if tokens is None else layer.out[torch.as_tensor(tokens)])
    return assert_close(got, ref, "out (%s)" % cfg.name, extra=extra)
