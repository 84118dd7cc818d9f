"""The three calls (dispatch, expert FFN, combine) captured once in a CUDA graph and replayed
on new inputs copied into the captured buffers: every replay equals an eager run of the same
inputs bit for bit, and the oracle on the final batch.  The calls never synchronise the host
and derive every launch size on the device, so one capture serves any routing."""
import dataclasses

import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from gen.device import make_case
from parity_util import check_out, geom_dict, check_routing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


@pytest.mark.parametrize("name", ["small_em", "small_rm", "small_flat", "pair_em", "tall_em"])
def test_graph_replay_matches_eager(name):
    base = gen.SMALL[name]
    cases = [make_case(base.with_(seed=40 + i, routing=r), "cuda")
             for i, r in enumerate(["uniform", "zipf", "dirichlet"])]
    cfg = base
    eager = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo)
    eager.set_weights(cases[0].w1, cases[0].w2)
    graphed = moe.MoELayer1GPU(cfg.W, cfg.Tr, cfg.tokens, cfg.H, cfg.E, cfg.k, cfg.I, cfg.layout, cfg.algo)
    graphed.set_weights(cases[0].w1, cases[0].w2)

    x = cases[0].x.clone()
    ids = cases[0].ids.clone()
    w = cases[0].w.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.forward(x, ids, w)          # first call outside capture (kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.forward(x, ids, w)

    for c in cases:
        x.copy_(c.x)
        ids.copy_(c.ids)
        w.copy_(c.w)
        g.replay()
        eager.forward(c.x, c.ids, c.w)
        torch.cuda.synchronize()
        assert graphed.status() == 0
        assert torch.equal(graphed.out.view(torch.int16), eager.out.view(torch.int16)), c.cfg.routing
    last = dataclasses.replace(cases[-1], w1_host=cases[0].w1_host, w2_host=cases[0].w2_host)
    rt = oracle.route(geom_dict(cfg), last.ids_np, last.w_np)
    check_routing(graphed, rt, cfg)
    check_out(graphed, last)
