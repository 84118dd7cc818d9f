"""Failure detection on the GPU without a fault: a device wait that can never complete gives
up after its limit, reports MOE_STATUS_TIMEOUT through the status word, and leaves the
context usable (a normal layer runs correctly afterwards)."""
import pytest
import torch

import combine_topk_ids_gb300 as moe
import gen
import oracle
from gen.device import make_case
from parity_util import check_out, check_routing, geom_dict, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


def test_wait_expiry_reports_timeout_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_selftest_wait_expiry(status)
    torch.cuda.synchronize()
    assert int(status.item()) & moe.STATUS_TIMEOUT
    # the context still works: a full layer, checked against the oracle
    cfg = gen.SMALL["small_em"]
    case = make_case(cfg, "cuda")
    layer = run_layer(case)
    assert layer.status() == 0
    rt = oracle.route(geom_dict(cfg), case.ids_np, case.w_np)
    check_routing(layer, rt, cfg)
    check_out(layer, case)
