"""Place one workload's seeded inputs on a torch device, plus the host copies the CPU
oracle reads.  Data marshalling only."""
from dataclasses import dataclass
from typing import Any, Callable, Union

import numpy as np

from .configs import MoeConfig
from .inputs import (expert_weights_numpy, gen_routing, gen_weights_numpy, gen_weights_torch, gen_x,
                     torch_bf16_to_bits, weights_on_host)


@dataclass
class Case:
    cfg: MoeConfig
    x: Any            # torch bf16 [T, H]
    ids: Any          # torch int64/int32 [T, k]
    w: Any            # torch float32 [T, k]
    w1: Any           # torch bf16 [E, 2I, H]
    w2: Any           # torch bf16 [E, H, I]
    x_bits: np.ndarray
    ids_np: np.ndarray
    w_np: np.ndarray
    w1_host: Union[np.ndarray, Callable[[int], np.ndarray]]   # uint16 bits, or per expert
    w2_host: Union[np.ndarray, Callable[[int], np.ndarray]]


def make_case(cfg: MoeConfig, device, ids_override=None) -> Case:
    """Inputs of `cfg` on `device`.  With device "cpu" and a weight set too large to draw on
    the host, no device weights are made (w1 = w2 = None) and the host copies are drawn
    with numpy one expert at a time on first use (values then differ from the GPU draw;
    this only serves timing the oracle)."""
    import torch
    import functools
    x_bits = gen_x(cfg)
    ids_np, w_np = gen_routing(cfg)
    if ids_override is not None:
        ids_np = np.ascontiguousarray(ids_override.astype(ids_np.dtype))
    if str(device) == "cpu" and not weights_on_host(cfg):
        one = functools.lru_cache(maxsize=None)(lambda e: expert_weights_numpy(cfg, e))
        w1 = w2 = None
        w1_host = lambda e: one(e)[0]  # noqa: E731
        w2_host = lambda e: one(e)[1]  # noqa: E731
    elif weights_on_host(cfg):
        w1_host, w2_host = gen_weights_numpy(cfg)
        w1 = torch.from_numpy(w1_host.view(np.int16)).view(torch.bfloat16).to(device)
        w2 = torch.from_numpy(w2_host.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        w1, w2 = gen_weights_torch(cfg, device)
        w1_host = lambda e: torch_bf16_to_bits(w1[e])  # noqa: E731
        w2_host = lambda e: torch_bf16_to_bits(w2[e])  # noqa: E731
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(device)
    ids = torch.from_numpy(ids_np).to(device)
    w = torch.from_numpy(w_np).to(device)
    return Case(cfg, x, ids, w, w1, w2, x_bits, ids_np, w_np, w1_host, w2_host)
