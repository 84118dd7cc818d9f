"""Seeded synthetic inputs and the workload registry (data only, no layer arithmetic)."""
from .configs import ACCURACY, ALL, CONFIGS, FP8, SMALL, LAYOUT_CODE, ALGO_CODE, MoeConfig  # noqa: F401
from .inputs import (expert_weights_numpy, gen_x, gen_routing, gen_weights_numpy, gen_weights_torch,  # noqa: F401
                     weights_on_host, f32_to_bf16_bits, bf16_bits_to_f32, torch_bf16_to_bits)
