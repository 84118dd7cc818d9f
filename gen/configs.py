"""Workload registry: the five MoE expert-parallel layer shapes plus small test shapes.

Notation follows the FlashInfer MoE-EP design page ("MoE-EP implementation & usage",
section 3 "Algorithm / layout contracts") and the Mooncake EP guide (Buffer.dispatch
parameters): W logical ranks ("world"), Tr tokens per rank
(num_max_dispatch_tokens_per_rank), E experts, k = top_k, H = hidden, I = FFN
intermediate size.  Token t belongs to logical rank t // Tr; expert e lives on logical
rank e // (E // W).

This module holds shapes and seeds only; it contains none of the layer's arithmetic.
"""
from dataclasses import dataclass, replace

LAYOUTS = ("EM", "RM", "FLAT")          # EXPERT_MAJOR, RANK_MAJOR, FLAT
LAYOUT_CODE = {"EM": 0, "RM": 1, "FLAT": 2}
ALGO_CODE = {"LL": 0, "HT": 1}


@dataclass(frozen=True)
class MoeConfig:
    name: str
    W: int            # logical ranks
    Tr: int           # max tokens per logical rank
    H: int            # hidden
    E: int            # experts (global)
    k: int            # top_k
    I: int            # FFN intermediate
    layout: str       # "EM" | "RM" | "FLAT"
    algo: str         # "LL" | "HT"
    routing: str      # "uniform" | "zipf" | "dirichlet"
    T: int = -1       # tokens in the batch; -1 means W*Tr
    zipf_s: float = 1.1
    dirichlet_alpha: float = 0.1
    seed: int = 0
    ids_dtype: str = "int64"
    mask_frac: float = 0.0   # fraction of picks replaced by -1 (masked picks)
    quant: str = "bf16"      # "bf16" | "fp8": FP8 dispatch and FP8 expert GEMMs
    expert_out: str = "fp32"  # "fp32" | "bf16": element type of expert_out
    act: str = "pair"        # "pair" | "bf16": the SwiGLU activation as GEMM2's operand

    @property
    def tokens(self) -> int:
        return self.W * self.Tr if self.T < 0 else self.T

    def with_(self, **kw) -> "MoeConfig":
        return replace(self, **kw)


# The five workloads of the layer (shapes of the pages' EP deployments; synthetic data).
CONFIGS = {
    "tiny_ll_em": MoeConfig("tiny_ll_em", W=2, Tr=32, H=256, E=8, k=2, I=512,
                            layout="EM", algo="LL", routing="uniform"),
    "mixtral_ll_em": MoeConfig("mixtral_ll_em", W=8, Tr=128, H=4096, E=8, k=2, I=14336,
                               layout="EM", algo="LL", routing="uniform"),
    "dsv3_ll_rm": MoeConfig("dsv3_ll_rm", W=8, Tr=128, H=7168, E=256, k=8, I=2048,
                            layout="RM", algo="LL", routing="zipf"),
    "dsv3_ht_flat": MoeConfig("dsv3_ht_flat", W=8, Tr=4096, H=7168, E=256, k=8, I=2048,
                              layout="FLAT", algo="HT", routing="uniform"),
    "ragged_em": MoeConfig("ragged_em", W=8, Tr=2048, H=2048, E=128, k=4, I=1024,
                           layout="EM", algo="LL", routing="dirichlet"),
}

# Mid-size shapes that the oracle finishes in seconds but that still span several
# 128-row tiles, several 256-column tiles and a ragged row tail, one per layout.
SMALL = {
    "small_em": MoeConfig("small_em", W=4, Tr=96, H=512, E=16, k=4, I=384,
                          layout="EM", algo="LL", routing="dirichlet", T=350),
    "small_rm": MoeConfig("small_rm", W=4, Tr=96, H=512, E=16, k=4, I=384,
                          layout="RM", algo="LL", routing="zipf", T=350),
    "small_flat": MoeConfig("small_flat", W=4, Tr=96, H=512, E=16, k=4, I=384,
                            layout="FLAT", algo="HT", routing="uniform", T=350),
}

# Shapes with many rows per expert (>= 192 on average), which take the two-SM GEMM tiles
# (256 rows per tile), still small enough for the oracle; ragged tails in every expert.
SMALL.update({
    "pair_em": MoeConfig("pair_em", W=2, Tr=384, H=512, E=4, k=2, I=384,
                         layout="EM", algo="LL", routing="uniform", T=700),
    "pair_rm": MoeConfig("pair_rm", W=2, Tr=384, H=384, E=4, k=2, I=256,
                         layout="RM", algo="LL", routing="zipf", T=700),
    "pair_flat": MoeConfig("pair_flat", W=2, Tr=384, H=512, E=4, k=3, I=384,
                           layout="FLAT", algo="HT", routing="uniform", T=700),
})

# Shapes with a long K loop (>= 4096: hidden for the first GEMM, intermediate for the
# second) and >= 512 rows per expert on average, which take the one-CTA 256-row GEMM
# tiles; ragged tails in every expert; H 384 gives 128-wide second-GEMM tiles.  The other
# dimension stays small so that the oracle finishes in seconds.
SMALL.update({
    "tall_em": MoeConfig("tall_em", W=2, Tr=560, H=4096, E=4, k=2, I=512,
                         layout="EM", algo="LL", routing="uniform", T=1100),
    "tall_rm": MoeConfig("tall_rm", W=2, Tr=560, H=384, E=4, k=2, I=4096,
                         layout="RM", algo="LL", routing="zipf", T=1100),
    "tall_flat": MoeConfig("tall_flat", W=2, Tr=560, H=512, E=4, k=2, I=4096,
                           layout="FLAT", algo="HT", routing="uniform", T=1100),
})

# Batches of more than 16384 picks, far above the single-CTA routing limit, which take the three-kernel
# multi-block routing path; narrow H and I keep the oracle fast.
SMALL.update({
    "blocks_em": MoeConfig("blocks_em", W=4, Tr=1100, H=256, E=16, k=4, I=128,
                           layout="EM", algo="HT", routing="dirichlet", T=4300),
    "blocks_rm": MoeConfig("blocks_rm", W=4, Tr=1100, H=256, E=16, k=4, I=128,
                           layout="RM", algo="LL", routing="zipf", T=4300),
    "blocks_flat": MoeConfig("blocks_flat", W=4, Tr=1100, H=256, E=16, k=4, I=128,
                             layout="FLAT", algo="HT", routing="uniform", T=4300, mask_frac=0.1),
})

# The same workloads with FP8 dispatch and FP8 expert GEMMs (use_fp8).
FP8 = {name + "_fp8": cfg.with_(name=name + "_fp8", quant="fp8") for name, cfg in CONFIGS.items()}

# The same workloads with bf16 expert_out (and the per-pick rows of RANK_MAJOR / FLAT).
EO16 = {name + "_eo16": cfg.with_(name=name + "_eo16", expert_out="bf16") for name, cfg in CONFIGS.items()}

# The same workloads with the single bf16 activation (one bf16 operand of the second GEMM
# instead of the default hi + lo pair).
ACT16 = {name + "_act16": cfg.with_(name=name + "_act16", act="bf16") for name, cfg in CONFIGS.items()}

# The shapes of the FlashInfer MoE-EP page's accuracy check ("MoE-EP implementation &
# usage", section 4 "Usage walkthrough" and section 5 "Correctness status"): 16 experts,
# top-8, hidden 8192, intermediate 2048, world 8; 128 tokens per rank for the two LL
# layouts, 4096 for HT FLAT.  The page does not state the routing; uniform distinct top-k
# is the plainest reading.  H = 8192 is the widest hidden of any test shape.
ACCURACY = {
    "fi_ll_em": MoeConfig("fi_ll_em", W=8, Tr=128, H=8192, E=16, k=8, I=2048,
                          layout="EM", algo="LL", routing="uniform"),
    "fi_ll_rm": MoeConfig("fi_ll_rm", W=8, Tr=128, H=8192, E=16, k=8, I=2048,
                          layout="RM", algo="LL", routing="uniform"),
    "fi_ht_flat": MoeConfig("fi_ht_flat", W=8, Tr=4096, H=8192, E=16, k=8, I=2048,
                            layout="FLAT", algo="HT", routing="uniform"),
}

ALL = {**CONFIGS, **SMALL, **FP8, **EO16, **ACT16, **ACCURACY}

# Smaller cases for detailed (multi-pass) profiler captures of the same kernels: 4
# experts, weights 0.7 GB (larger than L2), about 1.3 GB on the device.  ncu_em_small
# (512 rows per expert) takes the one-CTA 256-row bf16 tiles and is the FP8 profile case.
PROFILE = {
    "ncu_em_small": MoeConfig("ncu_em_small", W=4, Tr=256, H=4096, E=4, k=2, I=7168,
                              layout="EM", algo="LL", routing="uniform"),
    # 384 rows per expert: the 128-row tiles of the Mixtral-like decode workload
    "ncu_em_mid": MoeConfig("ncu_em_mid", W=4, Tr=192, H=4096, E=4, k=2, I=7168,
                            layout="EM", algo="LL", routing="uniform"),
    # >= 192 rows per expert with K, N <= 2048: the two-SM (cta_group::2) tiles of the
    # ragged workload; weights 201 MB, about 1.3 GB on the device
    "ncu_pair_small": MoeConfig("ncu_pair_small", W=4, Tr=1024, H=2048, E=16, k=4, I=1024,
                                layout="EM", algo="LL", routing="dirichlet"),
    "ncu_flat_small": MoeConfig("ncu_flat_small", W=8, Tr=512, H=7168, E=32, k=8, I=2048,
                                layout="FLAT", algo="HT", routing="uniform"),
}

PROFILE.update({name + "_fp8": cfg.with_(name=name + "_fp8", quant="fp8") for name, cfg in list(PROFILE.items())})

ALL.update(PROFILE)
