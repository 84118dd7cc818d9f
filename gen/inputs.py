"""Seeded synthetic inputs for the MoE layer, shared as data by the oracle and the GPU path.

Nothing here computes any step of the layer: it only draws x, topk_ids, topk_weights
and the expert weights W1 [E, 2I, H] / W2 [E, H, I] (shapes from the FlashInfer MoE-EP
page, section 4 "Usage walkthrough", step 1).

Recipe (one numpy PCG64 stream per tensor, spawned from SeedSequence(seed)):
  x               N(0, 1), rounded to bf16 (round-to-nearest-even), returned as uint16 bits
  topk_ids        uniform: k distinct experts per token (argsort of uniform scores)
                  zipf:    Gumbel-top-k on log p_e, p_e ~ (e+1)^-s (expert 0 hottest)
                  dirichlet: p ~ Dirichlet(alpha * 1_E), Gumbel-top-k on log max(p, 1e-300)
                  optional masking: a fraction of picks set to -1 (masked pick)
  topk_weights    softmax over the k picks of N(0,1) logits, float32
  W1, W2          N(0, 0.02) rounded to bf16.  Small tensors are drawn with numpy per
                  expert; tensors above NUMPY_WEIGHT_LIMIT elements are drawn on the
                  GPU with a seeded torch generator (no CPU oracle can afford to draw
                  11e9 normals), and the oracle receives host copies of the same values.
"""
import numpy as np

from .configs import MoeConfig

NUMPY_WEIGHT_LIMIT = 64 * 1024 * 1024  # elements of W1+W2 drawn on the host with numpy

_STREAM_X, _STREAM_IDS, _STREAM_W, _STREAM_W1, _STREAM_W2, _STREAM_MASK = range(6)


def _streams(seed: int):
    return np.random.SeedSequence(seed).spawn(6)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gen_x(cfg: MoeConfig) -> np.ndarray:
    """x [T, H] as bf16 bit patterns (uint16)."""
    rng = np.random.Generator(np.random.PCG64(_streams(cfg.seed)[_STREAM_X]))
    return f32_to_bf16_bits(rng.standard_normal((cfg.tokens, cfg.H), dtype=np.float32))


def _gumbel_topk(rng, logp: np.ndarray, T: int, k: int) -> np.ndarray:
    u = rng.random((T, logp.shape[0]))
    g = -np.log(-np.log(np.clip(u, 1e-300, 1.0)))
    return np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :k]


def gen_routing(cfg: MoeConfig):
    """topk_ids [T, k] (int64 or int32) and topk_weights [T, k] float32."""
    T, E, k = cfg.tokens, cfg.E, cfg.k
    st = _streams(cfg.seed)
    rng = np.random.Generator(np.random.PCG64(st[_STREAM_IDS]))
    if cfg.routing == "uniform":
        ids = np.argsort(rng.random((T, E)), axis=1, kind="stable")[:, :k]
    elif cfg.routing == "zipf":
        logp = -cfg.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
        ids = _gumbel_topk(rng, logp, T, k)
    elif cfg.routing == "dirichlet":
        p = rng.dirichlet(np.full(E, cfg.dirichlet_alpha))
        ids = _gumbel_topk(rng, np.log(np.maximum(p, 1e-300)), T, k)
    else:
        raise ValueError(cfg.routing)
    ids = ids.astype(np.int64)
    if cfg.mask_frac > 0:
        mrng = np.random.Generator(np.random.PCG64(st[_STREAM_MASK]))
        ids[mrng.random((T, k)) < cfg.mask_frac] = -1
    wrng = np.random.Generator(np.random.PCG64(st[_STREAM_W]))
    logits = wrng.standard_normal((T, k))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    if cfg.ids_dtype == "int32":
        ids = ids.astype(np.int32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(w)


def weights_on_host(cfg: MoeConfig) -> bool:
    return cfg.E * 3 * cfg.H * cfg.I <= NUMPY_WEIGHT_LIMIT


def expert_weights_numpy(cfg: MoeConfig, e: int):
    """Expert e's W1 [2I, H] and W2 [H, I] as bf16 bit patterns, from its own numpy streams."""
    st = _streams(cfg.seed)
    s1 = st[_STREAM_W1].spawn(cfg.E)[e]
    s2 = st[_STREAM_W2].spawn(cfg.E)[e]
    r1 = np.random.Generator(np.random.PCG64(s1))
    r2 = np.random.Generator(np.random.PCG64(s2))
    w1 = f32_to_bf16_bits(0.02 * r1.standard_normal((2 * cfg.I, cfg.H), dtype=np.float32))
    w2 = f32_to_bf16_bits(0.02 * r2.standard_normal((cfg.H, cfg.I), dtype=np.float32))
    return w1, w2


def gen_weights_numpy(cfg: MoeConfig):
    """W1 [E, 2I, H] and W2 [E, H, I] as bf16 bit patterns, one numpy stream per expert."""
    w1 = np.empty((cfg.E, 2 * cfg.I, cfg.H), dtype=np.uint16)
    w2 = np.empty((cfg.E, cfg.H, cfg.I), dtype=np.uint16)
    for e in range(cfg.E):
        w1[e], w2[e] = expert_weights_numpy(cfg, e)
    return w1, w2


def gen_weights_torch(cfg: MoeConfig, device):
    """W1, W2 as torch bf16 tensors on `device`; drawn on the GPU for large shapes."""
    import torch
    if weights_on_host(cfg):
        w1, w2 = gen_weights_numpy(cfg)
        return (torch.from_numpy(w1.view(np.int16)).view(torch.bfloat16).to(device),
                torch.from_numpy(w2.view(np.int16)).view(torch.bfloat16).to(device))
    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence(cfg.seed).generate_state(1)[0]))
    w1 = torch.empty((cfg.E, 2 * cfg.I, cfg.H), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((cfg.E, cfg.H, cfg.I), dtype=torch.bfloat16, device=device)
    for e in range(cfg.E):  # per expert keeps the fp32 temporary small
        w1[e] = (0.02 * torch.randn((2 * cfg.I, cfg.H), generator=g, device=device)).to(torch.bfloat16)
        w2[e] = (0.02 * torch.randn((cfg.H, cfg.I), generator=g, device=device)).to(torch.bfloat16)
    return w1, w2


def torch_bf16_to_bits(t) -> np.ndarray:
    """Host uint16 bit patterns of a torch bf16 tensor (for handing inputs to the oracle)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
