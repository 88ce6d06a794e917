"""Seeded synthetic inputs for the Gemma-4 26B-A4B feed-forward block.

This module only draws random tensors; it holds none of the block's arithmetic. Tests, the smoke
check and the benchmark use it for both the CUDA path and the oracle, which then receive the same
tensor values (the oracle gets host copies).

Recipe (per tensor, its own generator seeded with ``seed + 1000 * layer + tensor_id``):

  ===================  ==  ================================  =====  ==========================
  tensor               id  shape                             dtype  distribution
  ===================  ==  ================================  =====  ==========================
  x (layer input)       0  [T, H]                            bf16   N(0, 1)
  router_w              1  [E, H]                            fp32   N(0, 1), rows x c_e (skew)
  router_norm_w         2  [H]                               fp32   N(0, 0.1)
  per_expert_scale      3  [E]                               fp32   U(0.5, 1.5)
  gate_up               4  [E, 2I, H]                        bf16   N(0, 0.02)
  down                  5  [E, H, I]                         bf16   N(0, 0.02)
  dense_gate            6  [D, H]                            bf16   N(0, 0.02)
  dense_up              7  [D, H]                            bf16   N(0, 0.02)
  dense_down            8  [H, D]                            bf16   N(0, 0.02)
  pre_ff_ln ..          9  [H] each, ids 9..13 in the order  fp32   N(0, 0.1)
   post_ff_ln              pre, pre_2, post_1, post_2, post
  skew ranks           14  permutation of the E experts      int    uniform
  ===================  ==  ================================  =====  ==========================

Values are drawn in fp32 and rounded to bf16 (round to nearest even) where the tensor is bf16.
The small tensors (router, scales, norms, skew ranks) are always drawn on the CPU so they are the
same on every device. The large bf16 weights and x are drawn on the ``device`` argument: CPU and
CUDA generators give different streams for the same seed, so every comparison feeds both sides the
same drawn tensor, never a regenerated one.

Skewed routing: the router rows are multiplied by c_e = rank_e ** -1.1, where rank_e in 1..E is
expert e's place in a seeded random permutation. The Zipf exponent 1.1 is applied directly as the
row scale. Because x is symmetric about 0 and the router has no bias, a token and its negation pick
disjoint expert sets, so no expert can be chosen by more than about half the tokens (8x the mean
load for top-8 of 128); the tail experts with the smallest scales receive no tokens at all.
"""
import torch

GEMMA = {"hidden": 2816, "n_experts": 128, "top_k": 8, "moe_inter": 704, "dense_inter": 2112}
TENSOR_IDS = {"x": 0, "router_w": 1, "router_norm_w": 2, "per_expert_scale": 3, "gate_up": 4,
              "down": 5, "dense_gate": 6, "dense_up": 7, "dense_down": 8, "pre_ff_ln": 9,
              "pre_ff_ln_2": 10, "post_ff_ln_1": 11, "post_ff_ln_2": 12, "post_ff_ln": 13,
              "skew_ranks": 14}
ZIPF_S = 1.1
LAYER_SCALAR = 0.8


def _gen(seed: int, layer: int, name: str, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 1000 * int(layer) + TENSOR_IDS[name])
    return g


def _normal(shape, std, seed, layer, name, device, dtype):
    g = _gen(seed, layer, name, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_x(T: int, seed: int = 1234, layer: int = 0, device="cpu", dims=GEMMA) -> torch.Tensor:
    """Layer input [T, H] bf16 ~ N(0, 1)."""
    return _normal((T, dims["hidden"]), 1.0, seed, layer, "x", device, torch.bfloat16)


def skew_scales(seed: int = 1234, layer: int = 0, dims=GEMMA, s: float = ZIPF_S) -> torch.Tensor:
    """Row scales c_e = rank_e ** -s of the skewed-routing workload ([E] fp32, CPU)."""
    E = dims["n_experts"]
    perm = torch.randperm(E, generator=_gen(seed, layer, "skew_ranks"))
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    return rank.pow(-s).to(torch.float32)


def make_router_w(seed: int = 1234, layer: int = 0, device="cpu", skew: bool = False, dims=GEMMA) -> torch.Tensor:
    """The router matrix [E, H] fp32 ~ N(0, 1), rows scaled by c_e for the skewed workload. The
    same tensor make_weights draws, so a caller holding one layer's weights can switch it between
    uniform and skewed routing without drawing the expert weights again."""
    rw = _normal((dims["n_experts"], dims["hidden"]), 1.0, seed, layer, "router_w", "cpu", torch.float32)
    if skew:
        rw.mul_(skew_scales(seed, layer, dims)[:, None])
    return rw.to(device)


def make_weights(seed: int = 1234, layer: int = 0, device="cpu", full_layer: bool = True,
                 skew: bool = False, dims=GEMMA, layer_scalar: float = LAYER_SCALAR) -> dict:
    """One layer's weights as torch tensors on ``device`` (see the module docstring)."""
    H, E, I, D = dims["hidden"], dims["n_experts"], dims["moe_inter"], dims["dense_inter"]
    w = {}
    w["router_w"] = make_router_w(seed, layer, device, skew, dims)
    w["router_norm_w"] = _normal((H,), 0.1, seed, layer, "router_norm_w", "cpu", torch.float32).to(device)
    g = _gen(seed, layer, "per_expert_scale")
    w["per_expert_scale"] = (torch.rand(E, generator=g, dtype=torch.float32) + 0.5).to(device)
    w["gate_up"] = _normal((E, 2 * I, H), 0.02, seed, layer, "gate_up", device, torch.bfloat16)
    w["down"] = _normal((E, H, I), 0.02, seed, layer, "down", device, torch.bfloat16)
    if full_layer:
        w["dense_gate"] = _normal((D, H), 0.02, seed, layer, "dense_gate", device, torch.bfloat16)
        w["dense_up"] = _normal((D, H), 0.02, seed, layer, "dense_up", device, torch.bfloat16)
        w["dense_down"] = _normal((H, D), 0.02, seed, layer, "dense_down", device, torch.bfloat16)
        for name in ("pre_ff_ln", "pre_ff_ln_2", "post_ff_ln_1", "post_ff_ln_2", "post_ff_ln"):
            w[name] = _normal((H,), 0.1, seed, layer, name, "cpu", torch.float32).to(device)
    w["layer_scalar"] = float(layer_scalar)
    return w


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's bit patterns as a host numpy uint16 array (no rounding)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_arrays(weights: dict) -> dict:
    """Host numpy copies of a weights dict: float32 arrays, and uint16 bit patterns for bf16."""
    out = {}
    for k, v in weights.items():
        if isinstance(v, torch.Tensor):
            if v.dtype == torch.bfloat16:
                out[k] = bf16_bits(v)
            else:
                out[k] = v.detach().contiguous().cpu().numpy()
        else:
            out[k] = v
    return out
