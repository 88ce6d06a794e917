"""Tiny shapes and seeded draws for the oracle's CPU pin tests."""
import numpy as np

from mixture_experts_ffn_router_gb300 import synth

TINY = {"hidden": 16, "n_experts": 8, "top_k": 2, "moe_inter": 4, "dense_inter": 6}
SMALL = {"hidden": 64, "n_experts": 16, "top_k": 4, "moe_inter": 8, "dense_inter": 12}


def dims_of(shape: dict, full_layer: bool, router_reads_pre2: bool = False) -> dict:
    d = dict(shape)
    d["full_layer"] = int(full_layer)
    d["router_reads_pre2"] = int(router_reads_pre2)
    d["eps"] = 1e-6
    d["router_scale"] = shape["hidden"] ** -0.5
    return d


def case(shape: dict, T: int, seed: int, full_layer: bool = True, skew: bool = False,
         weight_std: float = None):
    """x bits and host weight arrays for a tiny case. weight_std rescales the bf16 weights so
    tiny hidden sizes give O(1) activations (the real 0.02 is sized for H = 2816)."""
    x = synth.bf16_bits(synth.make_x(T, seed=seed, dims=shape))
    w = synth.make_weights(seed=seed, full_layer=full_layer, skew=skew, dims=shape)
    if weight_std is not None:
        import torch
        for k in ("gate_up", "down", "dense_gate", "dense_up", "dense_down"):
            if k in w:
                w[k] = (w[k].float() * (weight_std / 0.02)).to(torch.bfloat16)
    return x, synth.host_arrays(w)


def bf16_round_f64(a: np.ndarray) -> np.ndarray:
    """Rounds float64 values to the nearest bf16 (ties to even), returned as float64."""
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().double().numpy()
