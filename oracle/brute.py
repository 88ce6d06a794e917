"""A second, independent float64 formulation of the block for tiny shapes (test infrastructure).

It shares nothing with moe_oracle.c but the definition on the pages. Where the C oracle loops over
the K selected experts of one token, this one forms every expert's output for every token with
einsum and contracts with a [T, E] matrix of router weights that is zero off the top-K — the
"compute all experts, mask to top-8" form of "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS
Inferentia2", section "The traceable trick". The router runs in float64 here (fp32 in the C
oracle), so the two agree to about 1e-6 relative wherever the top-K choice is clear.
GELU is torch's library routine (approximate="tanh"), the tanh form of "Porting Gemma-4 (2B / 4B /
12B) to AWS Inferentia2" §4.5.
"""
import numpy as np
import torch


def _gelu(a: np.ndarray) -> np.ndarray:
    return torch.nn.functional.gelu(torch.from_numpy(np.ascontiguousarray(a)), approximate="tanh").numpy()


def _rms(v: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * (1.0 + w.astype(np.float64))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def forward(dims: dict, x_bits: np.ndarray, weights: dict) -> dict:
    """dims/x_bits/weights as for oracle.forward. Returns out, moe, dense, logits, topk_idx, topk_w, gap."""
    H, E, K, I = dims["hidden"], dims["n_experts"], dims["top_k"], dims["moe_inter"]
    full = bool(dims.get("full_layer", 0))
    eps = float(np.float32(dims["eps"]))
    scale = float(np.float32(dims["router_scale"]))
    x = bf16_to_f64(x_bits).reshape(-1, H)
    T = x.shape[0]
    f64 = lambda k: np.asarray(weights[k], dtype=np.float64)

    n2 = _rms(x, weights["pre_ff_ln_2"], eps) if full else x
    xr = n2 if (full and dims.get("router_reads_pre2", 0)) else x
    r = _rms(xr, weights["router_norm_w"], eps) * scale
    logits = r @ f64("router_w").T                                   # [T, E]
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    order = np.argsort(-logits, axis=1, kind="stable")                # ties: lower id first
    top = order[:, :K]
    gap = (np.take_along_axis(logits, order[:, K - 1:K], 1) - np.take_along_axis(logits, order[:, K:K + 1], 1))[:, 0] \
        if K < E else np.zeros(T)
    M = np.zeros((T, E))
    rows = np.arange(T)[:, None]
    psel = p[rows, top]
    M[rows, top] = psel / psel.sum(axis=1, keepdims=True) * f64("per_expert_scale")[top]

    # Expert weights: bf16 bits, or float64 values given as gate_up_f64 / down_f64 (for instance the
    # dequantised int8 form of "Can it run on a smaller box?").
    gu = (f64("gate_up_f64") if "gate_up_f64" in weights else bf16_to_f64(weights["gate_up"])).reshape(E, 2 * I, H)
    dn = (f64("down_f64") if "down_f64" in weights else bf16_to_f64(weights["down"])).reshape(E, H, I)
    G = np.einsum("th,eih->tei", n2, gu[:, :I, :])
    U = np.einsum("th,eih->tei", n2, gu[:, I:, :])
    Y = np.einsum("tei,ehi->teh", _gelu(G) * U, dn)                 # every expert, every token
    moe = np.einsum("te,teh->th", M, Y)

    res = {"moe": moe, "logits": logits, "gap": gap,
           "topk_idx": np.sort(top, axis=1).astype(np.int32)}
    res["topk_w"] = np.take_along_axis(M, res["topk_idx"].astype(np.int64), 1)
    if full:
        D = dims["dense_inter"]
        n1 = _rms(x, weights["pre_ff_ln"], eps)
        Wg = bf16_to_f64(weights["dense_gate"]).reshape(D, H)
        Wu = bf16_to_f64(weights["dense_up"]).reshape(D, H)
        Wd = bf16_to_f64(weights["dense_down"]).reshape(H, D)
        dense = (_gelu(n1 @ Wg.T) * (n1 @ Wu.T)) @ Wd.T
        s = _rms(dense, weights["post_ff_ln_1"], eps) + _rms(moe, weights["post_ff_ln_2"], eps)
        res["dense"] = dense
        res["out"] = (x + _rms(s, weights["post_ff_ln"], eps)) * float(np.float32(weights["layer_scalar"]))
    else:
        res["out"] = moe
    return res
