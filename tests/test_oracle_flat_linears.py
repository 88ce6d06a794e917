"""The expert branch as two plain linears, sharded over ranks (CPU only).

The 26B-A4B post ("The traceable trick: compute all experts, mask to top-8") re-lays the experts
as two standard parallel linears: gate_up [128, 1408, 2816] flattened to [180224, 2816] and split
by rows (rank r of 8 owns experts 16r..16r+15), and down [128, 2816, 704] laid out as
[2816, 90112] and split by columns, the ranks' partial outputs then summed (the all-reduce). The
router is replicated and its top-k weights, which already carry the renormalisation and
per_expert_scale, mask the activations of the experts a token did not pick. The post checked that
form against the sparse one on the CPU and reports MAXDIFF about 2e-6 with cosine 1.0.

Here the same form, written with torch matmuls and torch's tanh GELU, is compared with the
oracle's experts-only output (the sparse sum over each token's 8 experts), using the oracle's own
routing: in float64 at small shapes to 1e-11 of the largest output, and at the model's shapes in
float32 within the post's 2e-6. A wrong flattening (down's columns feature-major instead of
expert-major, or gate and up rows swapped) misses by more than 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_router_gb300 import synth
from tests import tiny


def flat_two_linear(x, gate_up, down, topk_idx, topk_w, ranks, dtype):
    """x [T, H]; gate_up [E, 2I, H]; down [E, H, I]; routing [T, K]. Returns the sum over ranks."""
    E, I2, H = gate_up.shape
    I = I2 // 2
    T = x.shape[0]
    per = E // ranks
    wm = torch.zeros(T, E, dtype=dtype)
    wm.scatter_(1, torch.as_tensor(topk_idx).long(), torch.as_tensor(topk_w).to(dtype))
    gu = gate_up.reshape(E * I2, H)                      # column-parallel: rows of expert e together
    dn = down.permute(1, 0, 2).reshape(H, E * I)         # row-parallel: columns of expert e together
    xf = x.to(dtype)
    y = torch.zeros(T, H, dtype=dtype)
    for r in range(ranks):
        g = (xf @ gu[r * per * I2:(r + 1) * per * I2].to(dtype).T).reshape(T, per, I2)
        h = torch.nn.functional.gelu(g[..., :I], approximate="tanh") * g[..., I:]
        h = h * wm[:, r * per:(r + 1) * per, None]
        y += h.reshape(T, per * I) @ dn[:, r * per * I:(r + 1) * per * I].to(dtype).T
    return y


def _bf16(bits):
    return torch.from_numpy(np.asarray(bits).astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def test_flat_form_equals_the_sparse_sum_float64_small():
    shape = tiny.SMALL                                   # 16 experts: 8 ranks of 2
    x, w = tiny.case(shape, 24, 41, full_layer=False, weight_std=0.3)
    o = oracle.forward(tiny.dims_of(shape, full_layer=False), x, w, want=("out", "topk_idx", "topk_w"))
    E, H, I = shape["n_experts"], shape["hidden"], shape["moe_inter"]
    gate_up = _bf16(w["gate_up"]).reshape(E, 2 * I, H)
    down = _bf16(w["down"]).reshape(E, H, I)
    for ranks in (1, 2, 8):
        y = flat_two_linear(_bf16(x).reshape(-1, H), gate_up, down, o["topk_idx"], o["topk_w"], ranks, torch.float64)
        # The oracle's GELU uses the page's printed 0.7978845608 and torch's the exact sqrt(2/pi), 3e-12
        # apart relatively; through the expert MLP that leaves differences of a few 1e-12 here.
        np.testing.assert_allclose(y.numpy(), o["out"], rtol=0, atol=1e-11 * max(1.0, np.abs(o["out"]).max()))


def test_flat_form_at_model_shapes_within_the_posts_maxdiff():
    T = 4
    w = synth.make_weights(seed=21, device="cpu", full_layer=False)
    x = synth.make_x(T, seed=21, device="cpu")
    o = oracle.forward(oracle.gemma_dims(False), synth.bf16_bits(x), synth.host_arrays(w),
                       want=("out", "topk_idx", "topk_w"))
    y = flat_two_linear(x, w["gate_up"], w["down"], o["topk_idx"], o["topk_w"], 8, torch.float32).double().numpy()
    ref = o["out"]
    assert np.abs(y - ref).max() <= 2e-6
    cos = float((y.ravel() @ ref.ravel()) / (np.linalg.norm(y) * np.linalg.norm(ref)))
    assert cos == pytest.approx(1.0, abs=1e-9)


def test_wrong_flattenings_are_caught():
    # The same check with the two plausible layout mistakes: expert-interleaved down columns, and
    # gate and up rows swapped inside each expert.
    shape = tiny.SMALL
    x, w = tiny.case(shape, 24, 42, full_layer=False, weight_std=0.3)
    o = oracle.forward(tiny.dims_of(shape, full_layer=False), x, w, want=("out", "topk_idx", "topk_w"))
    E, H, I = shape["n_experts"], shape["hidden"], shape["moe_inter"]
    gate_up = _bf16(w["gate_up"]).reshape(E, 2 * I, H)
    down = _bf16(w["down"]).reshape(E, H, I)
    xs = _bf16(x).reshape(-1, H)
    # A [H, E*I] down whose columns run feature-major (i*E + e) instead of expert-major (e*I + i),
    # given back in the [E, H, I] form flat_two_linear lays out expert-major.
    interleaved = down.permute(1, 2, 0).reshape(H, I * E).reshape(H, E, I).permute(1, 0, 2)
    swapped = torch.cat([gate_up[:, I:], gate_up[:, :I]], dim=1)
    assert not torch.equal(interleaved, down) and not torch.equal(swapped, gate_up)
    for gu, dn in ((gate_up, interleaved), (swapped, down)):
        bad = flat_two_linear(xs, gu, dn, o["topk_idx"], o["topk_w"], 8, torch.float64)
        assert np.abs(bad.numpy() - o["out"]).max() > 1e-3
