"""Pins the oracle to facts that do not come from the oracle itself (CPU only).

Each test names what fixes the expected value: a closed form or identity of the mathematics, a
library routine, the pages' sparse == dense-masked identity, or an independent float64 brute force.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from tests import tiny


# ---------------------------------------------------------------- GELU (tanh form, Inferentia2 port §4.5)

XS = np.concatenate([np.linspace(-12, 12, 4801), [0.0, 1e-8, -1e-8, 30.0, -30.0]])


def test_gelu_odd_part_identity():
    # tanh is odd, so the tanh-form GELU satisfies g(x) - g(-x) = x exactly in real arithmetic.
    # A wrong sign, a dropped 0.5 or a dropped "1 +" breaks it.
    for x in XS:
        assert abs(oracle.gelu_tanh(x) - oracle.gelu_tanh(-x) - x) <= 1e-14 * max(1.0, abs(x))


def test_gelu_close_to_erf_gelu():
    # The tanh form approximates x * Phi(x) (Phi by math.erf) with a maximum error of 4.73e-4,
    # reached near x = -2.70. Dropping the cubic term raises it to 0.034.
    err = [abs(oracle.gelu_tanh(x) - 0.5 * x * (1 + math.erf(x / math.sqrt(2)))) for x in XS]
    assert max(err) <= 4.8e-4
    assert max(err) >= 4.6e-4
    assert abs(XS[int(np.argmax(err))] + 2.70) < 0.02


def test_gelu_matches_torch_tanh_gelu():
    # torch's library GELU with approximate="tanh" implements the same published formula with
    # sqrt(2/pi), which the page prints to 10 digits as 0.7978845608.
    ref = torch.nn.functional.gelu(torch.tensor(XS, dtype=torch.float64), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(x) for x in XS])
    assert np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))) < 1e-10


def test_gelu_special_values():
    assert oracle.gelu_tanh(0.0) == 0.0
    assert oracle.gelu_tanh(30.0) == 30.0          # tanh saturates to 1
    assert abs(oracle.gelu_tanh(-30.0)) < 1e-300
    h = 1e-6                                         # slope at 0 is 1/2
    assert abs((oracle.gelu_tanh(h) - oracle.gelu_tanh(-h)) / (2 * h) - 0.5) < 1e-9


# ---------------------------------------------------------------- Gemma RMSNorm

@pytest.mark.parametrize("c", [3.0, -0.25, 1e-4, 1234.5])
def test_rmsnorm_constant_vector_closed_form(c):
    n = 2816
    w = np.random.default_rng(1).normal(0, 0.1, n).astype(np.float32)
    got = oracle.rmsnorm(np.full(n, c), w, 1e-6)
    want = c / math.sqrt(c * c + 1e-6) * (1.0 + w.astype(np.float64))
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def test_rmsnorm_matches_torch_rms_norm():
    rng = np.random.default_rng(2)
    v = rng.normal(0, 3, 2816)
    w = rng.normal(0, 0.1, 2816).astype(np.float32)
    ref = torch.nn.functional.rms_norm(torch.tensor(v), (2816,), torch.tensor(1.0 + w.astype(np.float64)), eps=1e-6)
    np.testing.assert_allclose(oracle.rmsnorm(v, w, 1e-6), ref.numpy(), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- router

def _router_case(shape, T, seed, skew=False):
    x, w = tiny.case(shape, T, seed, full_layer=False, skew=skew)
    d = tiny.dims_of(shape, full_layer=False)
    o = oracle.forward(d, x, w, want=("logits", "probs", "topk_idx", "topk_w", "topk_w_renorm", "gap"))
    return d, x, w, o


@pytest.mark.parametrize("shape,seed", [(tiny.SMALL, 3), (tiny.TINY, 4)])
def test_router_logits_against_float64(shape, seed):
    d, x, w, o = _router_case(shape, 64, seed)
    xf = brute.bf16_to_f64(x).reshape(64, -1)
    r = xf / np.sqrt((xf ** 2).mean(1, keepdims=True) + 1e-6) * (1 + w["router_norm_w"]) * shape["hidden"] ** -0.5
    ref = r @ w["router_w"].astype(np.float64).T
    assert np.max(np.abs(o["logits"] - ref)) < 1e-5


def test_router_softmax_topk_renorm():
    d, x, w, o = _router_case(tiny.SMALL, 256, 5)
    E, K = d["n_experts"], d["top_k"]
    lg = o["logits"].astype(np.float64)
    # softmax of the oracle's own fp32 logits, in float64
    z = np.exp(lg - lg.max(1, keepdims=True))
    np.testing.assert_allclose(o["probs"], z / z.sum(1, keepdims=True), rtol=2e-6, atol=1e-9)
    # top-K: torch.topk of the logits gives the same set; the gap is K-th minus (K+1)-th value
    vals, idx = torch.topk(torch.tensor(o["logits"]), K + 1, dim=1)
    np.testing.assert_array_equal(o["topk_idx"], np.sort(idx[:, :K].numpy(), axis=1))
    np.testing.assert_array_equal(o["gap"], (vals[:, K - 1] - vals[:, K]).numpy())
    # renormalised weights sum to 1 before per_expert_scale; the scale multiplies them after
    assert np.max(np.abs(o["topk_w_renorm"].astype(np.float64).sum(1) - 1.0)) <= 1e-6
    np.testing.assert_array_equal(o["topk_w"], o["topk_w_renorm"] * w["per_expert_scale"][o["topk_idx"]])
    # closed form of the renormalised weights: exp(l_k) / sum over the selected exp(l_j)
    sel = np.take_along_axis(lg, o["topk_idx"].astype(np.int64), 1)
    cf = np.exp(sel - sel.max(1, keepdims=True))
    np.testing.assert_allclose(o["topk_w_renorm"], cf / cf.sum(1, keepdims=True), rtol=3e-6)
    assert (np.diff(o["topk_idx"], axis=1) > 0).all() and o["topk_idx"].max() < E


def test_router_ties_pick_lower_expert_id():
    shape = dict(tiny.TINY)
    x, w = tiny.case(shape, 4, 6, full_layer=False)
    rw = w["router_w"].copy()
    big = np.abs(rw).max() * 10
    rw[:] = 0.0
    # experts 2, 4 and 6 get the same row (bitwise-equal logits) that dominates the others
    rw[[2, 4, 6]] = big * np.sign(brute.bf16_to_f64(x)[0]).astype(np.float32)
    w["router_w"] = rw
    d = tiny.dims_of(shape, full_layer=False)
    o = oracle.forward(d, x[:1], w, want=("topk_idx", "gap", "logits"))
    assert o["logits"][0, 2] == o["logits"][0, 4] == o["logits"][0, 6]
    np.testing.assert_array_equal(o["topk_idx"][0], [2, 4])
    assert o["gap"][0] == 0.0


def test_all_experts_selected_is_plain_softmax():
    # K = E: no choice is made; the weights are the softmax times per_expert_scale.
    shape = dict(tiny.TINY, top_k=8)
    d, x, w, o = _router_case(shape, 16, 7)
    np.testing.assert_array_equal(o["topk_idx"], np.tile(np.arange(8), (16, 1)))
    np.testing.assert_allclose(o["topk_w_renorm"], o["probs"], rtol=1e-6)


# ---------------------------------------------------------------- experts

def test_identical_experts_reduce_to_one_mlp():
    # All experts equal and per_expert_scale = 1: the expert branch is sum_k w_k * MLP(x) with
    # sum_k w_k = 1, i.e. one plain MLP, evaluated here with torch float64 matmuls and GELU.
    shape = tiny.SMALL
    x, w = tiny.case(shape, 12, 8, full_layer=False, weight_std=0.3)
    E, I, H = shape["n_experts"], shape["moe_inter"], shape["hidden"]
    w["gate_up"] = np.tile(w["gate_up"][:1], (E, 1, 1))
    w["down"] = np.tile(w["down"][:1], (E, 1, 1))
    w["per_expert_scale"] = np.ones(E, np.float32)
    d = tiny.dims_of(shape, full_layer=False)
    o = oracle.forward(d, x, w, want=("out",))
    xt = torch.tensor(brute.bf16_to_f64(x).reshape(-1, H))
    gu = torch.tensor(brute.bf16_to_f64(w["gate_up"][0]).reshape(2 * I, H))
    dn = torch.tensor(brute.bf16_to_f64(w["down"][0]).reshape(H, I))
    ref = (torch.nn.functional.gelu(xt @ gu[:I].T, approximate="tanh") * (xt @ gu[I:].T)) @ dn.T
    np.testing.assert_allclose(o["out"], ref.numpy(), rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("full", [False, True])
def test_sparse_equals_dense_masked_bitwise_tiny(full):
    # "The traceable trick": every expert weighted by 0 off the top-K gives the same result.
    x, w = tiny.case(tiny.SMALL, 32, 9, full_layer=full, weight_std=0.3)
    d = tiny.dims_of(tiny.SMALL, full_layer=full)
    want = ("out", "moe", "y_slot", "h_slot")
    a = oracle.forward(d, x, w, want=want)
    b = oracle.forward(d, x, w, want=want, masked_dense=True)
    for k in want:
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.slow
def test_sparse_equals_dense_masked_bitwise_gemma_shapes():
    from mixture_experts_ffn_router_gb300 import synth
    x = synth.bf16_bits(synth.make_x(2, seed=11))
    w = synth.host_arrays(synth.make_weights(seed=11, full_layer=True))
    d = oracle.gemma_dims(full_layer=True)
    a = oracle.forward(d, x, w, want=("out", "moe"))
    b = oracle.forward(d, x, w, want=("out", "moe"), masked_dense=True)
    np.testing.assert_array_equal(a["moe"], b["moe"])
    np.testing.assert_array_equal(a["out"], b["out"])


# ---------------------------------------------------------------- whole layer vs the float64 brute force

@pytest.mark.parametrize("shape", [tiny.TINY, tiny.SMALL])
@pytest.mark.parametrize("full", [False, True])
@pytest.mark.parametrize("pre2", [False, True])
def test_layer_against_brute_force(shape, full, pre2):
    if pre2 and not full:
        pytest.skip("the router-input reading only differs in the full layer")
    T = 40
    x, w = tiny.case(shape, T, 12 + shape["hidden"], full_layer=full, weight_std=0.3)
    d = tiny.dims_of(shape, full_layer=full, router_reads_pre2=pre2)
    o = oracle.forward(d, x, w, want=("out", "moe", "topk_idx", "topk_w", "gap", "logits", "dense"))
    b = brute.forward(d, x, w)
    clear = b["gap"] > 1e-4                      # tokens whose top-K choice is not a near tie
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(o["topk_idx"][clear], b["topk_idx"][clear])
    np.testing.assert_allclose(o["topk_w"][clear], b["topk_w"][clear], rtol=2e-6)
    np.testing.assert_allclose(o["logits"], b["logits"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(o["out"][clear], b["out"][clear], rtol=1e-5, atol=1e-6)
    if full:
        np.testing.assert_allclose(o["dense"], b["dense"], rtol=1e-9, atol=1e-12)


def test_router_input_reading_changes_the_result():
    # The two readings of the router's input differ in the full layer, so the default is a choice.
    x, w = tiny.case(tiny.SMALL, 16, 13, full_layer=True, weight_std=0.3)
    a = oracle.forward(tiny.dims_of(tiny.SMALL, True, False), x, w, want=("logits",))
    b = oracle.forward(tiny.dims_of(tiny.SMALL, True, True), x, w, want=("logits",))
    assert np.max(np.abs(a["logits"] - b["logits"])) > 1e-3


# ---------------------------------------------------------------- norms, residual, layer_scalar

def _torch_rms(v, w):
    return torch.nn.functional.rms_norm(v, (v.shape[-1],), torch.tensor(1.0 + w.astype(np.float64)), eps=float(np.float32(1e-6)))


@pytest.mark.parametrize("zero", ["experts", "dense"])
def test_one_branch_zero_reduces_the_norm_chain(zero):
    # With one branch's weights all zero that branch is 0, its RMSNorm is 0, and the layer is
    # (x + N_post(N_other(branch))) * layer_scalar, evaluated here with torch's rms_norm.
    shape = tiny.SMALL
    x, w = tiny.case(shape, 10, 14, full_layer=True, weight_std=0.3)
    H, D = shape["hidden"], shape["dense_inter"]
    if zero == "experts":
        w["gate_up"] = np.zeros_like(w["gate_up"])
    else:
        w["dense_gate"] = np.zeros_like(w["dense_gate"])
    d = tiny.dims_of(shape, full_layer=True)
    o = oracle.forward(d, x, w, want=("out", "moe", "dense"))
    xt = torch.tensor(brute.bf16_to_f64(x).reshape(-1, H))
    if zero == "experts":
        assert np.all(o["moe"] == 0.0)
        s = _torch_rms(torch.tensor(o["dense"]), w["post_ff_ln_1"])
    else:
        assert np.all(o["dense"] == 0.0)
        s = _torch_rms(torch.tensor(o["moe"]), w["post_ff_ln_2"])
    ref = (xt + _torch_rms(s, w["post_ff_ln"])) * float(np.float32(w["layer_scalar"]))
    np.testing.assert_allclose(o["out"], ref.numpy(), rtol=1e-12, atol=1e-12)
    _ = D


def test_layer_scalar_scales_the_output():
    x, w = tiny.case(tiny.SMALL, 8, 15, full_layer=True, weight_std=0.3)
    d = tiny.dims_of(tiny.SMALL, full_layer=True)
    w1 = dict(w, layer_scalar=1.0)
    a = oracle.forward(d, x, w, want=("out",))["out"]
    b = oracle.forward(d, x, w1, want=("out",))["out"]
    np.testing.assert_array_equal(a, b * float(np.float32(0.8)))


# ---------------------------------------------------------------- permutation

@pytest.mark.parametrize("T,E,K,seed", [(1, 8, 2, 0), (37, 16, 4, 1), (300, 128, 8, 2), (0, 8, 2, 3)])
def test_permutation_is_the_stable_sort_by_expert(T, E, K, seed):
    rng = np.random.default_rng(seed)
    idx = np.sort(np.stack([rng.choice(E, K, replace=False) for _ in range(T)]), axis=1).astype(np.int32) \
        if T else np.zeros((0, K), np.int32)
    wt = rng.random((T, K)).astype(np.float32)
    p = oracle.permute(idx, wt, E)
    slots = sorted(range(T * K), key=lambda s: (idx.flat[s], s // K))
    np.testing.assert_array_equal(p["perm"], np.array([s // K for s in slots], np.int32))
    np.testing.assert_array_equal(p["w_sorted"], wt.flatten()[slots] if T else np.zeros(0, np.float32))
    np.testing.assert_array_equal(p["counts"], np.bincount(idx.flatten(), minlength=E))
    np.testing.assert_array_equal(p["offsets"], np.concatenate([[0], np.cumsum(p["counts"])]))
    pos = np.empty(T * K, np.int64)
    pos[slots] = np.arange(T * K)
    np.testing.assert_array_equal(p["slot_pos"].flatten(), pos)


def test_permutation_rejects_bad_expert_ids():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 9]], np.int32), None, 8)


def test_route_only_matches_forward():
    x, w = tiny.case(tiny.SMALL, 50, 16, full_layer=True, weight_std=0.3)
    for pre2 in (False, True):
        d = tiny.dims_of(tiny.SMALL, full_layer=True, router_reads_pre2=pre2)
        want = ("logits", "probs", "topk_idx", "topk_w", "topk_w_renorm", "gap")
        a = oracle.forward(d, x, w, want=want)
        b = oracle.forward(d, x, w, want=want, route_only=True)
        for k in want:
            np.testing.assert_array_equal(a[k], b[k])


# ---------------------------------------------------------------- degenerate cases

def test_empty_batch():
    x, w = tiny.case(tiny.SMALL, 0, 60, full_layer=True)
    o = oracle.forward(tiny.dims_of(tiny.SMALL, full_layer=True), x, w, want=("out", "topk_idx", "topk_w"))
    assert o["out"].shape == (0, tiny.SMALL["hidden"]) and o["topk_idx"].shape == (0, tiny.SMALL["top_k"])


def test_top_one_routing_is_one_scaled_expert():
    # With K = 1 the renormalised weight is exactly 1, so each token's expert branch is
    # per_expert_scale[e] times one plain expert MLP (torch fp64 matmuls, library tanh GELU).
    shape = dict(tiny.SMALL, top_k=1)
    x, w = tiny.case(shape, 20, 61, full_layer=False, weight_std=0.3)
    o = oracle.forward(tiny.dims_of(shape, full_layer=False), x, w, want=("out", "topk_idx", "topk_w", "topk_w_renorm"))
    assert (o["topk_w_renorm"] == 1.0).all()
    E, H, I = shape["n_experts"], shape["hidden"], shape["moe_inter"]
    xt = torch.tensor(brute.bf16_to_f64(x).reshape(-1, H))
    gu = torch.tensor(brute.bf16_to_f64(w["gate_up"]).reshape(E, 2 * I, H))
    dn = torch.tensor(brute.bf16_to_f64(w["down"]).reshape(E, H, I))
    for t in range(xt.shape[0]):
        e = int(o["topk_idx"][t, 0])
        g = gu[e] @ xt[t]
        h = torch.nn.functional.gelu(g[:I], approximate="tanh") * g[I:]
        ref = float(w["per_expert_scale"][e]) * (dn[e] @ h)
        np.testing.assert_allclose(o["out"][t], ref.numpy(), rtol=0, atol=1e-11 * max(1.0, ref.abs().max().item()))
