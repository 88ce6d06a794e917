"""Pins of the oracle's int8 expert form ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS
Inferentia2 — where every rank weighted the wrong experts", section "Can it run on a smaller box?":
per-channel symmetric int8 experts).

The quantiser (one scale per output row, scale = max |w| / 127, q = w / scale rounded to nearest
and clamped to [-127, 127]) is pinned by what any such quantiser must satisfy: the reconstruction
error bound, the row maximum landing on +-127, sign symmetry, exact reconstruction of values on
the quantisation grid, and zero rows. The layer with int8 experts is pinned against the float64
brute force (oracle/brute.py) run on the dequantised weights q * scale.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from tests import tiny


def _bf16(a) -> np.ndarray:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("std", [0.02, 1.0, 300.0])
def test_quantizer_error_bound_and_row_maximum(std):
    rng = np.random.default_rng(7)
    w = _bf16(rng.standard_normal((33, 300)) * std)
    q, s = oracle.quantize_int8(w)
    wf = _f32(w).astype(np.float64)
    # |q s - w| <= s/2, widened by the fp32 rounding of w / s (|w / s| <= 127, 2^-24 relative).
    err = np.abs(q.astype(np.float64) * s[:, None] - wf)
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-5)).all()
    # The largest magnitude of each row maps to +-127, and scale = max |w| / 127 in fp32.
    amax = np.abs(_f32(w)).max(axis=1)
    np.testing.assert_array_equal(s, (amax / np.float32(127.0)).astype(np.float32))
    assert (np.abs(q).max(axis=1) == 127).all()
    j = np.abs(wf).argmax(axis=1)
    assert (np.abs(q[np.arange(len(j)), j]) == 127).all()


def test_quantizer_is_symmetric():
    rng = np.random.default_rng(8)
    w = _bf16(rng.standard_normal((9, 64)))
    q1, s1 = oracle.quantize_int8(w)
    q2, s2 = oracle.quantize_int8(w ^ np.uint16(0x8000))   # every sign flipped
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_array_equal(q1, -q2)


def test_quantizer_reconstructs_grid_values_exactly():
    # Rows of n * 2^-k with integers |n| <= 127 and one entry +-127: scale is 2^-k and q is n.
    rng = np.random.default_rng(9)
    n = rng.integers(-126, 127, size=(6, 50))
    n[:, 3] = 127 * np.where(rng.random(6) < 0.5, 1, -1)
    k = np.arange(6)[:, None] + 3
    w = _bf16(n * np.exp2(-k.astype(np.float64)))
    q, s = oracle.quantize_int8(w)
    np.testing.assert_array_equal(q, n.astype(np.int8))
    np.testing.assert_array_equal(s, np.exp2(-k[:, 0].astype(np.float64)).astype(np.float32))


def test_quantizer_zero_row():
    w = np.zeros((2, 16), np.uint16)
    w[1, 5] = _bf16([0.5])[0]
    q, s = oracle.quantize_int8(w)
    assert s[0] == 0.0 and (q[0] == 0).all()
    assert q[1, 5] == 127 and (np.delete(q[1], 5) == 0).all()


def _int8_case(shape, T, seed, full):
    x, w = tiny.case(shape, T, seed, full_layer=full, weight_std=0.3)
    E, H, I = shape["n_experts"], shape["hidden"], shape["moe_inter"]
    gq, gs = oracle.quantize_int8(np.asarray(w["gate_up"]).reshape(E * 2 * I, H))
    dq, ds = oracle.quantize_int8(np.asarray(w["down"]).reshape(E * H, I))
    wq = dict(w)
    del wq["gate_up"], wq["down"]
    wq.update(gate_up_q=gq, gate_up_scale=gs, down_q=dq, down_scale=ds)
    wb = dict(w)
    wb["gate_up_f64"] = gq.astype(np.float64) * gs[:, None].astype(np.float64)
    wb["down_f64"] = dq.astype(np.float64) * ds[:, None].astype(np.float64)
    return x, w, wq, wb


@pytest.mark.parametrize("shape", [tiny.TINY, tiny.SMALL])
@pytest.mark.parametrize("full", [False, True])
def test_int8_layer_against_brute_force(shape, full):
    T = 40
    x, _, wq, wb = _int8_case(shape, T, 30 + shape["hidden"], full)
    d = tiny.dims_of(shape, full_layer=full)
    o = oracle.forward(d, x, wq, want=("out", "moe", "topk_idx"))
    b = brute.forward(d, x, wb)
    clear = b["gap"] > 1e-4
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(o["topk_idx"][clear], b["topk_idx"][clear])
    np.testing.assert_allclose(o["out"][clear], b["out"][clear], rtol=1e-5, atol=1e-6)


def test_int8_sparse_equals_dense_masked_bitwise():
    x, _, wq, _ = _int8_case(tiny.SMALL, 24, 41, True)
    d = tiny.dims_of(tiny.SMALL, full_layer=True)
    a = oracle.forward(d, x, wq, want=("out", "moe"))
    b = oracle.forward(d, x, wq, want=("out", "moe"), masked_dense=True)
    np.testing.assert_array_equal(a["moe"], b["moe"])
    np.testing.assert_array_equal(a["out"], b["out"])


def test_int8_layer_close_to_bf16_layer():
    # Each weight moves by at most scale/2 = max|w_row| / 254; the expert branch moves by about as
    # much relative to its size (about 1% for normal rows), well inside 3%.
    x, w, wq, _ = _int8_case(tiny.SMALL, 32, 43, False)
    d = tiny.dims_of(tiny.SMALL, full_layer=False)
    a = oracle.forward(d, x, w, want=("out", "gap"))["out"]
    b = oracle.forward(d, x, wq, want=("out",))["out"]
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-4 < rel < 3e-2
