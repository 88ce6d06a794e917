"""Pins of the oracle's MXFP4 expert form ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS
Inferentia2 — where every rank weighted the wrong experts", section "The fp4 rabbit hole": a
microscaling fp4 format, blocks of 32 fp4 values sharing one scale).

The quantiser follows the OCP Microscaling Formats (MX) v1.0 conversion: a power-of-two scale per
block of 32 consecutive elements, shared exponent floor(log2 max|w|) - 2, elements rounded to the
nearest E2M1 value with ties to even, saturating at 6. It is pinned by what that rule implies:
every block's maximum lands in [4, 8) scale units, values on the grid come back exactly, each
element is within half a grid step (or saturates to 6), midpoints go to the even code, the sign is
symmetric, and zero blocks give scale byte 0. The layer with MXFP4 experts is pinned against the
float64 brute force (oracle/brute.py) run on the dequantised weights.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from tests import tiny

FP4_SHAPE = {"hidden": 64, "n_experts": 16, "top_k": 4, "moe_inter": 32, "dense_inter": 12}


def _bf16(a) -> np.ndarray:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _block_scale(scales) -> np.ndarray:
    return np.repeat(np.exp2(np.asarray(scales, np.float64) - 127.0), 32, axis=1)


@pytest.mark.parametrize("std", [0.02, 1.0, 3e4])
def test_block_maximum_lands_in_four_to_eight_scale_units(std):
    rng = np.random.default_rng(11)
    # Rows whose magnitude varies over many octaves, so blocks take many different scales.
    w = _bf16(rng.standard_normal((40, 256)) * std * np.exp2(rng.integers(-6, 7, (40, 1))))
    codes, scales = oracle.quantize_mxfp4(w)
    amax = np.abs(_f64(w)).reshape(40, -1, 32).max(axis=2)
    units = amax / np.exp2(scales.astype(np.float64) - 127.0)
    assert ((units >= 4.0) & (units < 8.0)).all()


@pytest.mark.parametrize("std", [0.02, 1.0])
def test_error_bound_and_saturation(std):
    rng = np.random.default_rng(12)
    w = _bf16(rng.standard_normal((24, 512)) * std)
    codes, scales = oracle.quantize_mxfp4(w)
    dq = oracle.dequantize_mxfp4(codes, scales)
    X = _block_scale(scales)
    a = np.abs(_f64(w)) / X
    err = np.abs(dq - _f64(w)) / X
    # Half the gap of the E2M1 grid around the value: 0.25 below 2, 0.5 up to 4, 1 up to 6.
    bound = np.where(a <= 2.0, 0.25, np.where(a <= 4.0, 0.5, 1.0))
    inside = a <= 6.0
    assert (err[inside] <= bound[inside]).all()
    # Above 6 scale units the magnitude saturates to 6 with the element's sign.
    sat = ~inside
    assert sat.any()
    np.testing.assert_array_equal(np.abs(dq[sat]) / X[sat], 6.0)
    np.testing.assert_array_equal(np.sign(dq[sat]), np.sign(_f64(w)[sat]))


def test_grid_values_come_back_exactly():
    rng = np.random.default_rng(13)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rows, blocks = 16, 6
    mag = grid[rng.integers(0, 8, (rows, blocks, 32))]
    mag[:, :, 0] = rng.choice([4.0, 6.0], (rows, blocks))  # the block maximum fixes the scale
    sign = rng.choice([-1.0, 1.0], mag.shape)
    e = rng.integers(-20, 20, (rows, blocks, 1)).astype(np.float64)
    vals = (sign * mag * np.exp2(e)).reshape(rows, blocks * 32)
    w = _bf16(vals)
    codes, scales = oracle.quantize_mxfp4(w)
    np.testing.assert_array_equal(scales, (e[:, :, 0] + 127).astype(np.uint8))
    np.testing.assert_array_equal(oracle.dequantize_mxfp4(codes, scales), np.where(vals == 0, 0.0, vals))


def test_midpoints_go_to_the_even_code():
    # Block maximum 4 (scale 1): the midpoints between neighbouring E2M1 values and their codes.
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    want = [0, 2, 2, 4, 4, 6, 6]  # magnitude codes of 0, 1, 1, 2, 2, 4, 4
    row = np.zeros(32)
    row[0] = 4.0
    row[1:1 + len(mids)] = mids
    row[8:8 + len(mids)] = [-m for m in mids]
    codes, scales = oracle.quantize_mxfp4(_bf16(row[None, :]))
    assert scales[0, 0] == 127
    nib = np.stack([codes[0] & 15, codes[0] >> 4], axis=-1).reshape(-1)
    np.testing.assert_array_equal(nib[1:1 + len(mids)], want)
    neg = [c | 8 if c else 0 for c in want]
    np.testing.assert_array_equal(nib[8:8 + len(mids)], neg)


def test_symmetry():
    rng = np.random.default_rng(14)
    w = rng.standard_normal((8, 128)) * 0.05
    c1, s1 = oracle.quantize_mxfp4(_bf16(w))
    c2, s2 = oracle.quantize_mxfp4(_bf16(-w))
    np.testing.assert_array_equal(s1, s2)
    n1 = np.stack([c1 & 15, c1 >> 4], axis=-1)
    n2 = np.stack([c2 & 15, c2 >> 4], axis=-1)
    flipped = np.where(n1 & 7, n1 ^ 8, 0)
    np.testing.assert_array_equal(n2, flipped)


def test_zero_blocks():
    w = np.zeros((2, 64), np.uint16)
    w[1, 33] = _bf16([-0.75])[0]  # one nonzero element in the second block of row 1
    codes, scales = oracle.quantize_mxfp4(w)
    assert (scales[0] == 0).all() and (codes[0] == 0).all()
    assert scales[1, 0] == 0 and (codes[1, :16] == 0).all()
    # 0.75 = 1.5 * 2^-1: floor(log2 0.75) = -1, shared exponent -3, 0.75 = 6 scale units.
    assert scales[1, 1] == 124
    np.testing.assert_array_equal(oracle.dequantize_mxfp4(codes, scales)[1], _f64(w[1]))


def test_bad_arguments():
    with pytest.raises(ValueError):
        oracle.quantize_mxfp4(np.zeros((2, 48), np.uint16))


def _fp4_case(T, seed, full):
    x, w = tiny.case(FP4_SHAPE, T, seed, full_layer=full, weight_std=0.3)
    E, H, I = FP4_SHAPE["n_experts"], FP4_SHAPE["hidden"], FP4_SHAPE["moe_inter"]
    gc, gs = oracle.quantize_mxfp4(np.asarray(w["gate_up"]).reshape(E * 2 * I, H))
    dc, ds = oracle.quantize_mxfp4(np.asarray(w["down"]).reshape(E * H, I))
    wq = dict(w)
    del wq["gate_up"], wq["down"]
    wq.update(gate_up_f4=gc, gate_up_f4s=gs, down_f4=dc, down_f4s=ds)
    wb = dict(w)
    wb["gate_up_f64"] = oracle.dequantize_mxfp4(gc, gs)
    wb["down_f64"] = oracle.dequantize_mxfp4(dc, ds)
    return x, wq, wb


@pytest.mark.parametrize("full", [False, True])
def test_mxfp4_layer_against_brute_force(full):
    T = 40
    x, wq, wb = _fp4_case(T, 50, full)
    d = tiny.dims_of(FP4_SHAPE, full_layer=full)
    o = oracle.forward(d, x, wq, want=("out", "moe", "topk_idx"))
    b = brute.forward(d, x, wb)
    clear = b["gap"] > 1e-4
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(o["topk_idx"][clear], b["topk_idx"][clear])
    np.testing.assert_allclose(o["out"][clear], b["out"][clear], rtol=1e-5, atol=1e-6)


def test_mxfp4_sparse_equals_dense_masked_bitwise():
    x, wq, _ = _fp4_case(24, 51, True)
    d = tiny.dims_of(FP4_SHAPE, full_layer=True)
    a = oracle.forward(d, x, wq, want=("out", "moe"))
    b = oracle.forward(d, x, wq, want=("out", "moe"), masked_dense=True)
    np.testing.assert_array_equal(a["moe"], b["moe"])
    np.testing.assert_array_equal(a["out"], b["out"])
