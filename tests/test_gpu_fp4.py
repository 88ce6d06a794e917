"""MXFP4 experts on the GPU ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 — where
every rank weighted the wrong experts", section "The fp4 rabbit hole": a microscaling fp4 format,
32 fp4 values per block with one shared scale), through the C ABI (GB300 only).

* The device quantiser equals the oracle's bit for bit (codes and E8M0 scales).
* The layer with MXFP4 experts meets the block's acceptance rules against the oracle run on the
  same MXFP4 weights (routing, permutation, values).
* Argument checks of the quantiser and of the MXFP4 weight fields.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

FULL, MOE = B.MOE_FFN_FULL_LAYER, B.MOE_FFN_MOE_ONLY


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


def _device_quantize(w: torch.Tensor):
    rows, cols = w.shape
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    rc = B.moe_ffn_quantize_mxfp4(w.data_ptr(), rows, cols, codes.data_ptr(), scales.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == B.MOE_FFN_OK
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("cols", [2816, 704, 32])
def test_quantizer_matches_the_oracle_bitwise(cols):
    g = torch.Generator().manual_seed(cols + 1)
    rows = 515
    mag = torch.exp(torch.randn(rows, 1, generator=g) * 4.0)        # row scales over many octaves
    w = (torch.randn(rows, cols, generator=g) * mag).to(torch.bfloat16)
    w[3] = 0.0                                                         # all-zero blocks
    w[4, :32] = 0.0
    w[4, 5] = -3.0                                                     # a single nonzero entry
    w[5, :8] = torch.tensor([4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])  # midpoints at scale 1
    w[6, :8] = -w[5, :8]
    codes, scales = _device_quantize(w.cuda())
    co, so = oracle.quantize_mxfp4(synth.bf16_bits(w))
    np.testing.assert_array_equal(scales, so)
    np.testing.assert_array_equal(codes, co)


def test_quantizer_on_real_expert_rows():
    w = synth.make_weights(seed=78, device="cuda", full_layer=False)
    for name, cols in (("gate_up", 2816), ("down", 704)):
        rows = w[name].reshape(-1, cols)[:3 * 1408].contiguous()
        codes, scales = _device_quantize(rows)
        co, so = oracle.quantize_mxfp4(synth.bf16_bits(rows))
        np.testing.assert_array_equal(scales, so)
        np.testing.assert_array_equal(codes, co)


def test_quantizer_rejects_bad_arguments():
    w = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((4, 32), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 2), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert B.moe_ffn_quantize_mxfp4(w.data_ptr(), 4, 48, c.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_EINVAL
    assert B.moe_ffn_quantize_mxfp4(w.data_ptr() + 2, 4, 64, c.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_EALIGN
    assert B.moe_ffn_quantize_mxfp4(0, 4, 64, c.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_EINVAL
    assert B.moe_ffn_quantize_mxfp4(w.data_ptr(), 0, 64, c.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_OK


def _fp4_case(mode, T, seed):
    x, w = G.make_case(mode, T, seed)
    wq = B.quantize_experts_mxfp4(w)
    torch.cuda.synchronize()
    del wq["gate_up"], wq["down"]
    wh = G.host_weights(wq)                # the oracle sees only the MXFP4 experts
    return x, w, wq, wh


@pytest.mark.parametrize("mode,T", [(FULL, 64), (FULL, 1), (FULL, 33), (FULL, 200), (MOE, 8)])
def test_fp4_layer_against_the_oracle(mode, T):
    x, _, wq, wh = _fp4_case(mode, T, 1900 + T)
    run = G.Run(mode, x, wq)
    xb = synth.bf16_bits(x)
    ref = G.oracle_forward(mode, xb, wh)
    same = G.check_routing(run, ref)
    G.check_permutation(run)
    G.check_values(run.out_f64[same], ref["out"][same], "fp4 T=%d" % T)


def test_fp4_layer_sampled_1024():
    T = 1024
    x, _, wq, wh = _fp4_case(FULL, T, 2024)
    run = G.Run(FULL, x, wq)
    xb = synth.bf16_bits(x)
    route = G.oracle_route(FULL, xb, wh)
    same = G.check_routing(run, route)
    G.check_permutation(run)
    tok = np.unique(np.concatenate([np.random.default_rng(6).choice(T, 32, replace=False), [0, T - 1]]))
    ref = G.oracle_forward(FULL, xb, wh, tokens=tok, want=("out",))
    G.check_values(run.out_f64[tok][same[tok]], ref["out"][same[tok]], "fp4 T=1024")


def test_fp4_output_near_bf16_output():
    # MXFP4 moves each expert weight by up to a grid step of its block (saturation included); the
    # block's output moves by a few percent, more than int8's.
    x, w, wq, _ = _fp4_case(FULL, 64, 1950)
    a = G.Run(FULL, x, w).out_f64
    b = G.Run(FULL, x, wq).out_f64
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-3 < rel < 0.3


def test_fp4_fields_must_come_together_and_exclude_int8():
    x, w, wq, _ = _fp4_case(FULL, 16, 1960)
    m = B.MoeFFN(FULL, 16)
    out = torch.empty_like(x)
    st = torch.cuda.current_stream().cuda_stream
    ws = B.weights_struct(wq)
    ws.down_f4s = None
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), 16, ws, out.data_ptr(), st) == B.MOE_FFN_EINVAL
    both = B.quantize_experts_int8(dict(w))
    both.update({k: wq[k] for k in B.F4_FIELDS})
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), 16, B.weights_struct(both), out.data_ptr(), st) == B.MOE_FFN_EINVAL
