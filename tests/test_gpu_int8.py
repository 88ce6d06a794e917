"""int8 experts on the GPU ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 — where
every rank weighted the wrong experts", section "Can it run on a smaller box?": per-channel
symmetric int8 experts), through the C ABI (GB300 only).

* The device quantiser equals the oracle's bit for bit (q and scale).
* The layer with int8 experts meets the block's acceptance rules against the oracle run on the same
  int8 weights (routing, permutation, values).
* Argument checks of the quantiser and of the int8 weight fields.
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
    q = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    rc = B.moe_ffn_quantize_int8(w.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == B.MOE_FFN_OK
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("cols", [2816, 704, 8])
def test_quantizer_matches_the_oracle_bitwise(cols):
    g = torch.Generator().manual_seed(cols)
    rows = 515
    mag = torch.exp(torch.randn(rows, 1, generator=g) * 4.0)        # row scales over many octaves
    w = (torch.randn(rows, cols, generator=g) * mag).to(torch.bfloat16)
    w[3] = 0.0                                                         # an all-zero row
    w[4] = 0.0
    w[4, cols // 2] = -3.0                                             # a single nonzero entry
    w[5, :4] = torch.tensor([1.0, -1.0, 0.5, -0.5])                    # ties at the rounding midpoint
    q, s = _device_quantize(w.cuda())
    qo, so = oracle.quantize_int8(synth.bf16_bits(w))
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quantizer_on_real_expert_rows():
    w = synth.make_weights(seed=77, device="cuda", full_layer=False)
    for name, cols in (("gate_up", 2816), ("down", 704)):
        rows = w[name].reshape(-1, cols)[:3 * 1408].contiguous()
        q, s = _device_quantize(rows)
        qo, so = oracle.quantize_int8(synth.bf16_bits(rows))
        np.testing.assert_array_equal(q, qo)
        np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quantizer_rejects_bad_arguments():
    w = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((4, 64), dtype=torch.int8, device="cuda")
    s = torch.empty(4, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert B.moe_ffn_quantize_int8(w.data_ptr(), 4, 60, q.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_EINVAL
    assert B.moe_ffn_quantize_int8(w.data_ptr() + 2, 4, 64, q.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_EALIGN
    assert B.moe_ffn_quantize_int8(0, 4, 64, q.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_EINVAL
    assert B.moe_ffn_quantize_int8(w.data_ptr(), 0, 64, q.data_ptr(), s.data_ptr(), st) == B.MOE_FFN_OK


def _int8_case(mode, T, seed):
    x, w = G.make_case(mode, T, seed)
    wq = B.quantize_experts_int8(w)
    torch.cuda.synchronize()
    wh = G.host_weights(wq)
    del wh["gate_up"], wh["down"]          # the oracle sees only the int8 experts
    return x, w, wq, wh


@pytest.mark.parametrize("mode,T", [(FULL, 64), (FULL, 1), (FULL, 33), (FULL, 200), (MOE, 8)])
def test_int8_layer_against_the_oracle(mode, T):
    x, _, wq, wh = _int8_case(mode, T, 900 + T)
    run = G.Run(mode, x, wq)
    xb = synth.bf16_bits(x)
    ref = G.oracle_forward(mode, xb, wh)
    same = G.check_routing(run, ref)
    G.check_permutation(run)
    G.check_values(run.out_f64[same], ref["out"][same], "int8 T=%d" % T)


def test_int8_layer_sampled_1024():
    T = 1024
    x, _, wq, wh = _int8_case(FULL, T, 1024)
    run = G.Run(FULL, x, wq)
    xb = synth.bf16_bits(x)
    route = G.oracle_route(FULL, xb, wh)
    same = G.check_routing(run, route)
    G.check_permutation(run)
    tok = np.unique(np.concatenate([np.random.default_rng(5).choice(T, 32, replace=False), [0, T - 1]]))
    ref = G.oracle_forward(FULL, xb, wh, tokens=tok, want=("out",))
    G.check_values(run.out_f64[tok][same[tok]], ref["out"][same[tok]], "int8 T=1024")


def test_int8_output_close_to_bf16_output():
    # Each expert weight moves by at most max|row| / 254; the block's output moves by about 1%.
    x, w, wq, _ = _int8_case(FULL, 64, 950)
    a = G.Run(FULL, x, w).out_f64
    b = G.Run(FULL, x, wq).out_f64
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-4 < rel < 3e-2


def test_int8_fields_must_come_together():
    x, _, wq, _ = _int8_case(FULL, 16, 960)
    m = B.MoeFFN(FULL, 16)
    ws = B.weights_struct(wq)
    ws.down_scale = None
    out = torch.empty_like(x)
    rc = B.moe_ffn_forward(m.ctx, x.data_ptr(), 16, ws, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == B.MOE_FFN_EINVAL
