"""The allocation-free router-logits entry point, through the C ABI (GB300 only).

Some callers cannot allocate device memory when they call in: code running under a memory pool or
allocator it does not own, a plugin handed only a stream and its buffers, a real-time path where an
allocation (and the synchronisation cudaMalloc can imply) is not allowed. They use
moe_ffn_router_logits_noalloc, whose scratch is a fixed device array shared by every call. These
tests check that
  * two calls in a row give the logits that the regular entry point moe_ffn_forward computes for
    the same inputs, within the tolerance the routing checks use;
  * its logits are within 5e-5 of the oracle's fp32 logits, and the top-8 taken from them equals
    the oracle's choice on every token whose 8th/9th logit gap exceeds 1e-4;
  * two calls queued back to back on one stream, with different inputs and outputs and no
    synchronisation between them, each give their own inputs' logits;
  * after the first call on the device, further calls leave the device's free memory unchanged;
  * it rejects more tokens than its scratch holds.
The file sorts last so that a run stopping at its first failure has already run every other test;
it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

FULL = B.MOE_FFN_FULL_LAYER
SCALE = 2816 ** -0.5
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


def _noalloc(x, w, out, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = B.moe_ffn_router_logits_noalloc(x.data_ptr(), x.shape[0], w["router_w"].data_ptr(),
                                         w["router_norm_w"].data_ptr(), SCALE, EPS, out.data_ptr(), s)
    assert rc == B.MOE_FFN_OK, B.moe_ffn_status_string(rc)


def _top8(logits: np.ndarray) -> np.ndarray:
    """The 8 largest logits of each row (ties to the lower expert id), in ascending expert id."""
    order = np.lexsort((np.broadcast_to(np.arange(logits.shape[1]), logits.shape), -logits), axis=1)
    return np.sort(order[:, :8], axis=1)


@pytest.mark.parametrize("T", [64, 1000])
def test_noalloc_logits_match_the_regular_entry_point_twice(T):
    x, w = G.make_case(FULL, T, 1300 + T)
    m = B.MoeFFN(FULL, T)
    m.forward(x, w)
    torch.cuda.synchronize()
    ref = B.view_tensor(m.views().logits, (T, 128), torch.float32).cpu().numpy().astype(np.float64)
    out = torch.empty(T, 128, dtype=torch.float32, device="cuda")
    results = []
    for _ in range(2):
        out.fill_(float("nan"))
        _noalloc(x, w, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() < G.LOGIT_TOL
        results.append(got)
    np.testing.assert_array_equal(results[0], results[1])
    m.close()


@pytest.mark.parametrize("T", [64, 1000])
def test_noalloc_logits_match_the_oracle(T):
    x, w = G.make_case(FULL, T, 1500 + T)
    out = torch.empty(T, 128, dtype=torch.float32, device="cuda")
    _noalloc(x, w, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = G.oracle_route(FULL, synth.bf16_bits(x), G.host_weights(w))
    dl = np.abs(got.astype(np.float64) - ref["logits"].astype(np.float64)).max()
    assert dl < G.LOGIT_TOL, "logits differ from the oracle's by %.3e" % dl
    clear = ref["gap"] > G.GAP_MIN
    assert clear.sum() > 0.9 * T
    np.testing.assert_array_equal(_top8(got)[clear], ref["topk_idx"][clear])


def test_noalloc_back_to_back_calls_on_one_stream():
    T = 512
    xa, w = G.make_case(FULL, T, 1700)
    xb = synth.make_x(T, seed=1701, device="cuda")
    outs = [torch.full((T, 128), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    _noalloc(xa, w, outs[0])
    _noalloc(xb, w, outs[1])   # queued right behind the first call, no synchronisation between them
    torch.cuda.synchronize()
    hw = G.host_weights(w)
    for x, out in ((xa, outs[0]), (xb, outs[1])):
        ref = G.oracle_route(FULL, synth.bf16_bits(x), hw)
        dl = np.abs(out.cpu().numpy().astype(np.float64) - ref["logits"].astype(np.float64)).max()
        assert dl < G.LOGIT_TOL, "logits differ from the oracle's by %.3e" % dl


def test_noalloc_calls_leave_device_memory_unchanged():
    T = 256
    x, w = G.make_case(FULL, T, 1800)
    out = torch.empty(T, 128, dtype=torch.float32, device="cuda")
    _noalloc(x, w, out)          # the first call on the device does its one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        _noalloc(x, w, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "free device memory changed by %d bytes" % (free0 - free1)


def test_noalloc_rejects_more_tokens_than_its_scratch_holds():
    x, w = G.make_case(FULL, 1025, 1400)
    out = torch.empty(1025, 128, dtype=torch.float32, device="cuda")
    rc = B.moe_ffn_router_logits_noalloc(x.data_ptr(), 1025, w["router_w"].data_ptr(), w["router_norm_w"].data_ptr(),
                                         SCALE, EPS, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == B.MOE_FFN_ETOOBIG
