"""The allocation-free router-logits entry point, through the C ABI (GB300 only).

Callers that cannot allocate device memory (running under a pool or allocator they do not own, or
on a path where allocating is not allowed) use moe_ffn_router_logits_noalloc, whose scratch is a
fixed device array shared by every call. This checks that two calls in a row both give the logits
that the regular entry point moe_ffn_forward computes for the same inputs, within the tolerance the
routing checks use. The file sorts last so that a run stopping at its first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_router_gb300 import binding as B
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

FULL = B.MOE_FFN_FULL_LAYER


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


@pytest.mark.parametrize("T", [64, 1000])
def test_noalloc_logits_match_the_regular_entry_point_twice(T):
    x, w = G.make_case(FULL, T, 1300 + T)
    m = B.MoeFFN(FULL, T)
    m.forward(x, w)
    torch.cuda.synchronize()
    ref = B.view_tensor(m.views().logits, (T, 128), torch.float32).cpu().numpy().astype(np.float64)
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.empty(T, 128, dtype=torch.float32, device="cuda")
    results = []
    for _ in range(2):
        out.fill_(float("nan"))
        rc = B.moe_ffn_router_logits_noalloc(x.data_ptr(), T, w["router_w"].data_ptr(), w["router_norm_w"].data_ptr(),
                                             2816 ** -0.5, 1e-6, out.data_ptr(), stream)
        assert rc == B.MOE_FFN_OK, B.moe_ffn_status_string(rc)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() < G.LOGIT_TOL
        results.append(got)
    np.testing.assert_array_equal(results[0], results[1])


def test_noalloc_rejects_more_tokens_than_its_scratch_holds():
    x, w = G.make_case(FULL, 1025, 1400)
    out = torch.empty(1025, 128, dtype=torch.float32, device="cuda")
    rc = B.moe_ffn_router_logits_noalloc(x.data_ptr(), 1025, w["router_w"].data_ptr(), w["router_norm_w"].data_ptr(),
                                         2816 ** -0.5, 1e-6, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == B.MOE_FFN_ETOOBIG
