"""A bounded device wait runs out on the GPU (failure detection without a fault): the library's
self-test kernel waits on a barrier nothing arrives on, through the same helpers the forward's
kernels use, and must come back with the right status bits and timings; the GPU and a context
must stay usable afterwards."""
import pytest
import torch

from mixture_experts_ffn_router_gb300 import binding as B
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

WAIT_FULL, WAIT_EMPTY, DRAIN = (B.STATUS_BITS[k] for k in ("WAIT_FULL", "WAIT_EMPTY", "DRAIN"))


def test_bounded_waits_give_up_and_report():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rec = torch.full((6,), -1, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert B.moe_ffn_selftest_wait_expiry(status.data_ptr(), rec.data_ptr(), s) == B.MOE_FFN_OK
    torch.cuda.synchronize()
    word = int(status.item()) & 0xffffffff
    r = rec.cpu().tolist()
    # wait 1 gave up at the 2 s limit; wait 2 left through the abort flag without its own bit;
    # wait 3 (the exit drain, 1 ms limit) gave up too. None saw its phase complete.
    assert word & WAIT_FULL and word & DRAIN and not word & WAIT_EMPTY, B.decode_status(word)
    assert r[1] == 0 and r[3] == 0 and r[5] == 0, r
    assert 2.0e9 <= r[0] < 3.0e9, r
    assert r[2] < 1.0e8, r
    assert 1.0e6 <= r[4] < 1.0e8, r

    # The GPU is still usable: a forward right after runs clean and matches a fresh context.
    x, w = G.make_case(B.MOE_FFN_FULL_LAYER, 16, 1100)
    m = B.MoeFFN(B.MOE_FFN_FULL_LAYER, 16)
    a = m.forward(x, w).clone()
    torch.cuda.synchronize()
    assert m.status() == (B.MOE_FFN_OK, 0)
    b = B.MoeFFN(B.MOE_FFN_FULL_LAYER, 16).forward(x, w)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_selftest_rejects_null_pointers():
    assert B.moe_ffn_selftest_wait_expiry(0, 0, 0) == B.MOE_FFN_EINVAL
