"""The forward queues only kernels (no host synchronisation, no allocation), so a chain of layers
can be captured in a CUDA graph: replaying it gives bitwise the output of the same chain queued
eagerly, for bf16 and int8 experts (GB300 only)."""
import pytest
import torch

from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


@pytest.mark.parametrize("T,int8", [(64, False), (300, False), (64, True)])
def test_captured_chain_replays_bitwise(T, int8):
    layers = 3
    weights = [synth.make_weights(seed=40 + l, layer=l, device="cuda", full_layer=True) for l in range(layers)]
    if int8:
        weights = [B.quantize_experts_int8(w) for w in weights]
    x = synth.make_x(T, seed=41, device="cuda")
    ctxs = [B.MoeFFN(B.MOE_FFN_FULL_LAYER, T)]
    for _ in range(1, layers):
        ctxs.append(B.MoeFFN(B.MOE_FFN_FULL_LAYER, T, workspace=ctxs[0].workspace))
    wss = [B.weights_struct(w) for w in weights]
    bufs = [torch.empty_like(x), torch.empty_like(x)]

    def chain(stream):
        src = x
        for l in range(layers):
            dst = bufs[l % 2]
            rc = B.moe_ffn_forward(ctxs[l].ctx, src.data_ptr(), T, wss[l], dst.data_ptr(), stream.cuda_stream)
            assert rc == B.MOE_FFN_OK
            src = dst

    cur = torch.cuda.current_stream()
    chain(cur)
    torch.cuda.synchronize()
    eager = bufs[(layers - 1) % 2].clone()

    side = torch.cuda.Stream()
    side.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        chain(side)
    for b in bufs:
        b.zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bufs[(layers - 1) % 2], eager)
    assert ctxs[0].status() == (B.MOE_FFN_OK, 0)
