"""Expert-parallel shards of the block on one GB300, through the C ABI.

"Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2", section "The traceable trick":
rank r of n owns a contiguous group of experts, every rank takes the same top-8 choice, and the
ranks' partial expert outputs are summed (an all-reduce) before post_feedforward_layernorm_2. Here
the n shards run one after another on one GPU (moe_ffn_forward_shard), their partials are added in
rank order (the sum the all-reduce would form), and moe_ffn_finish_shards gives the block output.

Checks, on the same seeded inputs as the oracle:
  * every shard's expert choice and permutation equal the unsharded forward's;
  * each shard's fp32 partial matches the oracle's expert branch with per_expert_scale zero outside
    the shard (so the partials are the right pieces, not only a right sum);
  * the shared-MLP output of the rank that runs it matches the oracle's;
  * the finished block matches the oracle under the block's bar, and the unsharded forward closely;
  * one shard holding all 128 experts gives the unsharded forward bit for bit;
  * argument errors.
Sizes cover decode tiles (T=64), single-SM 128-token tiles (T=300), SM-pair prefill tiles with
skewed routing (T=3200: the gate_up GEMM copies only the shard's slots into sorted order) and the
experts-only mode.
"""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import synth
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

MOE, FULL = B.MOE_FFN_MOE_ONLY, B.MOE_FFN_FULL_LAYER


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()


def _masked(w_host: dict, begin: int, end: int) -> dict:
    ws = dict(w_host)
    pes = np.zeros_like(w_host["per_expert_scale"])
    pes[begin:end] = w_host["per_expert_scale"][begin:end]
    ws["per_expert_scale"] = pes
    return ws


def _run_shards(m, x, w, n):
    parts, dense, routes = [], None, []
    for r in range(n):
        b, e = B.expert_range(r, n)
        part, d = m.forward_shard(x, w, b, e, with_dense=(r == 0 and m.cfg.mode == FULL))
        torch.cuda.synchronize()
        rc, word = m.status()
        assert rc == B.MOE_FFN_OK, "device status 0x%x" % word
        v = m.views()
        T = x.shape[0]
        routes.append((G.fetch(v.topk_idx, (T, 8), torch.int32).numpy(), G.fetch(v.perm, (T * 8,), torch.int32).numpy()))
        parts.append((b, e, part.clone()))
        if d is not None:
            dense = d.clone()
    return parts, dense, routes


@pytest.mark.parametrize("mode,T,n,seed,skew", [(FULL, 64, 8, 2001, False), (FULL, 300, 2, 2002, False),
                                                (FULL, 3200, 8, 2003, True), (MOE, 200, 4, 2004, False)])
def test_shards_sum_to_the_block(mode, T, n, seed, skew):
    x, w = G.make_case(mode, T, seed, skew=skew)
    m = B.MoeFFN(mode, T)
    ref_run = G.Run(mode, x, w, ctx=m)
    full_out = ref_run.out.clone()
    parts, dense, routes = _run_shards(m, x, w, n)
    for idx, perm in routes:
        np.testing.assert_array_equal(idx, ref_run.topk_idx)
        np.testing.assert_array_equal(perm, ref_run.perm)
    moe_sum = parts[0][2].clone()
    for _, _, p in parts[1:]:
        moe_sum += p  # the exchange: what an all-reduce (sum) over the ranks forms, in rank order
    out = m.finish_shards(x, w, moe_sum, dense)
    torch.cuda.synchronize()

    xb, wh = synth.bf16_bits(x), G.host_weights(w)
    rng = np.random.default_rng(seed)
    tok = np.unique(np.concatenate([rng.choice(T, size=min(T, 24), replace=False), [0, T - 1]]))
    ref = G.oracle_forward(mode, xb, wh, tokens=tok, want=("out", "moe", "dense", "topk_idx", "gap", "logits",
                                                           "topk_w"))
    same = G.check_routing(ref_run, ref, tokens=tok)
    # each shard's partial against the oracle's expert branch of its experts alone
    for b, e, p in parts:
        r = G.oracle_forward(mode, xb, _masked(wh, b, e), tokens=tok, want=("moe",))
        got = p.cpu().numpy().astype(np.float64)[tok][same]
        G.check_values(got, r["moe"][same], "shard [%d, %d) partial" % (b, e))
    if mode == FULL:
        G.check_values(dense.cpu().numpy().astype(np.float64)[tok], ref["dense"], "shared-MLP output")
    got = G.bf16_to_f64(synth.bf16_bits(out))
    G.check_values(got[tok][same], ref["out"][same], "finished block, %d shards" % n)
    # against the unsharded forward: only the association of the fp32 expert sum differs
    frob, mx = G.errors(got, G.bf16_to_f64(synth.bf16_bits(full_out)))
    assert frob < 2e-3, "sharded vs unsharded rel Frobenius %.3e" % frob


@pytest.mark.parametrize("mode,T", [(FULL, 64), (FULL, 1100), (FULL, 3100), (MOE, 33)])
def test_one_shard_of_all_experts_is_the_forward(mode, T):
    x, w = G.make_case(mode, T, 2100 + T)
    m = B.MoeFFN(mode, T)
    full_out = m.forward(x, w).clone()
    part, dense = m.forward_shard(x, w, 0, 128, with_dense=(mode == FULL))
    out = m.finish_shards(x, w, part, dense)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), full_out.view(torch.int16))


def test_empty_shard_writes_zeros():
    T = 40
    x, w = G.make_case(FULL, T, 2200)
    m = B.MoeFFN(FULL, T)
    part, dense = m.forward_shard(x, w, 50, 50, with_dense=False)
    torch.cuda.synchronize()
    assert dense is None and torch.count_nonzero(part) == 0


def test_shard_argument_errors():
    T = 16
    x, w = G.make_case(FULL, T, 2300)
    m = B.MoeFFN(FULL, T)
    ws = B.weights_struct(w)
    s = torch.cuda.current_stream().cuda_stream
    part = torch.empty(T, 2816, dtype=torch.float32, device="cuda")
    dense = torch.empty_like(part)
    f = B.moe_ffn_forward_shard
    assert f(m.ctx, x.data_ptr(), T, ws, 10, 5, 0, part.data_ptr(), 0, s) == B.MOE_FFN_EINVAL     # begin > end
    assert f(m.ctx, x.data_ptr(), T, ws, 0, 129, 0, part.data_ptr(), 0, s) == B.MOE_FFN_EINVAL    # end > 128
    assert f(m.ctx, x.data_ptr(), T, ws, -1, 8, 0, part.data_ptr(), 0, s) == B.MOE_FFN_EINVAL     # begin < 0
    assert f(m.ctx, x.data_ptr(), T, ws, 0, 8, 1, part.data_ptr(), 0, s) == B.MOE_FFN_EINVAL      # dense_out NULL
    assert f(m.ctx, x.data_ptr(), T + 1, ws, 0, 8, 0, part.data_ptr(), 0, s) == B.MOE_FFN_ETOOBIG
    assert f(m.ctx, x.data_ptr(), T, ws, 0, 8, 0, part.data_ptr() + 4, 0, s) == B.MOE_FFN_EALIGN
    assert f(m.ctx, x.data_ptr(), T, ws, 0, 8, 1, part.data_ptr(), part.data_ptr(), s) == B.MOE_FFN_EINVAL  # overlap
    mo = B.MoeFFN(MOE, T)
    xo, wo = G.make_case(MOE, T, 2301)
    assert f(mo.ctx, xo.data_ptr(), T, B.weights_struct(wo), 0, 8, 1, part.data_ptr(), dense.data_ptr(), s) \
        == B.MOE_FFN_EINVAL  # no shared MLP in the experts-only mode
    fin = B.moe_ffn_finish_shards
    out = torch.empty_like(x)
    assert fin(m.ctx, x.data_ptr(), T, ws, part.data_ptr(), 0, out.data_ptr(), s) == B.MOE_FFN_EINVAL  # dense NULL
    assert fin(m.ctx, x.data_ptr(), T, ws, part.data_ptr(), dense.data_ptr(), x.data_ptr(), s) == B.MOE_FFN_EINVAL
    torch.cuda.synchronize()
    assert m.status() == (B.MOE_FFN_OK, 0)

