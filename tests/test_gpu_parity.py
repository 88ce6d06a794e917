"""CUDA path vs the oracle, through the C ABI, on the same seeded inputs (GB300 only).

Shapes: the five workloads of the block (experts-only T=8; full layer T=64; full layer T=4096
with skewed routing; the sweep's T values incl. the maximum 16384) plus ragged and degenerate
cases. Where the oracle cannot run every token in seconds, it runs the router on every token
(expert choice and the permutation are checked in full) and the whole block on a sample.
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
    B.lib()  # fails loudly if the library is missing


def _full_check(mode, T, seed, skew=False, label=""):
    x, w = G.make_case(mode, T, seed, skew=skew)
    run = G.Run(mode, x, w)
    wh = G.host_weights(w)
    xb = synth.bf16_bits(x)
    ref = G.oracle_forward(mode, xb, wh)
    same = G.check_routing(run, ref)
    G.check_permutation(run)
    frob, mx = G.check_values(run.out_f64[same], ref["out"][same], label)
    return run, ref, frob, mx


@pytest.mark.parametrize("T", [8, 1, 3, 31, 32, 33])
def test_moe_only_small(T):
    _full_check(MOE, T, 100 + T, label="moe-only T=%d" % T)


@pytest.mark.parametrize("T", [64, 1, 16, 17, 50, 65, 200])
def test_full_layer(T):
    # Up to 64 tokens the routing front end is one kernel in token groups of 16 (17 and 50 end in
    # a partly filled group); from 65 the router, top-k and scatter kernels run apart.
    _full_check(FULL, T, 200 + T, label="full T=%d" % T)


@pytest.mark.parametrize("T", [65, 300])
def test_moe_only_above_small_batches(T):
    # The experts-only block above 64 tokens: the router, top-k and scatter kernels run apart, and
    # the combine sums each token's 8 rows of y with no norms.
    _full_check(MOE, T, 150 + T, label="moe-only T=%d" % T)


def test_kernel_slots_by_batch_size():
    m = B.MoeFFN(FULL, 256)
    for T in (1, 17, 64):
        assert B.moe_ffn_kernel_slots(m.ctx, T) == [1, 4, 5, 6]
        assert [B.slot_name(k, T) for k in (1, 4)] == ["route_small", "gate_up_gemm"]
    for T in (65, 256):
        assert B.moe_ffn_kernel_slots(m.ctx, T) == [0, 1, 2, 3, 4, 5, 6]
        assert B.slot_name(1, T) == "router_logits"
    assert B.moe_ffn_kernel_slots(m.ctx, 0) == []


def _sampled_check(mode, T, seed, skew, n_sample, label):
    x, w = G.make_case(mode, T, seed, skew=skew)
    run = G.Run(mode, x, w)
    wh = G.host_weights(w)
    xb = synth.bf16_bits(x)
    route = G.oracle_route(mode, xb, wh)
    same = G.check_routing(run, route)
    G.check_permutation(run)
    rng = np.random.default_rng(seed)
    tok = np.sort(rng.choice(T, size=min(n_sample, T), replace=False))
    tok = np.unique(np.concatenate([tok, [0, T - 1]]))
    ref = G.oracle_forward(mode, xb, wh, tokens=tok, want=("out",))
    keep = same[tok]
    frob, mx = G.check_values(run.out_f64[tok][keep], ref["out"][keep], label)
    return run, route


def test_full_layer_prefill_skewed_4096():
    run, route = _sampled_check(FULL, 4096, 300, True, 48, "full T=4096 skewed")
    load = run.counts
    assert load.max() >= 6 * load.mean()      # a heavily loaded head ...
    assert (load == 0).sum() >= 8             # ... and experts with no tokens


@pytest.mark.parametrize("T", [256, 777, 1024, 1500])
def test_full_layer_sweep_sizes(T):
    _sampled_check(FULL, T, 400 + T, False, 32, "full T=%d" % T)


@pytest.mark.parametrize("T", [1100, 3100])
def test_moe_only_prefill_sized(T):
    # Experts only above 1024 tokens: token tiles of 256, the down GEMM on SM pairs; above 3072 the
    # gate_up GEMM too, with the expert input (x itself) copied into sorted-slot order and no
    # shared-MLP items to run meanwhile.
    _sampled_check(MOE, T, 460, False, 32, "moe-only T=%d" % T)


def test_full_layer_prefill_uniform_4096():
    # The sweep's T=4096 point: uniform routing, so nearly every expert gets two token tiles of 256
    # (the second one partly filled).
    run, _ = _sampled_check(FULL, 4096, 450, False, 32, "full T=4096 uniform")
    assert (run.counts > 0).sum() == 128


@pytest.mark.slow
def test_full_layer_max_sweep_16384():
    _sampled_check(FULL, 16384, 500, False, 24, "full T=16384")


@pytest.mark.slow
def test_full_layer_max_tokens_65536():
    # The largest batch a context accepts (MOE_FFN_MAX_TOKENS_LIMIT): 256 chunks of 256 tokens for
    # the counting sort, 524,288 slots, a 2.95 GB sorted copy of n2 in the y buffer.
    run, _ = _sampled_check(FULL, 65536, 510, False, 16, "full T=65536")
    assert run.counts.sum() == 65536 * 8


def test_all_tokens_identical_pick_the_same_experts():
    # Identical tokens choose the same 8 experts: 8 experts get all T tokens (several token tiles
    # each), the other 120 get none.
    T = 300
    x1, w = G.make_case(FULL, 1, 600)
    x = x1.expand(T, -1).contiguous()
    run = G.Run(FULL, x, w)
    assert (run.counts > 0).sum() == 8 and run.counts.max() == T
    G.check_permutation(run)
    ref = G.oracle_forward(FULL, synth.bf16_bits(x1), G.host_weights(w))
    if ref["gap"][0] > G.GAP_MIN:
        np.testing.assert_array_equal(run.topk_idx[0], ref["topk_idx"][0])
    np.testing.assert_array_equal(run.out_f64, np.broadcast_to(run.out_f64[:1], run.out_f64.shape))
    G.check_values(run.out_f64[:1], ref["out"], "identical tokens")


@pytest.mark.parametrize("T", [500, 2048])
def test_deterministic_bitwise(T):
    # The GEMMs hand out work items dynamically, so which CTA computes an item differs between
    # runs; each item is computed whole in a fixed order, so the output may not.
    x, w = G.make_case(FULL, T, 700)
    m = B.MoeFFN(FULL, T)
    a = m.forward(x, w).clone()
    b = m.forward(x, w).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_context_reuse_across_T_and_weights():
    # One context, calls with different T and different weights: each result equals a fresh run.
    # The sizes cross between the tensor-core router (T > 64) and the CUDA-core one, and repeat a
    # decode size, so every per-forward reset of the routing counters is exercised.
    m = B.MoeFFN(FULL, 256)
    for T, seed in [(256, 800), (17, 801), (130, 802), (64, 803), (64, 804), (1, 805)]:
        x, w = G.make_case(FULL, T, seed)
        a = m.forward(x, w).clone()
        fresh = B.MoeFFN(FULL, T).forward(x, w)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), fresh.view(torch.int16))
    assert m.status() == (B.MOE_FFN_OK, 0)


def test_error_paths():
    m = B.MoeFFN(FULL, 16)
    x, w = G.make_case(FULL, 16, 900)
    ws = B.weights_struct(w)
    out = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), 17, ws, out.data_ptr(), s) == B.MOE_FFN_ETOOBIG
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), -1, ws, out.data_ptr(), s) == B.MOE_FFN_EINVAL
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), 0, ws, out.data_ptr(), s) == B.MOE_FFN_OK
    assert B.moe_ffn_forward(m.ctx, x.data_ptr() + 2, 4, ws, out.data_ptr(), s) == B.MOE_FFN_EALIGN
    assert B.moe_ffn_forward(m.ctx, 0, 4, ws, out.data_ptr(), s) == B.MOE_FFN_EINVAL
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), 16, ws, x.data_ptr(), s) == B.MOE_FFN_EINVAL  # out aliases x
    bad = B.weights_struct(w)
    bad.dense_down = None
    assert B.moe_ffn_forward(m.ctx, x.data_ptr(), 4, bad, out.data_ptr(), s) == B.MOE_FFN_EINVAL
    cfg = B.make_config(FULL, 16)
    cfg.hidden = 4096
    assert B.moe_ffn_workspace_bytes(cfg) == 0
    torch.cuda.synchronize()
    assert m.status() == (B.MOE_FFN_OK, 0)


def test_all_zero_input_row():
    # A token whose input row is all zero: RMS is sqrt(eps), every logit is exactly 0, so all 128
    # experts tie and the tie rule picks experts 0..7 with equal renormalised weights (times
    # per_expert_scale); its expert inputs, expert outputs and shared-MLP output are zero, so the
    # post-norms give zero and the output row is (0 + 0) * layer_scalar = 0.
    T, z = 64, 5
    x, w = G.make_case(FULL, T, 1000)
    x[z].zero_()
    run, ref, _, _ = _full_check_inputs(FULL, x, w, "full T=64 with a zero row")
    np.testing.assert_array_equal(run.topk_idx[z], np.arange(8))
    np.testing.assert_array_equal(ref["topk_idx"][z], np.arange(8))
    assert run.gap[z] == 0.0 and (run.logits[z] == 0.0).all()
    pes = w["per_expert_scale"].cpu().numpy()[:8]
    np.testing.assert_allclose(run.topk_w[z], pes / 8.0, rtol=1e-6)
    assert (run.out_f64[z] == 0.0).all() and np.isfinite(run.out_f64).all()


@pytest.mark.parametrize("scale", [1e3, 1e-3])
def test_extreme_input_magnitudes(scale):
    # x scaled by 1e3 or 1e-3 (about 1e-6 mean square, the size of eps). The router and the
    # pre-norms see RMS-normalised rows, so the routing checks are unchanged; the output holds the
    # residual term x * layer_scalar, whose bf16 rounding is relative (half an ulp is 2^-9 of the
    # value), so the absolute bar grows by 2^-8 of the oracle's magnitude.
    T = 64
    x, w = G.make_case(FULL, T, 1100 + int(scale > 1))
    x = (x.float() * scale).to(torch.bfloat16)
    run, ref, frob, mx = _full_check_inputs(FULL, x, w, "full T=64, x * %g" % scale, rel_abs=2.0 ** -8)
    assert np.isfinite(run.out_f64).all()


def _full_check_inputs(mode, x, w, label, rel_abs=0.0):
    run = G.Run(mode, x, w)
    ref = G.oracle_forward(mode, synth.bf16_bits(x), G.host_weights(w))
    same = G.check_routing(run, ref)
    G.check_permutation(run)
    got, want = run.out_f64[same], ref["out"][same]
    frob, mx = G.errors(got, want)
    assert frob <= G.FROB_TOL, "%s rel Frobenius %.3e" % (label, frob)
    excess = np.abs(got - want) - (G.MAXABS_TOL + rel_abs * np.abs(want))
    assert (excess <= 0).all(), "%s max abs %.3e beyond the bar" % (label, mx)
    return run, ref, frob, mx
