"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI, run the oracle on
the same drawn tensors, and compare them under the block's acceptance rules.

Rules (the block's acceptance bar):
  * expert choice (the set of 8) bit-exact on every token whose 8th/9th oracle-logit gap > 1e-4;
    on the other tokens any choice is accepted whose experts all lie within 1e-4 of the oracle's
    8th logit (several answers are correct there);
  * router logits within 5e-5 (half the gap threshold) of the oracle's fp32 logits; renormalised,
    scaled weights within 2*max|logit difference| + 1e-6 relative on the tokens with the same
    choice (the softmax over the selected 8 moves log w by at most twice the logit shift);
  * the permutation (counts, offsets, perm, w_sorted, slot positions) bit-exact against the
    oracle's counting sort applied to the CUDA path's own choice;
  * the output within relative Frobenius error 1e-2 and max abs error 5e-2 of the fp64 oracle, on
    the tokens whose choice matches.
"""
import numpy as np
import torch

import oracle
from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import synth

GAP_MIN = 1e-4
LOGIT_TOL = 0.5 * GAP_MIN
W_RTOL_FLOOR = 1e-6
FROB_TOL = 1e-2
MAXABS_TOL = 5e-2


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def fetch(view_ptr, shape, dtype):
    return B.view_tensor(view_ptr, shape, dtype).cpu().clone()


class Run:
    """One CUDA-path forward and what it left in the workspace."""

    def __init__(self, mode, x, weights, max_tokens=None, ctx=None):
        T = x.shape[0]
        self.T = T
        self.mode = mode
        self.ctx = ctx or B.MoeFFN(mode, max_tokens or max(T, 1))
        self.out = self.ctx.forward(x, weights)
        torch.cuda.synchronize()
        rc, word = self.ctx.status()
        assert rc == B.MOE_FFN_OK, "device status word 0x%x" % word
        v = self.ctx.views()
        S = T * 8
        self.topk_idx = fetch(v.topk_idx, (T, 8), torch.int32).numpy()
        self.topk_w = fetch(v.topk_w, (T, 8), torch.float32).numpy()
        self.gap = fetch(v.gap, (T,), torch.float32).numpy()
        self.logits = fetch(v.logits, (T, 128), torch.float32).numpy()
        self.counts = fetch(v.counts, (128,), torch.int32).numpy()
        self.offsets = fetch(v.offsets, (129,), torch.int32).numpy()
        self.perm = fetch(v.perm, (S,), torch.int32).numpy()
        self.w_sorted = fetch(v.w_sorted, (S,), torch.float32).numpy()
        self.slot_pos = fetch(v.slot_pos, (T, 8), torch.int32).numpy()
        self.views = v
        self.out_f64 = bf16_to_f64(synth.bf16_bits(self.out))


def check_permutation(run: Run):
    p = oracle.permute(run.topk_idx, run.topk_w, 128)
    np.testing.assert_array_equal(run.counts, p["counts"])
    np.testing.assert_array_equal(run.offsets, p["offsets"])
    np.testing.assert_array_equal(run.perm, p["perm"])
    np.testing.assert_array_equal(run.w_sorted, p["w_sorted"])
    np.testing.assert_array_equal(run.slot_pos, p["slot_pos"])


def check_routing(run: Run, ref: dict, tokens=None):
    """ref: oracle router outputs for the tokens `tokens` (all if None). Returns the mask (over
    those tokens) of tokens whose choice equals the oracle's."""
    idx = run.topk_idx if tokens is None else run.topk_idx[tokens]
    w = run.topk_w if tokens is None else run.topk_w[tokens]
    same = (idx == ref["topk_idx"]).all(axis=1)
    clear = ref["gap"] > GAP_MIN
    bad = np.nonzero(clear & ~same)[0]
    assert bad.size == 0, "expert choice differs on %d clear tokens, e.g. %s" % (bad.size, bad[:5])
    lg = ref["logits"]
    for t in np.nonzero(~same)[0]:
        l8 = np.sort(lg[t])[::-1][7]
        assert (lg[t][idx[t]] >= l8 - GAP_MIN).all(), "token %d picked an expert far below the 8th logit" % t
    # Logits: fp32 sums of 2816 products in two different orders. Less than half the gap
    # threshold apart, so a gap above the threshold cannot be reversed.
    run_lg = run.logits if tokens is None else run.logits[tokens]
    dl = np.abs(run_lg.astype(np.float64) - lg).max(axis=1)
    assert dl.max() < LOGIT_TOL, "router logits differ by %.3e" % dl.max()
    # Weights: w_k = exp(l_k) / sum_j exp(l_j) over the 8 selected, so a perturbation of the
    # logits by at most dl moves log w_k by at most 2 dl; 1e-6 covers the fp32 division/scale.
    tol = (2.0 * dl + W_RTOL_FLOOR)[:, None]
    rel = np.abs(w.astype(np.float64) - ref["topk_w"]) / np.abs(ref["topk_w"])
    assert (rel[same] <= np.broadcast_to(tol, rel.shape)[same]).all(), "topk_w off by %.3e rel" % rel[same].max()
    return same


def errors(got: np.ndarray, want: np.ndarray):
    diff = got - want
    frob = float(np.linalg.norm(diff) / max(np.linalg.norm(want), 1e-300))
    return frob, float(np.abs(diff).max()) if diff.size else 0.0


def check_values(got: np.ndarray, want: np.ndarray, label=""):
    frob, mx = errors(got, want)
    assert frob <= FROB_TOL and mx <= MAXABS_TOL, "%s rel Frobenius %.3e, max abs %.3e" % (label, frob, mx)
    return frob, mx


def oracle_dims(mode):
    return oracle.gemma_dims(full_layer=(mode == B.MOE_FFN_FULL_LAYER))


def oracle_forward(mode, x_bits, w_host, tokens=None, want=("out", "topk_idx", "topk_w", "gap", "logits")):
    xs = x_bits if tokens is None else x_bits[tokens]
    return oracle.forward(oracle_dims(mode), xs, w_host, want=want)


def oracle_route(mode, x_bits, w_host):
    return oracle.forward(oracle_dims(mode), x_bits, w_host,
                          want=("topk_idx", "topk_w", "gap", "logits"), route_only=True)


def make_case(mode, T, seed, skew=False):
    full = mode == B.MOE_FFN_FULL_LAYER
    w = synth.make_weights(seed=seed, device="cuda", full_layer=full, skew=skew)
    x = synth.make_x(T, seed=seed, device="cuda")
    return x, w


def host_weights(w: dict) -> dict:
    return synth.host_arrays(w)
