"""Mutation check of the oracle's pins (CPU only).

The pins in test_oracle_pins.py, test_oracle_int8.py and test_oracle_fp4.py are meant to catch any
plausible mistake in the oracle: a dropped term, a wrong sign, index or stride, a transposed or
swapped operand, a wrong rounding rule. This test plants one such mistake at a time in a copy of
oracle/moe_oracle.c (never in the committed file), builds the copy with the oracle's own flags,
runs the pin files against it through MOE_ORACLE_LIB, and requires them to fail with an assertion
(pytest exit status 1: not a pass, not a crash). Every planted mistake keeps each access inside
its array, so a mutant can only give wrong values. An unmodified copy built the same way must
pass, which shows the harness itself is sound.

The mutants run in parallel subprocesses, one OpenMP thread each. The slow Gemma-shapes case of
the sparse == dense-masked identity is left out of these runs; every mutant below is caught by a
faster pin.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["tests/test_oracle_pins.py", "tests/test_oracle_int8.py", "tests/test_oracle_fp4.py"]
SLOW = "tests/test_oracle_pins.py::test_sparse_equals_dense_masked_bitwise_gemma_shapes"

# (name, exact text in moe_oracle.c, replacement). Each text occurs exactly once in the source.
MUTANTS = [
    # GELU, tanh form
    ("gelu_cubic_term_dropped", "0.7978845608 * (x + 0.044715 * x * x * x)", "0.7978845608 * (x)"),
    ("gelu_cubic_as_square", "0.044715 * x * x * x", "0.044715 * x * x"),
    ("gelu_sign_flipped", "(1.0 + tanh(", "(1.0 - tanh("),
    # RMSNorm, Gemma form
    ("rmsnorm_without_one_plus_w", "out[i] = v[i] * inv * (1.0 + (double)w[i])", "out[i] = v[i] * inv * ((double)w[i])"),
    ("rmsnorm_sum_not_mean", "1.0 / sqrt(ss / (double)n + eps)", "1.0 / sqrt(ss + eps)"),
    ("rmsnorm_eps_dropped", "1.0 / sqrt(ss / (double)n + eps)", "1.0 / sqrt(ss / (double)n)"),
    # router: its own norm, the scale, the projection
    ("router_norm_without_one_plus_w", "(1.0f + w->router_norm_w[h])", "(w->router_norm_w[h])"),
    ("router_scale_dropped", "(1.0f + w->router_norm_w[h]) * d->router_scale;", "(1.0f + w->router_norm_w[h]);"),
    ("router_rms_dropped", "r[h] = xin[h] * inv * (1.0f", "r[h] = xin[h] * (1.0f"),
    ("router_eps_dropped", "sqrtf(ss / (float)H + d->eps)", "sqrtf(ss / (float)H)"),
    ("router_matrix_read_column_major", "acc += r[h] * row[h];", "acc += r[h] * w->router_w[(size_t)h * E + e];"),
    # softmax, top-k, renormalisation, per_expert_scale
    ("softmax_not_normalised", "for (int e = 0; e < E; ++e) probs[e] = probs[e] / z;", ""),
    ("topk_ties_to_higher_id", "logits[e] > logits[best]) best = e;", "logits[e] >= logits[best]) best = e;"),
    ("topk_takes_smallest", "logits[e] > logits[best]) best = e;", "logits[e] < logits[best]) best = e;"),
    ("gap_from_the_largest", "logits[order[K - 1]] - logits[order[K]]", "logits[order[0]] - logits[order[K]]"),
    ("no_renormalisation", "wren[j] = probs[idx[j]] / s;", "wren[j] = probs[idx[j]];"),
    ("renormalised_over_all_experts", "for (int j = 0; j < K; ++j) s += probs[idx[j]];",
     "for (int j = 0; j < E; ++j) s += probs[j];"),
    ("gap_on_probabilities", "logits[order[K - 1]] - logits[order[K]]", "probs[order[K - 1]] - probs[order[K]]"),
    ("per_expert_scale_dropped", "wfin[j] = wren[j] * w->per_expert_scale[idx[j]];", "wfin[j] = wren[j];"),
    ("per_expert_scale_by_rank", "wfin[j] = wren[j] * w->per_expert_scale[idx[j]];", "wfin[j] = wren[j] * w->per_expert_scale[j];"),
    # expert MLP
    ("expert_gate_and_up_swapped", "hvec[i] = moe_oracle_gelu_tanh(g) * u;\n  }\n  const size_t d0",
     "hvec[i] = moe_oracle_gelu_tanh(u) * g;\n  }\n  const size_t d0"),
    ("expert_gate_up_stride", "const size_t g0 = (size_t)e * 2 * I;", "const size_t g0 = (size_t)e * I;"),
    ("expert_down_stride", "const size_t d0 = (size_t)e * H;", "const size_t d0 = (size_t)e * I;"),
    ("experts_read_raw_x", "expert_mlp(d, w, idx[k], n2, hv, y);", "expert_mlp(d, w, idx[k], xd, hv, y);"),
    ("experts_only_input_normed", "for (int h = 0; h < H; ++h) n2[h] = xd[h];",
     "moe_oracle_rmsnorm(xd, w->router_norm_w, H, (double)d->eps, n2);"),
    ("combine_without_per_expert_scale", "double c = (double)wfin[k] * y[h];", "double c = (double)wren[k] * y[h];"),
    ("masked_form_weights_unselected", "if (is_sel) we = (double)wfin[k];", "we = (double)wfin[k < K ? k : K - 1];"),
    # shared MLP
    ("dense_gate_and_up_swapped",
     "hvec[i] = moe_oracle_gelu_tanh(g) * u;\n  }\n  for (int h = 0; h < H; ++h) {\n    double acc = 0.0;\n    for (int i = 0; i < D;",
     "hvec[i] = moe_oracle_gelu_tanh(u) * g;\n  }\n  for (int h = 0; h < H; ++h) {\n    double acc = 0.0;\n    for (int i = 0; i < D;"),
    ("dense_down_transposed", "w->dense_down[(size_t)h * D + i]", "w->dense_down[(size_t)i * H + h]"),
    ("dense_reads_expert_input", "dense_mlp(d, w, n1, hv, dn);", "dense_mlp(d, w, n2, hv, dn);"),
    # norm chain, residual, layer_scalar
    ("pre_norms_swapped",
     "moe_oracle_rmsnorm(xd, w->pre_ff_ln, H, (double)d->eps, n1);\n        moe_oracle_rmsnorm(xd, w->pre_ff_ln_2,",
     "moe_oracle_rmsnorm(xd, w->pre_ff_ln_2, H, (double)d->eps, n1);\n        moe_oracle_rmsnorm(xd, w->pre_ff_ln,"),
    ("router_always_reads_pre_norm_2",
     "xin[h] = (d->full_layer && d->router_reads_pre2) ? (float)n2[h] : (float)xd[h];\n      float gap;\n      route_one(d, xin, w, r, logits, probs, idx, wren, wfin, &gap);\n\n",
     "xin[h] = (d->full_layer) ? (float)n2[h] : (float)xd[h];\n      float gap;\n      route_one(d, xin, w, r, logits, probs, idx, wren, wfin, &gap);\n\n"),
    ("post_norms_swapped",
     "moe_oracle_rmsnorm(dn, w->post_ff_ln_1, H, (double)d->eps, dn);\n        moe_oracle_rmsnorm(moe, w->post_ff_ln_2,",
     "moe_oracle_rmsnorm(dn, w->post_ff_ln_2, H, (double)d->eps, dn);\n        moe_oracle_rmsnorm(moe, w->post_ff_ln_1,"),
    ("expert_post_norm_skipped", "moe_oracle_rmsnorm(moe, w->post_ff_ln_2, H, (double)d->eps, moe);", ""),
    ("final_norm_skipped", "moe_oracle_rmsnorm(y, w->post_ff_ln, H, (double)d->eps, y);", ""),
    ("residual_dropped", "(xd[h] + y[h]) * (double)w->layer_scalar", "(y[h]) * (double)w->layer_scalar"),
    ("layer_scalar_before_residual", "(xd[h] + y[h]) * (double)w->layer_scalar", "(xd[h] + y[h] * (double)w->layer_scalar)"),
    # int8 experts
    ("int8_scale_over_128", "const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    ("int8_truncates", "v = rintf(bf16_to_f32(wr[c]) / s);", "v = truncf(bf16_to_f32(wr[c]) / s);"),
    ("int8_dequant_first_row_scale", "return (double)q[row * cols + col] * (double)scale[row];",
     "return (double)q[row * cols + col] * (double)scale[0];"),
    # MXFP4 experts
    ("fp4_exponent_off_by_one", "se = (ex - 1) - 2;", "se = ex - 2;"),
    ("fp4_emax_taken_as_3", "se = (ex - 1) - 2;", "se = (ex - 1) - 3;"),
    ("fp4_ties_to_odd", "(dk == db && (k & 1) == 0)", "(dk == db && (k & 1) == 1)"),
    ("fp4_nibbles_swapped_on_encode", "(uint8_t)(c0 | (c1 << 4))", "(uint8_t)(c1 | (c0 << 4))"),
    ("fp4_nibbles_swapped_on_decode", "const int code = (col & 1) ? (byte >> 4) : (byte & 15);",
     "const int code = (col & 1) ? (byte & 15) : (byte >> 4);"),
    ("fp4_grid_top_value_5", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}"),
    ("fp4_zero_keeps_its_sign", "return (best != 0 && v < 0) ? (best | 8) : best;",
     "return (v < 0) ? (best | 8) : best;"),
    ("fp4_decode_drops_sign", "return ldexp((code & 8) ? -mag : mag, e);", "return ldexp(mag, e);"),
    # permutation
    ("permute_tokens_descending",
     "for (int t = 0; t < T; ++t) {\n    for (int k = 0; k < K; ++k) {\n      int e = topk_idx[(size_t)t * K + k];",
     "for (int t = T - 1; t >= 0; --t) {\n    for (int k = 0; k < K; ++k) {\n      int e = topk_idx[(size_t)t * K + k];"),
    ("permute_stores_slot_not_token", "if (perm) perm[pos] = t;", "if (perm) perm[pos] = t * K + k;"),
    ("permute_weight_by_sorted_position", "w_sorted[pos] = topk_w[(size_t)t * K + k];", "w_sorted[pos] = topk_w[pos];"),
    ("permute_slot_position_one_late", "slot_pos[(size_t)t * K + k] = pos;", "slot_pos[(size_t)t * K + k] = next[e];"),
]

WORKERS = max(1, min(8, (os.cpu_count() or 2) - 1))


def _build_and_run(name, src, workdir):
    """Builds `src` as a copy of the oracle and runs the pin files against it."""
    d = os.path.join(workdir, name)
    os.makedirs(d)
    shutil.copy(os.path.join(ROOT, "oracle", "moe_oracle.h"), d)
    c = os.path.join(d, "moe_oracle.c")
    with open(c, "w") as f:
        f.write(src)
    so = os.path.join(d, "libmoe_oracle.so")
    cc = os.environ.get("CC", "gcc")
    b = subprocess.run([cc, *obuild.CFLAGS, c, "-o", so, "-lm"], capture_output=True, text=True)
    if b.returncode != 0:
        return ("build", b.returncode, b.stderr[-2000:])
    env = dict(os.environ, MOE_ORACLE_LIB=so, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", *PIN_FILES, "-x", "-q", "-p", "no:cacheprovider",
                        "--deselect", SLOW], cwd=ROOT, env=env, capture_output=True, text=True)
    return ("pins", r.returncode, r.stdout[-3000:] + r.stderr[-2000:])


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    with open(os.path.join(ROOT, "oracle", "moe_oracle.c")) as f:
        src = f.read()
    work = str(tmp_path_factory.mktemp("mutants"))
    jobs = {"unmodified": src}
    for name, old, new in MUTANTS:
        if src.count(old) == 1:
            jobs[name] = src.replace(old, new)
    with concurrent.futures.ThreadPoolExecutor(WORKERS) as ex:
        futs = {n: ex.submit(_build_and_run, n, s, work) for n, s in jobs.items()}
        return src, {n: f.result() for n, f in futs.items()}


def test_mutant_names_are_unique():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))


def test_unmodified_copy_passes_the_pins(results):
    _, res = results
    stage, rc, log = res["unmodified"]
    assert (stage, rc) == ("pins", 0), log


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(results, name, old, new):
    src, res = results
    assert src.count(old) == 1, "the text this mutant replaces is no longer unique in moe_oracle.c"
    stage, rc, log = res[name]
    assert stage == "pins", "mutant did not build: " + log
    assert rc == 1, "pins returned %d (0 = the mistake went unnoticed; other = not an assertion)\n%s" % (rc, log)
