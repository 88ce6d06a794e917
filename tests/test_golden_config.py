"""The block's shapes against the figures the pages print (tests/golden/gemma4_26b_a4b_config.txt).

The oracle, the C header, the binding and the synthetic-weight generator each carry the shapes of the
26B-A4B block; a mistyped dimension in any of them would make every parity test compare two wrong
programs. Here they are held against the printed configuration and against two figures the pages
derive from it: the shapes of the experts seen as two plain linears, and the bytes an int8 copy of
all 30 layers' experts saves over bf16 (one byte per expert weight).
"""
import os
import re

import pytest

import oracle
from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _golden():
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", "gemma4_26b_a4b_config.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            if "," in v:
                vals[k] = tuple(int(p) for p in v.split(","))
            else:
                try:
                    vals[k] = int(v)
                except ValueError:
                    try:
                        vals[k] = float(v)
                    except ValueError:
                        vals[k] = v
    return vals


G = _golden()
NAMES = ("hidden", "n_experts", "top_k", "moe_inter", "dense_inter")


def test_oracle_dims_are_the_printed_ones():
    d = oracle.gemma_dims(True)
    for k in NAMES:
        assert d[k] == G[k], k


def test_header_macros_are_the_printed_ones():
    with open(os.path.join(ROOT, "include", "moe_ffn.h")) as f:
        text = f.read()
    macros = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define MOE_FFN_(\w+) (\d+)\b", text)}
    for k in NAMES:
        assert macros[k.upper()] == G[k], k


def test_binding_and_generator_dims_are_the_printed_ones():
    assert (B.HIDDEN, B.N_EXPERTS, B.TOP_K, B.MOE_INTER, B.DENSE_INTER) == tuple(G[k] for k in NAMES)
    for k in NAMES:
        assert synth.GEMMA[k] == G[k], k


def test_expert_tensor_shapes():
    E, H, I = G["n_experts"], G["hidden"], G["moe_inter"]
    assert G["gate_up_shape"] == (E, 2 * I, H)      # gate rows and up rows fused
    assert G["down_shape"] == (E, H, I)
    assert G["gate_up_as_linear"] == (E * 2 * I, H)
    assert G["down_as_linear"] == (H, E * I)
    assert E // 8 == G["experts_per_rank_tp8"]


def test_int8_expert_saving_matches_the_shapes():
    """One byte saved per expert weight over all layers; the pages print it to 0.1 GB."""
    E, H, I, L = G["n_experts"], G["hidden"], G["moe_inter"], G["n_layers"]
    per_layer = E * 2 * I * H + E * H * I
    saving_gb = L * per_layer / 1e9
    assert saving_gb == pytest.approx(G["int8_expert_saving_gb"], abs=0.05)
    assert saving_gb / 2 == pytest.approx(G["int8_experts_per_rank_tp2_gb"], abs=0.05)


def test_activation_is_the_tanh_gelu():
    import numpy as np
    import torch
    assert G["activation"] == "gelu_pytorch_tanh"
    x = np.linspace(-6, 6, 97)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(v) for v in x])
    assert np.abs(got - ref).max() < 1e-10  # the oracle takes sqrt(2/pi) to the 10 digits a page prints
