"""The torch convenience layer of the binding rejects tensors of the wrong type, size, shape or
placement before anything reaches the library (CPU only: meta tensors carry dtype and shape without
memory, and are not CUDA tensors, so a well-formed one stops at the placement check)."""
import os
import re

import pytest
import torch

from mixture_experts_ffn_router_gb300 import binding as B
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
H, E, I, D = B.HIDDEN, B.N_EXPERTS, B.MOE_INTER, B.DENSE_INTER


def _meta_weights(full=True):
    w = {"router_w": torch.empty(E, H, device="meta"), "router_norm_w": torch.empty(H, device="meta"),
         "per_expert_scale": torch.empty(E, device="meta"),
         "gate_up": torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device="meta"),
         "down": torch.empty(E, H, I, dtype=torch.bfloat16, device="meta"), "layer_scalar": 0.8}
    if full:
        w["dense_gate"] = torch.empty(D, H, dtype=torch.bfloat16, device="meta")
        w["dense_up"] = torch.empty(D, H, dtype=torch.bfloat16, device="meta")
        w["dense_down"] = torch.empty(H, D, dtype=torch.bfloat16, device="meta")
        for n in ("pre_ff_ln", "pre_ff_ln_2", "post_ff_ln_1", "post_ff_ln_2", "post_ff_ln"):
            w[n] = torch.empty(H, device="meta")
    return w


def _header_fields():
    """(element type, element count) of each weight field, read from the comments of
    moe_ffn_weights in include/moe_ffn.h ("const T* name; /* [d0, d1, ...] ...")."""
    text = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    body = text[text.index("typedef struct moe_ffn_weights"):text.index("} moe_ffn_weights;")]
    types = {"float": torch.float32, "uint16_t": torch.bfloat16, "int8_t": torch.int8, "uint8_t": torch.uint8}
    out = {}
    for ctype, name, dims in re.findall(r"const (float|uint16_t|int8_t|uint8_t)\* (\w+);\s*/\* \[([0-9*, ]+)\]", body):
        n = 1
        for part in dims.split(","):
            for f in part.split("*"):
                n *= int(f)
        out[name] = (types[ctype], n)
    return out


def test_field_specs_are_the_header_shapes():
    spec = B._field_specs()
    assert set(spec) == set(B.WEIGHT_FIELDS + B.INT8_FIELDS + B.F4_FIELDS)
    header = _header_fields()
    # The five norm weights share one comment form ("[2816] fp32: ...") and are all listed.
    assert set(header) == set(spec)
    for f in spec:
        assert spec[f] == header[f], f


@pytest.mark.parametrize("full", [True, False])
def test_well_formed_weights_stop_only_at_placement(full):
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.weights_struct(_meta_weights(full))


@pytest.mark.parametrize("field,bad,msg", [
    ("gate_up", torch.empty(E, 2 * I, H, dtype=torch.float16, device="meta"), "must be torch.bfloat16"),
    ("router_w", torch.empty(E, H, dtype=torch.float64, device="meta"), "must be torch.float32"),
    ("down", torch.empty(E - 1, H, I, dtype=torch.bfloat16, device="meta"), "must hold"),
    ("post_ff_ln", torch.empty(H + 8, device="meta"), "must hold"),
    ("down_q", torch.empty(E * H, I, dtype=torch.uint8, device="meta"), "must be torch.int8"),
    ("gate_up_f4s", torch.empty(E * 2 * I, H // 16, dtype=torch.uint8, device="meta"), "must hold"),
])
def test_wrong_type_or_size_is_named(field, bad, msg):
    w = _meta_weights()
    w[field] = bad
    with pytest.raises(ValueError, match="weight %s %s" % (field, msg)):
        B.weights_struct(w)


def test_layer_scalar_is_required():
    w = _meta_weights()
    del w["layer_scalar"]
    for f in list(w):
        w[f] = None
    with pytest.raises(ValueError, match="layer_scalar"):
        B.weights_struct(w)


def test_forward_io_checks():
    x = torch.empty(5, H, dtype=torch.bfloat16, device="meta")
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.check_io(x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.check_io(x, torch.empty_like(x))
    with pytest.raises(ValueError, match="shape"):
        B.check_io(torch.empty(5, H // 2, dtype=torch.bfloat16, device="meta"))
    with pytest.raises(ValueError, match="shape"):
        B.check_io(torch.empty(5 * H, dtype=torch.bfloat16, device="meta"))
    with pytest.raises(ValueError, match="x must be torch.bfloat16"):
        B.check_io(torch.empty(5, H, device="meta"))
    with pytest.raises(ValueError, match="out must have the shape"):
        B.check_io(x, torch.empty(4, H, dtype=torch.bfloat16, device="meta"))
    with pytest.raises(ValueError, match="out must be torch.bfloat16"):
        B.check_io(x, torch.empty(5, H, device="meta"))
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.check_io(torch.empty(0, H, dtype=torch.bfloat16, device="meta"))


def test_expert_ranges_cover_the_experts_once():
    # The contiguous expert groups of the expert-parallel shards ("The traceable trick": rank r of 8
    # owns experts 16 r .. 16 r + 15): every expert exactly once, sizes within one of each other.
    assert [B.expert_range(r, 8) for r in range(8)] == [(16 * r, 16 * r + 16) for r in range(8)]
    for world in (1, 2, 3, 8, 16, 128):
        rs = [B.expert_range(r, world) for r in range(world)]
        assert rs[0][0] == 0 and rs[-1][1] == 128
        assert all(rs[i][1] == rs[i + 1][0] for i in range(world - 1))
        sizes = [e - b for b, e in rs]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
