"""The C ABI library builds, loads without a GPU and exports every entry point include/moe_ffn.h
declares; the ctypes binding's structures have the header's layout (CPU only, no compute calls)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from mixture_experts_ffn_router_gb300 import binding as B
from mixture_experts_ffn_router_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_ffn_[a-z_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return B.lib()


def test_header_declares_the_expected_entry_points():
    names = _declared_functions()
    for n in ("moe_ffn_init", "moe_ffn_forward", "moe_ffn_destroy", "moe_ffn_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_struct_layouts_match_the_header(tmp_path):
    src = tmp_path / "layout.c"
    exe = tmp_path / "layout"
    fields = {
        "moe_ffn_config": [f for f, _ in B.moe_ffn_config._fields_],
        "moe_ffn_weights": [f for f, _ in B.moe_ffn_weights._fields_],
        "moe_ffn_views": [f for f, _ in B.moe_ffn_views._fields_],
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_ffn.h"', "int main(void){"]
    for st, fs in fields.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (st, st))
        for f in fs:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (st, f, st, f))
    lines.append("return 0;}")
    src.write_text("\n".join(lines))
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(l.split() for l in out if l.strip())
    for st, fs in fields.items():
        cls = getattr(B, st)
        assert int(got[st]) == ctypes.sizeof(cls), st
        for f in fs:
            assert int(got["%s.%s" % (st, f)]) == getattr(cls, f).offset, (st, f)


def test_calls_that_need_no_device(lib):
    assert B.moe_ffn_status_string(B.MOE_FFN_EARCH).startswith("device is not")
    cfg = B.make_config(B.MOE_FFN_FULL_LAYER, 64)
    assert B.moe_ffn_workspace_bytes(cfg) > 64 * 8 * 2816 * 4
    bad = B.make_config(B.MOE_FFN_FULL_LAYER, 0)
    assert B.moe_ffn_workspace_bytes(bad) == 0
    bad = B.make_config(7, 64)
    assert B.moe_ffn_workspace_bytes(bad) == 0
    assert lib.moe_ffn_kernels_per_forward(None, 4) == B.MOE_FFN_EINVAL
    assert lib.moe_ffn_forward(None, None, 0, None, None, None) == B.MOE_FFN_EINVAL
    lib.moe_ffn_destroy(None)


def test_workspace_grows_with_max_tokens(lib):
    a = B.moe_ffn_workspace_bytes(B.make_config(B.MOE_FFN_FULL_LAYER, 64))
    b = B.moe_ffn_workspace_bytes(B.make_config(B.MOE_FFN_FULL_LAYER, 4096))
    c = B.moe_ffn_workspace_bytes(B.make_config(B.MOE_FFN_MOE_ONLY, 4096))
    assert a < c < b


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_LIB", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()
