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
    slots = (ctypes.c_int * 7)()
    assert lib.moe_ffn_kernel_slots(None, 4, slots, 7) == B.MOE_FFN_EINVAL
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


C_CALLER = r"""
#include <stdint.h>
#include <stdio.h>
#include "moe_ffn.h"

int main(void) {
  moe_ffn_config c = {MOE_FFN_HIDDEN, MOE_FFN_N_EXPERTS, MOE_FFN_TOP_K, MOE_FFN_MOE_INTER,
                      MOE_FFN_DENSE_INTER, MOE_FFN_FULL_LAYER, 64, 1e-6f, 0.018844459f};
  void* fake = (void*)(uintptr_t)4096; /* never dereferenced: every call below fails its checks first */
  printf("bytes %zu\n", moe_ffn_workspace_bytes(&c));
  printf("kernels %d\n", moe_ffn_kernels_per_forward(NULL, 4));
  printf("noalloc_toobig %d\n", moe_ffn_router_logits_noalloc(fake, 1025, fake, fake, 0.02f, 1e-6f, fake, NULL));
  printf("noalloc_align %d\n",
         moe_ffn_router_logits_noalloc((void*)(uintptr_t)4098, 4, fake, fake, 0.02f, 1e-6f, fake, NULL));
  printf("int8_cols %d\n", moe_ffn_quantize_int8(fake, 4, 7, fake, fake, NULL));
  printf("fp4_cols %d\n", moe_ffn_quantize_mxfp4(fake, 4, 48, fake, fake, NULL));
#ifdef WITH_INIT
  moe_ffn_ctx* ctx = (moe_ffn_ctx*)fake;
  int rc = moe_ffn_init(&ctx, &c, fake, moe_ffn_workspace_bytes(&c), 0);
  printf("init %d %d\n", rc, ctx == NULL);
  moe_ffn_destroy(ctx);
#endif
  printf("status %s\n", moe_ffn_status_string(MOE_FFN_ETOOBIG));
  return 0;
}
"""


def test_plain_c_caller_links_the_library(lib, tmp_path):
    # A C11 program, built with warnings as errors, includes the header and links the shared
    # library with no Python in between; the calls it makes fail their argument checks with the
    # header's status codes before any device work.
    import torch
    src = tmp_path / "caller.c"
    exe = tmp_path / "caller"
    src.write_text(C_CALLER)
    pkg = os.path.dirname(B.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", pkg, "-lmoe_ffn", "-Wl,-rpath," + pkg, "-o", str(exe)]
    if not torch.cuda.is_available():
        cmd.insert(1, "-DWITH_INIT")
    subprocess.run(cmd, check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout
    got = dict(l.split(" ", 1) for l in out.strip().split("\n"))
    assert int(got["bytes"]) == B.moe_ffn_workspace_bytes(B.make_config(B.MOE_FFN_FULL_LAYER, 64))
    assert int(got["kernels"]) == B.MOE_FFN_EINVAL
    assert int(got["noalloc_toobig"]) == B.MOE_FFN_ETOOBIG
    assert int(got["noalloc_align"]) == B.MOE_FFN_EALIGN
    assert int(got["int8_cols"]) == B.MOE_FFN_EINVAL
    assert int(got["fp4_cols"]) == B.MOE_FFN_EINVAL
    assert got["status"] == B.moe_ffn_status_string(B.MOE_FFN_ETOOBIG)
    if "init" in got:
        # No usable sm_103 device here: init reports a CUDA or architecture error and leaves NULL.
        rc, is_null = map(int, got["init"].split())
        assert rc in (B.MOE_FFN_ECUDA, B.MOE_FFN_EARCH) and is_null == 1


def test_status_bits_match_the_kernels():
    # The header's MOE_FFN_STATUS_* macros name the bits the kernels set (the kStatus* enum of the
    # PTX layer), one to one and with the same values.
    hdr = open(HEADER).read()
    macros = {m.group(1): int(m.group(2), 16) for m in
              re.finditer(r"#define MOE_FFN_STATUS_([A-Z_]+) (0x[0-9a-f]+)u", hdr)}
    ptx = open(os.path.join(ROOT, "mixture_experts_ffn_router_gb300", "csrc", "ptx.cuh")).read()
    enum = {m.group(1): 1 << int(m.group(2)) for m in re.finditer(r"kStatus(\w+) = 1u << (\d+)", ptx)}
    snake = {re.sub(r"(?<!^)(?=[A-Z])", "_", k).upper(): v for k, v in enum.items()}
    assert macros and macros == snake
    assert macros == B.STATUS_BITS
    assert B.decode_status(0x41) == ["WAIT_FULL", "DRAIN"] and B.decode_status(0) == []
    assert B.decode_status(0x102) == ["WAIT_EMPTY", "WAIT_COPY"]
    assert B.decode_status(0x202) == ["WAIT_EMPTY", "0x200"]
    # The status word of a forward holds nothing else.
    assert sum(macros.values()) == 0x1ff
