"""The CUDA path and the oracle stay independent (CPU only, by reading the sources).

Neither side imports, includes or links the other. Only the seeded input generator
(mixture_experts_ffn_router_gb300/synth.py, random draws and no block arithmetic) serves both, and
it is used by the tests and the benchmark, not by the oracle. bench.py touches the oracle only in
its CPU legs (the CPU baseline and the reference arm), and __graft_entry__ only to build it and in
smoke()'s comparison.
"""
import ast
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mixture_experts_ffn_router_gb300")


def _imports(path):
    """(module name, name of the enclosing top-level function or None) for every import."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            f = fn
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) and fn is None:
                f = child.name
            if isinstance(child, ast.Import):
                out.extend((a.name, f) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                mod = ("." * child.level) + (child.module or "")
                sep = "." if child.module else ""
                out.extend((mod + sep + a.name, f) for a in child.names)
            visit(child, f)

    visit(tree, None)
    return out


def _is_oracle(mod):
    return mod == "oracle" or mod.startswith("oracle.")


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        bad = [m for m, _ in _imports(path) if _is_oracle(m)]
        assert not bad, (path, bad)


def test_cuda_sources_reference_no_oracle_code():
    pat = re.compile(r"moe_oracle|oracle/|libmoe_oracle")
    for path in glob.glob(os.path.join(PKG, "csrc", "*")):
        text = open(path).read()
        assert not pat.search(text), path


def test_oracle_never_uses_the_cuda_path():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        bad = [m for m, _ in _imports(path) if m.startswith("mixture_experts_ffn_router_gb300")]
        assert not bad, (path, bad)
    pat = re.compile(r"#\s*include\s*[<\"](?!stdint\.h|stddef\.h|math\.h|stdlib\.h|string\.h|omp\.h|moe_oracle\.h)")
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")):
        text = open(path).read()
        assert not pat.search(text), path
        assert "moe_ffn" not in re.sub(r"/\*.*?\*/", "", text, flags=re.S), path


def test_bench_uses_the_oracle_only_in_its_cpu_legs():
    users = {f for m, f in _imports(os.path.join(ROOT, "bench.py")) if _is_oracle(m)}
    assert users and users <= {"oracle_tokens_per_s", "run_reference"}, users


def test_graft_entry_uses_the_oracle_only_to_build_it_and_in_smoke():
    users = {(m, f) for m, f in _imports(os.path.join(ROOT, "__graft_entry__.py")) if _is_oracle(m)}
    assert users and all(f in ("build", "smoke") for _, f in users), users
    assert all(m == "oracle.build" or m == "oracle" and f == "smoke" for m, f in users), users


def test_generator_holds_no_block_arithmetic():
    # synth.py draws random tensors; the block's operations (norms, softmax, top-k, GELU, matmul)
    # must not appear there, so that neither side can inherit a mistake from it.
    text = open(os.path.join(PKG, "synth.py")).read()
    for op in ("softmax", "topk", "gelu", "tanh", "rsqrt", "matmul", "einsum", "@ ", "rms_norm", "sort("):
        assert op not in text, op
