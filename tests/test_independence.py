"""The oracle and the CUDA path share no code (no GPU).

The product (the package, its CUDA sources and the C header) never imports,
includes or links anything under oracle/, and the oracle never reaches into
the product; bench.py touches the oracle only inside its CPU-baseline and
reference-arm functions.  The one module both sides read is the seeded input
generator (workloads.py), which holds none of the layer's arithmetic."""
import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mixture_experts_layer_capacity_b300")
ORACLE = os.path.join(ROOT, "oracle")


def _py_imports(path, top_level_only=False):
    tree = ast.parse(open(path).read(), path)
    nodes = tree.body if top_level_only else ast.walk(tree)
    out = set()
    for n in nodes:
        if isinstance(n, ast.Import):
            out |= {a.name.split(".")[0] for a in n.names}
        elif isinstance(n, ast.ImportFrom) and n.module:
            out.add(n.module.split(".")[0])
    return out


def _files(root, exts):
    for d, _, names in os.walk(root):
        if "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_never_imports_the_oracle():
    for f in _files(PKG, (".py",)):
        assert "oracle" not in _py_imports(f), f


def test_sources_never_include_across_the_boundary():
    inc = re.compile(r'^\s*#\s*include\s*[<"]([^">]+)[">]', re.M)
    for f in _files(PKG, (".cu", ".cuh", ".h", ".cpp", ".c")):
        for h in inc.findall(open(f).read()):
            assert "oracle" not in h, (f, h)
    for f in _files(ORACLE, (".c", ".h", ".cpp")):
        for h in inc.findall(open(f).read()):
            assert "moe.h" not in h and "csrc" not in h and "mixture_experts" not in h, (f, h)
    for f in _files(ORACLE, (".py",)):
        assert "mixture_experts_layer_capacity_b300" not in _py_imports(f), f


def test_bench_imports_the_oracle_only_in_its_baseline_legs():
    bench = os.path.join(ROOT, "bench.py")
    assert "oracle" not in _py_imports(bench, top_level_only=True)
    tree = ast.parse(open(bench).read())
    users = set()

    def visit(node, owner):
        for ch in ast.iter_child_nodes(node):
            if isinstance(ch, (ast.FunctionDef, ast.ClassDef)):
                visit(ch, f"{owner}.{ch.name}" if owner else ch.name)
            elif isinstance(ch, ast.Import) and any(a.name == "oracle" for a in ch.names):
                users.add(owner)
            else:
                visit(ch, owner)

    visit(tree, "")
    # the CPU-baseline sampler and the two arms' baseline legs
    assert users <= {"OracleSample.__init__", "run_reference", "run_ours"}, users


def test_loading_the_binding_leaves_the_oracle_unloaded():
    code = ("import sys; sys.path.insert(0, sys.argv[1]);"
            "from mixture_experts_layer_capacity_b300 import binding, sharded, workloads;"
            "binding.lib();"
            "print('oracle' in sys.modules)")
    r = subprocess.run([sys.executable, "-c", code, ROOT], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "False"


def test_input_generators_hold_no_layer_arithmetic():
    """workloads.py draws seeded tensors; it must not route, gate, or run an
    expert (no softmax, top-k, matmul or SiLU)."""
    tree = ast.parse(open(os.path.join(PKG, "workloads.py")).read())
    banned = {"softmax", "log_softmax", "topk", "sort", "argsort", "matmul", "mm", "bmm",
              "einsum", "silu", "sigmoid", "linear"}
    for n in ast.walk(tree):
        if isinstance(n, ast.Call):
            f = n.func
            name = f.attr if isinstance(f, ast.Attribute) else getattr(f, "id", "")
            assert name not in banned, name
        assert not (isinstance(n, ast.BinOp) and isinstance(n.op, ast.MatMult))
