"""The product path and the oracle are independent: the CUDA sources, the C header and the
Python binding never name the oracle, importing the binding loads no oracle module, the oracle
never imports the binding, and the shared input generator performs none of the method's
arithmetic (it imports neither side)."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bit_moe_expert_moet_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _imports(path):
    tree = ast.parse(open(path).read())
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.add(node.module.split(".")[0])
    return out


def test_product_sources_never_name_the_oracle():
    for f in list(_files(PKG, (".cu", ".cuh", ".py", ".h"))) + list(_files(os.path.join(ROOT, "include"), (".h",))):
        src = open(f).read()
        assert "oracle" not in src, f


def test_oracle_never_imports_the_product():
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        assert "bit_moe_expert_moet_gb300" not in _imports(f), f


def test_input_generator_imports_neither_side():
    imps = _imports(os.path.join(ROOT, "workloads.py"))
    assert "oracle" not in imps and "bit_moe_expert_moet_gb300" not in imps


def test_importing_the_binding_loads_no_oracle_module():
    code = ("import sys, __graft_entry__ as g; g.build(); import bit_moe_expert_moet_gb300; "
            "print(sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')))")
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip().splitlines()[-1] == "[]"
