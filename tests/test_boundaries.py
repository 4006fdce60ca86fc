"""Static checks of the separation between the product and its test oracle.

* The product (the package's Python modules, its CUDA sources and the C
  header) never imports, loads or includes the oracle.
* bench.py touches the oracle only in the CPU-baseline / reference leg (the
  OracleSample class), and __graft_entry__ only in build() (which compiles
  it) and the smoke check.
* No committed source reads from the untracked working folder.
"""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "quantized_optimizer_state_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d or "_build" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _oracle_imports(tree):
    """(node, enclosing function/class names) of every import of the oracle."""
    out = []

    def visit(node, scope):
        for child in ast.iter_child_nodes(node):
            s = scope + [child.name] if isinstance(child, (ast.FunctionDef, ast.ClassDef)) else scope
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                out.append((child, s))
            elif isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                out.append((child, s))
            visit(child, s)

    visit(tree, [])
    return out


def test_package_never_imports_the_oracle():
    for f in _files(PKG, (".py",)):
        src = open(f).read()
        assert not _oracle_imports(ast.parse(src)), f"{f} imports the oracle"
        assert "liboracle" not in src, f"{f} names the oracle's library"


def test_native_sources_never_include_the_oracle():
    for f in list(_files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h"))) + \
            list(_files(os.path.join(ROOT, "include"), (".h",))):
        src = open(f).read()
        assert not re.search(r'#\s*include\s*[<"][^>"]*oracle', src), f"{f} includes the oracle"
        assert "liboracle" not in src and "oracle_" not in src, f"{f} names oracle symbols"


def test_bench_and_entry_use_the_oracle_only_where_allowed():
    allowed = {"bench.py": {"OracleSample"}, "__graft_entry__.py": {"build", "_smoke_case"}}
    for name, scopes in allowed.items():
        tree = ast.parse(open(os.path.join(ROOT, name)).read())
        found = _oracle_imports(tree)
        assert found, f"{name}: expected its oracle leg"
        for node, scope in found:
            assert scopes & set(scope), f"{name}:{node.lineno} imports the oracle outside {sorted(scopes)}"


def test_no_source_reads_the_working_folder():
    pat = re.compile(r"""(^|[\s'"/(])_work(/|['"])""")
    srcs = [os.path.join(ROOT, n) for n in ("bench.py", "__graft_entry__.py")]
    srcs += list(_files(PKG, (".py", ".cu", ".cuh", ".h"))) + list(_files(os.path.join(ROOT, "tests"), (".py",)))
    srcs += list(_files(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")))
    for f in srcs:
        if os.path.abspath(f) == os.path.abspath(__file__):
            continue
        for i, line in enumerate(open(f), 1):
            assert not pat.search(line), f"{f}:{i} refers to the working folder"
