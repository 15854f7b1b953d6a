"""The oracle and the CUDA path share no code, and the product never calls the
oracle (a static scan of the sources; no GPU).

- Nothing under the package or ``include/`` names the oracle.
- Nothing under ``oracle/`` names the package, its headers or its sources.
- ``bench.py`` imports the oracle only inside its CPU-baseline helpers, and
  those are reached only from the CPU-baseline leg of the GPU arm and from
  the reference arm.
- ``__graft_entry__.py`` imports it only in ``build()`` (which compiles the
  checker) and ``smoke()`` (which checks against it).
- The package's Python calls no torch arithmetic: no CPU or library fallback
  stands in for a kernel.
"""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "w8a8_quantized_projections_gb300")
SOURCE_EXT = (".py", ".cu", ".cuh", ".h", ".c", ".cpp")


def _sources(*dirs):
    for d in dirs:
        for base, subdirs, files in os.walk(d):
            subdirs[:] = [s for s in subdirs if not s.startswith(("_build", "__pycache__"))]
            for f in files:
                if f.endswith(SOURCE_EXT):
                    yield os.path.join(base, f)


def test_product_never_names_the_oracle():
    for path in _sources(PKG, os.path.join(ROOT, "include")):
        text = open(path, encoding="utf-8").read()
        assert "oracle" not in text.lower(), path


def test_oracle_never_names_the_product():
    for path in _sources(os.path.join(ROOT, "oracle")):
        text = open(path, encoding="utf-8").read()
        for word in ("w8a8_quantized_projections_gb300", "clef.h", "clef_kernels", "csrc", "libclef.so"):
            assert word not in text, (path, word)


def _imports_of(tree, module):
    """(enclosing function name or None, node) for each import of module."""
    found = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == module for a in child.names):
                found.append(func)
            elif isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == module:
                found.append(func)
            visit(child, f)

    visit(tree, None)
    return found


def _callers(tree, name):
    """Names of the functions whose bodies call ``name``."""
    out = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and node.func.id == name:
                    out.add(fn.name)
    return out


def test_bench_imports_the_oracle_only_for_the_cpu_baseline():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read())
    where = set(_imports_of(tree, "oracle"))
    assert where == {"oracle_weights", "oracle_sample"}, where
    for helper in where:
        # the reference arm and the GPU arm's CPU-baseline leg (inside main)
        assert _callers(tree, helper) <= {"run_reference", "main"}, helper
    main = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "main")
    # inside main, every call of a helper sits under an `if` on the cpu-baseline switch
    parent = {c: n for n in ast.walk(main) for c in ast.iter_child_nodes(n)}
    calls = [c for c in ast.walk(main) if isinstance(c, ast.Call) and isinstance(c.func, ast.Name)
             and c.func.id in where]
    assert calls
    for call in calls:
        node, guarded = call, False
        while node in parent:
            node = parent[node]
            if isinstance(node, ast.If) and "no_cpu_baseline" in ast.unparse(node.test):
                guarded = True
        assert guarded, ast.unparse(call)


def test_entry_points_import_the_oracle_only_to_build_and_check():
    tree = ast.parse(open(os.path.join(ROOT, "__graft_entry__.py"), encoding="utf-8").read())
    assert set(_imports_of(tree, "oracle")) <= {"build", "smoke"}


# torch calls that would compute a step of the path (any of them in the package
# would be a fallback around the CUDA kernels)
COMPUTE = {"matmul", "mm", "bmm", "addmm", "einsum", "linear", "_int_mm", "_scaled_mm", "silu", "sigmoid",
           "exp", "softmax", "amax", "abs", "round", "clamp", "clip", "sum", "mul", "add", "div", "mul_",
           "add_", "div_", "hadamard", "fft", "functional", "rint"}


def test_package_python_computes_nothing_itself():
    """The binding and the layer runner only allocate, pack weights at set-up
    and marshal arguments; every step of the path runs in the library."""
    for path in _sources(PKG):
        if not path.endswith(".py"):
            continue
        tree = ast.parse(open(path, encoding="utf-8").read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Attribute) and node.attr in COMPUTE:
                raise AssertionError(f"{path}:{node.lineno}: .{node.attr}")
            if isinstance(node, ast.BinOp) and isinstance(node.op, ast.MatMult):
                raise AssertionError(f"{path}:{node.lineno}: @")
