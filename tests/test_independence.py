"""The oracle and the CUDA path share no code, and the product path never
reaches the oracle: checked on the sources' import statements.

* nothing under fp4_kv_cache_rope_gb300/ or synth/ imports `oracle`;
* nothing under oracle/ imports the product package;
* bench.py imports `oracle` only inside its CPU-baseline and reference-arm
  functions;
* no CUDA/C source includes a file from oracle/.
"""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PRODUCT = "fp4_kv_cache_rope_gb300"
BENCH_ORACLE_USERS = {"oracle_plan", "_score_fn", "cpu_baseline",
                      "reference_arm", "model_oracle_sample", "model_bench_cpu"}


def py_files(sub):
    for dirpath, _, files in os.walk(os.path.join(ROOT, sub)):
        if "__pycache__" in dirpath or "_build" in dirpath:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(dirpath, f)


def imported_modules(tree):
    """(module name, enclosing function name or None) of every import."""
    out = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, ast.Import):
                out.extend((a.name, func) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                mod = child.module or ""
                if child.level:  # relative import inside a package
                    mod = "." * child.level + mod
                out.append((mod, func))
            visit(child, f)

    visit(tree, None)
    return out


def top(name):
    return name.split(".")[0]


def test_product_and_generators_never_import_the_oracle():
    for sub in (PRODUCT, "synth"):
        for path in py_files(sub):
            mods = imported_modules(ast.parse(open(path).read()))
            assert all(top(m) != "oracle" for m, _ in mods), path


def test_oracle_never_imports_the_product():
    for path in py_files("oracle"):
        mods = imported_modules(ast.parse(open(path).read()))
        assert all(top(m) != PRODUCT for m, _ in mods), path
        # inputs come from the host generator, not from the module that lays
        # workloads out on the device through the CUDA path
        assert all(not m.startswith("synth.device") for m, _ in mods), path


def test_host_generator_stays_host_only():
    mods = imported_modules(ast.parse(open(os.path.join(ROOT, "synth", "host.py")).read()))
    assert all(top(m) not in (PRODUCT, "oracle") and not m.endswith("device") for m, _ in mods)


def test_bench_uses_the_oracle_only_in_its_cpu_legs():
    mods = imported_modules(ast.parse(open(os.path.join(ROOT, "bench.py")).read()))
    users = {f for m, f in mods if top(m) == "oracle"}
    assert users, "bench.py no longer times the oracle"
    assert users <= BENCH_ORACLE_USERS, users


def test_cuda_sources_include_nothing_from_the_oracle():
    csrc = os.path.join(ROOT, PRODUCT, "csrc")
    for f in os.listdir(csrc):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            for line in open(os.path.join(csrc, f)):
                if re.match(r"\s*#\s*include", line):
                    assert "oracle" not in line, (f, line)


def test_oracle_cpp_includes_nothing_from_the_product():
    """The C++ oracle includes only system headers: nothing from csrc/,
    include/ or the product package."""
    odir = os.path.join(ROOT, "oracle")
    srcs = [f for f in os.listdir(odir) if f.endswith((".c", ".cc", ".cpp", ".h", ".hpp"))]
    assert srcs, "no C++ oracle source"
    for f in srcs:
        for line in open(os.path.join(odir, f)):
            if re.match(r"\s*#\s*include", line):
                assert "<" in line and '"' not in line, (f, line)
