"""CPU checks of the separation between the product path and the oracle: the
library and its binding never reach the oracle (no CPU fallback can route
through it), the oracle never reaches the library, and the only Python code
that imports the oracle is the test-suite, the smoke entry point and the
benchmark's CPU legs."""
import ast
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Functions of bench.py that may run the oracle: its timed CPU sample, the CPU
# baseline and the reference arm.
BENCH_ORACLE_FUNCS = {"_oracle_sample", "cpu_baseline", "run_reference"}
SOURCE_DIRS = ("kda_prefill_gb300", "oracle", "tests", "include", "profiles")


def _tracked(pattern):
    out = subprocess.run(["git", "ls-files", pattern], cwd=ROOT, capture_output=True,
                         text=True)
    if out.returncode == 0 and out.stdout.strip():
        return out.stdout.split()
    # outside a git checkout: the source folders and the top-level files
    rx = re.compile(pattern.replace(".", r"\.").replace("*", ".*") + "$")
    found = [f for f in os.listdir(ROOT) if os.path.isfile(os.path.join(ROOT, f))]
    for top in SOURCE_DIRS:
        for d, dirs, files in os.walk(os.path.join(ROOT, top)):
            dirs[:] = [x for x in dirs if not x.startswith((".", "__"))]
            found += [os.path.relpath(os.path.join(d, f), ROOT) for f in files]
    return [rel for rel in found if rx.search(rel)]


def _imports(tree):
    """(module root, enclosing top-level function name or None) per import."""
    res = []

    def visit(node, func):
        for child in ast.iter_child_nodes(node):
            f = func
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) and func is None:
                f = child.name
            if isinstance(child, ast.Import):
                res.extend((a.name.split(".")[0], f) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.level == 0 and child.module:
                res.append((child.module.split(".")[0], f))
            visit(child, f)

    visit(tree, None)
    return res


def _parse(rel):
    return ast.parse(open(os.path.join(ROOT, rel)).read(), filename=rel)


def test_product_never_imports_the_oracle_or_the_tests():
    for rel in _tracked("kda_prefill_gb300/*.py"):
        mods = {m for m, _ in _imports(_parse(rel))}
        assert not mods & {"oracle", "tests", "bench"}, (rel, mods)


def test_oracle_never_imports_the_product():
    for rel in _tracked("oracle/*.py"):
        mods = {m for m, _ in _imports(_parse(rel))}
        assert not mods & {"kda_prefill_gb300", "tests", "bench"}, (rel, mods)


def test_only_tests_smoke_and_bench_cpu_legs_import_the_oracle():
    for rel in _tracked("*.py"):
        if rel.startswith(("tests/", "oracle/")) or rel == "__graft_entry__.py":
            continue
        for mod, func in _imports(_parse(rel)):
            if mod != "oracle":
                continue
            assert rel == "bench.py" and func in BENCH_ORACLE_FUNCS, (rel, func)


def test_native_sources_share_nothing_with_the_oracle():
    inc = re.compile(r'#\s*include\s*"([^"]+)"')
    for rel in _tracked("kda_prefill_gb300/csrc/*") + _tracked("include/*"):
        for name in inc.findall(open(os.path.join(ROOT, rel)).read()):
            assert "oracle" not in name, (rel, name)
    src = open(os.path.join(ROOT, "oracle", "kda_oracle.c")).read()
    for name in inc.findall(src):
        assert "kda" not in name, name  # standard headers only (angle brackets)


def test_nothing_tracked_refers_to_the_scratch_folder():
    for rel in _tracked("*.py") + _tracked("kda_prefill_gb300/csrc/*"):
        text = open(os.path.join(ROOT, rel)).read()
        if rel == "tests/test_separation.py":
            continue
        assert "_work/" not in text and "'_work'" not in text and '"_work"' not in text, rel


def test_product_uses_no_compiler_layer():
    """The compute path is the CUDA library: the package and the entry points
    import no Triton and call no torch.compile."""
    for rel in _tracked("kda_prefill_gb300/*.py") + ["__graft_entry__.py", "bench.py"]:
        tree = _parse(rel)
        mods = {m for m, _ in _imports(tree)}
        assert "triton" not in mods, rel
        for node in ast.walk(tree):
            if isinstance(node, ast.Attribute) and node.attr == "compile":
                assert not (isinstance(node.value, ast.Name) and node.value.id == "torch"), rel


def test_build_targets_sm_103a_only():
    from kda_prefill_gb300 import build as kbuild
    assert kbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-lineinfo" in kbuild._flags()
