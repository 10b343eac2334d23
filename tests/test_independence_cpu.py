"""The product path and the oracle share no code.

Static checks over the sources: no module of the package imports the oracle
(or the tests), the oracle imports nothing of the package but the seeded input
generators' data class, the CUDA sources include nothing from the oracle, and
in the benchmark only the CPU-baseline worker imports it.
"""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mla_split_kv_gb300")


def imports_of(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names += [(a.name, node) for a in node.names]
        elif isinstance(node, ast.ImportFrom):
            names.append((("." * node.level) + (node.module or ""), node))
    return tree, names


def test_package_never_imports_the_oracle_or_the_tests():
    for f in sorted(os.listdir(PKG)):
        if f.endswith(".py"):
            _, names = imports_of(os.path.join(PKG, f))
            for name, _ in names:
                assert not name.split(".")[0] in ("oracle", "tests"), (f, name)


def test_cuda_sources_include_nothing_of_the_oracle():
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        for line in text.splitlines():
            if line.lstrip().startswith("#include"):
                assert "oracle" not in line, (f, line)


def test_oracle_uses_only_the_input_generators_of_the_package():
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        if f.endswith(".py"):
            _, names = imports_of(os.path.join(odir, f))
            for name, _ in names:
                if name.startswith("mla_split_kv_gb300"):
                    assert name in ("mla_split_kv_gb300.inputs",), (f, name)


def test_bench_imports_the_oracle_only_in_the_cpu_worker():
    tree, names = imports_of(os.path.join(ROOT, "bench.py"))
    users = []
    for node in ast.walk(tree):
        if isinstance(node, ast.FunctionDef):
            for sub in ast.walk(node):
                if isinstance(sub, (ast.Import, ast.ImportFrom)):
                    mod = sub.module if isinstance(sub, ast.ImportFrom) else sub.names[0].name
                    if mod and mod.split(".")[0] == "oracle":
                        users.append(node.name)
    top = [n for n, node in names if n.split(".")[0] == "oracle" and node in tree.body]
    assert not top, "bench.py imports the oracle at module level"
    assert set(users) == {"_oracle_worker"}, users
