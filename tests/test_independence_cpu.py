"""The CUDA path and the oracle stay independent (CPU only, static).

The package never imports the oracle and the oracle never imports the
package or loads native code; the benchmark reaches the oracle only from
its CPU-baseline / reference code, and the build entry only from smoke();
no CUDA source mentions it."""
import ast
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_attention_prolog_gb300")


def _imports(tree):
    """(node, top-level module name) of every import in the tree."""
    out = []
    for n in ast.walk(tree):
        if isinstance(n, ast.Import):
            out += [(n, a.name.split(".")[0]) for a in n.names]
        elif isinstance(n, ast.ImportFrom) and n.level == 0 and n.module:
            out.append((n, n.module.split(".")[0]))
    return out


def _parents(tree):
    par = {}
    for n in ast.walk(tree):
        for c in ast.iter_child_nodes(n):
            par[c] = n
    return par


def _enclosing(node, par, kind):
    while node in par:
        node = par[node]
        if isinstance(node, kind):
            return node
    return None


def test_package_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        tree = ast.parse(open(path).read())
        assert all(mod != "oracle" for _, mod in _imports(tree)), path


def test_oracle_imports_neither_the_package_nor_native_code():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        tree = ast.parse(open(path).read())
        mods = {mod for _, mod in _imports(tree)}
        assert "sparse_attention_prolog_gb300" not in mods, path
        assert "ctypes" not in mods and "torch" not in mods, path


def test_cuda_sources_do_not_mention_the_oracle():
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*")):
        assert "oracle" not in open(path).read().lower(), path


def test_bench_and_entry_reach_the_oracle_only_from_their_baseline_code():
    allowed = {
        "bench.py": {"oracle_step", "run_act_quant", "run_int8_gemm", "run_mhc", "run_mla", "prolog_cpu_baseline",
                     "prefill_cpu_baseline", "ragged_cpu_baseline", "dia_cpu_baseline",
                     "int8_gemm_tc_cpu_baseline"},
        "__graft_entry__.py": {"smoke"},
    }
    for name, fns in allowed.items():
        tree = ast.parse(open(os.path.join(ROOT, name)).read())
        par = _parents(tree)
        for node, mod in _imports(tree):
            if mod != "oracle":
                continue
            fn = _enclosing(node, par, ast.FunctionDef)
            assert fn is not None and fn.name in fns, f"{name}:{node.lineno}"
            if fn.name.startswith("run_"):  # a standalone-operator bench: only its CPU-baseline branch
                cond = _enclosing(node, par, ast.If)
                assert cond is not None and "no_cpu_baseline" in ast.unparse(cond.test), f"{name}:{node.lineno}"
