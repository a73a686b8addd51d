"""The product package and the oracle stay apart.

The oracle is test infrastructure.  The library, its binding and the
workload generators must neither import it nor include or link any of its
sources, so that every parity test compares two independent computations.
Loading the binding must leave no oracle module in the process.
"""
import ast
import pathlib
import re
import subprocess
import sys

ROOT = pathlib.Path(__file__).resolve().parents[1]
PKG = ROOT / "packed_variable_length_varlen_gb300"
ORACLE = ROOT / "oracle"


def _product_files(suffixes):
    return sorted(p for p in PKG.rglob("*") if p.suffix in suffixes and "_build" not in p.parts)


def test_package_python_never_imports_the_oracle():
    files = _product_files({".py"})
    assert files, "no package sources found"
    for f in files:
        tree = ast.parse(f.read_text(), filename=str(f))
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            elif isinstance(node, ast.Call) and getattr(node.func, "id", "") == "__import__":
                names = [getattr(a, "value", "") for a in node.args[:1]]
            else:
                continue
            for n in names:
                assert not str(n).split(".")[0] == "oracle", "%s imports %s" % (f.name, n)


def test_native_sources_never_reach_the_oracle():
    oracle_files = {p.name for p in ORACLE.iterdir() if p.is_file()}
    inc = re.compile(r'^\s*#\s*include\s*[<"]([^">]+)[">]', re.M)
    files = _product_files({".cu", ".cuh", ".h", ".c", ".cc", ".cpp"}) + sorted((ROOT / "include").glob("*.h"))
    assert files, "no native sources found"
    for f in files:
        text = f.read_text()
        for target in inc.findall(text):
            assert "oracle" not in target and pathlib.PurePath(target).name not in oracle_files, \
                "%s includes %s" % (f.name, target)


def test_build_script_compiles_no_oracle_source():
    text = (PKG / "build.py").read_text()
    assert "oracle" not in text
    assert "varlen_oracle" not in text


def test_loading_the_binding_loads_no_oracle_module():
    from packed_variable_length_varlen_gb300 import build
    build.build()
    code = ("import sys\n"
            "import packed_variable_length_varlen_gb300.varlen_attn as va\n"
            "import packed_variable_length_varlen_gb300.workloads\n"
            "bad = sorted(m for m in sys.modules if m == 'oracle' or m.startswith('oracle.'))\n"
            "print(','.join(bad))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "", "oracle modules loaded: " + r.stdout
