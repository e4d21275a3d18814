"""The oracle and the CUDA path share no code (no GPU needed): nothing in the
package imports, includes or loads the oracle, and the oracle neither
includes the kernels' headers nor names the package or its library."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_wise_kv_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(top, exts):
    for dirpath, dirnames, files in os.walk(top):
        dirnames[:] = [d for d in dirnames if not d.startswith(("_", "."))]
        for f in files:
            if f.endswith(exts):
                path = os.path.join(dirpath, f)
                with open(path, encoding="utf-8") as fh:
                    yield os.path.relpath(path, ROOT), fh.read()


def test_package_never_uses_the_oracle():
    uses = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b)|oracle/|\borc_\w+\(|liboracle", re.M)
    for rel, text in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        assert not uses.search(text), rel


def test_oracle_never_uses_the_package():
    uses = re.compile(r"block_wise_kv_gb300|csrc/|libdllm|#include\s+\"(sm103|kernels|attn_common|norm|tmap)\.cuh\"|"
                      r"#include\s+\"dllm\.h\"")
    for rel, text in _sources(ORACLE, (".py", ".cpp", ".h", ".c")):
        assert not uses.search(text), rel


def test_bench_and_smoke_load_the_oracle_only_in_their_cpu_legs():
    """bench.py loads the oracle only for its CPU baseline / reference arm, and the package's
    entry point only in build() (which compiles it) and smoke(): imports of it sit inside
    those functions, never at module level."""
    for rel in ("bench.py", "__graft_entry__.py"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            text = fh.read()
        top_level = [ln for ln in text.splitlines() if re.match(r"(import\s+oracle|from\s+oracle\b)", ln)]
        assert not top_level, (rel, top_level)
