"""The product path and the oracle share no code: neither imports, includes
or loads the other, and the one module both use (the seeded input
generator) holds none of the attention arithmetic.  Checked statically on
the sources."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "exact_attention_39_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(folder, exts):
    for dirpath, _, files in os.walk(folder):
        if "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith(exts):
                path = os.path.join(dirpath, f)
                with open(path, encoding="utf-8") as fh:
                    yield path, fh.read()


def test_product_never_touches_the_oracle():
    found = []
    for path, src in _sources(PKG, (".py", ".cu", ".cuh", ".h")):
        if re.search(r"^\s*(import|from)\s+oracle\b", src, re.M) or \
                re.search(r"#\s*include\s*[<\"][^>\"]*oracle", src) or \
                "liboracle" in src or "attn_oracle" in src:
            found.append(path)
    assert not found, found


def test_oracle_never_touches_the_product():
    found = []
    for path, src in _sources(ORACLE, (".py", ".c", ".h")):
        if re.search(r"^\s*(import|from)\s+exact_attention_39_gb300\b", src, re.M) or \
                re.search(r"#\s*include\s*[<\"][^>\"]*(fa\.h|fa_\w+\.cuh|ptx\.cuh)", src) or \
                "libfa_sm103" in src or "csrc" in src:
            found.append(path)
    assert not found, found


def test_input_generator_holds_no_attention_arithmetic():
    with open(os.path.join(PKG, "workloads.py"), encoding="utf-8") as fh:
        src = fh.read()
    code = re.sub(r'"""(.|\n)*?"""', "", src)          # docstrings may name the op
    code = "\n".join(line.split("#", 1)[0] for line in code.splitlines())
    for word in ("softmax", "logsumexp", "matmul", "einsum", ".exp(", "exp2", " @ ",
                 "import oracle", "binding"):
        assert word not in code, word
