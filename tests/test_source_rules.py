"""Static checks of the CUDA sources (no GPU needed).

A kernel launched with programmatic stream serialization (`launch_pdl`) may start while
the previous kernel on the stream is still writing its inputs; it must execute
`griddep_wait()` before it reads any memory.  One test finds every kernel that
`launch_pdl` can launch and checks that `griddep_wait();` comes first in its body, with
nothing before it that indexes or dereferences memory.  Another checks the code hash that
keys the committed DRAM-traffic measurements."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "global_causal_gqa_gb300", "csrc")


def _sources():
    out = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, f)) as fh:
                out[f] = fh.read()
    return out


def _strip_comments(src):
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def _pdl_kernels(srcs):
    """Names of the __global__ functions passed to launch_pdl, resolving a local
    `auto kern = ...` that selects among template instances."""
    names = set()
    for text in srcs.values():
        text = _strip_comments(text)
        for m in re.finditer(r"\blaunch_pdl\(\s*([A-Za-z_]\w*)", text):
            arg = m.group(1)
            if arg == "kern":
                # the nearest preceding `auto kern = ...;` in the same file
                defs = [d for d in re.finditer(r"auto\s+kern\s*=([^;]*);", text)
                        if d.start() < m.start()]
                assert defs, "launch_pdl(kern) without a visible definition of kern"
                names |= set(re.findall(r"\b(\w+_kernel)\s*<", defs[-1].group(1)))
            elif arg != "kern" and not arg.startswith("void"):
                names.add(arg)
    return names


def _kernel_body(srcs, name):
    for text in srcs.values():
        text = _strip_comments(text)
        m = re.search(r"__global__[^;{]*?\b" + re.escape(name) + r"\s*\(", text)
        if not m:
            continue
        i = text.index("{", m.end())
        depth, j = 0, i
        while True:
            if text[j] == "{":
                depth += 1
            elif text[j] == "}":
                depth -= 1
                if depth == 0:
                    return text[i + 1:j]
            j += 1
    raise AssertionError(f"kernel {name} not found")


def test_pdl_kernels_found():
    names = _pdl_kernels(_sources())
    assert {"kv_append_kernel", "decode_partial_kernel", "decode_combine_kernel"} <= names


@pytest.mark.parametrize("name", sorted(_pdl_kernels(_sources())))
def test_pdl_kernel_waits_before_reading(name):
    body = _kernel_body(_sources(), name)
    k = body.find("griddep_wait();")
    assert k >= 0, f"{name} is launched by launch_pdl but never calls griddep_wait()"
    before = body[:k]
    assert "[" not in before and "->" not in before, \
        f"{name} touches memory before griddep_wait(): {before.strip()!r}"


def test_code_hash_ignores_comments_only(tmp_path):
    """The DRAM-traffic records are keyed on the hash of a source's code: a comment or
    blank-line edit keeps it, any code edit changes it."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// head\n__global__ void k(int *p) {\n    p[0] = 1;  // store\n}\n")
    h = bench.code_sha256(str(a))
    a.write_text("/* other\n   words */\n__global__ void k(int *p) {\n\n    p[0] = 1;\n}\n")
    assert bench.code_sha256(str(a)) == h
    a.write_text("__global__ void k(int *p) {\n    p[0] = 2;\n}\n")
    assert bench.code_sha256(str(a)) != h
