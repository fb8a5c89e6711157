"""Static rules of the device code, checked on the sources (no GPU):
nothing that traps, no multicast, the Blackwell tensor-core path only, and
every poll of an mbarrier bounded by the global timer."""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "exact_attention_39_gb300", "csrc")


def _strip_comments(src):
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return "\n".join(line.split("//", 1)[0] for line in src.splitlines())


def _sources():
    out = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
                out[f] = _strip_comments(fh.read())
    return out


@pytest.mark.parametrize("pattern", [r"__trap", r"\btrap\s*;", r"\bbrkpt\b",
                                     r"(?<!static_)\bassert\s*\(", r"multicast",
                                     r"\bwgmma\b", r"\bmma\.sync\b", r"\bwmma\b"])
def test_forbidden_device_constructs_absent(pattern):
    hits = [f for f, src in _sources().items() if re.search(pattern, src)]
    assert not hits, (pattern, hits)


def test_tensor_core_and_tma_path_present():
    src = "\n".join(_sources().values())
    for needle in ("tcgen05.mma", "tcgen05.alloc", "tcgen05.ld", "cp.async.bulk.tensor",
                   "mbarrier.try_wait"):
        assert needle in src, needle


def _functions_calling(src, callee):
    """Bodies (brace-matched) of the functions whose body calls ``callee``."""
    bodies = []
    for m in re.finditer(r"\)\s*(?:const\s*)?\{", src):
        depth, i = 0, m.end() - 1
        while i < len(src):
            depth += {"{": 1, "}": -1}.get(src[i], 0)
            if depth == 0:
                break
            i += 1
        body = src[m.end():i]
        if callee in body:
            bodies.append(body)
    return bodies


def test_every_mbarrier_poll_is_bounded_by_the_global_timer():
    # The PTX wrapper itself is one try_wait; every loop around it lives in
    # a function that reads %globaltimer and gives up after timeout_ns.
    loops = 0
    for f, src in _sources().items():
        if f == "ptx.cuh":
            continue
        for body in _functions_calling(src, "mbar_try_wait("):
            # a block that polls in a loop must carry the time limit with it
            if re.search(r"for\s*\(|while\s*\(", body):
                loops += 1
                assert "globaltimer_ns()" in body and "timeout_ns" in body, body[:200]
    assert loops >= 2
    # no other unbounded loop form anywhere in the device code
    for f, src in _sources().items():
        for m in re.finditer(r"for\s*\(\s*;\s*;\s*\)|while\s*\(\s*(true|1)\s*\)", src):
            tail = src[m.end():m.end() + 400]
            assert "globaltimer_ns()" in tail and "timeout_ns" in tail, (f, tail[:200])
