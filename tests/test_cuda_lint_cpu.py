"""Source checks of the CUDA kernels, on CPU. A full-mask warp collective (shuffle,
ballot, match, reduction, __syncwarp) needs every lane of the warp; inside a loop whose
index starts at the lane (`for (int v = lane; v < n; v += 32)`), the lanes without an
item in the last pass skip it and the result is undefined. Every such collective must
sit outside those loops."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "expert_token_dispatch_gemm_b300", "csrc")
COLLECTIVE = re.compile(r"__(shfl\w*_sync|ballot_sync|match_any_sync|match_all_sync|"
                        r"reduce_\w+_sync|any_sync|all_sync|syncwarp)\s*\(")
LANE_LOOP = re.compile(r"for\s*\(\s*(?:int|unsigned|int64_t|size_t)?\s*\w+\s*=\s*lane\b[^;]*;")


def strip_comments(src):
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def loop_body(src, start):
    """The text of the loop statement beginning at `start` (a `for (`): its braced body,
    or its single statement."""
    i = src.index("(", start)
    depth = 0
    while True:                      # the loop header's parentheses
        if src[i] == "(":
            depth += 1
        elif src[i] == ")":
            depth -= 1
            if depth == 0:
                break
        i += 1
    j = i + 1
    while src[j].isspace():
        j += 1
    if src[j] != "{":
        return src[j:src.index(";", j) + 1]
    depth = 0
    k = j
    while True:
        if src[k] == "{":
            depth += 1
        elif src[k] == "}":
            depth -= 1
            if depth == 0:
                return src[j:k + 1]
        k += 1


def lane_loop_collectives(src):
    src = strip_comments(src)
    found = []
    for m in LANE_LOOP.finditer(src):
        body = loop_body(src, m.start())
        for c in COLLECTIVE.finditer(body):
            found.append((src.count("\n", 0, m.start()) + 1, c.group(0)))
    return found


def test_the_check_finds_a_collective_in_a_lane_loop():
    bad = """for (int v = lane; v < nvec; v += 32) {
        const int s = __shfl_sync(0xffffffffu, my_slot, j);
    }"""
    good = """const int s = __shfl_sync(0xffffffffu, my_slot, j);
    for (int v = lane; v < nvec; v += 32) acc += s;"""
    assert lane_loop_collectives(bad) and not lane_loop_collectives(good)


@pytest.mark.parametrize("name", sorted(n for n in os.listdir(CSRC) if n.endswith((".cu", ".cuh"))))
def test_no_warp_collective_inside_a_lane_indexed_loop(name):
    assert lane_loop_collectives(open(os.path.join(CSRC, name)).read()) == []
