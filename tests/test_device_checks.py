"""The range predicates behind the debug library's on-chip offset checks
(csrc/checks.cuh), built for the host with g++ and compared with the plain
integer definition of "inside the region" over boundary and overflow cases.

The checked draft kernel itself runs in tests/test_gpu_faults.py.
"""

import itertools
import os
import random
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "rank_markov_draft_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "checks.cuh"
int main() {
  unsigned a, b, c, d, e;
  char kind;
  while (std::scanf(" %c %u %u %u %u %u", &kind, &a, &b, &c, &d, &e) == 6) {
    if (kind == 's')
      std::printf("%d %u\n", dspark::span_ok(a, b, c) ? 1 : 0, dspark::span_or_first(a, b, c));
    else
      std::printf("%d %u\n", dspark::tmem_span_ok(a, b, c, d, e) ? 1 : 0,
                  dspark::tmem_or_first(a, b, c, d, e));
  }
  return 0;
}
"""

U32 = 2 ** 32


def span_inside(off, length, limit):
    return 0 <= off and off + length <= limit


def tmem_inside(rel, width, lo, hi, lane0):
    lane, col = rel >> 16, rel & 0xFFFF
    return lane == lane0 and lo <= col and col + width <= hi


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = tmp_path_factory.mktemp("checks")
    src, exe = d / "checks_host.cpp", d / "checks_host"
    src.write_text(PROGRAM)
    subprocess.run([cxx, "-std=c++17", "-O1", "-D__host__=", "-D__device__=", "-I", CSRC,
                    str(src), "-o", str(exe)], check=True)

    def run(lines):
        out = subprocess.run([str(exe)], input="\n".join(lines) + "\n", capture_output=True,
                             text=True, check=True).stdout.split("\n")
        return [tuple(int(x) for x in line.split()) for line in out if line.strip()]
    return run


def test_shared_memory_span_predicate(checker):
    rng = random.Random(5)
    limits = [0, 1, 16, 5120, 16384, 98304, 232448, U32 - 1]
    cases = []
    for limit in limits:
        for off, length in itertools.product(
                [0, 1, 15, 16, limit // 2, limit - 16, limit - 1, limit, limit + 1,
                 U32 - 16, U32 - 1], [0, 1, 16, 128, 512, limit, limit + 1, U32 - 1]):
            if 0 <= off < U32 and 0 <= length < U32:
                cases.append((off, length, limit))
    for _ in range(2000):
        limit = rng.randrange(U32)
        cases.append((rng.randrange(U32), rng.randrange(limit + 1), limit))
    got = checker([f"s {o} {n} {m} 0 0" for o, n, m in cases])
    assert len(got) == len(cases)
    for (off, length, limit), (ok, off_used) in zip(cases, got):
        assert ok == int(span_inside(off, length, limit)), (off, length, limit)
        # a failed check redirects the access to the region's start
        assert off_used == (off if ok else 0)


def test_tensor_memory_span_predicate(checker):
    # the draft kernel's regions: accumulators in columns [0, 384), the operand in
    # [384, 512); warps reach the lane quadrant 32 q, the MMA lane 0
    regions = [(0, 384), (384, 512), (0, 512), (100, 100)]
    cases = []
    for (lo, hi), lane0, lane in itertools.product(regions, [0, 32, 64, 96],
                                                    [0, 32, 64, 96, 127, 128]):
        for col, width in itertools.product([0, 1, lo - 1, lo, hi - 64, hi - 32, hi - 8,
                                             hi - 1, hi, hi + 32, 0xFFFF],
                                            [1, 8, 16, 32, 64, 128, 0xFFFF]):
            if 0 <= col <= 0xFFFF:
                cases.append(((lane << 16) | col, width, lo, hi, lane0))
    got = checker([f"t {r} {w} {lo} {hi} {l0}" for r, w, lo, hi, l0 in cases])
    assert len(got) == len(cases)
    for (rel, width, lo, hi, lane0), (ok, rel_used) in zip(cases, got):
        assert ok == int(tmem_inside(rel, width, lo, hi, lane0)), (hex(rel), width, lo, hi, lane0)
        assert rel_used == (rel if ok else (lane0 << 16) | lo)


def test_release_build_compiles_the_checks_away():
    """The release library defines no DSPARK_DEVICE_CHECKS; only the checked twin of
    the draft unit is compiled with it (the build script's flag list)."""
    from rank_markov_draft_gb300 import build
    assert build.CHECKED == "draft.cu" and build.CHECKED in build.SOURCES
    text = open(os.path.join(CSRC, "checks.cuh")).read()
    assert "#ifdef DSPARK_DEVICE_CHECKS" in text
