"""How repops_host_alloc sizes and places a request (csrc/hostmem_plan.h),
compiled as host code with g++ and checked on CPU against the rule it states:
a request of at least a quarter of a huge page becomes whole huge pages at a
huge-page-aligned start inside a reservation one huge page larger; a smaller
request, or any where huge pages are off (huge == base page), whole base pages
at a base-page start; empty and unmappable requests refused; and the aligned
block always lies inside the reservation, head + block + tail covering it."""
import os
import random
import shutil
import subprocess

import pytest

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "verifiable_repops_gemm_gb300", "csrc")

DRIVER = r"""
#include "hostmem_plan.h"
#include <cstdio>
int main() {
    unsigned long long bytes, pg, huge, raw;
    while (std::scanf("%llu %llu %llu %llu", &bytes, &pg, &huge, &raw) == 4) {
        repops::HostAllocPlan p;
        if (!repops::host_alloc_plan(bytes, size_t(pg), size_t(huge), &p)) { std::printf("refused\n"); continue; }
        uintptr_t start; size_t head, tail;
        repops::host_alloc_trim(uintptr_t(raw), p, &start, &head, &tail);
        std::printf("%llu %llu %llu %d %llu %llu %llu\n", (unsigned long long)p.len, (unsigned long long)p.align,
                    (unsigned long long)p.span, int(p.in_huge), (unsigned long long)start,
                    (unsigned long long)head, (unsigned long long)tail);
    }
    return 0;
}
"""

SIZE_MAX = (1 << 64) - 1


@pytest.fixture(scope="module")
def planner(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("hostmem_plan")
    src, exe = d / "drv.cpp", d / "drv"
    src.write_text(DRIVER)
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-I", HEADER_DIR, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "warning" not in r.stderr, r.stderr

    def run(cases):
        inp = "".join("%d %d %d %d\n" % c for c in cases)
        out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True).stdout.split("\n")
        return [None if line == "refused" else tuple(int(x) for x in line.split()) for line in out[:len(cases)]]
    return run


def up(x, u):
    return (x + u - 1) // u * u


def cases():
    rng = random.Random(11)
    out = []
    for pg in (4096, 65536):
        for huge in (pg, 2 << 20, 512 << 20):
            sizes = {1, pg - 1, pg, pg + 1, huge // 4 - 1, huge // 4, huge // 4 + 1, huge - 1, huge, huge + 1,
                     3 * (256 << 20), 1 << 30, (16 << 30) + 17}
            sizes |= {rng.randrange(1, 1 << 36) for _ in range(20)}
            for b in sorted(x for x in sizes if x > 0):
                for _ in range(3):
                    raw = rng.randrange(1 << 20, 1 << 46) // pg * pg
                    out.append((b, pg, huge, raw))
    return out


def test_sizing_and_placement_follow_the_rule(planner):
    cs = cases()
    for (b, pg, huge, raw), got in zip(cs, planner(cs)):
        assert got is not None, (b, pg, huge)
        length, align, span, in_huge, start, head, tail = got
        want_huge = huge > pg and b >= huge // 4
        unit = huge if want_huge else pg
        assert in_huge == int(want_huge), (b, pg, huge)
        assert length == up(b, unit) and length >= b and length - b < unit, (b, pg, huge)
        assert align == unit and span == length + (huge if want_huge else 0), (b, pg, huge)
        # the aligned block lies inside the reservation; nothing is lost
        assert start % align == 0 and raw <= start and start + length <= raw + span, (b, pg, huge, raw)
        assert head + length + tail == span and head % pg == 0 and tail % pg == 0, (b, pg, huge, raw)


def test_empty_and_unmappable_requests_are_refused(planner):
    huge = 512 << 20
    got = planner([(0, 65536, huge, 1 << 30), (SIZE_MAX // 2 - huge + 1, 65536, huge, 1 << 30),
                   (SIZE_MAX, 4096, 4096, 1 << 30), (SIZE_MAX // 2 - huge, 65536, huge, 1 << 30)])
    assert got[0] is None and got[1] is None and got[2] is None
    assert got[3] is not None       # the largest request the rule accepts still plans without overflow
