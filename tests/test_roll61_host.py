"""The rolling hash's modular helpers (csrc/roll61.cuh), compiled as host code.

The kernels' arithmetic modulo the Mersenne prime P = 2^61 - 1 replaces the
products by the base B = 2^32 + 15 with 61-bit rotations and folds each step's
sum once.  These functions are __host__ __device__, so g++ can build them with
the CUDA qualifiers defined away; the results are checked against Python's
exact integers: (h*B + w) mod P for a Horner step and (h*B - w_out*B^W + w_in)
mod P for a window slide, on seeded random residues and on the extremes
(0, 1, P - 1, words 0 and 2^32 - 1) where the unreduced sums are largest.
"""
import os
import random
import shutil
import subprocess

import pytest

P = (1 << 61) - 1
B = (1 << 32) + 15
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "verifiable_repops_gemm_gb300", "csrc", "roll61.cuh")

DRIVER = r"""
#define __host__
#define __device__
#define __forceinline__ inline
#include "roll61.cuh"
#include <cstdio>
#include <cstring>
#include <cinttypes>
#include <vector>
int main(int argc, char **argv) {
    unsigned long long h, wo, wi, bw;
    if (argc > 1 && std::strcmp(argv[1], "row") == 0) {
        // W, B^W mod P, n, then n words: every window's hash, Horner then slides
        unsigned long long W, n;
        if (std::scanf("%llu %llu %llu", &W, &bw, &n) != 3) return 1;
        std::vector<uint32_t> w(n);
        for (auto &x : w) { unsigned long long v; if (std::scanf("%llu", &v) != 1) return 1; x = uint32_t(v); }
        h = 0;
        for (unsigned long long k = 0; k < W; ++k) h = repops::roll61::push(h, w[k]);
        std::printf("%" PRIu64 "\n", uint64_t(h));
        for (unsigned long long i = 1; i + W <= n; ++i) {
            h = repops::roll61::slide(h, w[i - 1], w[i + W - 1], bw);
            std::printf("%" PRIu64 "\n", uint64_t(h));
        }
        return 0;
    }
    while (std::scanf("%llu %llu %llu %llu", &h, &wo, &wi, &bw) == 4)
        std::printf("%" PRIu64 " %" PRIu64 "\n", repops::roll61::push(h, uint32_t(wi)),
                    repops::roll61::slide(h, uint32_t(wo), uint32_t(wi), bw));
    return 0;
}
"""


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    d = tmp_path_factory.mktemp("roll61")
    src = d / "drv.cpp"
    src.write_text(DRIVER)
    exe = d / "drv"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    return str(exe)


def _cases():
    rng = random.Random(61)
    hs = [0, 1, 2, P - 1, P - 2, 1 << 60, (1 << 32) - 1, 1 << 32]
    ws = [0, 1, (1 << 32) - 1, 1 << 31]
    bws = [0, 1, P - 1, B, (1 << 32) - 1, 1 << 32]
    out = [(h, wo, wi, bw) for h in hs for wo in ws for wi in ws for bw in bws]
    for _ in range(20000):
        out.append((rng.randrange(P), rng.randrange(1 << 32), rng.randrange(1 << 32), rng.randrange(P)))
    return out


def test_push_and_slide_match_exact_integers(helper):
    cases = _cases()
    text = "\n".join("%d %d %d %d" % c for c in cases) + "\n"
    res = subprocess.run([helper], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
    assert len([r for r in res if r]) == len(cases)
    for (h, wo, wi, bw), line in zip(cases, res):
        push, slide = (int(x) for x in line.split())
        assert push == (h * B + wi) % P
        assert slide == (h * B - wo * bw + wi) % P


def test_rolled_row_equals_horner_of_every_window(helper):
    # a row rolled with push() then slide() gives every window's value of the
    # definition sum_t w[i+t] * B^(W-1-t) mod P; B^W from pow()
    rng = random.Random(7)
    row = [rng.choice([0, (1 << 32) - 1, rng.randrange(1 << 32)]) for _ in range(400)]
    for W in (1, 2, 5, 32, 100, 400):
        text = "%d %d %d\n%s\n" % (W, pow(B, W, P), len(row), " ".join(map(str, row)))
        got = [int(x) for x in subprocess.run([helper, "row"], input=text, capture_output=True, text=True,
                                              check=True).stdout.split()]
        want = [sum(row[i + t] * pow(B, W - 1 - t, P) for t in range(W)) % P for i in range(len(row) - W + 1)]
        assert got == want
