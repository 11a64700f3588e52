"""Host check of the multiply-shift division the kernels use for run-time
divisors (FastDiv in csrc/lsa_internal.h: Granlund and Montgomery, "Division
by invariant integers using multiplication").  The header is compiled as
host C++ and every quotient is compared with exact integer division: all
divisors up to 4096 against boundary and random dividends, then large and
power-of-two divisors.  The device form differs only in taking the high
32 bits with __umulhi, which is the same product's upper half.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

SRC = r"""
#include <cstdio>
#include <cstdint>
#include "lsa_internal.h"
using namespace lsa;
static uint64_t state = 0x9e3779b97f4a7c15ull;
static uint32_t rnd() { state ^= state << 13; state ^= state >> 7; state ^= state << 17; return (uint32_t)state; }
static long bad = 0, checked = 0;
static void check(uint32_t d, uint32_t x, const FastDiv &f) {
    ++checked;
    const uint32_t q = fdiv(x, f), r = fmodu(x, f);
    if (q != x / d || r != x % d) { if (bad < 5) printf("d=%u x=%u q=%u r=%u\n", d, x, q, r); ++bad; }
}
static void divisor(uint32_t d, int nrand) {
    const FastDiv f = make_fastdiv(d);
    if (f.d != d) { printf("d=%u stored %u\n", d, f.d); ++bad; }
    const uint32_t top = 0x7fffffffu;
    for (uint32_t x = 0; x < 2048; ++x) check(d, x, f);
    for (uint32_t k = 0; k < 64; ++k) { check(d, top - k, f); }
    for (uint64_t m = d; m <= top; m += (uint64_t)d * 977 + 1) { check(d, (uint32_t)m, f); if (m) check(d, (uint32_t)m - 1, f); }
    for (uint64_t q = 1; q * d <= top; q *= 3) { check(d, (uint32_t)(q * d), f); check(d, (uint32_t)(q * d - 1), f); }
    for (int i = 0; i < nrand; ++i) check(d, rnd() & top, f);
}
int main() {
    for (uint32_t d = 1; d <= 4096; ++d) divisor(d, 200);
    for (int i = 0; i < 2000; ++i) divisor((rnd() & 0x7fffffffu) | 1u, 200);
    for (int l = 0; l < 31; ++l) { divisor(1u << l, 500); divisor((1u << l) + 1, 500); if (l > 1) divisor((1u << l) - 1, 500); }
    divisor(0x7fffffffu, 2000);
    printf("checked %ld bad %ld\n", checked, bad);
    return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                    reason="needs g++ and the CUDA headers")
def test_fastdiv_matches_integer_division(tmp_path):
    src = tmp_path / "fastdiv.cpp"
    src.write_text(SRC)
    exe = tmp_path / "fastdiv"
    csrc = os.path.join(ROOT, "sparse_attention_decode_block_gb300", "csrc")
    subprocess.run(["g++", "-O2", "-std=c++17", "-I" + csrc, "-I" + CUDA_INC, "-I" + os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    print(r.stdout, file=sys.stderr)
    assert r.returncode == 0, r.stdout
    assert "bad 0" in r.stdout
