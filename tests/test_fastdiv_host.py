"""The multiply-and-shift division the kernels use to decode their work items
(csrc/fastdiv.h), checked on the CPU against C++'s own integer division: a
small program built with the host compiler from the same header runs every
divisor up to 4096, the divisors around each power of two and seeded large
ones, against numerators at and around every multiple boundary and at the
top of the range."""
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "attention_variant_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <initializer_list>
#include "fastdiv.h"

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint32_t next_u32() { // xorshift64*
    state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
    return uint32_t((state * 0x2545F4914F6CDD1Dull) >> 32);
}

static long bad = 0, checked = 0;
static void check(int32_t n, const fl::FastDiv &f) {
    if (n < 0) return;
    ++checked;
    if (fl::fast_div(n, f) != n / f.d) {
        if (bad < 5) std::printf("mismatch n=%d d=%d got %d\n", n, f.d, fl::fast_div(n, f));
        ++bad;
    }
}

static void divisor(int32_t d) {
    const fl::FastDiv f = fl::make_fastdiv(d);
    if (f.m < 0x80000000u) { std::printf("multiplier below 2^31 for d=%d\n", d); ++bad; }
    const int32_t top = 0x7fffffff;
    for (int32_t n : {0, 1, d - 1, d, d + 1, top, top - 1, top - d, top - d + 1}) check(n, f);
    // around the multiples near the top of the range and at seeded places
    const int32_t q_top = top / d;
    for (int32_t q = q_top; q > q_top - 4 && q >= 0; --q)
        for (int32_t e = -1; e <= 1; ++e) check(int32_t(int64_t(q) * d + e), f);
    for (int i = 0; i < 64; ++i) {
        const int32_t q = int32_t(next_u32() % uint32_t(q_top + 1));
        for (int32_t e = -1; e <= 1; ++e) check(int32_t(int64_t(q) * d + e), f);
        check(int32_t(next_u32() >> 1), f);
    }
}

int main() {
    for (int32_t d = 1; d <= 4096; ++d) divisor(d);
    for (int s = 1; s < 31; ++s)
        for (int32_t e = -2; e <= 2; ++e) {
            const int64_t d = (int64_t(1) << s) + e;
            if (d >= 1 && d < (int64_t(1) << 31)) divisor(int32_t(d));
        }
    divisor(0x7fffffff);
    for (int i = 0; i < 2000; ++i) divisor(int32_t((next_u32() >> 1) | 1u));
    // small numerators exhaustively for the divisors the kernels meet most
    for (int32_t d : {1, 2, 3, 5, 7, 8, 16, 64, 112, 128, 152, 1024})
        for (int32_t n = 0; n < (1 << 20); ++n) check(n, fl::make_fastdiv(d));
    std::printf("checked %ld bad %ld\n", checked, bad);
    return bad == 0 ? 0 : 1;
}
"""


def test_fast_division_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "fastdiv_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
