"""The multiply-shift division by invariant divisors (csrc/fastdiv.h) that the
one-kernel decode layer uses for its work shares and chunk cursors: checked
against plain integer division over the divisors and numerators the kernel can
see (Granlund and Montgomery, "Division by Invariant Integers using
Multiplication", PLDI 1994, unsigned case).  Host build of the same header."""
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(__file__), "..", "bit_quantized_expert_moe_gb300", "csrc")

PROG = r"""
#include "fastdiv.h"
#include <cstdio>
int main() {
    unsigned long long bad = 0, n = 0;
    for (uint32_t d = 1; d <= 4096; ++d) {
        const moe::FastDiv f = moe::make_fastdiv(d);
        for (uint32_t x = 0; x < 20000; ++x, ++n) bad += moe::fd_div(x, f) != x / d;
        for (uint32_t x = 0x7FFFFFFFu - 20000; x < 0x7FFFFFFFu; ++x, ++n) bad += moe::fd_div(x, f) != x / d;
        uint32_t r = 0;
        const uint32_t q = moe::fd_divmod(123456789u, f, &r);
        bad += (q != 123456789u / d) || (r != 123456789u % d);
    }
    // large divisors (grid sizes times work, feature counts)
    for (uint32_t d = 4097; d < (1u << 30); d = d * 3 + 7) {
        const moe::FastDiv f = moe::make_fastdiv(d);
        for (uint32_t x = 0; x < 0x7FFFFFFFu - 1000003u; x += 1000003u, ++n) bad += moe::fd_div(x, f) != x / d;
    }
    std::printf("%llu %llu\n", n, bad);
    return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_fastdiv_matches_integer_division(tmp_path):
    src = tmp_path / "fd.cpp"
    exe = tmp_path / "fd"
    src.write_text(PROG)
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    n, bad = map(int, out.stdout.split())
    assert out.returncode == 0 and bad == 0 and n > 10_000_000
