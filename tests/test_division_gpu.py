"""The corrected reciprocal quotient used by the per-16 E4M3 fake
quantisation (x / s as rn(x * r) plus one exact-residual correction, r the
hardware's approximate reciprocal of s, or rn(1/6) for the scale itself)
equals the IEEE division for every operand pair it can meet: every finite
bf16 numerator by every positive E4M3 scale and by 6 (the scale's own
divisor), wherever the quotient is below 2^120 (the quantiser's quotients
are at most 9, or below 2^128 / 448 when the scale saturates), except below
2^-60, where the residual may underflow and the quotient be an ulp off; the
E2M1 code taken from the quotient is the same for every pair.  The check
program includes the library's header, so it tests the same function the
kernel runs."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_corrected_quotient_matches_ieee_division(tmp_path):
    exe = tmp_path / "div_check"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "fp4_sparse_attention_fp4idx_gb300", "csrc"),
                    "-o", str(exe), os.path.join(ROOT, "tests", "cuda", "div_check.cu")],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    first = out.splitlines()[0].split()
    assert first[0::2] == ["checked", "mismatches", "skipped", "tiny", "codes", "packed"], out
    checked, bad, skipped, tiny, codes, packed = (int(x) for x in first[1::2])
    assert checked + skipped == 127 * 65536, out
    # every finite numerator by 6, and most pairs by the E4M3 scales
    assert checked > 120 * 65536, out
    assert bad == tiny, out  # quotients differ only below 2^-60
    assert codes == 0, out
    assert packed == 0, out  # the f32x2 form the kernel runs gives the same quotients
    print(out.splitlines()[0])
