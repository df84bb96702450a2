"""The quantizer kernels' division method, checked on the host (no GPU): one
FMA correction of the reciprocal product gives the correctly rounded IEEE
quotient (Markstein's theorem) in the domain the kernels use it in (scales in
[2^-80, 2^100], quotients of 2^-12 and up: every one that can give a nonzero
FP8 or E2M1 code), on 2 * 10^7 seeded pairs, all-ones and all-zero
significands included.  The C file is compiled without contraction, so only the explicit
fmaf calls fuse."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("seed", [1, 2])
def test_fma_corrected_quotient_is_correctly_rounded(tmp_path, seed):
    exe = tmp_path / "fma_quotient_check"
    subprocess.run(["cc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe),
                    os.path.join(HERE, "fma_quotient_check.c"), "-lm"], check=True)
    out = subprocess.run([str(exe), "10000000", str(seed)], check=True, capture_output=True, text=True).stdout
    assert int(out.strip()) == 0
