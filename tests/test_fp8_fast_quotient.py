"""The FP8 dispatch kernel computes the group scale amax/448 and divides by
it with one multiply and two fused multiply-adds each (Markstein's
correction with the correctly rounded reciprocal) instead of a full IEEE
division.  This checks, on the CPU with IEEE fmaf, that the scale equals the
IEEE quotient for every finite bf16 amax, and that the E4M3 code of each
quotient equals the code of the IEEE quotient for every bf16 x and bf16
amax >= 2^-60 with |x| <= amax (every fourth amax here; the stride-1 run
covers ~1e9 pairs)."""
import os
import subprocess

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("stride", [4])
def test_fast_quotient_gives_ieee_e4m3_codes(tmp_path, stride):
    exe = tmp_path / "fp8_quotient_check"
    src = os.path.join(HERE, "fp8_quotient_check.c")
    oracle_src = os.path.join(os.path.dirname(HERE), "oracle", "ep_oracle.c")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-o", str(exe), src, oracle_src, "-lm"],
                   check=True, capture_output=True)
    r = subprocess.run([str(exe), str(stride)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    words = r.stdout.split()
    pairs, bad, scale_bad = words[1], words[3], words[5]
    assert int(bad) == 0 and int(scale_bad) == 0 and int(pairs) > 2e8
