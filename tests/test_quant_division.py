"""The GPU quantizer divides by the tile scale with a correctly rounded
reciprocal and one FMA residual correction instead of a full IEEE divide.
Inputs are bf16, so the method is checked here against IEEE division for
every (amax, x) pair with |x| <= amax and amax >= 2^-90 (the range where the
kernel uses it; smaller tiles take the IEEE divide), and the tile scale
amax / 448 (constant reciprocal plus one correction) for every finite bf16
amax. The GPU parity tests
then confirm the codes bit for bit against the oracle."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_reciprocal_division_matches_ieee_for_all_bf16_pairs(tmp_path):
    exe = tmp_path / "quant_division_check"
    src = os.path.join(HERE, "csrc", "quant_division_check.c")
    # -ffp-contract=off keeps each step a separately rounded fp32 operation;
    # fmaf is the correctly rounded C99 fused multiply-add.
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
                    "-o", str(exe), src, "-lm"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    pairs, bad, scale_bad = int(out[0]), int(out[1]), int(out[2])
    assert pairs > 1_000_000_000
    assert bad == 0
    assert scale_bad == 0
