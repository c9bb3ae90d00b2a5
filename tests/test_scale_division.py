"""The group scale fl32(max(amax, 1e-10) / 448) is computed on the GPU without
a division (a corrected reciprocal product, see csrc/bfp8_e4m3.cuh div448).
Pinned here exhaustively: for every fp32 value in the scale's domain the
method equals the IEEE quotient (host division, correctly rounded).  The GPU
quantisation tests then check the codes and scales bit for bit against the
oracle's IEEE division."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_corrected_reciprocal_equals_ieee_division_on_every_scale(tmp_path):
    exe = tmp_path / "div448_check"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe),
                    os.path.join(HERE, "helpers", "div448_check.c"), "-lm"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
