"""CPU proofs behind the quantizer's division shortcuts in the library: the
division by 127 of the group scale, by Markstein's correction step from the
correctly rounded reciprocal RN(1/127), equals the IEEE quotient for every
finite non-negative binary32 (exhaustive; the device uses the same IEEE
binary32 operations, so the result carries over).  The GPU tests compare the
device helpers with __fdiv_rn directly."""
import os
import subprocess



from conftest import ROOT


def test_div127_markstein_is_the_ieee_quotient_everywhere(tmp_path):
    exe = str(tmp_path / "div127")
    src = os.path.join(ROOT, "tests", "csrc", "div127_check.c")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-o", exe, src, "-lm"], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=900).stdout.split()
    assert out[0] == "0", f"{out[0]} mismatches, first at bits {out[1]}"
