"""The write kernels divide their scales by constants (127, 448, 7 for the
per-token-head scales of max(amax, 1e-8); 15 and 3 for KVarN's max - min) with
Markstein's correction step instead of an IEEE division.  This checks, on the
CPU and over every fp32 input of each range, that the result equals the IEEE
quotient.  CPU only; about a minute."""
import os
import platform
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def test_constant_division_is_the_ieee_quotient_for_every_input():
    src = os.path.join(HERE, "c", "const_division_check.c")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "check")
        flags = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]
        if platform.machine() in ("x86_64", "AMD64"):
            flags.append("-mfma")             # a hardware fused multiply-add for fmaf
        subprocess.run(["gcc", *flags, "-o", exe, src, "-lm"], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=900).stdout
    rows = [line.split() for line in out.splitlines() if line.strip()]
    assert [float(r[0]) for r in rows] == [127.0, 448.0, 7.0, 15.0, 3.0]
    for d, first, bad in rows:
        assert int(bad) == 0, f"x / {d} from {first}: {bad} inputs differ from the IEEE quotient"
