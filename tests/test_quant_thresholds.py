"""The page kernel's 2-bit decision thresholds against the quantizer's definition, on the CPU.

tests/host/threshold_check.cu includes the kernel's own threshold code (kvq::qthr in
kvq_quantizer.cuh, host-compiled) and checks, for 4000 groups of 32 fp16 values from eight
distributions (standard normal, an outlier channel, subnormal and tiny ranges, magnitudes up to
the fp16 maximum, all-negative groups, powers of two of both signs), that every fp16 value between
a group's minimum and maximum gets the same code from the thresholds as from
clamp(rint(fl(fl(x - z) / s)), 0, 3) in plain fp32 -- about 10^8 values; and that the division of
a group's range by L = 3, 7, 15 (a rounded reciprocal product with one exact-remainder correction)
equals the IEEE division for every significand of a binade and every subnormal quotient.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_thresholds_give_the_exact_codes(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = tmp_path / "threshold_check"
    src = os.path.join(ROOT, "tests", "host", "threshold_check.cu")
    csrc = os.path.join(ROOT, "bit_asymmetric_kv_kvq_gb300", "csrc")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-Xcompiler", "-ffp-contract=off", "-I", csrc, "-I",
                    os.path.join(ROOT, "include"), "-o", str(exe), src], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("checked ")
