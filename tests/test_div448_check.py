"""The identity the fp8 kernels compute a block's scale with: amax / 448
rounded to nearest from one multiply and one remainder correction, equal to
IEEE division for every binary32 amax in [2^-120, FLT_MAX]
(tests/div448_check.c; the full run, step 1, covers all 2.08e9 values).

Here a sample (every 4096th bit pattern); the uncorrected product must fail
(the check can see a wrong quotient), and so must the method below 2^-120,
where the kernels divide instead."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    out = tmp_path_factory.mktemp("div448") / "div448_check"
    subprocess.run([shutil.which("gcc") or "gcc", "-O2", "-ffp-contract=off", "-std=c11",
                    os.path.join(HERE, "div448_check.c"), "-o", str(out), "-lm"], check=True)
    return str(out)


def _run(exe, *args):
    out = subprocess.run([exe, *args], check=True, capture_output=True, text=True).stdout.split()
    return {out[i]: int(out[i + 1]) for i in range(0, len(out), 2)}


def test_corrected_product_is_ieee_division(exe):
    r = _run(exe, "4096")
    assert r["cases"] > 500_000 and r["mismatches"] == 0, r


def test_uncorrected_product_is_detected(exe):
    assert _run(exe, "4096", "nocorr")["mismatches"] > 0


def test_method_fails_below_its_range(exe):
    assert _run(exe, "16", "below")["mismatches"] > 0
