"""The identity the fp8 dispatch kernels quantise bf16 rows with: one
remainder correction of RN(x * RN(1/scale)) gives RN(x / scale) for every
bf16 x and every binary32 scale in [2^-60, 2^60] (tests/quotient_check.c).

The CPU run here covers a sample of scale significands at nine exponents
(every 2^14-th: 512 per exponent, 1.6e8 cases, a few seconds); the full run
(step 1) covers every binary32 significand.  Two controls must fail, so that
the check is seen to detect a wrong result: the uncorrected product, and the
steps run on +x (which turn x = -0 into +0)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(tmp_path, *args):
    exe = tmp_path / "quotient_check"
    subprocess.run([shutil.which("gcc") or "gcc", "-O2", "-ffp-contract=off", "-std=c11",
                    os.path.join(HERE, "quotient_check.c"), "-o", str(exe), "-lm"], check=True)
    out = subprocess.run([str(exe), *args], check=True, capture_output=True, text=True).stdout.split()
    return {out[i]: int(out[i + 1]) for i in range(0, len(out), 2)}


@pytest.fixture(scope="module")
def tmp(tmp_path_factory):
    return tmp_path_factory.mktemp("quot")


def test_corrected_quotient_is_exact(tmp):
    r = _run(tmp, "16384")
    assert r["cases"] > 100_000_000
    assert r["exact_mismatches"] == 0 and r["small_failures"] == 0, r


def test_uncorrected_product_is_detected(tmp):
    r = _run(tmp, "65536", "nocorr")
    assert r["exact_mismatches"] > 0, r


def test_lost_zero_sign_is_detected(tmp):
    r = _run(tmp, "65536", "unsigned")
    assert r["small_failures"] > 0 and r["exact_mismatches"] == 0, r
