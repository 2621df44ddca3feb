"""The router's softmax arithmetic: float-float (binary32 pairs) with a
table-driven Cody-Waite reduced exponential gives every weight within one fp32 ulp
of RN32 of the binary64 softmax, which is what the oracle computes
(tests/router_ff_check.c restates the kernel's steps in C with fmaf).

The exponential is checked on every 997th binary32 argument in [-64, 0] and
on 2.4e6 differences of random logits (relative error about 2^-36), and the
weights on 3e5 random rows with K = 1..32 (a few seconds).  Two controls must
fail, so that the check is seen to detect a wrong result: a reduction by the
leading part of ln 2 alone, and a sum of the exponentials in binary32."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    out = tmp_path_factory.mktemp("rff") / "router_ff_check"
    subprocess.run([shutil.which("gcc") or "gcc", "-O2", "-ffp-contract=off", "-std=c11",
                    os.path.join(HERE, "router_ff_check.c"), "-o", str(out), "-lm"], check=True)
    return out


def _run(exe, *args):
    out = subprocess.run([str(exe), *args], check=True, capture_output=True, text=True).stdout.split()
    return {out[i]: float(out[i + 1]) for i in range(0, len(out), 2)}


def _weights(rows):
    return rows * 16.5          # K uniform in 1..32


def test_float_float_softmax_within_one_ulp(exe):
    r = _run(exe, "997", "300000")
    assert r["exp_cases"] > 3_000_000
    assert r["exp_err_log2"] < -35, r
    assert r["ulp2plus"] == 0, r
    assert r["ulp1"] <= 1e-3 * _weights(r["rows"]), r


@pytest.mark.parametrize("ulps", [-2, -1, 1, 2])
def test_quotient_independent_of_reciprocal_error(exe, ulps):
    """The kernel's 1/S_h comes from the approximate reciprocal: with y
    moved by up to 2 ulps from RN(1/S_h) the weights stay within one ulp,
    at the same rate."""
    r = _run(exe, "9973", "300000", f"rcp{ulps}")
    assert r["ulp2plus"] == 0, r
    assert r["ulp1"] <= 1e-3 * _weights(r["rows"]), r


def test_reduction_without_low_parts_is_detected(exe):
    r = _run(exe, "9973", "100000", "noL2")
    assert r["exp_err_log2"] > -20 and r["ulp2plus"] > 0, r


def test_binary32_sum_is_detected(exe):
    r = _run(exe, "9973", "300000", "f32sum")
    assert r["ulp1"] > 1e-2 * _weights(r["rows"]), r
