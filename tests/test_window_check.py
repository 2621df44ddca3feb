"""The bracketing window the activation kernel quantises fp32 values with
(tests/window_check.c): where RN(x RN(r(1 - 2^-20))) and RN(x RN(r(1 + 2^-20)))
give the same E4M3 byte, r = RN(1/scale), that byte is e4m3(RN(x / scale)).
fp32 inputs cannot be enumerated, so the check samples 2e6 pairs, half of
them on or next to E4M3 midpoints.  A control (no window: both ends at r)
must produce wrong bytes, and the checker's own E4M3 encoder is compared
with torch's float8_e4m3fn cast first."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    out = tmp_path_factory.mktemp("window") / "window_check"
    subprocess.run([shutil.which("gcc") or "gcc", "-O2", "-ffp-contract=off", "-std=c11",
                    os.path.join(HERE, "window_check.c"), "-o", str(out), "-lm"], check=True)
    return str(out)


def _run(exe, *args):
    out = subprocess.run([exe, *args], check=True, capture_output=True, text=True).stdout.split()
    return {out[i]: int(out[i + 1]) for i in range(0, len(out), 2)}


def test_encoder_matches_torch(exe):
    bits = np.arange(65536, dtype=np.uint32) << 16                 # every bf16 value
    v = bits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 464)]
    codes = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = ((codes[:-1] + codes[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e3))])
    v = np.concatenate([v, near, -near]).astype(np.float32)
    got = np.frombuffer(subprocess.run([exe, "encode"], input=v.tobytes(), capture_output=True,
                                       check=True).stdout, np.uint8)
    ref = torch.from_numpy(np.clip(v, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert got.size == v.size and np.array_equal(got, ref)


def test_window_bytes_are_exact(exe):
    r = _run(exe, "2000000", "7")
    assert r["mismatches"] == 0, r
    assert 0 < r["agree"] < r["cases"], r        # both outcomes occur


def test_no_window_is_detected(exe):
    assert _run(exe, "500000", "7", "noshrink")["mismatches"] > 0
