"""The SiLU table the activation kernel stages in shared memory, against the
oracle's SiLU, on the CPU.

The build generates the table (csrc/silu_table_gen.cpp, a host program) for
the 8192 bf16 gates with 2^-25 <= |g| < 128; entry i is the gate with sign
i >> 12 and magnitude bits (i & 0xFFF) + 0x3300.  Every entry must equal the
oracle's SiLU of its gate bit for bit.  Outside the table the kernel uses
closed forms, pinned here against the oracle over every other finite bf16
gate: g * 0.5 below 2^-25, g from 128 up, and -0 from -128 down."""
import re

import numpy as np

import oracle
from combine_moe_dispatch_gb300 import buildlib


def _f32(bits):
    return np.asarray(bits, np.uint32).view(np.float32)


def _bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def test_table_equals_oracle_silu():
    path = buildlib.generate_table()
    with open(path) as f:
        words = [int(w, 16) for w in re.findall(r"0x([0-9a-f]{8})u", f.read())]
    assert len(words) == 8192
    i = np.arange(8192, dtype=np.uint32)
    gate_bits = ((i >> 12) << 15) | ((i & 0xFFF) + 0x3300)
    g = _f32(gate_bits << 16)
    assert np.all(np.abs(g[:4096]) >= 2.0 ** -25) and np.all(np.abs(g) < 128)
    ref = _bits(oracle.silu_f32(g))
    bad = np.nonzero(ref != np.asarray(words, np.uint32))[0]
    assert bad.size == 0, f"{bad.size} entries differ, first gate {g[bad[0]]!r}"


def test_closed_forms_outside_the_table():
    pats = np.arange(65536, dtype=np.uint32)
    finite = (pats & 0x7F80) != 0x7F80
    mag = pats & 0x7FFF
    g = _f32(pats << 16)
    small = finite & (mag < 0x3300)                       # |g| < 2^-25
    big_pos = finite & (mag >= 0x4300) & (pats < 0x8000)  # g >= 128
    big_neg = finite & (mag >= 0x4300) & (pats >= 0x8000) # g <= -128
    for sel, form in [(small, lambda x: x * np.float32(0.5)),
                      (big_pos, lambda x: x),
                      (big_neg, lambda x: np.full_like(x, -0.0))]:
        got = _bits(oracle.silu_f32(g[sel]))
        assert np.array_equal(got, _bits(form(g[sel])))
