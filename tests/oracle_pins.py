"""Checks that pin the CPU oracle to facts other than its own code.

Every check takes an ``oracle.Oracle`` (the real build, or a deliberately
broken copy compiled by ``test_oracle_mutants.py``) and raises
AssertionError when the oracle disagrees with:

* library routines that implement a special case of the same definition
  (torch's bf16 and float8_e4m3fn casts, numpy's stable argsort),
* brute force written differently from the oracle (nearest value in the
  full E4M3 code table; exhaustive routings of tiny shapes),
* closed forms and invariants (sum of counts = N*K; offsets end at the count;
  slot_of and src_of are inverse maps; identity experts return x),
* error bounds (combine within half a bf16 ulp plus the fp32 fma-chain error
  of the exact fp64 sum; E4M3 dequantisation within half a grid step),
* worked examples under ``tests/golden/`` (derivations in each file).
"""
from __future__ import annotations

import itertools
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# fixture parsing
# ---------------------------------------------------------------------------

def _ints(s):
    return [int(t, 0) for t in s.split()]


def read_kv(name):
    """Parse a golden file of ``key: values`` lines (``#`` comments).  Keys
    that repeat (``case:``) start a new record."""
    recs, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split(":", 1)
            key, val = key.strip(), val.strip()
            if key == "case" and cur:
                recs.append(cur)
                cur = {}
            cur[key] = val
    if cur:
        recs.append(cur)
    return recs


# ---------------------------------------------------------------------------
# independent references (library routines and brute force)
# ---------------------------------------------------------------------------

def torch_bf16_bits(v):
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def torch_e4m3_bits(v):
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def e4m3_table():
    """Values of all 256 E4M3 codes, decoded by torch."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_nearest(v):
    """Brute force: the non-negative finite code nearest to |v| (ties to the
    even code), signed like v; |v| >= 448 saturates.  NaN not handled."""
    v = np.asarray(v, np.float32)
    tab = e4m3_table()[:0x7F]                 # codes 0x00..0x7E, increasing
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - tab[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best                           # one code, or two on a tie
    idx = np.where(cand.sum(axis=1) == 1, cand.argmax(axis=1), 0)
    two = cand.sum(axis=1) == 2
    if two.any():
        lo = cand[two].argmax(axis=1)          # the tie is between lo and lo+1
        idx[two] = np.where(lo % 2 == 0, lo, lo + 1)
    code = idx.astype(np.uint8)
    code[a >= 448.0] = 0x7E
    sign = np.signbit(v)
    return np.where(sign, code | 0x80, code).astype(np.uint8)


def plan_by_sort(R, T, E, K, topk_idx):
    """Plan outputs from numpy's stable argsort of the flattened routing."""
    flat = np.asarray(topk_idx, np.int64).ravel()
    order = np.argsort(flat, kind="stable")      # entries grouped by expert, in (g,k) order
    cnt = np.bincount(flat, minlength=E).astype(np.int32)
    start = np.concatenate([[0], np.cumsum(cnt)[:-1]])
    slot = np.empty(flat.size, np.int64)
    slot[order] = np.arange(flat.size) - start[flat[order]]
    off = np.zeros((E, R + 1), np.int32)
    for e in range(E):
        pos = np.sort(np.nonzero(flat == e)[0])
        off[e] = np.searchsorted(pos, np.arange(R + 1) * T * K)
    return cnt, off, slot.reshape(-1, K).astype(np.int32), order, start


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def _probe_floats():
    rng = np.random.default_rng(1234)
    all_bf16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    rand_bits = rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    normals = rng.standard_normal(100000).astype(np.float32)
    # exact bf16 midpoints (ties) and their neighbours
    up = np.arange(0, 65536, 7, dtype=np.uint32) << 16
    ties = (up | 0x8000).view(np.float32)
    near = np.concatenate([(up | 0x7FFF).view(np.float32), (up | 0x8001).view(np.float32)])
    v = np.concatenate([all_bf16, rand_bits, normals, ties, near])
    return v[~np.isnan(v)]


def check_bf16(o):
    v = _probe_floats()
    got = o.f32_to_bf16(v)
    assert np.array_equal(got, torch_bf16_bits(v)), "f32->bf16 differs from torch's cast"
    nan = np.array([np.nan, -np.nan], np.float32)
    back = o.bf16_to_f32(o.f32_to_bf16(nan))
    assert np.isnan(back).all(), "NaN must stay NaN"
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = o.bf16_to_f32(bits)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got.view(np.uint32)[~both_nan], ref.view(np.uint32)[~both_nan]), \
        "bf16->f32 differs from torch's widening"


def check_e4m3_decode(o):
    tab = e4m3_table()
    got = o.e4m3_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    nan = np.isnan(tab)
    assert np.array_equal(np.isnan(got), nan), "E4M3 NaN codes"
    assert np.array_equal(got[~nan], tab[~nan]), "E4M3 decode differs from torch"
    assert nan.sum() == 2 and np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])


def _e4m3_probe():
    with np.errstate(all="ignore"):
        return _e4m3_probe_values()


def _e4m3_probe_values():
    rng = np.random.default_rng(99)
    tab = e4m3_table()[:0x7F]
    mids = (tab[:-1] + tab[1:]) / 2                      # exact ties
    eps = np.abs(mids) * 2.0**-20
    all_bf16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    v = np.concatenate([
        mids, mids + eps, mids - eps, -mids, tab, -tab,
        all_bf16, all_bf16 * np.float32(128.0), all_bf16 * np.float32(2.0**-7),
        rng.standard_normal(50000) * 200, rng.standard_normal(20000) * 2.0**-8,
        [0.0, -0.0, 448.0, -448.0, 449.0, 463.99, 464.0, 465.0, 479.0, 480.0, 1e30,
         -1e30, np.inf, -np.inf, 2.0**-9, 2.0**-10, 1.5 * 2.0**-9, 2.0**-6, 2.0**-6 - 2.0**-10],
    ]).astype(np.float32)
    return v[~np.isnan(v)]


def check_e4m3_encode(o):
    v = _e4m3_probe()
    got = o.f32_to_e4m3(v)
    brute = e4m3_nearest(v)
    bad = np.nonzero(got != brute)[0]
    assert bad.size == 0, f"E4M3 encode differs from nearest-code search at {v[bad[:5]]}: " \
                          f"{got[bad[:5]]} vs {brute[bad[:5]]}"
    lib = torch_e4m3_bits(np.clip(v, -448.0, 448.0))
    bad = np.nonzero(got != lib)[0]
    assert bad.size == 0, f"E4M3 encode differs from torch's cast at {v[bad[:5]]}"
    q = o.f32_to_e4m3(np.array([np.nan, -np.nan], np.float32))
    assert set((q & 0x7F).tolist()) == {0x7F}, "NaN -> NaN code"


# ---------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------

def _check_plan_matches_sort(o, R, T, E, K, cap, idx):
    st, cnt, off, slot, src = o.plan(R, T, E, K, cap, idx)
    rcnt, roff, rslot, order, start = plan_by_sort(R, T, E, K, idx)
    assert np.array_equal(cnt, rcnt), "counts"
    assert np.array_equal(off, roff), "rank offsets"
    assert np.array_equal(slot, rslot), "slots"
    exp_st = 0 if rcnt.max(initial=0) <= cap else 2
    assert st == exp_st, f"status {st} != {exp_st}"
    for e in range(E):
        members = order[start[e]:start[e] + rcnt[e]]
        n = min(rcnt[e], cap)
        assert np.array_equal(src[e, :n], members[:n]), "src_of"
        assert (src[e, n:] == -1).all(), "src_of written beyond count/capacity"


def check_plan_exhaustive(o):
    shapes = [(1, 3, 3, 2, 6), (3, 1, 4, 2, 3), (2, 2, 2, 2, 8), (2, 1, 3, 3, 2), (1, 2, 4, 1, 2)]
    for R, T, E, K, cap in shapes:
        N = R * T
        for combo in itertools.product(range(E), repeat=N * K):
            idx = np.array(combo, np.int32).reshape(N, K)
            _check_plan_matches_sort(o, R, T, E, K, cap, idx)


def check_plan_random(o):
    rng = np.random.default_rng(7)
    for R, T, E, K in [(4, 33, 16, 4), (8, 64, 256, 8), (3, 100, 384, 8), (5, 17, 8, 2), (1, 1, 1, 1)]:
        N = R * T
        keys = rng.random((N, E))
        idx = np.argsort(keys, axis=1)[:, :K].astype(np.int32)
        _check_plan_matches_sort(o, R, T, E, K, N, idx)
        # invariants, stated without the sort
        st, cnt, off, slot, src = o.plan(R, T, E, K, N, idx)
        assert st == 0 and cnt.sum() == N * K, "sum of counts must equal R*T*K"
        assert (cnt <= N).all(), "distinct experts: a count is at most N"
        assert np.array_equal(off[:, R], cnt) and (off[:, 0] == 0).all()
        assert (np.diff(off, axis=1) >= 0).all(), "offsets are a cumulative sum"
        flat = idx.ravel()
        for e in range(E):
            row = src[e, :cnt[e]]
            assert (np.diff(row) > 0).all(), "src_of strictly increasing"
            assert (flat[row] == e).all()
            assert np.array_equal(slot.ravel()[row], np.arange(cnt[e])), "slot_of o src_of = id"


def check_plan_empty(o):
    """An empty batch: the definitions give zero counts and offsets."""
    st, cnt, off, slot, src = o.plan(3, 0, 5, 2, 4, np.zeros((0, 2), np.int32))
    assert st == 0 and (cnt == 0).all() and (off == 0).all() and (src == -1).all()


def _routed_mask(R, T, K, topk_idx, num_tokens):
    idx = np.asarray(topk_idx, np.int64).reshape(R * T, K)
    t = np.arange(R * T) % T
    r = np.arange(R * T) // T
    nt = np.full(R, T) if num_tokens is None else np.clip(np.asarray(num_tokens), 0, T)
    return (t < nt[r])[:, None] & (idx != -1)


def plan_masked_by_sort(R, T, E, K, topk_idx, num_tokens):
    """Masked plan from numpy: the routed entries' positions, then a stable
    argsort of their experts."""
    routed = _routed_mask(R, T, K, topk_idx, num_tokens).ravel()
    flat = np.asarray(topk_idx, np.int64).ravel()
    pos = np.nonzero(routed)[0]
    ex = flat[pos]
    order = np.argsort(ex, kind="stable")
    cnt = np.bincount(ex, minlength=E).astype(np.int32)
    start = np.concatenate([[0], np.cumsum(cnt)[:-1]]).astype(np.int64)
    slot = np.full(flat.size, -1, np.int64)
    slot[pos[order]] = np.arange(pos.size) - start[ex[order]]
    off = np.zeros((E, R + 1), np.int32)
    for e in range(E):
        off[e] = np.searchsorted(np.sort(pos[ex == e]), np.arange(R + 1) * T * K)
    src_rows = [pos[order][start[e]:start[e] + cnt[e]] for e in range(E)]
    return cnt, off, slot.reshape(-1, K).astype(np.int32), src_rows


def check_plan_masked(o):
    rng = np.random.default_rng(71)
    shapes = [(1, 2, 2, 2), (2, 1, 2, 2), (3, 1, 3, 1), (2, 2, 2, 1)]
    for R, T, E, K in shapes:                      # exhaustive over ids in {-1..E-1}
        N = R * T
        for combo in itertools.product(range(-1, E), repeat=N * K):
            idx = np.array(combo, np.int32).reshape(N, K)
            nt = rng.integers(-1, T + 2, R).astype(np.int32)   # includes out-of-range counts
            for num_tokens in (None, nt):
                st, cnt, off, slot, src = o.plan_masked(R, T, E, K, N * K, idx, num_tokens)
                rc, ro, rs, rows = plan_masked_by_sort(R, T, E, K, idx, num_tokens)
                assert st == 0, f"status {st}"
                assert np.array_equal(cnt, rc) and np.array_equal(off, ro), "masked counts/offsets"
                assert np.array_equal(slot, rs), "masked slots"
                for e in range(E):
                    assert np.array_equal(src[e, :cnt[e]], rows[e]), "masked src_of"
    for R, T, E, K in [(4, 50, 16, 4), (8, 33, 256, 8)]:   # random, larger
        idx = np.argsort(rng.random((R * T, E)), axis=1)[:, :K].astype(np.int32)
        idx[rng.random(idx.shape) < 0.2] = -1
        nt = rng.integers(0, T + 1, R).astype(np.int32)
        st, cnt, off, slot, src = o.plan_masked(R, T, E, K, R * T, idx, nt)
        rc, ro, rs, rows = plan_masked_by_sort(R, T, E, K, idx, nt)
        assert st == 0 and np.array_equal(cnt, rc) and np.array_equal(off, ro)
        assert np.array_equal(slot, rs)
        assert cnt.sum() == _routed_mask(R, T, K, idx, nt).sum(), "counts = routed entries"
    # ids of padding tokens are ignored, routed out-of-range ids are errors
    idx = np.array([[0, 1], [5, 9]], np.int32)
    assert o.plan_masked(1, 2, 2, 2, 4, idx, np.array([1], np.int32))[0] == 0
    assert o.plan_masked(1, 2, 2, 2, 4, idx, np.array([2], np.int32))[0] == 1
    # hand-worked fixture
    g = read_kv("plan_masked.txt")[0]
    R, T, E, K, cap = (int(g[k]) for k in ("R", "T", "E", "K", "cap"))
    idx = np.array(_ints(g["topk_idx"]), np.int32).reshape(R * T, K)
    st, cnt, off, slot, src = o.plan_masked(R, T, E, K, cap, idx,
                                            np.array(_ints(g["num_tokens"]), np.int32))
    assert st == int(g["status"])
    assert cnt.tolist() == _ints(g["expert_num_tokens"]), "fixture counts"
    assert off.ravel().tolist() == _ints(g["expert_rank_offsets"]), "fixture offsets"
    assert slot.ravel().tolist() == _ints(g["slot_of"]), "fixture slots"
    assert src.ravel().tolist() == _ints(g["src_of"]), "fixture src_of"


def check_plan_errors(o):
    idx = np.array([[0, 1], [2, 3]], np.int32)
    for bad in (-1, 4, 1 << 20):
        b = idx.copy()
        b[1, 0] = bad
        st, cnt, off, slot, src = o.plan(1, 2, 4, 2, 2, b)
        assert st == 1, "bad expert id -> BAD_EXPERT"
        assert (cnt == -1).all() and (slot == -1).all() and (src == -1).all(), \
            "nothing written on BAD_EXPERT"


def check_plan_golden(o):
    for name in ("plan_small.txt", "plan_small_capacity.txt"):
        g = read_kv(name)[0]
        R, T, E, K, cap = (int(g[k]) for k in ("R", "T", "E", "K", "cap"))
        idx = np.array(_ints(g["topk_idx"]), np.int32).reshape(R * T, K)
        st, cnt, off, slot, src = o.plan(R, T, E, K, cap, idx)
        assert st == int(g["status"]), f"{name}: status"
        assert cnt.tolist() == _ints(g["expert_num_tokens"]), f"{name}: counts"
        assert off.ravel().tolist() == _ints(g["expert_rank_offsets"]), f"{name}: offsets"
        assert slot.ravel().tolist() == _ints(g["slot_of"]), f"{name}: slots"
        assert src.ravel().tolist() == _ints(g["src_of"]), f"{name}: src_of"


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------

def _routing(rng, N, E, K):
    return np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)


def check_dispatch_bf16(o):
    rng = np.random.default_rng(3)
    R, T, E, K, H = 2, 40, 6, 3, 136
    N = R * T
    idx = _routing(rng, N, E, K)
    x = rng.integers(0, 65536, (N, H), dtype=np.uint16)
    st, cnt, off, slot, src = o.plan(R, T, E, K, N, idx)
    sentinel = np.uint16(0xA5A5)
    out = np.full((E, N, H), sentinel, np.uint16)
    o.dispatch_bf16(x, idx, slot, E, N, out=out)
    for g in range(N):
        for k in range(K):
            assert np.array_equal(out[idx[g, k], slot[g, k]], x[g]), "row copied bit for bit"
    for e in range(E):
        assert (out[e, cnt[e]:] == sentinel).all(), "rows beyond the count untouched"


def check_fp8_golden(o):
    for name in ("fp8_block.txt", "fp8_division.txt"):
        _check_fp8_golden_file(o, name)


def _check_fp8_golden_file(o, name):
    g = read_kv(name)[0]
    H = int(g["H"])
    x = np.zeros(H, np.uint16)
    pairs = _ints(g["x"])
    for i, b in zip(pairs[0::2], pairs[1::2]):
        x[i] = b
    q_exp = np.zeros(H, np.uint8)
    pairs = _ints(g["q"])
    for i, b in zip(pairs[0::2], pairs[1::2]):
        q_exp[i] = b
    sc_exp = np.array(_ints(g["scale"]), np.uint32)
    q, sc = o.quant_row_e4m3(x)
    bad = np.nonzero(q != q_exp)[0]
    assert bad.size == 0, f"{name}: bytes differ at {bad.tolist()}: {q[bad]} vs {q_exp[bad]}"
    assert np.array_equal(sc.view(np.uint32), sc_exp), f"{name}: scales {sc}"


def check_fp8_properties(o):
    """Pins that hold for any row: the block maximum maps to +-448, the scale
    times 448 recovers the maximum to within one fp32 rounding, every value
    dequantises to within half an E4M3 grid step (plus the rounding of the
    division), zero blocks give scale 0 and q = +0."""
    rng = np.random.default_rng(11)
    H = 1024
    for trial in range(40):
        f = rng.standard_normal(H).astype(np.float32) * np.float32(10.0 ** rng.uniform(-30, 30))
        if trial % 5 == 0:
            f[256:384] = 0.0                 # a zero block
        row = torch_bf16_bits(f)
        xv = torch.from_numpy(row.view(np.int16)).view(torch.bfloat16).float().numpy()
        q, sc = o.quant_row_e4m3(row)
        deq = e4m3_table()[q].astype(np.float64)
        for b in range(H // 128):
            blk = xv[b * 128:(b + 1) * 128].astype(np.float64)
            amax = np.abs(blk).max()
            s = float(sc[b])
            if amax == 0:
                assert s == 0.0 and (q[b * 128:(b + 1) * 128] == 0).all(), "zero block"
                continue
            assert abs(s * 448.0 - amax) <= amax * 2.0**-23, "scale = amax/448"
            j = np.abs(blk).argmax()
            assert (q[b * 128 + j] & 0x7F) == 0x7E, "block max maps to 448"
            t = blk / s                                       # exact target in fp64
            step = np.where(np.abs(t) < 2.0**-6, 2.0**-9,
                            2.0 ** (np.floor(np.log2(np.maximum(np.abs(t), 2.0**-6))) - 3))
            err = np.abs(deq[b * 128:(b + 1) * 128] - np.clip(t, -448, 448))
            assert (err <= 0.5 * step + np.abs(t) * 2.0**-23).all(), "E4M3 rounding bound"


def check_fp8_partial_block(o):
    """A row whose length is not a multiple of 128 has ceil(H/128) blocks, the
    last one short ("Lower latency and higher throughput with multi-node
    DeepSeek deployment", Quantization: scales M x ceil_div(K, 128)).  The
    short block must quantise exactly as the same elements followed by zeros
    up to 128 (zeros change neither the maximum nor any other element's
    byte), which is the full-block path pinned above; an all-zero short block
    has scale 0."""
    rng = np.random.default_rng(29)
    for H in (16, 144, 400, 7200):
        nb = (H + 127) // 128
        for trial in range(6):
            f = rng.standard_normal(H).astype(np.float32) * np.float32(10.0 ** rng.uniform(-3, 3))
            if trial == 0:
                f[(nb - 1) * 128:] = 0.0              # an all-zero short block
            if trial == 1:
                f[(nb - 1) * 128:] *= np.float32(1e4)  # the short block holds the row's maximum
            row = torch_bf16_bits(f)
            q, sc = o.quant_row_e4m3(row)
            assert q.shape == (H,) and sc.shape == (nb,), "ceil(H/128) scales"
            padded = np.zeros(nb * 128, np.uint16)
            padded[:H] = row
            qp, scp = o.quant_row_e4m3(padded)
            assert np.array_equal(q, qp[:H]), f"H={H}: short block bytes as if zero-padded"
            assert np.array_equal(sc.view(np.uint32), scp.view(np.uint32)), f"H={H}: scales"
            if trial == 0:
                assert sc[-1] == 0.0 and (q[(nb - 1) * 128:] == 0).all(), "zero short block"


def check_dispatch_fp8(o):
    rng = np.random.default_rng(5)
    R, T, E, K, H = 3, 21, 5, 2, 384
    N = R * T
    idx = _routing(rng, N, E, K)
    x = torch_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    st, cnt, off, slot, src = o.plan(R, T, E, K, N, idx)
    out = np.full((E, N, H), 0xA5, np.uint8)
    sc = np.full((E, N, H // 128), np.float32(-7.0), np.float32)
    o.dispatch_fp8(x, idx, slot, E, N, out=out, out_scale=sc)
    for g in range(N):
        q, s = o.quant_row_e4m3(x[g])
        for k in range(K):
            e, sl = idx[g, k], slot[g, k]
            assert np.array_equal(out[e, sl], q) and np.array_equal(sc[e, sl], s), \
                "quantised row and scales written to every slot of the token"
    for e in range(E):
        assert (out[e, cnt[e]:] == 0xA5).all() and (sc[e, cnt[e]:] == -7.0).all()


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

def check_combine_golden(o):
    for c in read_kv("combine_small.txt"):
        w = np.array(_ints(c["w"]), np.uint32).view(np.float32)
        v = np.array(_ints(c["v"]), np.uint16)
        K, H = w.size, 8
        ey = np.repeat(v[:, None, None], H, axis=2).astype(np.uint16)    # [E=K, cap=1, H]
        idx = np.arange(K, dtype=np.int32)[None, :]
        slot = np.zeros((1, K), np.int32)
        y = o.combine(ey, idx, slot, w[None, :])
        assert (y == int(c["y"], 0)).all(), f"combine golden case {c['case']}: {hex(y[0, 0])}"


def _combine_case(o, rng, R, T, E, K, H):
    N = R * T
    idx = _routing(rng, N, E, K)
    z = rng.standard_normal((N, K))
    w = (np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)).astype(np.float32)
    st, cnt, off, slot, src = o.plan(R, T, E, K, N, idx)
    return N, idx, w, slot, cnt


def check_combine_identity(o):
    """Identity experts (expert_y = dispatched x) with weights summing to 1
    return x exactly; K = 1 with weight 1 is a pure gather."""
    rng = np.random.default_rng(21)
    R, T, E, K, H = 2, 24, 7, 3, 264
    N, idx, w, slot, cnt = _combine_case(o, rng, R, T, E, K, H)
    x = torch_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    ey = o.dispatch_bf16(x, idx, slot, E, N)
    y = o.combine(ey, idx, slot, w)
    assert np.array_equal(y, x), "identity experts must return x"
    # fp8 payload through identity experts: y = bf16(q * scale)
    H8 = 256
    x8 = torch_bf16_bits(rng.standard_normal((N, H8)).astype(np.float32))
    q, sc = o.dispatch_fp8(x8, idx, slot, E, N)
    deq = (e4m3_table()[q] * np.repeat(sc.astype(np.float64), 128, axis=2)).astype(np.float32)
    ey8 = torch_bf16_bits(deq)
    y8 = o.combine(ey8, idx, slot, w)
    first = ey8[idx[:, 0], slot[:, 0]]
    assert np.array_equal(y8, first), "identity experts on the fp8 payload"
    # pure gather
    idx1 = idx[:, :1].copy()
    st, cnt1, off1, slot1, src1 = o.plan(R, T, E, 1, N, idx1)
    ey1 = torch_bf16_bits(rng.standard_normal((E, N, H)).astype(np.float32))
    y1 = o.combine(ey1, idx1, slot1, np.ones((N, 1), np.float32))
    assert np.array_equal(y1, ey1[idx1[:, 0], slot1[:, 0]]), "K=1, w=1 is a gather"


def check_combine_bound(o):
    """|y - S| <= half a bf16 ulp of S plus the fp32 fma-chain error bound,
    where S is the weighted sum in fp64 (error bound of the arithmetic)."""
    rng = np.random.default_rng(31)
    for R, T, E, K, H in [(2, 16, 9, 4, 128), (1, 40, 32, 8, 72)]:
        N, idx, w, slot, cnt = _combine_case(o, rng, R, T, E, K, H)
        ey = torch_bf16_bits(rng.standard_normal((E, N, H)).astype(np.float32))
        y = o.combine(ey, idx, slot, w)
        eyf = torch.from_numpy(ey.view(np.int16)).view(torch.bfloat16).double().numpy()
        rows = eyf[idx, slot]                                 # [N, K, H]
        terms = w.astype(np.float64)[:, :, None] * rows
        S = terms.sum(axis=1)
        A = np.abs(terms).sum(axis=1)
        yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy()
        e = np.floor(np.log2(np.maximum(np.abs(S), 2.0**-126)))
        half_ulp = 2.0 ** (e - 8)
        bound = half_ulp + (K + 1) * 2.0**-24 * A * 1.01 + 2.0**-133
        assert (np.abs(yf - S) <= bound).all(), "combine outside the fp32 error bound"


def check_combine_shared(o):
    """Hand-worked cases; a zero shared output reduces to combine exactly
    (+0 + x = x for every non-NaN x); the fp64 error bound with the shared
    term; and the shared output alone when no entry is routed."""
    for c in read_kv("combine_shared.txt"):
        w = np.array(_ints(c["w"]), np.uint32).view(np.float32)
        v = np.array(_ints(c["v"]), np.uint16)
        K, H = w.size, 8
        ey = np.repeat(v[:, None, None], H, axis=2).astype(np.uint16)
        sh = np.full((1, H), int(c["shared"], 0), np.uint16)
        y = o.combine_shared(ey, np.arange(K, dtype=np.int32)[None, :], np.zeros((1, K), np.int32),
                             w[None, :], sh)
        assert (y == int(c["y"], 0)).all(), f"combine_shared case {c['case']}: {hex(y[0, 0])}"
    rng = np.random.default_rng(41)
    R, T, E, K, H = 2, 20, 9, 4, 64
    N, idx, w, slot, cnt = _combine_case(o, rng, R, T, E, K, H)
    ey = torch_bf16_bits(rng.standard_normal((E, N, H)).astype(np.float32))
    zero = np.zeros((N, H), np.uint16)
    assert np.array_equal(o.combine_shared(ey, idx, slot, w, zero), o.combine(ey, idx, slot, w))
    sh = torch_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    y = o.combine_shared(ey, idx, slot, w, sh)
    eyf = torch.from_numpy(ey.view(np.int16)).view(torch.bfloat16).double().numpy()
    shf = torch.from_numpy(sh.view(np.int16)).view(torch.bfloat16).double().numpy()
    terms = w.astype(np.float64)[:, :, None] * eyf[idx, slot]
    S = shf + terms.sum(axis=1)
    A = np.abs(shf) + np.abs(terms).sum(axis=1)
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).double().numpy()
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(S), 2.0**-126))) - 8)
    assert (np.abs(yf - S) <= half_ulp + (K + 1) * 2.0**-24 * A * 1.01 + 2.0**-133).all()
    none = np.full((N, K), -1, np.int32)
    assert np.array_equal(o.combine_shared(ey, none, none, w, sh), sh), "no routed entry: y = shared"


def check_router(o):
    """Hand-worked cases; indices against numpy's lexsort (descending logit,
    then ascending index); weights within 1 fp32 ulp of a numpy fp64 softmax
    over the chosen logits (the two fp64 exps may differ in the last bit);
    weights sum to 1 and do not increase."""
    for c in read_kv("router.txt"):
        E, K = int(c["E"]), int(c["K"])
        lg = np.array(_ints(c["logits"]), np.uint32).view(np.float32).reshape(1, E)
        idx, w = o.router_topk(lg, K)
        assert idx[0].tolist() == _ints(c["topk_idx"]), f"router case {c['case']}: {idx}"
        assert w.view(np.uint32)[0].tolist() == _ints(c["topk_weights"]), f"router case {c['case']}: {w}"
    rng = np.random.default_rng(61)
    for N, E, K in [(200, 8, 2), (100, 256, 8), (50, 384, 8), (30, 7, 7), (64, 64, 1)]:
        lg = rng.standard_normal((N, E)).astype(np.float32) * 3
        lg[: N // 2] = np.round(lg[: N // 2])               # many ties
        idx, w = o.router_topk(lg, K)
        ref = np.stack([np.lexsort((np.arange(E), -lg[g]))[:K] for g in range(N)]).astype(np.int32)
        assert np.array_equal(idx, ref), "router indices"
        sel = np.take_along_axis(lg, ref, axis=1).astype(np.float64)
        z = np.exp(sel - sel[:, :1])
        wr = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
        d = np.abs(w.view(np.int32).astype(np.int64) - wr.view(np.int32).astype(np.int64))
        assert d.max() <= 1, "router weights vs fp64 softmax"
        assert (np.abs(w.astype(np.float64).sum(axis=1) - 1) <= K * 2.0**-24).all()
        assert (np.diff(w, axis=1) <= 0).all(), "weights follow the logit order"


def _ulps(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    a = np.where(a < 0, -(a & 0x7FFFFFFF), a)
    b = np.where(b < 0, -(b & 0x7FFFFFFF), b)
    return np.abs(a - b)


def check_exp_silu(o):
    """The fixed binary32 exp within 1 ulp of fp64 exp rounded to binary32,
    exact at 0, saturating outside [-87.33, 88.72], monotone; SiLU within 4
    ulp of the fp64 definition x / (1 + e^-x)."""
    rng = np.random.default_rng(81)
    x = np.concatenate([np.linspace(-87.3, 88.7, 20001), rng.uniform(-87.3, 88.7, 5000),
                        rng.standard_normal(5000), [0.0, 1.0, -1.0, 0.5, 1e-8, -1e-8]]).astype(np.float32)
    e = o.exp_f32(x)
    assert _ulps(e, np.exp(x.astype(np.float64)).astype(np.float32)).max() <= 1, "exp within 1 ulp"
    assert o.exp_f32([0.0])[0] == 1.0
    assert np.isinf(o.exp_f32([88.75])[0]) and o.exp_f32([-87.4])[0] == 0.0
    xs = np.sort(x)
    assert (np.diff(o.exp_f32(xs)) >= 0).all(), "exp is monotone"
    g = np.concatenate([rng.standard_normal(20000) * 4, np.linspace(-80, 80, 4001)]).astype(np.float32)
    si = o.silu_f32(g)
    gd = g.astype(np.float64)
    ref = (gd / (1.0 + np.exp(-gd))).astype(np.float32)
    assert _ulps(si, ref).max() <= 4, "silu within 4 ulp"
    assert o.silu_f32([0.0])[0] == 0.0


def check_silu_mul_quant(o):
    """Rows below clamp(count, 0, cap) only; a = SiLU(gate) * up from the
    first and second halves of each row; every dequantised value within half
    an E4M3 step (plus the SiLU error) of the fp64 reference; zero blocks
    give scale 0 and q = 0."""
    rng = np.random.default_rng(91)
    E, cap, I = 5, 6, 256
    h = torch_bf16_bits((rng.standard_normal((E, cap, 2 * I)) * 2).astype(np.float32))
    h[2, 0, :128] = 0                                  # zero gate block -> zero block
    cnt = np.array([3, 0, 2, 9, -4], np.int32)         # beyond cap and negative clamp
    q = np.full((E, cap, I), 0xA5, np.uint8)
    sc = np.full((E, cap, I // 128), -3.0, np.float32)
    o.silu_mul_quant(h, cnt, q, sc)
    hf = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).double().numpy()
    tab = e4m3_table()
    for e in range(E):
        rows = min(max(int(cnt[e]), 0), cap)
        assert (q[e, rows:] == 0xA5).all() and (sc[e, rows:] == -3.0).all(), "rows beyond the count"
        for s_ in range(rows):
            gate, up = hf[e, s_, :I], hf[e, s_, I:]
            a = gate / (1 + np.exp(-gate)) * up
            for b in range(I // 128):
                blk = a[b * 128:(b + 1) * 128]
                amax = np.abs(blk).max()
                if amax == 0:
                    assert sc[e, s_, b] == 0 and (q[e, s_, b * 128:(b + 1) * 128] == 0).all()
                    continue
                s = float(sc[e, s_, b])
                assert abs(s * 448 - amax) <= amax * 2.0**-20, "scale from the block maximum"
                t = blk / s
                step = np.where(np.abs(t) < 2.0**-6, 2.0**-9,
                                2.0 ** (np.floor(np.log2(np.maximum(np.abs(t), 2.0**-6))) - 3))
                deq = tab[q[e, s_, b * 128:(b + 1) * 128]]
                assert (np.abs(deq - np.clip(t, -448, 448)) <= 0.5 * step + np.abs(t) * 2.0**-19).all()
    assert (sc[2, 0, 0] == 0) and (q[2, 0, :128] == 0).all(), "zero gate -> zero block"


def check_silu_partial_block(o):
    """An intermediate size that is not a multiple of 128 gives ceil(I/128)
    scale blocks per row, the last one short (the same reading as the
    dispatch's).  Metamorphic pin: the result equals that of rows whose gate
    and up halves are zero-padded to a multiple of 128 (SiLU(0) * 0 = 0
    changes no block maximum), truncated back; an all-zero short block has
    scale 0."""
    rng = np.random.default_rng(93)
    E, cap = 3, 4
    cnt = np.array([4, 1, 3], np.int32)
    for I in (16, 144, 400):
        nb, Ip = (I + 127) // 128, ((I + 127) // 128) * 128
        g = rng.standard_normal((E, cap, I)).astype(np.float32) * 2
        u = rng.standard_normal((E, cap, I)).astype(np.float32)
        g[0, 1, (nb - 1) * 128:] = 0.0                     # an all-zero short block
        h = torch_bf16_bits(np.concatenate([g, u], axis=2))
        q, sc = o.silu_mul_quant(h, cnt)
        assert q.shape == (E, cap, I) and sc.shape == (E, cap, nb), "ceil(I/128) scales"
        gp = np.zeros((E, cap, Ip), np.float32)
        up = np.zeros((E, cap, Ip), np.float32)
        gp[..., :I], up[..., :I] = g, u
        hp = torch_bf16_bits(np.concatenate([gp, up], axis=2))
        qp, scp = o.silu_mul_quant(hp, cnt)
        assert np.array_equal(q, qp[..., :I]), f"I={I}: short block bytes as if zero-padded"
        assert np.array_equal(sc.view(np.uint32), scp.view(np.uint32)), f"I={I}: scales"
        assert sc[0, 1, nb - 1] == 0 and (q[0, 1, (nb - 1) * 128:] == 0).all(), "zero short block"


ALL_CHECKS = [
    check_bf16, check_e4m3_decode, check_e4m3_encode,
    check_plan_exhaustive, check_plan_random, check_plan_empty, check_plan_masked,
    check_plan_errors,
    check_plan_golden,
    check_dispatch_bf16, check_fp8_golden, check_fp8_properties, check_fp8_partial_block,
    check_dispatch_fp8,
    check_combine_golden, check_combine_identity, check_combine_bound, check_combine_shared,
    check_router, check_exp_silu, check_silu_mul_quant, check_silu_partial_block,
]
