"""Run the CUDA path on one set of inputs and compare it with the CPU oracle.

Used by the ``-m gpu`` parity tests and by ``__graft_entry__.smoke()``.
Everything the oracle sees comes from the seeded generator or from the
oracle itself; nothing it compares against is derived from the CUDA path.

Checks per call:
* plan: counts, offsets, slot_of bit-exact; src_of rows below the count.
* dispatch: the row at the oracle's (expert, slot) of every entry equals
  x[g] (bf16) or the oracle's quantised row and scales (fp8), bit for bit;
  every row at or beyond an expert's count still holds the 0xA5 sentinel.
* combine: within 1 bf16 ulp of the oracle (and the number of elements that
  are not bit-identical is reported); expert_y rows beyond each count are
  NaN, so any stray read would surface as NaN in y.
With ``fused=True`` the plan and the dispatch are one moe_plan_dispatch
call, checked the same way; after a data error it may have written rows of
valid entries below cap, so there only "no row outside [0, min(count, cap))
was written" is checked.
"""
from __future__ import annotations

import numpy as np
import torch

import combine_moe_dispatch_gb300 as moe
import oracle
from combine_moe_dispatch_gb300 import inputs

SENTINEL_BYTE = 0xA5
SENTINEL_SCALE = -1234.5
NAN_BF16 = 0x7FC0


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in bf16 units in the last place (sign-magnitude ordered)."""
    def ordered(u):
        u = u.astype(np.int32)
        mag = u & 0x7FFF
        return np.where(u & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def populated_mask(cnt: np.ndarray, cap: int) -> torch.Tensor:
    c = torch.from_numpy(cnt.astype(np.int64)).cuda()
    return torch.arange(cap, device="cuda")[None, :] < c[:, None]


def rows_touched(buf: torch.Tensor, E: int, cap: int) -> torch.Tensor:
    """[E, cap] bool: row differs from the all-0xA5 sentinel (chunked)."""
    b = buf.view(torch.uint8).view(E, cap, -1)
    out = torch.empty((E, cap), dtype=torch.bool, device=buf.device)
    step = max(1, (1 << 30) // max(1, cap * b.shape[2]))
    for e0 in range(0, E, step):
        out[e0:e0 + step] = (b[e0:e0 + step] != SENTINEL_BYTE).any(dim=-1)
    return out


class Result(dict):
    pass


def run_case(R, T, H, E, K, cap, idx: np.ndarray, x: np.ndarray, w: np.ndarray,
             payloads=("bf16", "fp8"), expert_y="host", combine_tokens=None, seed=0,
             expect_status=None, masked=False, num_tokens=None, fused=False,
             idx_device=None, early_x=False) -> Result:
    """Run plan/dispatch/combine on the GPU and compare with the oracle.
    ``expert_y``: "host" (seeded numpy, full [E,cap,H]) or "device" (seeded
    torch generator on the GPU, for shapes too large for the host).
    ``combine_tokens``: token ids the oracle recomputes (None = all).
    ``fused``: plan and dispatch through moe_plan_dispatch.
    ``idx_device``: the device copy of ``idx`` to pass (e.g. a view that is
    not 16-byte aligned); default a fresh tensor.
    ``early_x``: dispatch through moe_dispatch_ex(MOE_DISPATCH_EARLY_X)."""
    N = R * T
    res = Result(mismatch={}, max_ulp=0, not_bit_exact=0)
    if masked:
        st_o, cnt, off, slot_o, src_o = oracle.plan_masked(R, T, E, K, cap, idx, num_tokens)
        nt_d = None if num_tokens is None else dev(np.asarray(num_tokens, np.int32))
    else:
        st_o, cnt, off, slot_o, src_o = oracle.plan(R, T, E, K, cap, idx)

    def do_plan(buf):
        if masked:
            buf.plan_masked(idx_d, nt_d)
        else:
            buf.plan(idx_d)
    if expect_status is None:
        expect_status = {oracle.OK: moe.Status.OK, oracle.CAPACITY: moe.Status.CAPACITY,
                         oracle.BAD_EXPERT: moe.Status.BAD_EXPERT}[st_o]
    idx_d = dev(idx.astype(np.int32)) if idx_device is None else idx_device
    x_d = dev(x)
    w_d = dev(w.astype(np.float32))
    e_t = idx_d.long().view(-1)
    s_t = dev(slot_o.astype(np.int64)).view(-1) if N else None
    bf16_buf = None

    for payload in payloads:
        code = {"bf16": moe.PAYLOAD_BF16, "fp8": moe.PAYLOAD_FP8_E4M3,
                "fp8t": moe.PAYLOAD_FP8_E4M3_TSCALE}[payload]
        shape = moe.make_shape(R, T, H, E, K, cap, code)
        buf = moe.Buffers(shape, expert_y=False)
        buf.expert_x.view(torch.uint8).fill_(SENTINEL_BYTE)
        if buf.expert_x_scale is not None:
            buf.expert_x_scale.fill_(SENTINEL_SCALE)
        buf.src_of.fill_(-1)
        if fused:
            assert not masked
            buf.plan_dispatch(x_d, idx_d)
        else:
            do_plan(buf)
        st = moe.read_status(buf.workspace)
        assert st == expect_status, f"plan status {st!r}, expected {expect_status!r}"
        if expect_status == moe.Status.BAD_EXPERT and fused:
            return res
        if expect_status == moe.Status.BAD_EXPERT:
            buf.dispatch(x_d, idx_d, early_x=early_x)
            torch.cuda.synchronize()
            assert not rows_touched(buf.expert_x, E, cap).any(), "dispatch wrote after BAD_EXPERT"
            return res
        g_cnt = buf.expert_num_tokens.cpu().numpy()
        assert np.array_equal(g_cnt, cnt), "expert_num_tokens"
        assert np.array_equal(buf.expert_rank_offsets.cpu().numpy(), off), "expert_rank_offsets"
        assert np.array_equal(buf.slot_of.cpu().numpy(), slot_o), "slot_of"
        g_src = buf.src_of.cpu().numpy()
        for e in range(E):
            n = min(int(cnt[e]), cap)
            assert np.array_equal(g_src[e, :n], src_o[e, :n]), f"src_of row {e}"
        if not fused:
            buf.dispatch(x_d, idx_d, early_x=early_x)
        torch.cuda.synchronize()
        touched = rows_touched(buf.expert_x, E, cap)
        if expect_status == moe.Status.CAPACITY and fused:
            below = populated_mask(np.minimum(cnt, cap), cap)
            assert not (touched & ~below).any(), "fused call wrote a row outside [0, min(count, cap))"
            continue
        if expect_status == moe.Status.CAPACITY:
            assert not touched.any(), "dispatch wrote rows although the plan reported CAPACITY"
            continue
        assert torch.equal(touched, populated_mask(cnt, cap)), "rows written outside [0, count)"
        if N == 0:
            continue
        sel = (slot_o.reshape(-1) >= 0)
        sel_d = dev(sel)
        got = buf.expert_x[e_t[sel_d], s_t[sel_d]]
        if payload == "bf16":
            got = host_u16(got)
            exp = np.repeat(x, K, axis=0)[sel]
            assert np.array_equal(got, exp), "bf16 dispatch rows"
            bf16_buf = buf
        else:
            q_o, sc_o = oracle.dispatch_fp8(x, np.zeros((N, 1), np.int32),
                                            np.arange(N, dtype=np.int32)[:, None], 1, N)
            got_q = got.cpu().numpy()
            exp_q = np.repeat(q_o[0], K, axis=0)[sel]
            bad = np.nonzero((got_q != exp_q).any(axis=1))[0]
            assert bad.size == 0, f"fp8 bytes differ in {bad.size} rows (first entry {bad[:4]})"
            # the scales as [E, cap, H/128] whatever the layout
            sc_rows = buf.expert_x_scale.transpose(1, 2) if payload == "fp8t" else buf.expert_x_scale
            got_s = sc_rows[e_t[sel_d], s_t[sel_d]].cpu().numpy()
            exp_s = np.repeat(sc_o[0], K, axis=0)[sel]
            assert np.array_equal(got_s.view(np.uint32), exp_s.view(np.uint32)), "fp8 scales"
            pop = populated_mask(cnt, cap)
            assert bool((sc_rows[~pop] == SENTINEL_SCALE).all()), "scales beyond count"

    # combine (bf16 expert outputs), reusing the plan of a bf16 buffer
    if expect_status != moe.Status.OK or N == 0:
        return res
    if bf16_buf is None:
        shape = moe.make_shape(R, T, H, E, K, cap, moe.PAYLOAD_BF16)
        bf16_buf = moe.Buffers(shape, expert_y=False, expert_x=False)
        do_plan(bf16_buf)
        assert moe.read_status(bf16_buf.workspace) == moe.Status.OK
    if expert_y == "host":
        ey = inputs.expert_outputs(E, cap, H, seed)
        keep = np.arange(cap)[None, :] < cnt[:, None]
        ey[~keep] = NAN_BF16
        ey_d = dev(ey)
    else:
        ey_d = inputs.expert_outputs_device(E, cap, H, seed)
        ey_d[~populated_mask(cnt, cap)] = float("nan")
    bf16_buf.y.view(torch.int16).fill_(0x7FC1)
    bf16_buf.combine(idx_d, w_d, expert_y=ey_d)
    y = host_u16(bf16_buf.y)
    G = np.arange(N) if combine_tokens is None else np.asarray(combine_tokens)
    if expert_y == "host":
        y_o = oracle.combine(ey, idx, slot_o, w)[G]
    else:
        routed = slot_o[G] >= 0
        e_g = np.where(routed, idx[G], 0).astype(np.int64)
        s_g = np.where(routed, slot_o[G], 0).astype(np.int64)
        rows = host_u16(ey_d[dev(e_g).view(-1), dev(s_g).view(-1)])
        nG = len(G)
        y_o = oracle.combine(rows.reshape(1, nG * K, H), np.zeros((nG, K), np.int32),
                             np.where(routed, np.arange(nG * K).reshape(nG, K), -1).astype(np.int32),
                             w[G])
    yg = y[G]
    assert not np.isnan((yg.astype(np.uint32) << 16).view(np.float32)).any(), \
        "NaN in y: a row beyond an expert's count was read"
    d = bf16_ulp_diff(yg, y_o)
    res["max_ulp"] = int(d.max(initial=0))
    res["not_bit_exact"] = int((d != 0).sum())
    assert res["max_ulp"] <= 1, f"combine differs by {res['max_ulp']} bf16 ulp"
    return res
