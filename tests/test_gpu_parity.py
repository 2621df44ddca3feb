"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Small shapes (whole outputs compared) span several plan tiles per rank,
ragged last tiles, ragged hidden segments, K = 1 and K = 32, E = 1 and
E = 2048, duplicate experts per token, and an empty batch.  The five
workloads run at full size in the launch configuration the benchmark times;
there the oracle recomputes every plan output and dispatched row, and the
combine output of all tokens (or of a seeded sample of 1024 tokens when the
expert outputs are generated on the device)."""
import zlib

import numpy as np
import pytest
import torch

from combine_moe_dispatch_gb300 import inputs
from combine_moe_dispatch_gb300.configs import WORKLOADS
import gpu_check

pytestmark = pytest.mark.gpu


def _rand_case(seed, R, T, H, E, K, distinct=True):
    rng = np.random.default_rng(seed)
    N = R * T
    if distinct:
        idx = np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)
    else:
        idx = rng.integers(0, E, (N, K)).astype(np.int32)
    x = inputs.to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    z = rng.standard_normal((N, K))
    w = (np.exp(z) / np.exp(z).sum(1, keepdims=True)).astype(np.float32)
    return idx, x, w


SMALL = [
    # name, R, T, H, E, K, payloads
    ("tiles_ragged_k5", 2, 500, 392, 37, 5, ("bf16",)),
    ("tiles_ragged_fp8", 3, 300, 640, 64, 8, ("bf16", "fp8")),
    ("k_equals_e", 5, 7, 128, 3, 3, ("bf16", "fp8")),
    ("one_expert", 2, 33, 256, 1, 1, ("bf16", "fp8")),
    ("k32", 1, 50, 256, 40, 32, ("bf16", "fp8")),
    ("many_ranks", 64, 40, 256, 16, 2, ("bf16",)),
    ("many_tiles", 1, 20000, 128, 96, 8, ("fp8",)),
    ("e2048", 1, 256, 256, 2048, 8, ("bf16", "fp8")),
    ("h8", 3, 17, 8, 5, 2, ("bf16",)),
    # fp8 rows that are not a multiple of 128 long: the last scale block is
    # short (H = 16: one block of 16; 144: 128 + 16; 400: 3 x 128 + 16;
    # 7200: 56 x 128 + 32, eight tasks of four block pairs, the last partial)
    ("short_block_h16", 2, 40, 16, 8, 2, ("fp8", "fp8t")),
    ("short_block_h144", 3, 50, 144, 16, 4, ("bf16", "fp8", "fp8t")),
    ("short_block_h400", 2, 64, 400, 37, 5, ("fp8", "fp8t")),
    ("short_block_h7200", 2, 48, 7200, 64, 8, ("fp8", "fp8t")),
]


@pytest.mark.parametrize("name,R,T,H,E,K,payloads", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes(name, R, T, H, E, K, payloads):
    idx, x, w = _rand_case(zlib.crc32(name.encode()), R, T, H, E, K)
    res = gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, payloads)
    assert res["not_bit_exact"] == 0, f"expected bit-exact combine, {res}"


def _fp8_edge_rows(H=256):
    """Rows that stress the e4m3 rounding: the hand-worked fixture rows, rows
    whose quotients x/scale are exact E4M3 midpoints (scale a power of two),
    one bf16 step either side of a midpoint, and scales so small that the
    reciprocal overflows."""
    import oracle_pins
    rows = []
    for name in ("fp8_block.txt", "fp8_division.txt"):
        g = oracle_pins.read_kv(name)[0]
        r = np.zeros(H, np.uint16)
        v = [int(t, 0) for t in g["x"].split()]
        for i, b in zip(v[0::2], v[1::2]):
            r[i] = b
        rows.append(r)
    tab = oracle_pins.e4m3_table()[:0x7F]
    mids = ((tab[:-1] + tab[1:]) / 2).astype(np.float64)
    rng = np.random.default_rng(17)
    for k in (-20, -3, 0, 5, 30):
        s = 2.0 ** k
        for sign in (1.0, -1.0):
            m = rng.choice(mids, H)
            vals = sign * m * s
            vals[::128] = 448.0 * s                           # every block: scale = 2^k
            rows.append(inputs.to_bf16_bits(vals.astype(np.float32)))
            b = inputs.to_bf16_bits(vals.astype(np.float32)).astype(np.int32)
            step = rng.choice([-1, 1], H)
            step[::128] = 0
            rows.append((b + step).astype(np.uint16))          # one bf16 ulp off the midpoint
    for amax in (2.0 ** -130, 3.0 * 2.0 ** -128, 1e-38):      # reciprocal of the scale overflows
        vals = rng.standard_normal(H) * amax / 4
        vals[0] = amax
        rows.append(inputs.to_bf16_bits(vals.astype(np.float32)))
    return np.stack(rows)


def test_fp8_rounding_edge_rows():
    x = _fp8_edge_rows()
    N = x.shape[0]
    R, T, H, E, K = 1, N, x.shape[1], 5, 2
    rng = np.random.default_rng(3)
    idx = np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)
    w = inputs.weights(N, K, 3)
    gpu_check.run_case(R, T, H, E, K, N, idx, x, w, ("fp8",))


def _fp8_scale_range_rows(H=1024):
    """Rows of 8 blocks (one 4-pair task each) whose block scales 2^k sit on
    both sides of 2^-60 and 2^60, the range where the kernels take the
    quotient without dividing: quotients at E4M3 midpoints and one bf16 step
    either side, rows all in range, rows with one block out of range, rows
    all out of range."""
    tab = __import__("oracle_pins").e4m3_table()[:0x7F]
    mids = ((tab[:-1] + tab[1:]) / 2).astype(np.float64)
    rng = np.random.default_rng(29)
    plans = [(-60, -59, 59, 60, -60, 60, 0, 3),      # every block in range
             (0, 3, -61, 5, -2, 1, 7, -4),           # one block below the range
             (2, 62, -1, 0, 4, -3, 6, 1),            # one block above the range
             (-61, -62, 61, 62, -70, 70, -61, 61),   # every block out of range
             (-60, -61, 60, 61, -59, -62, 59, 62)]   # alternating at the edges
    rows = []
    for ks in plans:
        for sign in (1.0, -1.0):
            vals = np.empty(H)
            top = np.zeros(H, bool)
            for b, k in enumerate(ks):
                blk = sign * rng.choice(mids, 128) * 2.0 ** k
                j = b * 128 + int(rng.integers(0, 128))
                vals[b * 128:(b + 1) * 128] = blk
                vals[j] = sign * 448.0 * 2.0 ** k              # scale = 2^k
                top[j] = True
            bits = inputs.to_bf16_bits(vals.astype(np.float32))
            rows.append(bits)
            step = rng.choice([-1, 1], H)
            step[top] = 0                                   # keep each block's scale
            rows.append((bits.astype(np.int32) + step).astype(np.uint16))   # one bf16 step off
    return np.stack(rows)


@pytest.mark.parametrize("fused", [False, True], ids=["dispatch", "plan_dispatch"])
def test_fp8_scale_range_edges(fused):
    x = _fp8_scale_range_rows()
    N = x.shape[0]
    R, T, H, E, K = 1, N, x.shape[1], 6, 2
    rng = np.random.default_rng(5)
    idx = np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)
    w = inputs.weights(N, K, 5)
    gpu_check.run_case(R, T, H, E, K, N, idx, x, w, ("fp8",), fused=fused)


def test_fp8_long_task_list():
    """More than 3 tasks per warp of the 3-blocks-per-SM grid (12000 tasks of
    1024 elements against 3648 warps on 152 SMs): the fp8 dispatch runs at 4
    blocks per SM.  Whole outputs compared."""
    R, T, H, E, K = 4, 750, 4096, 16, 2
    idx, x, w = _rand_case(41, R, T, H, E, K)
    gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, ("fp8",))


def test_duplicate_experts_per_token():
    idx, x, w = _rand_case(5, 2, 64, 256, 4, 4, distinct=False)
    gpu_check.run_case(2, 64, 256, 4, 4, 2 * 64 * 4, idx, x, w, ("bf16", "fp8"))


def test_empty_batch():
    R, T, H, E, K = 3, 0, 256, 8, 2
    idx = np.zeros((0, K), np.int32)
    x = np.zeros((0, H), np.uint16)
    w = np.zeros((0, K), np.float32)
    gpu_check.run_case(R, T, H, E, K, 4, idx, x, w, ("bf16", "fp8"))


def test_tight_capacity_is_exact_fit():
    # cap equal to the largest count: every row of the busiest expert is used
    idx, x, w = _rand_case(9, 2, 200, 256, 8, 2)
    cap = int(np.bincount(idx.ravel(), minlength=8).max())
    gpu_check.run_case(2, 200, 256, 8, 2, cap, idx, x, w, ("bf16", "fp8"))


def test_repeated_calls_reuse_workspace():
    # the same buffers through several plans of different routings
    import combine_moe_dispatch_gb300 as moe
    R, T, H, E, K = 4, 300, 256, 32, 4
    shape = moe.make_shape(R, T, H, E, K, R * T)
    buf = moe.Buffers(shape, expert_y=False)
    import oracle
    for seed in range(6):
        idx, x, w = _rand_case(100 + seed, R, T, H, E, K)
        buf.plan(gpu_check.dev(idx))
        assert moe.read_status(buf.workspace) == moe.Status.OK
        st, cnt, off, slot, src = oracle.plan(R, T, E, K, R * T, idx)
        assert np.array_equal(buf.slot_of.cpu().numpy(), slot)
        assert np.array_equal(buf.expert_rank_offsets.cpu().numpy(), off)


def test_both_plan_paths_share_one_workspace():
    """The single-cluster plan (small shapes) and the multi-tile plan (here
    20000 tokens, beyond one cluster) alternate on one workspace."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    shapes = [(4, 300, 32, 4), (1, 20000, 32, 8), (8, 128, 256, 8), (1, 20000, 32, 8)]
    ws = torch.zeros(max(moe.workspace_size(moe.make_shape(R, T, 256, E, K, R * T))
                         for R, T, E, K in shapes), dtype=torch.uint8, device="cuda")
    for i, (R, T, E, K) in enumerate(shapes):
        shape = moe.make_shape(R, T, 256, E, K, R * T)
        idx, _, _ = _rand_case(50 + i, R, T, 8, E, K)
        b = moe.Buffers(shape, expert_x=False, expert_y=False)
        moe.plan(shape, gpu_check.dev(idx), b.expert_num_tokens, b.expert_rank_offsets, b.slot_of,
                 b.src_of, ws)
        assert moe.read_status(ws) == moe.Status.OK
        st, cnt, off, slot, src = oracle.plan(R, T, E, K, R * T, idx)
        assert np.array_equal(b.slot_of.cpu().numpy(), slot)
        assert np.array_equal(b.expert_rank_offsets.cpu().numpy(), off)
        assert np.array_equal(b.expert_num_tokens.cpu().numpy(), cnt)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3_decode", "dsv3_prefill", "kimi_decode"])
def test_workload_full_size(name):
    """Every workload at its full size, in the bench's launch configuration:
    every plan output, every dispatched row, and the combine of every token.
    Where expert_y is too large for the host (E*cap*H > 2^28) it is drawn on
    the device, and only the N*K routed rows (at most 0.94 GB, at prefill)
    come back for the oracle."""
    wl = WORKLOADS[name]
    d = inputs.make(wl, 0)
    big = wl.E * wl.cap * wl.H > (1 << 28)
    payloads = wl.payloads
    res = gpu_check.run_case(wl.R, wl.T, wl.H, wl.E, wl.K, wl.cap, d["topk_idx"], d["x"],
                             d["topk_weights"], payloads,
                             expert_y="device" if big else "host", combine_tokens=None)
    print(name, res)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("R,T,H,E,K,status", [
    (2, 96, 512, 16, 4, "ok"), (3, 300, 1536, 64, 8, "ok"), (8, 128, 7168, 256, 8, "ok"),
    (2, 64, 256, 8, 2, "capacity"), (2, 64, 256, 8, 2, "bad_expert")])
def test_dispatch_early_x(R, T, H, E, K, status):
    """moe_dispatch_ex with MOE_DISPATCH_EARLY_X right after moe_plan (the
    order it is meant for): the same rows, bytes and scales as the oracle,
    and nothing written after a failed plan."""
    idx, x, w = _rand_case(91, R, T, H, E, K)
    cap = R * T
    if status == "capacity":
        cap = int(np.bincount(idx.ravel(), minlength=E).max()) - 1
    if status == "bad_expert":
        idx[R * T // 2, 0] = E
    gpu_check.run_case(R, T, H, E, K, cap, idx, x, w, ("bf16", "fp8"), early_x=True)


def test_fp8_scales_offset_by_4_bytes():
    """A scale array 4 bytes past a 16-byte boundary: the scales must still
    land exactly (bulk copies need 16-byte alignment, so they are not used)."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    R, T, H, E, K = 2, 96, 512, 8, 2
    idx, x, w = _rand_case(77, R, T, H, E, K)
    cap = R * T
    shape = moe.make_shape(R, T, H, E, K, cap, moe.PAYLOAD_FP8_E4M3)
    b = moe.Buffers(shape, expert_x=True, expert_y=False)
    raw = torch.full((E * cap * (H // 128) + 4,), -5.0, dtype=torch.float32, device="cuda")
    sc = raw[1:1 + E * cap * (H // 128)]
    assert sc.data_ptr() % 16 == 4
    idx_d = gpu_check.dev(idx)
    b.plan(idx_d)
    moe.dispatch(shape, gpu_check.dev(x), idx_d, b.slot_of, b.expert_x, sc, b.workspace)
    st, cnt, off, slot, src = oracle.plan(R, T, E, K, cap, idx)
    q_o, sc_o = oracle.dispatch_fp8(x, idx, slot, E, cap)
    got = sc.view(E, cap, H // 128).cpu().numpy()
    for e in range(E):
        assert np.array_equal(got[e, :cnt[e]].view(np.uint32), sc_o[e, :cnt[e]].view(np.uint32))
        assert (got[e, cnt[e]:] == -5.0).all()
    assert np.array_equal(b.expert_x.cpu().numpy()[0, :cnt[0]], q_o[0, :cnt[0]])


MASKED = [
    # name, R, T, H, E, K  (the last two take the multi-tile plan)
    ("masked_cluster", 4, 100, 256, 16, 4),
    ("masked_dsv3_like", 8, 128, 512, 256, 8),
    ("masked_many_tiles", 1, 20000, 128, 32, 8),
    ("masked_e2048", 2, 128, 256, 2048, 8),
]


@pytest.mark.parametrize("name,R,T,H,E,K", MASKED, ids=[c[0] for c in MASKED])
def test_masked_ragged_routing(name, R, T, H, E, K):
    """moe_plan_masked: ragged ranks (num_tokens, including 0, T and values
    outside [0, T]) and masked entries (id -1) through plan, dispatch (both
    payloads) and combine, against the oracle's masked plan."""
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    idx, x, w = _rand_case(zlib.crc32(name.encode()) + 1, R, T, H, E, K)
    idx[rng.random(idx.shape) < 0.15] = -1
    nt = rng.integers(0, T + 1, R).astype(np.int32)
    nt[0] = T
    if R > 2:
        nt[1], nt[2] = 0, T + 7
    # ids of tokens beyond num_tokens are never read: fill them with garbage
    t = np.arange(R * T) % T
    pad = t >= np.clip(nt, 0, T)[np.arange(R * T) // T]
    idx[pad] = 1 << 20
    res = gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, ("bf16", "fp8"),
                             masked=True, num_tokens=nt)
    assert res["not_bit_exact"] == 0


def test_masked_without_num_tokens():
    idx, x, w = _rand_case(3, 2, 64, 256, 8, 2)
    idx[::3, 1] = -1
    idx[5] = -1                                        # a token with no routed entry: y = +0
    res = gpu_check.run_case(2, 64, 256, 8, 2, 128, idx, x, w, ("bf16",), masked=True)
    assert res["not_bit_exact"] == 0


def test_masked_full_size_dsv3_decode():
    wl = WORKLOADS["dsv3_decode"]
    d = inputs.make(wl, 0)
    rng = np.random.default_rng(11)
    idx = d["topk_idx"].copy()
    idx[rng.random(idx.shape) < 0.1] = -1
    nt = rng.integers(wl.T // 2, wl.T + 1, wl.R).astype(np.int32)
    gpu_check.run_case(wl.R, wl.T, wl.H, wl.E, wl.K, wl.cap, idx, d["x"], d["topk_weights"],
                       ("bf16", "fp8"), expert_y="device", masked=True, num_tokens=nt)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("R,T,H,E,K", [(2, 64, 256, 8, 2), (3, 50, 392, 37, 5), (8, 128, 7168, 256, 8)])
def test_combine_shared(R, T, H, E, K):
    """moe_combine_shared against the oracle, bit for bit, including tokens
    with no routed entry (y = shared) and in place (y = shared_y)."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    idx, x, w = _rand_case(R * T + K, R, T, H, E, K)
    idx[::7] = -1
    N, cap = R * T, R * T
    shape = moe.make_shape(R, T, H, E, K, cap)
    b = moe.Buffers(shape, expert_x=False, expert_y=False)
    idx_d = gpu_check.dev(idx)
    b.plan_masked(idx_d)
    st, cnt, off, slot, src = oracle.plan_masked(R, T, E, K, cap, idx)
    ey = inputs.expert_outputs_device(E, cap, H, 5)
    ey[~gpu_check.populated_mask(cnt, cap)] = float("nan")
    sh = inputs.hidden_states(N, H, 9)
    sh_d = gpu_check.dev(sh)
    moe.combine_shared(shape, ey, idx_d, b.slot_of, gpu_check.dev(w), sh_d, b.y, b.workspace)
    routed = slot >= 0
    e_g = np.where(routed, idx, 0).astype(np.int64)
    s_g = np.where(routed, slot, 0).astype(np.int64)
    rows = gpu_check.host_u16(ey[gpu_check.dev(e_g).view(-1), gpu_check.dev(s_g).view(-1)])
    y_o = oracle.combine_shared(rows.reshape(1, N * K, H), np.zeros((N, K), np.int32),
                                np.where(routed, np.arange(N * K).reshape(N, K), -1).astype(np.int32),
                                w, sh)
    assert np.array_equal(gpu_check.host_u16(b.y), y_o)
    # in place: the shared output buffer receives y
    moe.combine_shared(shape, ey, idx_d, b.slot_of, gpu_check.dev(w), sh_d, sh_d, b.workspace)
    assert np.array_equal(gpu_check.host_u16(sh_d), y_o)
    assert moe.read_status(b.workspace) == moe.Status.OK


@pytest.mark.parametrize("N,E,K", [(64, 8, 2), (1024, 256, 8), (4096, 384, 8), (500, 1024, 32),
                                   (33, 7, 7), (300, 64, 1), (5000, 256, 8), (3000, 8, 2)])
def test_router_topk(N, E, K):
    """moe_router_topk against the oracle: indices bit for bit (including
    many exact ties), weights within 1 fp32 ulp (the kernel computes them in
    float-float, the oracle in fp64: the two round the same value to
    neighbouring floats at most); then the router's output through moe_plan.
    Up to one token per warp of one block per SM the kernel keeps two
    candidates per lane; the larger N here take the one-candidate variant."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    rng = np.random.default_rng(N + E + K)
    lg = (rng.standard_normal((N, E)) * 3).astype(np.float32)
    lg[: N // 3] = np.round(lg[: N // 3])
    lg[N // 3: N // 2, : E // 2] = -np.inf
    shape = moe.make_shape(1, N, 256, E, K, N)
    idx_d = torch.empty((N, K), dtype=torch.int32, device="cuda")
    w_d = torch.empty((N, K), dtype=torch.float32, device="cuda")
    moe.router_topk(shape, gpu_check.dev(lg), idx_d, w_d)
    idx_o, w_o = oracle.router_topk(lg, K)
    assert np.array_equal(idx_d.cpu().numpy(), idx_o)
    d = np.abs(w_d.cpu().numpy().view(np.int32).astype(np.int64) - w_o.view(np.int32).astype(np.int64))
    assert d.max() <= 1, f"router weights differ by {d.max()} ulp"
    b = moe.Buffers(shape, expert_x=False, expert_y=False)
    b.plan(idx_d)
    st, cnt, off, slot, src = oracle.plan(1, N, E, K, N, idx_o)
    assert moe.read_status(b.workspace) == moe.Status.OK
    assert np.array_equal(b.slot_of.cpu().numpy(), slot)


def test_router_topk_wide_spread():
    """Logit differences on both sides of -64, where the kernel leaves the
    float-float exponential for fp64 (weights down to subnormal and zero),
    and rows whose chosen logits are all equal: the same indices as the
    oracle and weights within 1 ulp."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    E, K = 256, 8
    rng = np.random.default_rng(11)
    offsets = np.array([0.0, -10.0, -63.9, -64.0, -64.1, -80.0, -100.0, -150.0], np.float32)
    rows = []
    for t in range(64):
        lg = (rng.standard_normal(E) * 0.01 - 400.0).astype(np.float32)
        top = rng.choice(E, size=K, replace=False)
        lg[top] = np.float32(rng.standard_normal() * 3) + offsets * (1.0 + 0.01 * (t % 5))
        rows.append(lg)
    rows.append(np.full(E, 1.5, np.float32))               # every logit equal
    rows.append(np.where(np.arange(E) % 2 == 0, -np.inf, 0.0).astype(np.float32))
    lg = np.stack(rows)
    N = lg.shape[0]
    shape = moe.make_shape(1, N, 256, E, K, N)
    idx_d = torch.empty((N, K), dtype=torch.int32, device="cuda")
    w_d = torch.empty((N, K), dtype=torch.float32, device="cuda")
    moe.router_topk(shape, gpu_check.dev(lg), idx_d, w_d)
    idx_o, w_o = oracle.router_topk(lg, K)
    assert np.array_equal(idx_d.cpu().numpy(), idx_o)
    d = np.abs(w_d.cpu().numpy().view(np.int32).astype(np.int64) - w_o.view(np.int32).astype(np.int64))
    assert d.max() <= 1, f"router weights differ by {d.max()} ulp"
    assert (w_o < np.float32(1.2e-38)).any() and (w_o == 0).any()   # subnormal and zero weights occur


def test_router_topk_unaligned_logits():
    """Logits that start 4 bytes past a 16-byte boundary (the kernel's
    16-byte loads are skipped for them): the same result as the oracle."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    N, E, K = 257, 256, 8
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((N, E)).astype(np.float32)
    flat = torch.empty(N * E + 4, dtype=torch.float32, device="cuda")
    flat[1:1 + N * E] = torch.from_numpy(lg.ravel()).cuda()
    lg_d = flat[1:1 + N * E].view(N, E)
    assert lg_d.data_ptr() % 16 == 4
    shape = moe.make_shape(1, N, 256, E, K, N)
    idx_d = torch.empty((N, K), dtype=torch.int32, device="cuda")
    w_d = torch.empty((N, K), dtype=torch.float32, device="cuda")
    moe.router_topk(shape, lg_d, idx_d, w_d)
    idx_o, w_o = oracle.router_topk(lg, K)
    assert np.array_equal(idx_d.cpu().numpy(), idx_o)
    d = np.abs(w_d.cpu().numpy().view(np.int32).astype(np.int64) - w_o.view(np.int32).astype(np.int64))
    assert d.max() <= 1


TSCALE = [
    # name, R, T, H, E, K
    ("tscale_small", 3, 300, 640, 64, 8),
    ("tscale_ragged_pairs", 2, 64, 1536, 16, 4),
]


@pytest.mark.parametrize("name,R,T,H,E,K", TSCALE, ids=[c[0] for c in TSCALE])
def test_fp8_transposed_scales(name, R, T, H, E, K):
    """PAYLOAD_FP8_E4M3_TSCALE (scales [E, H/128, cap], as a grouped GEMM
    reads them), through moe_plan + moe_dispatch and through
    moe_plan_dispatch: the same bytes and scales as the oracle."""
    idx, x, w = _rand_case(zlib.crc32(name.encode()), R, T, H, E, K)
    gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, ("fp8t",))
    gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, ("fp8t",), fused=True)


def test_fp8_transposed_scales_full_size_dsv3_decode():
    wl = WORKLOADS["dsv3_decode"]
    d = inputs.make(wl, 0)
    for fused in (False, True):
        gpu_check.run_case(wl.R, wl.T, wl.H, wl.E, wl.K, wl.cap, d["topk_idx"], d["x"],
                           d["topk_weights"], ("fp8t",), expert_y="device", fused=fused)
    torch.cuda.empty_cache()
