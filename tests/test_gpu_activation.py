"""moe_silu_mul_quant (SiLU(gate) * up, then 1x128 E4M3) against the oracle,
through the C ABI, bit for bit: every E4M3 byte and every fp32 scale of the
rows below each expert's clamped count, and the 0xA5 / sentinel-scale
contents of every other row (the kernel must not touch them)."""
import numpy as np
import pytest
import torch

from combine_moe_dispatch_gb300 import inputs
from combine_moe_dispatch_gb300.configs import WORKLOADS
import gpu_check

pytestmark = pytest.mark.gpu


def _buffers(E, cap, I):
    q = torch.full((E, cap, I), gpu_check.SENTINEL_BYTE, dtype=torch.uint8, device="cuda")
    sc = torch.full((E, cap, (I + 127) // 128), gpu_check.SENTINEL_SCALE, dtype=torch.float32,
                    device="cuda")
    return q, sc


def _workspace(moe, shape):
    ws = torch.empty(moe.workspace_size(shape), dtype=torch.uint8, device="cuda")
    moe.workspace_init(ws)
    return ws


def _edge_rows(I):
    """Rows that reach the corners of e^x and of the quantiser: SiLU of
    large negative gates (e^-g overflows: SiLU = -0), gates next to the 2^128
    rescaling step, large positive gates (SiLU = g), all-zero blocks, and a
    block whose largest |a| sits at an E4M3 rounding midpoint."""
    rows = []
    g = np.linspace(-88.8, -86.0, 2 * I).astype(np.float32)[:I]
    rows.append((g, np.ones(I, np.float32)))
    rows.append((np.linspace(80.0, 100.0, I).astype(np.float32), np.full(I, 0.5, np.float32)))
    z = np.zeros(I, np.float32)
    if I >= 256:
        z[128:256] = np.linspace(-3, 3, 128)
    rows.append((z, np.ones(I, np.float32)))                      # block 0 all zero
    rows.append((np.full(I, -200.0, np.float32), np.ones(I, np.float32)))  # every a = -0
    u = np.ones(I, np.float32)
    rows.append((np.tile(np.linspace(-10, 10, 128), I // 128).astype(np.float32), u))
    out = []
    for gg, uu in rows:
        out.append(np.concatenate([inputs.to_bf16_bits(gg), inputs.to_bf16_bits(uu)]))
    return np.stack(out)


def _check(moe, E, cap, I, h_host, counts, q, sc):
    import oracle
    q_o = np.full((E, cap, I), gpu_check.SENTINEL_BYTE, np.uint8)
    sc_o = np.full((E, cap, (I + 127) // 128), gpu_check.SENTINEL_SCALE, np.float32)
    oracle.silu_mul_quant(h_host, counts, q_o, sc_o)
    q_g = q.cpu().numpy()
    sc_g = sc.cpu().numpy()
    bad = np.argwhere(q_g != q_o)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[0]}"
    assert np.array_equal(sc_g.view(np.uint32), sc_o.view(np.uint32))


@pytest.mark.parametrize("I", [128, 384, 512, 1408, 2048, 4096])
def test_silu_mul_quant_small(I):
    """Hand-set counts: zero, negative, above capacity and partial; I spans
    the 1-, 2- and 4-block-pair task shapes and a ragged last task."""
    import combine_moe_dispatch_gb300 as moe
    E, cap = 6, 12
    counts = np.array([3, 0, 12, 15, -4, 7], np.int32)
    h = inputs.gate_up(E, cap, I, seed=I)
    h[1, 0:5] = _edge_rows(I)          # rows of a count-0 expert: must stay untouched
    h[5, 0:5] = _edge_rows(I)
    shape = moe.make_shape(1, 16, 256, E, 2, cap)
    ws = _workspace(moe, shape)
    q, sc = _buffers(E, cap, I)
    moe.silu_mul_quant(shape, I, gpu_check.dev(h), gpu_check.dev(counts), q, sc, ws)
    _check(moe, E, cap, I, h, counts, q, sc)
    assert moe.read_status(ws) == moe.Status.OK


def test_silu_mul_quant_after_plan():
    """Counts produced on the device by moe_plan feed the activation without
    a host round trip."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    R, T, E, K, I = 2, 300, 16, 4, 512
    cap = R * T
    rng = np.random.default_rng(3)
    idx = np.argsort(rng.random((R * T, E)), axis=1)[:, :K].astype(np.int32)
    shape = moe.make_shape(R, T, 256, E, K, cap)
    b = moe.Buffers(shape, expert_x=False, expert_y=False)
    b.plan(gpu_check.dev(idx))
    st, cnt, off, slot, src = oracle.plan(R, T, E, K, cap, idx)
    h = inputs.gate_up(E, cap, I, seed=11)
    q, sc = _buffers(E, cap, I)
    h_d = gpu_check.dev(h)
    moe.silu_mul_quant(shape, I, h_d, b.expert_num_tokens, q, sc, b.workspace)
    _check(moe, E, cap, I, h, cnt, q, sc)


def test_silu_mul_quant_skips_on_plan_error():
    """A failed plan (capacity) leaves the activation buffers untouched."""
    import combine_moe_dispatch_gb300 as moe
    R, T, E, K, I = 1, 64, 4, 2, 256
    cap = 8
    idx = np.zeros((T, K), np.int32)
    idx[:, 1] = 1
    shape = moe.make_shape(R, T, 256, E, K, cap)
    b = moe.Buffers(shape, expert_x=False, expert_y=False)
    b.plan(gpu_check.dev(idx), check=False)
    h = gpu_check.dev(inputs.gate_up(E, cap, I, seed=2))
    q, sc = _buffers(E, cap, I)
    moe.silu_mul_quant(shape, I, h, b.expert_num_tokens, q, sc, b.workspace)
    torch.cuda.synchronize()
    assert moe.read_status(b.workspace) == moe.Status.CAPACITY
    assert bool((q == gpu_check.SENTINEL_BYTE).all())
    assert bool((sc == gpu_check.SENTINEL_SCALE).all())


def test_silu_mul_quant_rejects_bad_arguments():
    import combine_moe_dispatch_gb300 as moe
    E, cap, I = 2, 4, 256
    shape = moe.make_shape(1, 4, 256, E, 1, cap)
    ws = _workspace(moe, shape)
    h = torch.zeros((E, cap, 2 * I), dtype=torch.bfloat16, device="cuda")
    cnt = torch.zeros(E, dtype=torch.int32, device="cuda")
    q, sc = _buffers(E, cap, I)
    assert moe.silu_mul_quant(shape, 200, h, cnt, q, sc, ws, check=False) == moe.Status.UNSUPPORTED
    assert moe.silu_mul_quant(shape, 0, h, cnt, q, sc, ws, check=False) == moe.Status.INVALID_ARG
    qv = q.view(-1)[1:]
    assert moe.silu_mul_quant(shape, I, h, cnt, qv, sc, ws, check=False) == moe.Status.ALIGNMENT
    torch.cuda.synchronize()
    assert bool((q == gpu_check.SENTINEL_BYTE).all())


def test_silu_mul_quant_full_size_dsv3_decode():
    """DeepSeek-V3-shaped decode layer (E=256, capacity 1024, intermediate
    2048 per expert): counts from moe_plan of the seeded routing; every
    populated row compared with the oracle (rows gathered compactly), and
    every unpopulated row checked untouched."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    wl = WORKLOADS["dsv3_decode"]
    I = 2048
    idx = inputs.routing(wl, 0)
    shape = moe.make_shape(wl.R, wl.T, wl.H, wl.E, wl.K, wl.cap)
    b = moe.Buffers(shape, expert_x=False, expert_y=False)
    b.plan(gpu_check.dev(idx))
    st, cnt, off, slot, src = oracle.plan(wl.R, wl.T, wl.E, wl.K, wl.cap, idx)
    h = inputs.gate_up_device(wl.E, wl.cap, I, seed=4)
    q, sc = _buffers(wl.E, wl.cap, I)
    moe.silu_mul_quant(shape, I, h, b.expert_num_tokens, q, sc, b.workspace)
    pop = gpu_check.populated_mask(cnt, wl.cap)
    rows = gpu_check.host_u16(h[pop])
    n = rows.shape[0]
    q_o, sc_o = oracle.silu_mul_quant(rows.reshape(1, n, 2 * I), np.array([n], np.int32))
    assert np.array_equal(q[pop].cpu().numpy(), q_o[0])
    assert np.array_equal(sc[pop].cpu().numpy().view(np.uint32), sc_o[0].view(np.uint32))
    assert bool((q[~pop] == gpu_check.SENTINEL_BYTE).all())
    assert bool((sc[~pop] == gpu_check.SENTINEL_SCALE).all())
    assert moe.read_status(b.workspace) == moe.Status.OK


def test_silu_mul_quant_every_bf16_gate():
    """Every finite bf16 gate value, one binade per 128-element block (so
    each block's scale is set by gates of one magnitude), with up = 1 and
    up = -3: bytes and scales equal the oracle's.  NaN and infinite gates are
    left out (the sign of a NaN is not defined across implementations)."""
    import combine_moe_dispatch_gb300 as moe
    I = 2048
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    pats[(pats & 0x7F80) == 0x7F80] = 0
    gate = pats.reshape(-1, I)                                  # 32 rows
    rows = []
    for u in (1.0, -3.0):
        up = np.full_like(gate, inputs.to_bf16_bits(np.array([u], np.float32))[0])
        rows.append(np.concatenate([gate, up], axis=1))
    h = np.concatenate(rows)[None]                              # [1, 64, 2I]
    E, cap = 1, h.shape[1]
    counts = np.array([cap], np.int32)
    shape = moe.make_shape(1, 16, 256, E, 1, cap)
    ws = _workspace(moe, shape)
    q, sc = _buffers(E, cap, I)
    moe.silu_mul_quant(shape, I, gpu_check.dev(h), gpu_check.dev(counts), q, sc, ws)
    _check(moe, E, cap, I, h, counts, q, sc)


def test_silu_mul_quant_midpoint_rich_rows():
    """Gates >= 128 have SiLU(g) = g exactly; with up values of 1 to 3
    significant bits, a = g * up keeps few significant bits, and like bf16
    activations its quotients a / scale land next to an E4M3 rounding
    midpoint often (the kernel then divides those bytes alone).  The rows are
    checked to contain such bytes, and the kernel's output against the
    oracle."""
    import combine_moe_dispatch_gb300 as moe
    import oracle
    rng = np.random.default_rng(17)
    E, cap, I = 3, 16, 1024
    g = inputs.to_bf16_bits(rng.uniform(128, 4096, (E, cap, I)).astype(np.float32))
    coarse = np.array([0.5, 0.75, 1.0, 1.25, 1.5, 2.0, 3.0], np.float32)
    u = inputs.to_bf16_bits((rng.choice(coarse, (E, cap, I)) *
                             rng.choice([-1.0, 1.0], (E, cap, I))).astype(np.float32))
    h = np.concatenate([g, u], axis=2)
    counts = np.array([cap, 9, cap], np.int32)
    # how often the window test is undecided, emulated in binary32 on the host
    a = (oracle.bf16_to_f32(g) * oracle.bf16_to_f32(u)).astype(np.float32).reshape(-1, 128)
    amax = np.abs(a).max(axis=1)
    r = (np.float32(1) / (amax / np.float32(448)).astype(np.float32)).astype(np.float32)
    q = (a * r[:, None]).astype(np.float32)
    lo = oracle.f32_to_e4m3((q * np.float32(1 - 2**-20)).astype(np.float32))
    hi = oracle.f32_to_e4m3((q * np.float32(1 + 2**-20)).astype(np.float32))
    assert (lo != hi).sum() > 50, "the rows must exercise the per-byte division"
    shape = moe.make_shape(1, 16, 256, E, 1, cap)
    ws = _workspace(moe, shape)
    qd, sc = _buffers(E, cap, I)
    moe.silu_mul_quant(shape, I, gpu_check.dev(h), gpu_check.dev(counts), qd, sc, ws)
    _check(moe, E, cap, I, h, counts, qd, sc)


@pytest.mark.parametrize("I", [16, 144, 400, 2064])
@pytest.mark.parametrize("tscale", [False, True])
def test_silu_mul_quant_short_last_block(I, tscale):
    """An intermediate size that is not a multiple of 128 (I % 16 == 0):
    ceil(I/128) scales per row, the last block short.  Rows where the short
    block is all zero, and where it holds the row's largest value; every
    byte and scale bit for bit, untouched rows still the sentinel."""
    import combine_moe_dispatch_gb300 as moe
    E, cap = 5, 9
    nb = (I + 127) // 128
    counts = np.array([4, 0, 9, 11, 2], np.int32)
    h = inputs.gate_up(E, cap, I, seed=I + 7)
    hf = np.zeros((2, 2 * I), np.float32)
    hf[:, I:] = 1.0
    hf[0, :I] = np.linspace(-3, 3, I)
    hf[0, (nb - 1) * 128:I] = 0.0                            # short block all zero
    hf[1, :I] = np.linspace(-3, 3, I)
    hf[1, I - 1] = 40.0                                      # short block holds the maximum
    h[0, 0:2] = inputs.to_bf16_bits(hf)
    pay = moe.PAYLOAD_FP8_E4M3_TSCALE if tscale else moe.PAYLOAD_FP8_E4M3
    shape = moe.make_shape(1, 16, 256, E, 2, cap, pay)
    ws = _workspace(moe, shape)
    q = torch.full((E, cap, I), gpu_check.SENTINEL_BYTE, dtype=torch.uint8, device="cuda")
    sdims = (E, nb, cap) if tscale else (E, cap, nb)
    sc = torch.full(sdims, gpu_check.SENTINEL_SCALE, dtype=torch.float32, device="cuda")
    moe.silu_mul_quant(shape, I, gpu_check.dev(h), gpu_check.dev(counts), q, sc, ws)
    _check(moe, E, cap, I, h, counts, q, sc.transpose(1, 2) if tscale else sc)
    assert moe.read_status(ws) == moe.Status.OK


@pytest.mark.parametrize("I", [384, 2048])
def test_silu_mul_quant_transposed_scales(I):
    """PAYLOAD_FP8_E4M3_TSCALE: the same bytes, the scales stored [E, I/128,
    cap]; compared with the oracle's [E, cap, I/128] scales transposed, and
    every scale of an unwritten row still the sentinel."""
    import combine_moe_dispatch_gb300 as moe
    E, cap = 6, 12
    counts = np.array([3, 0, 12, 15, -4, 7], np.int32)
    h = inputs.gate_up(E, cap, I, seed=I + 1)
    shape = moe.make_shape(1, 16, 256, E, 2, cap, moe.PAYLOAD_FP8_E4M3_TSCALE)
    ws = _workspace(moe, shape)
    q = torch.full((E, cap, I), gpu_check.SENTINEL_BYTE, dtype=torch.uint8, device="cuda")
    sc_t = torch.full((E, I // 128, cap), gpu_check.SENTINEL_SCALE, dtype=torch.float32, device="cuda")
    moe.silu_mul_quant(shape, I, gpu_check.dev(h), gpu_check.dev(counts), q, sc_t, ws)
    _check(moe, E, cap, I, h, counts, q, sc_t.transpose(1, 2))
    assert moe.read_status(ws) == moe.Status.OK
