"""moe_plan_dispatch (the plan and the dispatch in one launch) against the CPU
oracle, element by element, through the C ABI.

The fused path is taken up to 16384 routed entries; the shapes here cover
one and many tasks per block, several blocks per token and tokens per block,
ragged rows, K = 1 and K = 32, E = 1 and E = 2048 (several experts owned by
each block), many ranks (long offsets rows), duplicate experts, a routing
table that is not 16-byte aligned (no bulk copy), the decode-sized
workloads at full size (Kimi-K2's 32768 entries are beyond the limit: two
launches, same results), data errors, repeated calls on one workspace, and
capture in a CUDA graph."""
import zlib

import numpy as np
import pytest
import torch

import combine_moe_dispatch_gb300 as moe
import gpu_check
import oracle
from combine_moe_dispatch_gb300 import inputs
from combine_moe_dispatch_gb300.configs import WORKLOADS

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
    ("one_task_per_block", 1, 64, 256, 8, 2, ("bf16", "fp8")),
    ("ragged_k5", 2, 500, 392, 37, 5, ("bf16",)),
    ("ragged_fp8", 3, 300, 640, 64, 8, ("bf16", "fp8")),
    ("k_equals_e", 5, 7, 128, 3, 3, ("bf16", "fp8")),
    ("one_expert", 2, 33, 256, 1, 1, ("bf16", "fp8")),
    ("k32", 1, 50, 256, 40, 32, ("bf16", "fp8")),
    ("many_ranks", 64, 40, 256, 16, 2, ("bf16",)),
    ("one_token_per_rank_k1", 64, 1, 256, 8, 1, ("bf16", "fp8")),  # a rank boundary every entry
    ("one_token_per_rank_k3", 40, 1, 256, 8, 3, ("bf16",)),
    ("e2048", 1, 256, 256, 2048, 8, ("bf16", "fp8")),
    ("h8", 3, 17, 8, 5, 2, ("bf16",)),
    ("wide_rows", 2, 96, 7168, 64, 4, ("bf16", "fp8")),
    ("two_pairs_per_task", 2, 64, 1536, 16, 4, ("bf16", "fp8")),     # 12 blocks: 3 tasks of 2 pairs
    ("ten_pairs_per_row", 1, 48, 2560, 24, 2, ("bf16", "fp8")),      # 20 blocks: 5 tasks of 2 pairs
    ("at_the_limit", 2, 1024, 256, 128, 8, ("bf16", "fp8")),
    ("beyond_the_limit", 2, 1025, 256, 128, 8, ("bf16", "fp8")),
    # fp8 rows that are not a multiple of 128 long: the last scale block is
    # short (H = 16: one block of 16; 144: 128 + 16; 400: 3 x 128 + 16;
    # 7200: 56 x 128 + 32, eight tasks of four block pairs, the last partial)
    ("short_block_h16", 2, 40, 16, 8, 2, ("fp8", "fp8t")),
    ("short_block_h144", 3, 50, 144, 16, 4, ("bf16", "fp8", "fp8t")),
    ("short_block_h400", 2, 64, 400, 37, 5, ("fp8", "fp8t")),
    ("short_block_h7200", 2, 48, 7200, 64, 8, ("fp8", "fp8t")),
]


@pytest.mark.parametrize("name,R,T,H,E,K,payloads", SMALL, ids=[c[0] for c in SMALL])
def test_fused_small_shapes(name, R, T, H, E, K, payloads):
    idx, x, w = _rand_case(zlib.crc32(name.encode()), R, T, H, E, K)
    res = gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, payloads, fused=True)
    assert res["not_bit_exact"] == 0, f"expected bit-exact combine, {res}"


def test_fused_duplicate_experts_per_token():
    idx, x, w = _rand_case(5, 2, 64, 256, 4, 4, distinct=False)
    gpu_check.run_case(2, 64, 256, 4, 4, 2 * 64 * 4, idx, x, w, ("bf16", "fp8"), fused=True)


def test_fused_routing_table_not_16_byte_aligned():
    R, T, H, E, K = 2, 200, 512, 32, 3
    idx, x, w = _rand_case(8, R, T, H, E, K)
    raw = torch.zeros(R * T * K + 1, dtype=torch.int32, device="cuda")
    raw[1:] = gpu_check.dev(idx.reshape(-1))
    view = raw[1:].view(R * T, K)
    assert view.data_ptr() % 16 == 4
    gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, ("bf16", "fp8"), fused=True,
                       idx_device=view)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3_decode", "kimi_decode"])
def test_fused_workload_full_size(name):
    wl = WORKLOADS[name]
    d = inputs.make(wl, 0)
    big = wl.E * wl.cap * wl.H > (1 << 28)
    payloads = ("bf16", "fp8")
    res = gpu_check.run_case(wl.R, wl.T, wl.H, wl.E, wl.K, wl.cap, d["topk_idx"], d["x"],
                             d["topk_weights"], payloads, fused=True,
                             expert_y="device" if big else "host", combine_tokens=None)
    print(name, res)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("bad", [-1, 8, 1 << 30])
def test_fused_bad_expert(bad):
    idx, x, w = _rand_case(1, 2, 100, 256, 8, 2)
    idx[150, 1] = bad
    gpu_check.run_case(2, 100, 256, 8, 2, 200, idx, x, w, ("bf16", "fp8"), fused=True)
    # a valid call on the same workspace clears the status
    shape = moe.make_shape(2, 100, 256, 8, 2, 200)
    buf = moe.Buffers(shape, expert_y=False)
    buf.plan_dispatch(gpu_check.dev(x), gpu_check.dev(idx))
    assert moe.read_status(buf.workspace) == moe.Status.BAD_EXPERT
    idx[150, 1] = 3 if idx[150, 0] != 3 else 4
    buf.plan_dispatch(gpu_check.dev(x), gpu_check.dev(idx))
    assert moe.read_status(buf.workspace) == moe.Status.OK


def test_fused_capacity_overflow():
    idx, x, w = _rand_case(2, 4, 128, 256, 16, 4)
    cap = int(np.bincount(idx.ravel(), minlength=16).max()) - 1
    gpu_check.run_case(4, 128, 256, 16, 4, cap, idx, x, w, ("bf16", "fp8"), fused=True)


def test_fused_repeated_calls_and_mixed_with_plan():
    """One workspace through fused calls, plain plans and the multi-tile plan
    in turn: each call's status and outputs are its own."""
    R, T, H, E, K = 4, 300, 256, 32, 4
    shape = moe.make_shape(R, T, H, E, K, R * T)
    buf = moe.Buffers(shape, expert_y=False)
    big = moe.make_shape(1, 20000, H, E, 8, 20000)
    ws = torch.zeros(max(moe.workspace_size(shape), moe.workspace_size(big)), dtype=torch.uint8,
                     device="cuda")
    bb = moe.Buffers(big, expert_x=False, expert_y=False)
    for seed in range(6):
        idx, x, w = _rand_case(100 + seed, R, T, H, E, K)
        if seed == 3:
            idx[7, 0] = E                       # one failing call in the middle
        moe.plan_dispatch(shape, gpu_check.dev(x), gpu_check.dev(idx), buf.expert_num_tokens,
                          buf.expert_rank_offsets, buf.slot_of, buf.src_of, buf.expert_x, None, ws)
        st = moe.read_status(ws)
        if seed == 3:
            assert st == moe.Status.BAD_EXPERT
            continue
        assert st == moe.Status.OK
        _, cnt, off, slot, src = oracle.plan(R, T, E, K, R * T, idx)
        assert np.array_equal(buf.slot_of.cpu().numpy(), slot)
        assert np.array_equal(buf.expert_rank_offsets.cpu().numpy(), off)
        assert np.array_equal(buf.expert_num_tokens.cpu().numpy(), cnt)
        got = gpu_check.host_u16(buf.expert_x[gpu_check.dev(idx.astype(np.int64)).view(-1),
                                              gpu_check.dev(slot.astype(np.int64)).view(-1)])
        assert np.array_equal(got, np.repeat(x, K, axis=0))
        if seed % 2 == 0:                       # the multi-tile plan on the same workspace
            bidx, _, _ = _rand_case(200 + seed, 1, 20000, 8, E, 8)
            moe.plan(big, gpu_check.dev(bidx), bb.expert_num_tokens, bb.expert_rank_offsets,
                     bb.slot_of, bb.src_of, ws)
            assert moe.read_status(ws) == moe.Status.OK
            _, _, _, bslot, _ = oracle.plan(1, 20000, E, 8, 20000, bidx)
            assert np.array_equal(bb.slot_of.cpu().numpy(), bslot)


def test_fused_in_cuda_graph():
    R, T, H, E, K = 8, 128, 1024, 64, 8
    shape = moe.make_shape(R, T, H, E, K, R * T, moe.PAYLOAD_FP8_E4M3)
    buf = moe.Buffers(shape, expert_y=False)
    idx_s = torch.zeros((R * T, K), dtype=torch.int32, device="cuda")
    x_s = torch.zeros((R * T, H), dtype=torch.bfloat16, device="cuda")
    first, _, _ = _rand_case(10, R, T, H, E, K)
    idx_s.copy_(gpu_check.dev(first))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        buf.plan_dispatch(x_s, idx_s)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        buf.plan_dispatch(x_s, idx_s)
    for seed in (11, 12):
        idx, x, w = _rand_case(seed, R, T, H, E, K)
        idx_s.copy_(gpu_check.dev(idx))
        x_s.copy_(gpu_check.dev(x))
        g.replay()
        torch.cuda.synchronize()
        assert moe.read_status(buf.workspace) == moe.Status.OK
        _, cnt, off, slot, src = oracle.plan(R, T, E, K, R * T, idx)
        assert np.array_equal(buf.slot_of.cpu().numpy(), slot)
        q_o, sc_o = oracle.dispatch_fp8(x, idx, slot, E, R * T)
        for e in range(E):
            n = int(cnt[e])
            assert np.array_equal(buf.expert_x[e, :n].cpu().numpy(), q_o[e, :n])
            assert np.array_equal(buf.expert_x_scale[e, :n].cpu().numpy().view(np.uint32),
                                  sc_o[e, :n].view(np.uint32))


@pytest.mark.parametrize("s", [1.2, 2.5])
def test_fused_zipf_skewed_routing(s):
    """Zipf-skewed routing at a decode size: the hot experts appear in every
    block's run, so their counts take many same-address shared atomics and
    warp 0 ranks long stretches of one expert."""
    R, T, H, E, K = 8, 128, 512, 256, 8
    rng = np.random.default_rng(int(s * 10))
    idx = inputs._zipf_topk(rng, R * T, E, K, s)
    x = inputs.hidden_states(R * T, H, 3)
    w = inputs.weights(R * T, K, 3)
    res = gpu_check.run_case(R, T, H, E, K, R * T, idx, x, w, ("bf16", "fp8"), fused=True)
    assert res["not_bit_exact"] == 0


def test_fused_every_token_to_the_same_experts():
    """The worst skew: every token routes to experts 0..K-1 in the same
    order, so each of them receives N rows (cap = N) and every block's run
    holds only those K experts."""
    R, T, H, E, K = 4, 256, 256, 64, 8
    N = R * T
    idx = np.tile(np.arange(K, dtype=np.int32), (N, 1))
    x = inputs.hidden_states(N, H, 4)
    w = inputs.weights(N, K, 4)
    res = gpu_check.run_case(R, T, H, E, K, N, idx, x, w, ("bf16", "fp8"), fused=True)
    assert res["not_bit_exact"] == 0
    # and the separate plan and dispatch on the same routing
    res = gpu_check.run_case(R, T, H, E, K, N, idx, x, w, ("bf16", "fp8"))
    assert res["not_bit_exact"] == 0


def test_fused_empty_batch():
    """T = 0: zero counts and offsets, status OK, nothing dispatched."""
    R, T, H, E, K = 3, 0, 256, 8, 2
    idx = np.zeros((0, K), np.int32)
    x = np.zeros((0, H), np.uint16)
    w = np.zeros((0, K), np.float32)
    gpu_check.run_case(R, T, H, E, K, 4, idx, x, w, ("bf16", "fp8"), fused=True)
