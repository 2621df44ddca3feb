"""Error paths on the GPU, all made on the host or by a bounded wait that is
allowed to run out; nothing here faults, traps or hangs the GPU.

* expert ids out of range -> BAD_EXPERT, dispatch and combine write nothing;
* more rows than the capacity -> CAPACITY with exact counts/offsets/slots;
* the test hook withholds one tile's counts in the multi-tile plan, so the
  other tiles' bounded waits give up after 50 ms and the plan reports
  TIMEOUT; the next plan on the same workspace is correct again;
* misaligned arguments are rejected before anything is enqueued;
* plan + dispatch + combine captured in a CUDA graph and replayed."""
import numpy as np
import pytest
import torch

import combine_moe_dispatch_gb300 as moe
import gpu_check
import oracle
from combine_moe_dispatch_gb300 import inputs

pytestmark = pytest.mark.gpu


def _case(seed, R, T, H, E, K):
    rng = np.random.default_rng(seed)
    N = R * T
    idx = np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)
    x = inputs.to_bf16_bits(rng.standard_normal((N, H)).astype(np.float32))
    w = rng.random((N, K)).astype(np.float32)
    return idx, x, w


@pytest.mark.parametrize("bad", [-1, 8, 1 << 30])
def test_bad_expert(bad):
    idx, x, w = _case(1, 2, 100, 256, 8, 2)
    idx[150, 1] = bad
    gpu_check.run_case(2, 100, 256, 8, 2, 200, idx, x, w, ("bf16", "fp8"))
    # combine after a failed plan writes nothing
    shape = moe.make_shape(2, 100, 256, 8, 2, 200)
    buf = moe.Buffers(shape)
    buf.plan(gpu_check.dev(idx))
    buf.y.view(torch.int16).fill_(0x1234)
    buf.combine(gpu_check.dev(idx), gpu_check.dev(w))
    assert moe.read_status(buf.workspace) == moe.Status.BAD_EXPERT
    assert bool((buf.y.view(torch.int16) == 0x1234).all())
    # a valid plan on the same workspace clears the status
    idx[150, 1] = 3 if idx[150, 0] != 3 else 4
    buf.plan(gpu_check.dev(idx))
    assert moe.read_status(buf.workspace) == moe.Status.OK


def test_capacity_overflow():
    idx, x, w = _case(2, 4, 128, 256, 16, 4)
    cap = int(np.bincount(idx.ravel(), minlength=16).max()) - 1
    res = gpu_check.run_case(4, 128, 256, 16, 4, cap, idx, x, w, ("bf16", "fp8"))
    assert res["max_ulp"] == 0


def test_timeout_hook_and_recovery():
    # 20000 tokens x 8 experts is beyond one cluster, so the plan runs as 157
    # tiles that wait on each other (the hook only affects those waits)
    R, T, H, E, K = 1, 20000, 128, 32, 8
    idx, x, w = _case(3, R, T, H, E, K)
    shape = moe.make_shape(R, T, H, E, K, R * T)
    buf = moe.Buffers(shape, expert_y=False)
    moe.workspace_set_debug(buf.workspace, 1, 50_000_000)
    buf.plan(gpu_check.dev(idx))
    assert moe.read_status(buf.workspace) == moe.Status.TIMEOUT
    buf.expert_x.view(torch.int16).fill_(0x5A5A)
    buf.dispatch(gpu_check.dev(x), gpu_check.dev(idx))
    torch.cuda.synchronize()
    assert bool((buf.expert_x.view(torch.int16) == 0x5A5A).all()), "dispatch ran after TIMEOUT"
    moe.workspace_set_debug(buf.workspace, 0, 0)
    buf.plan(gpu_check.dev(idx))
    assert moe.read_status(buf.workspace) == moe.Status.OK
    st, cnt, off, slot, src = oracle.plan(R, T, E, K, R * T, idx)
    assert np.array_equal(buf.slot_of.cpu().numpy(), slot)


def test_misaligned_arguments_rejected():
    shape = moe.make_shape(2, 8, 256, 8, 2, 16)
    buf = moe.Buffers(shape)
    idx = gpu_check.dev(np.zeros((16, 2), np.int32))
    x = torch.zeros(16 * 256 + 8, dtype=torch.bfloat16, device="cuda")
    st = moe.dispatch(shape, x[1:], idx, buf.slot_of, buf.expert_x, None, buf.workspace, check=False)
    assert st == moe.Status.ALIGNMENT
    i32 = torch.zeros(64, dtype=torch.int32, device="cuda")
    st = moe.plan(shape, idx, i32.view(torch.int8)[1:].view(torch.int8), buf.expert_rank_offsets,
                  buf.slot_of, buf.src_of, buf.workspace, check=False)
    assert st == moe.Status.ALIGNMENT
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    st = moe.plan(shape, idx, buf.expert_num_tokens, buf.expert_rank_offsets, buf.slot_of,
                  buf.src_of, small, check=False)
    assert st == moe.Status.WORKSPACE


def test_cuda_graph_capture_and_replay():
    R, T, H, E, K = 4, 64, 512, 16, 4
    shape = moe.make_shape(R, T, H, E, K, R * T)
    buf = moe.Buffers(shape)
    idx_s = torch.zeros((R * T, K), dtype=torch.int32, device="cuda")
    x_s = torch.zeros((R * T, H), dtype=torch.bfloat16, device="cuda")
    w_s = torch.zeros((R * T, K), dtype=torch.float32, device="cuda")
    first, _, _ = _case(10, R, T, H, E, K)
    idx_s.copy_(gpu_check.dev(first))
    buf.expert_y.copy_(gpu_check.dev(inputs.expert_outputs(E, R * T, H, 4)))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # warm-up outside capture
        buf.plan(idx_s); buf.dispatch(x_s, idx_s); buf.combine(idx_s, w_s)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        buf.plan(idx_s)
        buf.dispatch(x_s, idx_s)
        buf.combine(idx_s, w_s)
    ey = buf.expert_y.view(torch.int16).cpu().numpy().view(np.uint16)
    for seed in (11, 12, 13):
        idx, x, w = _case(seed, R, T, H, E, K)
        idx_s.copy_(gpu_check.dev(idx)); x_s.copy_(gpu_check.dev(x)); w_s.copy_(gpu_check.dev(w))
        g.replay()
        torch.cuda.synchronize()
        assert moe.read_status(buf.workspace) == moe.Status.OK
        st, cnt, off, slot, src = oracle.plan(R, T, E, K, R * T, idx)
        assert np.array_equal(buf.slot_of.cpu().numpy(), slot)
        got = gpu_check.host_u16(buf.expert_x[gpu_check.dev(idx.astype(np.int64)).view(-1),
                                              gpu_check.dev(slot.astype(np.int64)).view(-1)])
        assert np.array_equal(got, np.repeat(x, K, axis=0))
        y_o = oracle.combine(ey, idx, slot, w)
        assert gpu_check.bf16_ulp_diff(gpu_check.host_u16(buf.y), y_o).max() <= 1
