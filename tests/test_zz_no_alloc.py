"""moe_plan_noalloc, the plan entry point for callers that cannot allocate
device memory (its scratch is a static array inside the library), against
moe_plan on the same inputs: several calls in a row, each compared output by
output.  Plan outputs are integers, so the comparison is bit-exact, as in the
other plan tests.

The shapes cover both plan kernels: the single-cluster plan (DeepSeek-V3
decode and prefill sizes, a small ragged shape) and the multi-tile plan,
whose bounded cross-block waits depend on the counters and per-tile flags
that this entry point clears in the static array before every call (2048
experts; 20000 tokens).  A call that ends in a device error is followed by
clean calls on the same array, and an empty batch needs no routes.  Kept in
its own file, collected last."""
import numpy as np
import pytest
import torch

import combine_moe_dispatch_gb300 as moe

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH = 1 << 20


def _routing(seed, N, E, K):
    rng = np.random.default_rng(seed)
    return np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)


def _outputs(shape, device="cuda"):
    R, T, E, K, cap = (shape.num_ranks, shape.tokens_per_rank, shape.num_experts,
                       shape.top_k, shape.capacity)
    i32 = dict(dtype=torch.int32, device=device)
    return (torch.full((E,), -7, **i32), torch.full((E, R + 1), -7, **i32),
            torch.full((R * T, K), -7, **i32), torch.full((E, cap), -7, **i32))


def _compare(shape, ref, idx, status, tag):
    """moe_plan into ``ref`` and moe_plan_noalloc into fresh outputs, both on
    ``idx``; every output must agree bit for bit, and both must report OK."""
    ref.src_of.fill_(-7)
    ref.plan(idx)
    assert moe.read_status(ref.workspace) == moe.Status.OK, f"{tag}: moe_plan status"
    cnt, off, slot, src = _outputs(shape)
    status.fill_(-1)
    moe.plan_noalloc(shape, idx, cnt, off, slot, src, status)
    torch.cuda.synchronize()
    assert int(status.item()) == int(moe.Status.OK), f"{tag}: status"
    assert torch.equal(cnt, ref.expert_num_tokens), f"{tag}: counts"
    assert torch.equal(off, ref.expert_rank_offsets), f"{tag}: offsets"
    assert torch.equal(slot, ref.slot_of), f"{tag}: slots"
    assert torch.equal(src, ref.src_of), f"{tag}: src_of"


# (R, T, H, E, K): DeepSeek-V3 decode and prefill (single-cluster plan), a
# small ragged shape, and two multi-tile shapes (E > 1024; 20000 tokens)
SHAPES = [(8, 128, 7168, 256, 8), (16, 512, 7168, 256, 8), (3, 300, 256, 64, 8),
          (2, 64, 256, 2048, 8), (4, 5000, 256, 256, 8)]


@pytest.mark.parametrize("R,T,H,E,K", SHAPES)
def test_noalloc_plan_matches_moe_plan(R, T, H, E, K):
    shape = moe.make_shape(R, T, H, E, K, R * T)
    assert moe.workspace_size(shape) <= NOALLOC_SCRATCH
    ref = moe.Buffers(shape, expert_x=False, expert_y=False)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((1, 2, 3)):            # calls in a row on the same array
        idx = torch.from_numpy(_routing(seed, R * T, E, K)).cuda()
        _compare(shape, ref, idx, status, f"call {call}")


@pytest.mark.parametrize("R,T,H,E,K", [(8, 128, 7168, 256, 8), (2, 64, 256, 2048, 8)])
def test_noalloc_recovers_after_a_device_error(R, T, H, E, K):
    """An out-of-range expert id: the plan's BAD_EXPERT reaches status_out,
    and the next valid calls on the same static array are OK and exact."""
    shape = moe.make_shape(R, T, H, E, K, R * T)
    ref = moe.Buffers(shape, expert_x=False, expert_y=False)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    bad = _routing(7, R * T, E, K)
    bad[R * T // 2, K - 1] = E                        # one id just past the last expert
    cnt, off, slot, src = _outputs(shape)
    moe.plan_noalloc(shape, torch.from_numpy(bad).cuda(), cnt, off, slot, src, status)
    torch.cuda.synchronize()
    assert int(status.item()) == int(moe.Status.BAD_EXPERT)
    for call, seed in enumerate((8, 9)):
        idx = torch.from_numpy(_routing(seed, R * T, E, K)).cuda()
        _compare(shape, ref, idx, status, f"after the error, call {call}")


def test_noalloc_empty_batch():
    """T = 0: no routes are read (topk_idx and slot_of may be NULL), counts
    and offsets come out zero and the status OK."""
    R, E, K = 4, 32, 4
    shape = moe.make_shape(R, 0, 256, E, K, 16)
    i32 = dict(dtype=torch.int32, device="cuda")
    cnt = torch.full((E,), -7, **i32)
    off = torch.full((E, R + 1), -7, **i32)
    src = torch.full((E, 16), -7, **i32)
    status = torch.full((1,), -1, **i32)
    moe.plan_noalloc(shape, None, cnt, off, None, src, status)
    torch.cuda.synchronize()
    assert int(status.item()) == int(moe.Status.OK)
    assert int(cnt.abs().sum()) == 0 and int(off.abs().sum()) == 0


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # 64 ranks x 1 tile x 2048 experts x 2 rows x 4 B > 1 MiB
    shape = moe.make_shape(64, 16, 256, 2048, 8, 1024)
    assert moe.workspace_size(shape) > NOALLOC_SCRATCH
    cnt, off, slot, src = _outputs(shape)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = moe.plan_noalloc(shape, torch.zeros((64 * 16, 8), dtype=torch.int32, device="cuda"),
                          cnt, off, slot, src, status, check=False)
    assert st == moe.Status.WORKSPACE
