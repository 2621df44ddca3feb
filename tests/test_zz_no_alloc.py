"""moe_plan_noalloc, the plan entry point for callers that cannot allocate
device memory (its scratch is a static array inside the library), against
moe_plan on the same inputs: two calls in a row, each compared output by
output.  Plan outputs are integers, so the comparison is bit-exact, as in the
other plan tests.  Kept in its own file, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import combine_moe_dispatch_gb300 as moe

pytestmark = pytest.mark.gpu


def _routing(seed, N, E, K):
    rng = np.random.default_rng(seed)
    return np.argsort(rng.random((N, E)), axis=1)[:, :K].astype(np.int32)


def _outputs(shape, device="cuda"):
    R, T, E, K, cap = (shape.num_ranks, shape.tokens_per_rank, shape.num_experts,
                       shape.top_k, shape.capacity)
    i32 = dict(dtype=torch.int32, device=device)
    return (torch.full((E,), -7, **i32), torch.full((E, R + 1), -7, **i32),
            torch.full((R * T, K), -7, **i32), torch.full((E, cap), -7, **i32))


@pytest.mark.parametrize("R,T,H,E,K", [(8, 128, 7168, 256, 8), (3, 300, 256, 64, 8)])
def test_noalloc_plan_matches_moe_plan(R, T, H, E, K):
    shape = moe.make_shape(R, T, H, E, K, R * T)
    ref = moe.Buffers(shape, expert_x=False, expert_y=False)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((1, 2)):              # two calls in a row
        idx = torch.from_numpy(_routing(seed, R * T, E, K)).cuda()
        ref.src_of.fill_(-7)
        ref.plan(idx)
        assert moe.read_status(ref.workspace) == moe.Status.OK
        cnt, off, slot, src = _outputs(shape)
        status.fill_(-1)
        moe.plan_noalloc(shape, idx, cnt, off, slot, src, status)
        torch.cuda.synchronize()
        assert int(status.item()) == int(moe.Status.OK), f"call {call}: status"
        assert torch.equal(cnt, ref.expert_num_tokens), f"call {call}: counts"
        assert torch.equal(off, ref.expert_rank_offsets), f"call {call}: offsets"
        assert torch.equal(slot, ref.slot_of), f"call {call}: slots"
        assert torch.equal(src, ref.src_of), f"call {call}: src_of"


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # 64 ranks x 1 tile x 2048 experts x 2 rows x 4 B > 1 MiB
    shape = moe.make_shape(64, 16, 256, 2048, 8, 1024)
    assert moe.workspace_size(shape) > (1 << 20)
    cnt, off, slot, src = _outputs(shape)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = moe.plan_noalloc(shape, torch.zeros((64 * 16, 8), dtype=torch.int32, device="cuda"),
                          cnt, off, slot, src, status, check=False)
    assert st == moe.Status.WORKSPACE
