"""The seeded input generator: deterministic, shaped like the workloads, and
with the routing structure each workload names.  CPU only."""
import numpy as np
import pytest

from combine_moe_dispatch_gb300 import inputs
from combine_moe_dispatch_gb300.configs import WORKLOADS


def test_deterministic_and_seed_dependent():
    wl = WORKLOADS["tiny"]
    a, b, c = inputs.make(wl, 0), inputs.make(wl, 0), inputs.make(wl, 1)
    for k in a:
        assert np.array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k])


@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3_decode", "dsv3_prefill", "kimi_decode"])
def test_routing_shapes_and_distinct_experts(name):
    wl = WORKLOADS[name]
    idx = inputs.routing(wl, 0)
    assert idx.shape == (wl.N, wl.K) and idx.dtype == np.int32
    assert idx.min() >= 0 and idx.max() < wl.E
    s = np.sort(idx, axis=1)
    assert (np.diff(s, axis=1) > 0).all(), "K distinct experts per token"
    w = inputs.weights(wl.N, wl.K, 0)
    assert w.dtype == np.float32 and (w > 0).all()
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


def test_zipf_skew_matches_popularity():
    wl = WORKLOADS["dsv3_prefill"]
    idx = inputs.routing(wl, 0)
    cnt = np.bincount(idx.ravel(), minlength=wl.E)
    # Zipf(1.2) over 256 experts, K=8 without replacement: the most popular
    # expert is picked by most tokens, the least popular by few.
    assert cnt.max() > 0.6 * wl.N
    assert cnt.min() < 0.05 * wl.N
    uni = inputs.routing(WORKLOADS["dsv3_decode"], 0)
    ucnt = np.bincount(uni.ravel(), minlength=256)
    assert ucnt.max() < 3 * ucnt.mean()


def test_kimi_half_uniform_half_zipf():
    wl = WORKLOADS["kimi_decode"]
    idx = inputs.routing(wl, 0)
    t = np.arange(wl.N) % wl.T
    lo = np.bincount(idx[t < wl.T // 2].ravel(), minlength=wl.E)
    hi = np.bincount(idx[t >= wl.T // 2].ravel(), minlength=wl.E)
    assert hi.max() > 3 * lo.max()


def test_hidden_states_are_bf16_normal():
    x = inputs.hidden_states(256, 512, 0)
    assert x.dtype == np.uint16
    f = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1) < 0.02
