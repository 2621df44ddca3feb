"""moe_dispatch right after a kernel that writes x and lets its dependents
start early (griddepcontrol.launch_dependents at entry, then a delay, then
the writes): the default dispatch waits for that kernel before reading x, so
every row it writes is the new x's, checked against the oracle.

The same sequence with MOE_DISPATCH_EARLY_X (whose contract the producer
breaks on purpose) is run as a control: it shows whether the producer really
overlapped the dispatch.  Its rows may be stale, so they are only counted."""
import os
import subprocess
import warnings

import numpy as np
import pytest
import torch

import combine_moe_dispatch_gb300 as moe
import oracle
from combine_moe_dispatch_gb300 import inputs
from combine_moe_dispatch_gb300.configs import WORKLOADS

import gpu_check

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
DELAY_NS = 30_000


@pytest.fixture(scope="module")
def producer(tmp_path_factory):
    import ctypes
    out = str(tmp_path_factory.mktemp("pdl") / "libpdl_producer.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", "-o", out, os.path.join(HERE, "pdl_producer.cu")],
                   check=True)
    lib = ctypes.CDLL(out)
    fn = lib.launch_produce_x
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_ulonglong,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _expected_rows(payload, x_new, K, sel):
    """The oracle's dispatched rows (and fp8 scales) of every routed entry,
    in (g, k) order, from the new x."""
    N = x_new.shape[0]
    if payload == "bf16":
        return np.repeat(x_new, K, axis=0)[sel], None
    q, sc = oracle.dispatch_fp8(x_new, np.zeros((N, 1), np.int32),
                                np.arange(N, dtype=np.int32)[:, None], 1, N)
    return np.repeat(q[0], K, axis=0)[sel], np.repeat(sc[0], K, axis=0)[sel]


def _run(producer, buf, x_d, x_old_d, x_new_d, idx_d, early):
    x_d.copy_(x_old_d)
    buf.expert_x.view(torch.uint8).fill_(gpu_check.SENTINEL_BYTE)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    n16 = x_d.numel() * 2 // 16
    assert producer(x_d.data_ptr(), x_new_d.data_ptr(), n16, DELAY_NS, stream.cuda_stream) == 0
    buf.dispatch(x_d, idx_d, early_x=early)
    torch.cuda.synchronize()
    assert moe.read_status(buf.workspace) == moe.Status.OK


@pytest.mark.parametrize("payload", ["bf16", "fp8"])
def test_dispatch_waits_for_an_early_triggering_producer(producer, payload):
    wl = WORKLOADS["dsv3_decode"]
    R, T, H, E, K, N = wl.R, wl.T, wl.H, wl.E, wl.K, wl.N
    d = inputs.make(wl, 0)
    idx = d["topk_idx"]
    x_old = d["x"]
    x_new = inputs.hidden_states(N, H, seed=1)
    assert not np.array_equal(x_old, x_new)
    code = moe.PAYLOAD_BF16 if payload == "bf16" else moe.PAYLOAD_FP8_E4M3
    shape = moe.make_shape(R, T, H, E, K, N, code)
    buf = moe.Buffers(shape, expert_y=False)
    idx_d = gpu_check.dev(idx)
    buf.plan(idx_d)
    assert moe.read_status(buf.workspace) == moe.Status.OK
    st, cnt, off, slot, src = oracle.plan(R, T, E, K, N, idx)
    sel = slot.reshape(-1) >= 0
    e_t = idx_d.long().view(-1)
    s_t = gpu_check.dev(slot.astype(np.int64)).view(-1)
    exp_rows, exp_sc = _expected_rows(payload, x_new, K, sel)
    x_old_d, x_new_d = gpu_check.dev(x_old), gpu_check.dev(x_new)
    x_d = torch.empty_like(x_old_d)

    def rows():
        got = buf.expert_x[e_t, s_t]
        got = gpu_check.host_u16(got) if payload == "bf16" else got.cpu().numpy()
        sc = None if payload == "bf16" else buf.expert_x_scale[e_t, s_t].cpu().numpy()
        return got, sc

    for rep in range(3):
        _run(producer, buf, x_d, x_old_d, x_new_d, idx_d, early=False)
        got, sc = rows()
        bad = np.nonzero((got != exp_rows).any(axis=1))[0]
        assert bad.size == 0, f"rep {rep}: {bad.size} rows dispatched from stale x (first {bad[:4]})"
        if sc is not None:
            assert np.array_equal(sc.view(np.uint32), exp_sc.view(np.uint32)), f"rep {rep}: scales"

    # the control: with the early read the first rows may come from the old x
    _run(producer, buf, x_d, x_old_d, x_new_d, idx_d, early=True)
    got, _ = rows()
    stale = int((got != exp_rows).any(axis=1).sum())
    print(f"{payload}: early read, {stale} of {got.shape[0]} rows from the old x")
    if stale == 0:
        warnings.warn("the producer did not overlap the dispatch; the ordering check was vacuous")
