"""Host logic of bench.py that the reported numbers rest on, without a GPU:
the algorithmic bytes of each call (the roofline's numerator), and the code
hash that ties a recorded DRAM-traffic line to the kernel source it was
measured on."""
import os

import bench
from combine_moe_dispatch_gb300.configs import WORKLOADS


def test_algorithmic_bytes_follow_the_formulas():
    for wl in WORKLOADS.values():
        N, H, E, K, R = wl.N, wl.H, wl.E, wl.K, wl.R
        cb = bench.call_bytes(wl)
        plan = N * K * 4 * 3 + E * 4 + E * (R + 1) * 4          # idx in; slot_of, src_of, counts, offsets out
        assert cb["plan"] == plan
        assert cb["dispatch_bf16"] == N * H * 2 + 2 * N * K * 4 + N * K * H * 2
        assert cb["dispatch_fp8"] == N * H * 2 + 2 * N * K * 4 + N * K * H + N * K * (H // 128) * 4
        assert cb["combine"] == N * K * H * 2 + 3 * N * K * 4 + N * H * 2
        for p in ("bf16", "fp8"):
            assert cb["plan_dispatch_" + p] == cb["plan"] + cb["dispatch_" + p]


def test_deepseek_v3_decode_bytes():
    # the figures the roofline of the bench's default workload divides by
    cb = bench.call_bytes(WORKLOADS["dsv3_decode"])
    assert round(cb["dispatch_bf16"] / 1e6, 1) == 132.2
    assert round(cb["dispatch_fp8"] / 1e6, 1) == 75.3
    assert round(cb["combine"] / 1e6, 1) == 132.2
    assert cb["plan_dispatch_bf16"] == 132_294_656


def test_code_hash_ignores_comments_only():
    src = "int f(int a) {\n  // add one\n  return a + 1; /* the sum */\n}\n"
    recommented = "/* f: a + 1 */\nint f(int a) {\n  return a + 1;   // done\n}\n"
    changed = "int f(int a) {\n  return a + 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(recommented)
    assert bench._code_only(src) != bench._code_only(changed)


def test_recorded_traffic_lines_parse():
    # every line names a call the bench times, on a known workload
    calls = set(bench.KERNEL_SOURCES)
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.md")) as f:
        lines = [l.split() for l in f if l.strip().startswith("traffic ")]
    assert lines and all(len(l) == 5 and l[1] in calls and l[2] in WORKLOADS and int(l[3]) > 0
                         for l in lines)
