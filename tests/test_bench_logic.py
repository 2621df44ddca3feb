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
        assert cb["dispatch_fp8"] == N * H * 2 + 2 * N * K * 4 + N * K * H + N * K * ((H + 127) // 128) * 4
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


def test_step_moves_the_bytes_of_every_row():
    # the step's calls (fused plan + bf16 dispatch, the early-reading fp8
    # dispatch, combine) move exactly the bytes of the rows a1-a6
    for wl in WORKLOADS.values():
        cb = bench.call_bytes(wl)
        assert (sum(cb[bench.base_call(c)] for c in bench.step_sequence(wl))
                == sum(cb[c] for c in bench.step_calls(wl)))
    assert bench.base_call("dispatch_fp8_early") == "dispatch_fp8"
    assert bench.base_call("combine") == "combine"


def test_dispatch_incl_plan_reports_both_two_launch_orders():
    wl = WORKLOADS["dsv3_decode"]
    cb = bench.call_bytes(wl)
    ms = {"plan_dispatch_fp8": 0.016, "plan+dispatch_fp8": 0.018, "plan+dispatch_fp8_early": 0.017}
    d = bench.dispatch_incl_plan(["plan", "dispatch_fp8"], ms, cb, 6782.4)
    b = cb["plan"] + cb["dispatch_fp8"]
    assert abs(d["fp8"]["us"] - 16.0) < 1e-9
    assert abs(d["fp8"]["frac_of_peak"] - b / 16e-6 / 1e9 / 6782.4) < 1e-12
    assert abs(d["fp8"]["two_launches_us"] - 17.0) < 1e-9
    assert abs(d["fp8"]["two_launches_default_us"] - 18.0) < 1e-9
    assert set(bench.EXTRA_WORKLOADS) <= set(WORKLOADS)
