"""The pins are not vacuous: each plausible mistake planted in a copy of the
oracle's C source (a dropped term, a wrong index, a wrong rounding rule, ...)
must make at least one pin in ``oracle_pins`` fail.  Mutants are compiled
into a temporary directory on the CPU; the real oracle is untouched."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import oracle_pins

# (name, text in moe_oracle.c, replacement).  Every occurrence of the text is
# replaced (the same mistake made consistently).
MUTANTS = [
    ("bf16_ties_away", "(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    ("bf16_truncate", "upper += 1u;", "upper += 0u;"),
    ("bf16_widen_shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("e4m3_floor", "rint(a / spacing)", "floor(a / spacing)"),
    ("e4m3_ties_away", "rint(a / spacing)", "round(a / spacing)"),
    ("e4m3_subnormal_spacing", "if (k < -6) k = -6;", "if (k < -7) k = -7;"),
    ("e4m3_no_saturation", "if (a >= 448.0) return", "if (a >= 480.0) return"),
    ("e4m3_zero_sign", "if (a == 0.0) return sign;", "if (a == 0.0) return 0;"),
    ("e4m3_decode_bias", "ex - 7);", "ex - 8);"),
    ("plan_slot_from_one", "int s = fill[e];\n      fill[e] += 1;", "fill[e] += 1;\n      int s = fill[e] - (e == 0);"),
    ("plan_k_descending", "for (int k = 0; k < K; ++k) {\n      int e = topk_idx[g * K + k];\n      int s = fill[e];",
     "for (int k = K - 1; k >= 0; --k) {\n      int e = topk_idx[g * K + k];\n      int s = fill[e];"),
    ("plan_offsets_inclusive", "g < (int64_t)r * T;", "g <= (int64_t)r * T && g < N;"),
    ("plan_src_drops_k", "src_of[(int64_t)e * cap + s] = (int32_t)(g * K + k);",
     "src_of[(int64_t)e * cap + s] = (int32_t)(g * K);"),
    ("plan_no_capacity_status", "else status = ORACLE_CAPACITY;", "else status = ORACLE_OK;"),
    ("plan_wrong_error_code", "return ORACLE_BAD_EXPERT;", "return ORACLE_CAPACITY;"),
    ("masked_rank0_count", "int64_t nt = num_tokens[r];", "int64_t nt = num_tokens[0];"),
    ("masked_counts_padding", "    if (t >= nt) return 0;", "    if (t > nt) return 0;"),
    ("masked_routes_minus_one", "  return topk_idx[g * K + k] != -1;", "  return topk_idx[g * K + k] != -2;"),
    ("dispatch_bf16_swap_pairs", "dst[h] = x[g * H + h];", "dst[h] = x[g * H + (h ^ 1)];"),
    ("quant_scale_447", "float s = amax / 448.0f;", "float s = amax / 447.0f;"),
    ("quant_amax_drops_last", "for (int i = b * 128; i < end; ++i) {\n      float a",
     "for (int i = b * 128; i < end - 1; ++i) {\n      float a"),
    ("quant_partial_block_dropped", "const int nb = (H + 127) / 128;", "const int nb = H / 128;"),
    ("quant_partial_block_scale_128", "    float s = amax / 448.0f;\n    scale[b] = s;",
     "    float s = (end - b * 128 < 128 ? amax * 0.5f : amax) / 448.0f;\n    scale[b] = s;"),
    ("quant_zero_block_one", "if (amax == 0.0f) q[i] = 0x00;", "if (amax == 0.0f) q[i] = 0x01;"),
    ("quant_reciprocal", "oracle_bf16_to_f32(row[i]) / s);", "oracle_bf16_to_f32(row[i]) * (448.0f / amax));"),
    ("dispatch_fp8_scale_index", "expert_x_scale[row * nb + b] = sc[b];", "expert_x_scale[row * nb] = sc[b];"),
    ("combine_weight_index", "fmaf(topk_weights[g * K + k], v, acc)", "fmaf(topk_weights[g * K], v, acc)"),
    ("combine_drop_last_k", "acc = fmaf(topk_weights[g * K + k], v, acc);",
     "if (k + 1 < K) acc = fmaf(topk_weights[g * K + k], v, acc);"),
    ("combine_mul_then_add", "acc = fmaf(topk_weights[g * K + k], v, acc);",
     "acc = topk_weights[g * K + k] * v + acc;"),
    ("combine_k_descending", "float acc = 0.0f;\n      for (int k = 0; k < K; ++k) {",
     "float acc = 0.0f;\n      for (int k = K - 1; k >= 0; --k) {"),
    ("combine_acc_negzero", "float acc = 0.0f;", "float acc = -0.0f;"),
    ("shared_ignored", "float acc = oracle_bf16_to_f32(shared[g * H + h]);", "float acc = 0.0f;"),
    ("router_ties_higher_index", "  return (ia > ib) - (ia < ib);", "  return (ia < ib) - (ia > ib);"),
    ("router_ascending", "  if (la > lb) return -1;\n  if (la < lb) return 1;", "  if (la > lb) return 1;\n  if (la < lb) return -1;"),
    ("router_no_max_shift", "      z[k] = exp((double)router_row[order[k]] - m);", "      z[k] = exp((double)router_row[order[k]]);"),
    ("router_float_softmax", "      topk_weights[g * K + k] = (float)(z[k] / sum);", "      topk_weights[g * K + k] = (float)z[k] / (float)sum + 1e-7f;"),
    ("exp_no_ln2_lo", "  r = fmaf(-n, ln2_lo, r);", "  r = r;"),
    ("exp_floor", "  const float n = rintf(x * log2e);", "  const float n = floorf(x * log2e);"),
    ("exp_short_polynomial", "  float p = 1.98412701e-04f;", "  float p = 0.0f;"),
    ("silu_sign", "  return g / (1.0f + oracle_exp_f32(-g));", "  return g / (1.0f + oracle_exp_f32(g));"),
    ("silu_gate_up_swapped", "        const float g = oracle_bf16_to_f32(h[i]);\n        const float u = oracle_bf16_to_f32(h[I + i]);",
     "        const float u = oracle_bf16_to_f32(h[i]);\n        const float g = oracle_bf16_to_f32(h[I + i]);"),
    ("silu_count_off_by_one", "    for (int s = 0; s < rows; ++s) {", "    for (int s = 0; s + 1 < rows; ++s) {"),
    ("silu_partial_block_dropped", "  const int nb = (I + 127) / 128;", "  const int nb = I / 128;"),
    ("silu_partial_block_amax", "        for (int i = b * 128; i < end; ++i) {\n          const float v = fabsf(a[i]);",
     "        for (int i = b * 128; i < (end - b * 128 < 128 ? end - 1 : end); ++i) {\n          const float v = fabsf(a[i]);"),
    ("shared_after_rounding",
     "      y[g * H + h] = oracle_f32_to_bf16(acc); /* shared + routed, one rounding */",
     "      y[g * H + h] = oracle_f32_to_bf16(oracle_bf16_to_f32(oracle_f32_to_bf16(acc - "
     "oracle_bf16_to_f32(shared[g * H + h]))) + oracle_bf16_to_f32(shared[g * H + h]));"),
]


def _first_failure(o):
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            return check.__name__
    return None


def test_real_oracle_passes_every_pin():
    assert _first_failure(oracle.default()) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mdir = tmp_path / name
    mdir.mkdir()
    shutil.copy(oracle.HDR, mdir / "moe_oracle.h")
    (mdir / "moe_oracle.c").write_text(src.replace(old, new))
    lib = str(mdir / "libmutant.so")
    subprocess.run(oracle.gcc_command(str(mdir / "moe_oracle.c"), lib, str(mdir)), check=True)
    with np.errstate(all="ignore"):
        caught = _first_failure(oracle.Oracle(lib))
    assert caught is not None, f"no pin catches the planted mistake {name}"
