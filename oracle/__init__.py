"""CPU oracle for MoE token dispatch and combine: TEST INFRASTRUCTURE ONLY.

This package wraps ``moe_oracle.c``, a plain single-threaded C implementation
of the definitions (the header ``moe_oracle.h`` states what each function
computes and which page and section it follows).  Only the tests, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import it.  The CUDA library never calls it and shares no code with it.

Arrays are numpy: bf16 values travel as ``uint16`` bit patterns and e4m3
values as ``uint8`` bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
HDR = os.path.join(HERE, "moe_oracle.h")
LIB = os.path.join(HERE, "libmoe_oracle.so")

OK, BAD_EXPERT, CAPACITY, BAD_SHAPE = 0, 1, 2, 3


def gcc_command(src: str, out: str, include_dir: str = HERE) -> list:
    """Plain IEEE binary32 arithmetic: no fast-math, and no contraction of
    a*b+c into an fma except where the C source calls fmaf() itself."""
    return ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-I", include_dir, "-o", out, src, "-lm"]


def build(src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle into a shared library (default: next to its source)."""
    subprocess.run(gcc_command(src, out), check=True)
    return out


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return t < os.path.getmtime(SRC) or t < os.path.getmtime(HDR)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """The oracle's entry points over numpy arrays, bound to one build of the
    library (the default build, or a test's deliberately broken copy)."""

    def __init__(self, lib_path: str = LIB):
        lib = ctypes.CDLL(lib_path)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.oracle_plan.argtypes = [I, I, I, I, I, P, P, P, P, P]
        lib.oracle_plan.restype = I
        lib.oracle_plan_masked.argtypes = [I, I, I, I, I, P, P, P, P, P, P]
        lib.oracle_plan_masked.restype = I
        lib.oracle_dispatch_bf16.argtypes = [I, I, I, I, I, P, P, P, P]
        lib.oracle_dispatch_bf16.restype = None
        lib.oracle_quant_row_e4m3.argtypes = [I, P, P, P]
        lib.oracle_quant_row_e4m3.restype = None
        lib.oracle_dispatch_fp8.argtypes = [I, I, I, I, I, P, P, P, P, P]
        lib.oracle_dispatch_fp8.restype = None
        lib.oracle_combine.argtypes = [I, I, I, I, I, P, P, P, P, P]
        lib.oracle_combine.restype = None
        lib.oracle_combine_shared.argtypes = [I, I, I, I, I, P, P, P, P, P, P]
        lib.oracle_combine_shared.restype = None
        lib.oracle_router_topk.argtypes = [I, I, I, P, P, P]
        lib.oracle_router_topk.restype = None
        lib.oracle_exp_f32.argtypes = [ctypes.c_float]
        lib.oracle_exp_f32.restype = ctypes.c_float
        lib.oracle_silu_f32.argtypes = [ctypes.c_float]
        lib.oracle_silu_f32.restype = ctypes.c_float
        lib.oracle_silu_mul_quant.argtypes = [I, I, I, P, P, P, P]
        lib.oracle_silu_mul_quant.restype = None
        for name in ("oracle_bf16_to_f32_n", "oracle_f32_to_bf16_n",
                     "oracle_e4m3_to_f32_n", "oracle_f32_to_e4m3_n"):
            getattr(lib, name).argtypes = [I64, P, P]
            getattr(lib, name).restype = None
        self.lib = lib
        self.path = lib_path

    # --- number formats ------------------------------------------------------
    def bf16_to_f32(self, bits) -> np.ndarray:
        b = _c(bits, np.uint16)
        out = np.empty(b.shape, np.float32)
        self.lib.oracle_bf16_to_f32_n(b.size, _ptr(b), _ptr(out))
        return out

    def f32_to_bf16(self, vals) -> np.ndarray:
        v = _c(vals, np.float32)
        out = np.empty(v.shape, np.uint16)
        self.lib.oracle_f32_to_bf16_n(v.size, _ptr(v), _ptr(out))
        return out

    def e4m3_to_f32(self, codes) -> np.ndarray:
        c = _c(codes, np.uint8)
        out = np.empty(c.shape, np.float32)
        self.lib.oracle_e4m3_to_f32_n(c.size, _ptr(c), _ptr(out))
        return out

    def f32_to_e4m3(self, vals) -> np.ndarray:
        v = _c(vals, np.float32)
        out = np.empty(v.shape, np.uint8)
        self.lib.oracle_f32_to_e4m3_n(v.size, _ptr(v), _ptr(out))
        return out

    # --- the method ----------------------------------------------------------
    def plan(self, R: int, T: int, E: int, K: int, cap: int, topk_idx):
        """Return (status, expert_num_tokens[E], expert_rank_offsets[E,R+1],
        slot_of[N,K], src_of[E,cap]).  Entries the oracle does not write keep
        -1 (``src_of`` beyond each count; everything on BAD_EXPERT)."""
        idx = _c(topk_idx, np.int32).reshape(R * T, K)
        cnt = np.full(E, -1, np.int32)
        off = np.full((E, R + 1), -1, np.int32)
        slot = np.full((R * T, K), -1, np.int32)
        src = np.full((E, cap), -1, np.int32)
        st = self.lib.oracle_plan(R, T, E, K, cap, _ptr(idx), _ptr(cnt), _ptr(off),
                                  _ptr(slot), _ptr(src))
        return st, cnt, off, slot, src

    def plan_masked(self, R: int, T: int, E: int, K: int, cap: int, topk_idx, num_tokens=None):
        """As ``plan`` for ragged ranks (``num_tokens[R]``, None = all T) and
        masked entries (expert id -1)."""
        idx = _c(topk_idx, np.int32).reshape(R * T, K)
        nt = None if num_tokens is None else _c(num_tokens, np.int32)
        cnt = np.full(E, -1, np.int32)
        off = np.full((E, R + 1), -1, np.int32)
        slot = np.full((R * T, K), -7, np.int32)
        src = np.full((E, cap), -1, np.int32)
        st = self.lib.oracle_plan_masked(R, T, E, K, cap, _ptr(idx), None if nt is None else _ptr(nt),
                                         _ptr(cnt), _ptr(off), _ptr(slot), _ptr(src))
        return st, cnt, off, slot, src

    def dispatch_bf16(self, x_bits, topk_idx, slot_of, E: int, cap: int, out=None):
        x = _c(x_bits, np.uint16)
        N, H = x.shape
        idx = _c(topk_idx, np.int32)
        slot = _c(slot_of, np.int32)
        if out is None:
            out = np.zeros((E, cap, H), np.uint16)
        self.lib.oracle_dispatch_bf16(N, H, E, idx.shape[1], cap, _ptr(x), _ptr(idx),
                                      _ptr(slot), _ptr(out))
        return out

    def quant_row_e4m3(self, row_bits):
        r = _c(row_bits, np.uint16)
        H = r.shape[0]
        q = np.empty(H, np.uint8)
        sc = np.empty((H + 127) // 128, np.float32)
        self.lib.oracle_quant_row_e4m3(H, _ptr(r), _ptr(q), _ptr(sc))
        return q, sc

    def dispatch_fp8(self, x_bits, topk_idx, slot_of, E: int, cap: int,
                     out=None, out_scale=None):
        x = _c(x_bits, np.uint16)
        N, H = x.shape
        idx = _c(topk_idx, np.int32)
        slot = _c(slot_of, np.int32)
        if out is None:
            out = np.zeros((E, cap, H), np.uint8)
        if out_scale is None:
            out_scale = np.zeros((E, cap, (H + 127) // 128), np.float32)
        self.lib.oracle_dispatch_fp8(N, H, E, idx.shape[1], cap, _ptr(x), _ptr(idx),
                                     _ptr(slot), _ptr(out), _ptr(out_scale))
        return out, out_scale

    def combine(self, expert_y_bits, topk_idx, slot_of, topk_weights):
        ey = _c(expert_y_bits, np.uint16)
        E, cap, H = ey.shape
        idx = _c(topk_idx, np.int32)
        N, K = idx.shape
        slot = _c(slot_of, np.int32)
        w = _c(topk_weights, np.float32)
        y = np.empty((N, H), np.uint16)
        self.lib.oracle_combine(N, H, E, K, cap, _ptr(ey), _ptr(idx), _ptr(slot),
                                _ptr(w), _ptr(y))
        return y


    def combine_shared(self, expert_y_bits, topk_idx, slot_of, topk_weights, shared_bits):
        ey = _c(expert_y_bits, np.uint16)
        E, cap, H = ey.shape
        idx = _c(topk_idx, np.int32)
        N, K = idx.shape
        slot = _c(slot_of, np.int32)
        w = _c(topk_weights, np.float32)
        sh = _c(shared_bits, np.uint16)
        y = np.empty((N, H), np.uint16)
        self.lib.oracle_combine_shared(N, H, E, K, cap, _ptr(ey), _ptr(idx), _ptr(slot), _ptr(w),
                                       _ptr(sh), _ptr(y))
        return y


    def router_topk(self, logits, K: int):
        lg = _c(logits, np.float32)
        N, E = lg.shape
        idx = np.empty((N, K), np.int32)
        w = np.empty((N, K), np.float32)
        self.lib.oracle_router_topk(N, E, K, _ptr(lg), _ptr(idx), _ptr(w))
        return idx, w


    def exp_f32(self, x) -> np.ndarray:
        x = np.asarray(x, np.float32).ravel()
        return np.array([self.lib.oracle_exp_f32(float(v)) for v in x], np.float32)

    def silu_f32(self, x) -> np.ndarray:
        x = np.asarray(x, np.float32).ravel()
        return np.array([self.lib.oracle_silu_f32(float(v)) for v in x], np.float32)

    def silu_mul_quant(self, expert_h_bits, expert_num_tokens, act_q=None, act_scale=None):
        h = _c(expert_h_bits, np.uint16)
        E, cap, I2 = h.shape
        I = I2 // 2
        cnt = _c(expert_num_tokens, np.int32)
        if act_q is None:
            act_q = np.zeros((E, cap, I), np.uint8)
        if act_scale is None:
            act_scale = np.zeros((E, cap, (I + 127) // 128), np.float32)
        self.lib.oracle_silu_mul_quant(E, cap, I, _ptr(h), _ptr(cnt), _ptr(act_q), _ptr(act_scale))
        return act_q, act_scale


_default = None


def default() -> Oracle:
    """The oracle built from this directory's source (compiled on first use
    when the library is missing or older than its source)."""
    global _default
    if _default is None:
        if _stale(LIB):
            build()
        _default = Oracle(LIB)
    return _default


def __getattr__(name):
    # Module-level shortcuts: oracle.plan(...), oracle.combine(...), ...
    if name in ("bf16_to_f32", "f32_to_bf16", "e4m3_to_f32", "f32_to_e4m3", "plan", "plan_masked",
                "dispatch_bf16", "quant_row_e4m3", "dispatch_fp8", "combine", "combine_shared", "router_topk", "exp_f32", "silu_f32",
                "silu_mul_quant"):
        return getattr(default(), name)
    raise AttributeError(name)
