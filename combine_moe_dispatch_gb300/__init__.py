"""GB300-native MoE token dispatch and combine.

A thin ctypes binding over ``libmoe_gb300.so`` (C ABI in
``include/moe_dispatch.h``).  The functions keep the C names without the
``moe_`` prefix and only marshal arguments: torch tensors become device
pointers, the stream becomes the current torch stream.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback, and a
missing library raises ``LibraryNotBuilt``.

    from combine_moe_dispatch_gb300 import Shape, PAYLOAD_FP8_E4M3, plan, dispatch, combine
"""
from __future__ import annotations

import ctypes
import enum
import os

from . import buildlib as _build

PAYLOAD_BF16 = 0
PAYLOAD_FP8_E4M3 = 1
PAYLOAD_FP8_E4M3_TSCALE = 2   # E4M3 bytes, scales [E, ceil(H/128), cap]
# moe_dispatch_ex flag: x was final before the kernel preceding the dispatch began
DISPATCH_EARLY_X = 1


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    ALIGNMENT = 3
    BAD_EXPERT = 4
    CAPACITY = 5
    TIMEOUT = 6
    CUDA = 7
    WORKSPACE = 8


class MoEError(RuntimeError):
    def __init__(self, status: Status, where: str):
        super().__init__(f"{where}: {Status(status).name} ({status_string(status)})")
        self.status = Status(status)


class LibraryNotBuilt(RuntimeError):
    pass


class Shape(ctypes.Structure):
    """moe_shape: R ranks x T tokens, hidden H, E experts, top-K, capacity, payload."""
    _fields_ = [("num_ranks", ctypes.c_int32), ("tokens_per_rank", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("payload", ctypes.c_int32)]

    @property
    def N(self) -> int:
        return self.num_ranks * self.tokens_per_rank

    @property
    def fp8(self) -> bool:
        return self.payload != PAYLOAD_BF16

    def __repr__(self):
        return (f"Shape(R={self.num_ranks}, T={self.tokens_per_rank}, H={self.hidden}, "
                f"E={self.num_experts}, K={self.top_k}, cap={self.capacity}, "
                f"payload={['bf16', 'fp8', 'fp8, transposed scales'][self.payload]})")


def make_shape(R, T, H, E, K, cap, payload=PAYLOAD_BF16) -> Shape:
    return Shape(R, T, H, E, K, cap, payload)


LIB_PATH = _build.LIB
# Entry points declared in include/moe_dispatch.h, with their C signatures.
_P, _S, _U32, _U64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64
_SP = ctypes.POINTER(Shape)
SIGNATURES = {
    "moe_workspace_size": ([_SP], _S),
    "moe_workspace_init": ([_P, _S, _P], ctypes.c_int),
    "moe_plan": ([_SP, _P, _P, _P, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_dispatch": ([_SP, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_dispatch_ex": ([_SP, _P, _P, _P, _P, _P, _P, _P, _U32], ctypes.c_int),
    "moe_combine": ([_SP, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_read_status": ([_P, _P, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "moe_workspace_set_debug": ([_P, _U32, _U64, _P], ctypes.c_int),
    "moe_plan_noalloc": ([_SP, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_plan_masked": ([_SP, _P, _P, _P, _P, _P, _P, _P, _S, _P], ctypes.c_int),
    "moe_combine_shared": ([_SP, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_router_topk": ([_SP, _P, _P, _P, _P], ctypes.c_int),
    "moe_silu_mul_quant": ([_SP, ctypes.c_int32, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "moe_plan_dispatch": ([_SP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P], ctypes.c_int),
}

_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmoe_gb300.so (built by ``build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise LibraryNotBuilt(
            f"{path} not found: build it with `python -m combine_moe_dispatch_gb300.buildlib` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def build(force: bool = False) -> str:
    return _build.build(force=force)


# --- marshalling helpers -----------------------------------------------------

def _ptr(t) -> int:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(st: int, where: str, check: bool) -> Status:
    st = Status(st)
    if check and st != Status.OK:
        raise MoEError(st, where)
    return st


def status_string(status) -> str:
    return load_library().moe_status_string(int(status)).decode()


# --- the C ABI, one function each --------------------------------------------

def workspace_size(shape: Shape) -> int:
    return load_library().moe_workspace_size(ctypes.byref(shape))


def workspace_init(workspace, stream=None, check=True) -> Status:
    st = load_library().moe_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream))
    return _check(st, "moe_workspace_init", check)


def plan(shape: Shape, topk_idx, expert_num_tokens, expert_rank_offsets, slot_of, src_of,
         workspace, stream=None, check=True) -> Status:
    st = load_library().moe_plan(ctypes.byref(shape), _ptr(topk_idx), _ptr(expert_num_tokens),
                                 _ptr(expert_rank_offsets), _ptr(slot_of), _ptr(src_of),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream))
    return _check(st, "moe_plan", check)


def plan_masked(shape: Shape, topk_idx, num_tokens, expert_num_tokens, expert_rank_offsets,
                slot_of, src_of, workspace, stream=None, check=True) -> Status:
    st = load_library().moe_plan_masked(ctypes.byref(shape), _ptr(topk_idx), _ptr(num_tokens),
                                        _ptr(expert_num_tokens), _ptr(expert_rank_offsets),
                                        _ptr(slot_of), _ptr(src_of), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream))
    return _check(st, "moe_plan_masked", check)


def dispatch(shape: Shape, x, topk_idx, slot_of, expert_x, expert_x_scale, workspace,
             stream=None, check=True, early_x=False) -> Status:
    """moe_dispatch; with ``early_x`` moe_dispatch_ex(MOE_DISPATCH_EARLY_X),
    for callers whose x was final before the preceding kernel began."""
    if early_x:
        st = load_library().moe_dispatch_ex(ctypes.byref(shape), _ptr(x), _ptr(topk_idx),
                                            _ptr(slot_of), _ptr(expert_x), _ptr(expert_x_scale),
                                            _ptr(workspace), _stream(stream), DISPATCH_EARLY_X)
        return _check(st, "moe_dispatch_ex", check)
    st = load_library().moe_dispatch(ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(slot_of),
                                     _ptr(expert_x), _ptr(expert_x_scale), _ptr(workspace),
                                     _stream(stream))
    return _check(st, "moe_dispatch", check)


def dispatch_ex(shape: Shape, x, topk_idx, slot_of, expert_x, expert_x_scale, workspace,
                flags: int, stream=None, check=True) -> Status:
    st = load_library().moe_dispatch_ex(ctypes.byref(shape), _ptr(x), _ptr(topk_idx),
                                        _ptr(slot_of), _ptr(expert_x), _ptr(expert_x_scale),
                                        _ptr(workspace), _stream(stream), flags)
    return _check(st, "moe_dispatch_ex", check)


def plan_dispatch(shape: Shape, x, topk_idx, expert_num_tokens, expert_rank_offsets, slot_of,
                  src_of, expert_x, expert_x_scale, workspace, stream=None, check=True) -> Status:
    """moe_plan followed by moe_dispatch, in one launch where the shape allows."""
    st = load_library().moe_plan_dispatch(ctypes.byref(shape), _ptr(x), _ptr(topk_idx),
                                          _ptr(expert_num_tokens), _ptr(expert_rank_offsets),
                                          _ptr(slot_of), _ptr(src_of), _ptr(expert_x),
                                          _ptr(expert_x_scale), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    return _check(st, "moe_plan_dispatch", check)


def combine(shape: Shape, expert_y, topk_idx, slot_of, topk_weights, y, workspace,
            stream=None, check=True) -> Status:
    st = load_library().moe_combine(ctypes.byref(shape), _ptr(expert_y), _ptr(topk_idx),
                                    _ptr(slot_of), _ptr(topk_weights), _ptr(y), _ptr(workspace),
                                    _stream(stream))
    return _check(st, "moe_combine", check)


def plan_noalloc(shape: Shape, topk_idx, expert_num_tokens, expert_rank_offsets, slot_of, src_of,
                 status_out, stream=None, check=True) -> Status:
    """moe_plan for callers that cannot allocate: scratch in the library's
    static device array; the plan's status goes to the device int32
    ``status_out``."""
    st = load_library().moe_plan_noalloc(ctypes.byref(shape), _ptr(topk_idx),
                                         _ptr(expert_num_tokens), _ptr(expert_rank_offsets),
                                         _ptr(slot_of), _ptr(src_of), _ptr(status_out),
                                         _stream(stream))
    return _check(st, "moe_plan_noalloc", check)


def combine_shared(shape: Shape, expert_y, topk_idx, slot_of, topk_weights, shared_y, y, workspace,
                   stream=None, check=True) -> Status:
    st = load_library().moe_combine_shared(ctypes.byref(shape), _ptr(expert_y), _ptr(topk_idx),
                                           _ptr(slot_of), _ptr(topk_weights), _ptr(shared_y),
                                           _ptr(y), _ptr(workspace), _stream(stream))
    return _check(st, "moe_combine_shared", check)


def router_topk(shape: Shape, logits, topk_idx, topk_weights, stream=None, check=True) -> Status:
    st = load_library().moe_router_topk(ctypes.byref(shape), _ptr(logits), _ptr(topk_idx),
                                        _ptr(topk_weights), _stream(stream))
    return _check(st, "moe_router_topk", check)


def silu_mul_quant(shape: Shape, intermediate: int, expert_h, expert_num_tokens, act_q, act_scale,
                   workspace, stream=None, check=True) -> Status:
    st = load_library().moe_silu_mul_quant(ctypes.byref(shape), intermediate, _ptr(expert_h),
                                           _ptr(expert_num_tokens), _ptr(act_q), _ptr(act_scale),
                                           _ptr(workspace), _stream(stream))
    return _check(st, "moe_silu_mul_quant", check)


def read_status(workspace, stream=None) -> Status:
    out = ctypes.c_int(0)
    st = load_library().moe_read_status(_ptr(workspace), _stream(stream), ctypes.byref(out))
    _check(st, "moe_read_status", True)
    return Status(out.value)


def workspace_set_debug(workspace, flags: int, timeout_ns: int = 0, stream=None, check=True) -> Status:
    st = load_library().moe_workspace_set_debug(_ptr(workspace), flags, timeout_ns, _stream(stream))
    return _check(st, "moe_workspace_set_debug", check)


# --- buffers -----------------------------------------------------------------

class Buffers:
    """Device buffers of one shape, allocated with torch (the library itself
    allocates nothing).  ``expert_x`` is uint8 [E, cap, H] for the fp8
    payloads, bf16 otherwise; ``expert_x_scale`` is [E, cap, ceil(H/128)], or
    [E, ceil(H/128), cap] for PAYLOAD_FP8_E4M3_TSCALE, and None for bf16."""

    def __init__(self, shape: Shape, device="cuda", expert_y: bool = True, expert_x: bool = True):
        import torch
        R, T, H, E, K, cap = (shape.num_ranks, shape.tokens_per_rank, shape.hidden,
                              shape.num_experts, shape.top_k, shape.capacity)
        N = R * T
        i32 = dict(dtype=torch.int32, device=device)
        self.shape = shape
        self.expert_num_tokens = torch.zeros(E, **i32)
        self.expert_rank_offsets = torch.zeros((E, R + 1), **i32)
        self.slot_of = torch.zeros((N, K), **i32)
        self.src_of = torch.zeros((E, cap), **i32)
        ws = workspace_size(shape)
        if ws == 0:
            raise MoEError(Status.UNSUPPORTED, f"workspace_size({shape})")
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)
        if not expert_x:
            self.expert_x = self.expert_x_scale = None
        elif shape.fp8:
            self.expert_x = torch.empty((E, cap, H), dtype=torch.uint8, device=device)
            nb = (H + 127) // 128                      # the last block is short when H % 128 != 0
            sdims = (E, nb, cap) if shape.payload == PAYLOAD_FP8_E4M3_TSCALE else (E, cap, nb)
            self.expert_x_scale = torch.empty(sdims, dtype=torch.float32, device=device)
        else:
            self.expert_x = torch.empty((E, cap, H), dtype=torch.bfloat16, device=device)
            self.expert_x_scale = None
        self.y = torch.empty((N, H), dtype=torch.bfloat16, device=device)
        self.expert_y = (torch.empty((E, cap, H), dtype=torch.bfloat16, device=device)
                         if expert_y else None)

    def plan(self, topk_idx, stream=None, check=True):
        return plan(self.shape, topk_idx, self.expert_num_tokens, self.expert_rank_offsets,
                    self.slot_of, self.src_of, self.workspace, stream, check)

    def plan_masked(self, topk_idx, num_tokens=None, stream=None, check=True):
        return plan_masked(self.shape, topk_idx, num_tokens, self.expert_num_tokens,
                           self.expert_rank_offsets, self.slot_of, self.src_of, self.workspace,
                           stream, check)

    def dispatch(self, x, topk_idx, stream=None, check=True, early_x=False):
        return dispatch(self.shape, x, topk_idx, self.slot_of, self.expert_x, self.expert_x_scale,
                        self.workspace, stream, check, early_x)

    def plan_dispatch(self, x, topk_idx, stream=None, check=True):
        return plan_dispatch(self.shape, x, topk_idx, self.expert_num_tokens,
                             self.expert_rank_offsets, self.slot_of, self.src_of, self.expert_x,
                             self.expert_x_scale, self.workspace, stream, check)

    def combine(self, topk_idx, topk_weights, expert_y=None, stream=None, check=True):
        ey = self.expert_y if expert_y is None else expert_y
        return combine(self.shape, ey, topk_idx, self.slot_of, topk_weights, self.y,
                       self.workspace, stream, check)
