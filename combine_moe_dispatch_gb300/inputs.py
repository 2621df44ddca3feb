"""Seeded synthetic inputs for MoE dispatch and combine.

This module only draws random data.  It holds none of the method's
arithmetic (no counting, slotting, packing, quantising or weighted sums), so
both the CUDA path and the CPU oracle can consume exactly the same bytes.

Recipe (numpy ``default_rng``; one independent child stream per quantity,
spawned from ``SeedSequence(seed)`` in the order x, routing, logits,
expert outputs, gate/up projections, ragged batches, router logits):

* ``x``: N(0,1) in float32, rounded to bf16 by torch's CPU cast (round to
  nearest even).  Returned as ``uint16`` bit patterns.
* routing, "uniform": each token takes K distinct experts uniformly at
  random (the first K of a random permutation of the E expert ids).
* routing, "zipf": expert popularity p_j proportional to 1/j^s for rank
  j = 1..E, ranks assigned to expert ids by a seeded permutation; each token
  draws K distinct experts without replacement with probability
  proportional to p (Gumbel-top-K on log p, which is sequential weighted
  sampling without replacement), in the order drawn.
* routing, "half_uniform_half_zipf": tokens t < T/2 of every rank routed
  "uniform", tokens t >= T/2 routed "zipf".
* weights: softmax over the K chosen experts of N(0,1) logits, computed in
  float64 and stored as float32 (the router's probabilities).
* expert outputs: N(0,1) rounded to bf16, like ``x``.
* gate/up projections (the first expert GEMM's output, [E, cap, 2I]): the
  gate half N(0, 2^2), the up half N(0,1), rounded to bf16.
* ragged batches: valid tokens per logical rank uniform in [T/2, T]; a
  seeded fraction of the routed entries replaced by -1 (masked); the entries
  of tokens beyond a rank's count hold arbitrary expert ids.
* router logits [N, E]: N(0,1) in float32.
"""
from __future__ import annotations

import numpy as np

from .configs import Workload

_STREAMS = ("x", "routing", "logits", "expert_y", "gate_up", "ragged", "router")


def _rng(seed: int, what: str) -> np.random.Generator:
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return np.random.default_rng(children[_STREAMS.index(what)])


def to_bf16_bits(a) -> np.ndarray:
    """float32 -> bf16 bit patterns via torch's CPU cast (nearest even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def hidden_states(N: int, H: int, seed: int = 0) -> np.ndarray:
    """x[N, H] as bf16 bits."""
    return to_bf16_bits(_rng(seed, "x").standard_normal((N, H), dtype=np.float32))


def _uniform_topk(rng: np.random.Generator, n: int, E: int, K: int) -> np.ndarray:
    return np.argsort(rng.random((n, E)), axis=1, kind="stable")[:, :K].astype(np.int32)


def _zipf_topk(rng: np.random.Generator, n: int, E: int, K: int, s: float) -> np.ndarray:
    perm = rng.permutation(E)
    logp = np.empty(E, np.float64)
    logp[perm] = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    keys = logp[None, :] + rng.gumbel(size=(n, E))
    return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)


def routing(wl: Workload, seed: int = 0) -> np.ndarray:
    """topk_idx[N, K] int32 (K distinct experts per token)."""
    rng = _rng(seed, "routing")
    if wl.routing == "uniform":
        return _uniform_topk(rng, wl.N, wl.E, wl.K)
    if wl.routing == "zipf":
        return _zipf_topk(rng, wl.N, wl.E, wl.K, wl.zipf_s)
    if wl.routing == "half_uniform_half_zipf":
        uni = _uniform_topk(rng, wl.N, wl.E, wl.K)
        zipf = _zipf_topk(rng, wl.N, wl.E, wl.K, wl.zipf_s)
        t = np.arange(wl.N) % wl.T
        return np.where((t < wl.T // 2)[:, None], uni, zipf).astype(np.int32)
    raise ValueError(f"unknown routing {wl.routing!r}")


def weights(N: int, K: int, seed: int = 0) -> np.ndarray:
    """topk_weights[N, K] float32: softmax of N(0,1) logits over the K chosen."""
    z = _rng(seed, "logits").standard_normal((N, K))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def expert_outputs(E: int, cap: int, H: int, seed: int = 0) -> np.ndarray:
    """expert_y[E, cap, H] as bf16 bits, every row N(0,1) (host; small shapes)."""
    return to_bf16_bits(_rng(seed, "expert_y").standard_normal((E, cap, H), dtype=np.float32))


def expert_outputs_device(E: int, cap: int, H: int, seed: int = 0, device="cuda"):
    """expert_y[E, cap, H] bf16 drawn on the device with a seeded torch
    generator (large shapes, where a host copy would not fit).  Deterministic
    for a given seed and device type."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn((E, cap, H), generator=gen, device=device, dtype=torch.bfloat16)


def gate_up(E: int, cap: int, I: int, seed: int = 0) -> np.ndarray:
    """expert_h[E, cap, 2I] as bf16 bits: gate half N(0, 4), up half N(0, 1)."""
    z = _rng(seed, "gate_up").standard_normal((E, cap, 2 * I), dtype=np.float32)
    z[..., :I] *= 2.0
    return to_bf16_bits(z)


def gate_up_device(E: int, cap: int, I: int, seed: int = 0, device="cuda"):
    """As ``gate_up`` drawn on the device with a seeded torch generator
    (bf16 N(0,1), the gate half then doubled: exact in bf16)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    z = torch.randn((E, cap, 2 * I), generator=gen, device=device, dtype=torch.bfloat16)
    z[..., :I] *= 2
    return z


def ragged_batch(R: int, T: int, topk_idx: np.ndarray, E: int, mask_frac: float = 1 / 32,
                 seed: int = 0):
    """(num_tokens[R] int32, topk_idx with masked and garbage entries)."""
    rng = _rng(seed, "ragged")
    nt = rng.integers(T // 2, T + 1, size=R).astype(np.int32)
    idx = np.array(topk_idx, dtype=np.int32, copy=True)
    K = idx.shape[1]
    idx[rng.random(idx.shape) < mask_frac] = -1
    t = np.arange(R * T) % T
    beyond = t >= np.repeat(nt, T)
    idx[beyond] = rng.integers(-(1 << 20), 1 << 20, size=(int(beyond.sum()), K)).astype(np.int32)
    return nt, idx


def router_logits(N: int, E: int, seed: int = 0) -> np.ndarray:
    """logits[N, E] float32, N(0,1)."""
    return _rng(seed, "router").standard_normal((N, E), dtype=np.float32)


def make(wl: Workload, seed: int = 0) -> dict:
    """Host inputs of one workload: x, topk_idx, topk_weights."""
    return {
        "x": hidden_states(wl.N, wl.H, seed),
        "topk_idx": routing(wl, seed),
        "topk_weights": weights(wl.N, wl.K, seed),
    }
