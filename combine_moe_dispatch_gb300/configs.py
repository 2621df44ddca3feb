"""The MoE layer shapes the library is checked and measured on.

Each workload is one MoE layer seen from one GPU whose HBM holds ``R``
logical ranks of ``T`` tokens each.  Sizes follow the model families the
pages deploy: DeepSeek-V3 (hidden 7168, 256 routed experts, top-8: "Lower
latency and higher throughput with multi-node DeepSeek deployment", Expert
Parallelism; "Enabling trillion-parameter models on AWS EFA",
Dispatch/Combine Latency), Kimi-K2 (hidden 7168) and Mixtral 8x7B
("Efficient and portable mixture-of-experts communication", Introduction).
The expert FFN intermediate sizes (``inter``: 2048 per routed expert for
DeepSeek-V3 and Kimi-K2, 14336 for Mixtral) are not on the pages; they are
the published model configurations of those families, used only to size the
activation between the expert GEMMs.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    R: int            # logical ranks
    T: int            # tokens per rank
    H: int            # hidden size
    E: int            # experts
    K: int            # experts per token
    cap: int          # rows per expert in the padded buffers
    payloads: tuple   # dispatch payloads exercised: "bf16", "fp8"
    routing: str      # "uniform", "zipf", or "half_uniform_half_zipf"
    zipf_s: float = 0.0
    description: str = ""
    inter: int = 0    # expert FFN intermediate size (activation between the expert GEMMs)
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return self.R * self.T


WORKLOADS = {
    "tiny": Workload(
        "tiny", R=1, T=64, H=256, E=8, K=2, cap=64, payloads=("bf16",),
        routing="uniform", inter=256,
        description="1 logical rank x 64 tokens, H=256, E=8, top-2, capacity 64, bf16"),
    "mixtral": Workload(
        "mixtral", R=8, T=512, H=4096, E=8, K=2, cap=8 * 512 * 2, payloads=("bf16",),
        routing="uniform", inter=14336,
        description="Mixtral-8x7B-shaped MoE layer: 8 logical ranks x 512 tokens, H=4096, "
                    "E=8, top-2, capacity 8192, bf16"),
    "dsv3_decode": Workload(
        "dsv3_decode", R=8, T=128, H=7168, E=256, K=8, cap=1024, payloads=("bf16", "fp8"),
        routing="uniform", inter=2048,
        description="DeepSeek-V3-shaped decode MoE layer: 8 logical ranks x 128 tokens, "
                    "H=7168, E=256, top-8, capacity 1024, bf16 and fp8-e4m3 dispatch, "
                    "bf16 combine"),
    "dsv3_prefill": Workload(
        "dsv3_prefill", R=16, T=512, H=7168, E=256, K=8, cap=8192, payloads=("fp8",),
        routing="zipf", zipf_s=1.2, inter=2048,
        description="DeepSeek-V3-shaped prefill MoE layer, Zipf(1.2) expert popularity: "
                    "16 logical ranks x 512 tokens, H=7168, E=256, top-8, capacity 8192, "
                    "fp8-e4m3 dispatch, bf16 combine"),
    "kimi_decode": Workload(
        "kimi_decode", R=32, T=128, H=7168, E=384, K=8, cap=4096, payloads=("bf16",),
        routing="half_uniform_half_zipf", zipf_s=1.0, inter=2048,
        description="Kimi-K2-shaped decode MoE layer: 32 logical ranks x 128 tokens, "
                    "H=7168, E=384, top-8, capacity 4096, half uniform / half Zipf(1.0) "
                    "routing, bf16"),
}
