"""Named workload shapes for the decode path (sizes only, no arithmetic).

Each entry is a pre-LN GPT-style layer or stack: hidden H, heads nh (head_dim
d = H / nh), FFN width F, number of layers, batch rows, cached positions and
decode steps.  The 7B-shaped fp16 stack at batch 1 is the headline bench
workload.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    heads: int
    ffn: int
    layers: int
    batches: tuple
    past: int            # cached positions before the first decode step
    steps: int           # decode steps
    weight_dtype: str    # "f16" | "bf16" | "i8"
    act_dtype: str = "f16"
    quant_group: int = 64
    seed: int = 1000

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads


WORKLOADS = {
    # One layer, H=256, 4 heads (d=64), FFN 1024, batch 1, 32 cached positions.
    "layer256": Workload("layer256", 256, 4, 1024, 1, (1,), 32, 1, "f16", seed=1000),
    # GPT-Neo-2.7B-shaped: 32 layers, H=2560, 20 heads, FFN 10240, 128 cached, 64 steps.
    "neo2p7b": Workload("neo2p7b", 2560, 20, 10240, 32, (1,), 128, 64, "f16", seed=1001),
    # 7B-shaped: 32 layers, H=4096, 32 heads, FFN 16384, 512 cached, 64 steps.
    "gpt7b": Workload("gpt7b", 4096, 32, 16384, 32, (1, 4, 8), 512, 64, "f16", seed=1002),
    # One 4096-hidden layer's four skinny GEMMs, batch rows 1..64.
    "sweep4096": Workload("sweep4096", 4096, 32, 16384, 1, (1, 2, 4, 8, 16, 32, 64), 512, 1,
                          "f16", seed=1003),
    # 13B-shaped MoQ int8 (group 64): 40 layers, H=5120, 40 heads, FFN 20480, 1024 cached.
    "moq13b": Workload("moq13b", 5120, 40, 20480, 40, (1, 16), 1024, 64, "i8", seed=1004),
}


def weight_bytes_per_layer(w: Workload) -> int:
    """Bytes of one layer's parameters as stored (weights + biases + LN + scales)."""
    H, F = w.hidden, w.ffn
    n_w = 3 * H * H + H * H + F * H + H * F
    n_small = 3 * H + H + F + H + 4 * H  # biases + LN gamma/beta
    if w.weight_dtype == "i8":
        return n_w + 2 * (n_w // w.quant_group) + 2 * n_small
    return 2 * n_w + 2 * n_small
