"""Seeded synthetic inputs, shared by the device path's tests/bench and the oracle.

This module draws random tensors and nothing else: it holds none of the layer's
arithmetic.  Every tensor is ``torch.randn`` from its own ``torch.Generator``
seeded with (seed, tensor id), scaled and shifted in float32, then rounded to
the storage dtype (round to nearest even).  The same call therefore returns the
same bytes on the same device type; the CPU and CUDA generators give different
streams, so a test hands one set of bytes to both the device path and the
oracle rather than regenerating it.

Distributions follow the workload definitions (weights ~ N(0, 0.02), biases ~
N(0, 0.01), LayerNorm gamma = 1 + N(0, 0.1), beta ~ N(0, 0.1), hidden input and
KV cache ~ N(0, 1)).
"""
from __future__ import annotations

import torch

# Tensor ids: one per named tensor so each one has its own stream.
_IDS = {
    "ln1_g": 1, "ln1_b": 2, "w_qkv": 3, "b_qkv": 4, "w_o": 5, "b_o": 6,
    "ln2_g": 7, "ln2_b": 8, "w_fc1": 9, "b_fc1": 10, "w_fc2": 11, "b_fc2": 12,
    "k_cache": 20, "v_cache": 21, "x": 30,
}


def _gen(seed: int, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(tensor_id) * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def normal(shape, mean, std, seed, tensor_id, dtype=torch.float16, device="cpu"):
    """mean + std * N(0, 1), drawn in float32 and rounded to ``dtype``."""
    g = _gen(seed, tensor_id, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def layer_params(hidden, ffn, seed, layer=0, dtype=torch.float16, device="cpu",
                 w_std=0.02, b_std=0.01, ln_std=0.1):
    """Weights of one layer, [out][in] row-major, in the storage ``dtype``.

    Returns a dict keyed like the oracle's LAYER_PARAM_NAMES.
    """
    H, F = hidden, ffn
    shapes = {
        "ln1_g": (H,), "ln1_b": (H,), "w_qkv": (3 * H, H), "b_qkv": (3 * H,),
        "w_o": (H, H), "b_o": (H,), "ln2_g": (H,), "ln2_b": (H,),
        "w_fc1": (F, H), "b_fc1": (F,), "w_fc2": (H, F), "b_fc2": (H,),
    }
    out = {}
    lseed = int(seed) * 1009 + int(layer)
    for name, shp in shapes.items():
        tid = _IDS[name]
        if name.startswith("w_"):
            out[name] = normal(shp, 0.0, w_std, lseed, tid, dtype, device)
        elif name.startswith("b_"):
            out[name] = normal(shp, 0.0, b_std, lseed, tid, dtype, device)
        elif name.endswith("_g"):
            out[name] = normal(shp, 1.0, ln_std, lseed, tid, dtype, device)
        else:  # LayerNorm beta
            out[name] = normal(shp, 0.0, ln_std, lseed, tid, dtype, device)
    return out


def kv_cache(batch, heads, max_len, head_dim, seed, layer=0, dtype=torch.float16,
             device="cpu"):
    """K and V caches [B][nh][max_len][d], every position ~ N(0, 1)."""
    lseed = int(seed) * 1009 + int(layer)
    shp = (batch, heads, max_len, head_dim)
    return (normal(shp, 0.0, 1.0, lseed, _IDS["k_cache"], dtype, device),
            normal(shp, 0.0, 1.0, lseed, _IDS["v_cache"], dtype, device))


def hidden(batch, tokens, hidden_size, seed, step=0, dtype=torch.float16, device="cpu"):
    """Layer input [B][T][H] ~ N(0, 1); ``step`` gives each decode step its own draw."""
    return normal((batch, tokens, hidden_size), 0.0, 1.0, int(seed) * 131 + int(step),
                  _IDS["x"], dtype, device)
