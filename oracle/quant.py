"""MoQ-style symmetric per-group int8 weight quantisation (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: page "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核
与 MoQ 量化支持", §5.2 "推理侧：面向量化模型的高性能内核": int8 inference runs
kernels that dequantise the weights without dedicated int8 hardware, with the
grouping set by ``quantization_setting=(quantize_groups, mlp_extra_grouping)``.
The page fixes neither the group shape nor the rounding.  Readings taken:
  * groups are runs of ``group`` consecutive weights along K (the input axis)
    of one output row; default 64;
  * scale s = max|w| / 127 computed as an IEEE float32 division of the exact
    float32 value of max|w| by 127, then rounded to float16 (round to nearest,
    ties to even);
  * code q = clamp(round_half_even(w / s), -127, 127) with w / s an IEEE
    float32 division (a true division, not a multiply by 1/s);
  * a group whose max|w| is 0 gets s = 0 and all codes 0;
  * dequantised weight = q * s, exact (float64 here).
Both decisions (the scale and the code) are taken in float32, the precision of
the device kernel; the tests show that float64 would give the same integers.
"""
from __future__ import annotations

import numpy as np


def fp16_scale_from_amax(amax):
    """Scale for a group whose largest magnitude is ``amax`` (float16 input).

    float32(amax) / 127 in float32, rounded to float16.  Returns float16.
    """
    a32 = np.asarray(amax, dtype=np.float16).astype(np.float32)
    return (a32 / np.float32(127.0)).astype(np.float16)


def quantize_int8(w, group=64):
    """Quantise a float16 weight matrix [N][K] in groups of ``group`` along K.

    Returns (codes int8 [N][K], scales float16 [N][K // group]).
    """
    w16 = np.asarray(w, dtype=np.float16)
    N, K = w16.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    wg = w16.astype(np.float32).reshape(N, K // group, group)
    amax = np.abs(wg).max(axis=-1)
    s16 = fp16_scale_from_amax(amax.astype(np.float16))
    s32 = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(s32 > 0, wg / np.where(s32 > 0, s32, np.float32(1.0)), np.float32(0.0))
    q = np.clip(np.rint(r), -127, 127).astype(np.int8)
    return q.reshape(N, K), s16


def dequantize_int8(codes, scales, group=64):
    """w = q * s exactly, as float64 [N][K]."""
    q = np.asarray(codes, dtype=np.int8).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    N, K = q.shape
    return (q.reshape(N, K // group, group) * s[..., None]).reshape(N, K)
