"""Residual-MoE (PR-MoE) FFN block: plain float64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source page, cited as [P3]: "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、
PR-MoE 优化与 init_inference 全解析", section "用 PR-MoE 结构进一步提速并降低推理
成本": the residual structure (mlp_type 'residual') with per-layer expert counts,
and the configuration table (moe.type standard / residual, moe_experts).  The
page gives no formula.  Reading taken, the plainest one for a residual MoE with
top-1 routing, for rows x [R, H]:
  h = LayerNorm2(x)                       (biased variance, affine after)
  p = softmax(h W_g^T)                    (W_g [E][H], no bias)
  e = argmax_j p_j                        (ties: the lowest index)
  y = x + MLP(h) + p_e * Expert_e(h)
where MLP and every expert are GeLU(tanh) FFNs: W2 GeLU(W1 h + b1) + b2.
"""
from __future__ import annotations

import numpy as np

from .layer import gelu_tanh, layer_norm, linear, softmax


def ffn(h, w1, b1, w2, b2):
    """One GeLU FFN: W2 GeLU(W1 h + b1) + b2 (weights [out][in])."""
    return linear(gelu_tanh(linear(h, w1, b1)), w2, b2)


def residual_moe_ffn(x, p, eps=1e-5, experts=None):
    """The residual-MoE FFN block over rows x [R, H] (float64).

    p: dict with ln2_g, ln2_b [H]; w_gate [E][H]; the dense MLP w_fc1 [F][H],
    b_fc1 [F], w_fc2 [H][F], b_fc2 [H]; the experts we_fc1 [E][F][H],
    be_fc1 [E][F], we_fc2 [E][H][F], be_fc2 [E][H].
    experts: optional [R] expert indices to use instead of the argmax (to
    evaluate the block at a choice made elsewhere, e.g. at a near-tie).
    Returns a dict: y [R, H], expert [R] (the argmax), logits [R, E],
    weight [R] (p at the expert used), h [R, H].
    """
    x = np.asarray(x, dtype=np.float64)
    h = layer_norm(x, p["ln2_g"], p["ln2_b"], eps)
    logits = linear(h, p["w_gate"])
    probs = softmax(logits, axis=-1)
    e_arg = np.argmax(logits, axis=-1)          # first maximum = lowest index on ties
    e_use = e_arg if experts is None else np.asarray(experts)
    y = x + ffn(h, p["w_fc1"], p["b_fc1"], p["w_fc2"], p["b_fc2"])
    weight = np.empty(x.shape[0])
    for r in range(x.shape[0]):
        e = int(e_use[r])
        weight[r] = probs[r, e]
        y[r] += weight[r] * ffn(h[r], p["we_fc1"][e], p["be_fc1"][e], p["we_fc2"][e], p["be_fc2"][e])
    return dict(y=y, expert=e_arg, logits=logits, weight=weight, h=h)
