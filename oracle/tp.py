"""Tensor-sliced (Megatron-style) layer: plain float64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source page, cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
算子融合推理内核与 MoQ 量化支持".  §3.2 states that the layer's attention (Attn)
and feed-forward (FF) blocks are split across GPUs in the Megatron-LM manner,
with one cross-GPU all-reduce after each block; §3.1 (second fusion principle)
makes each all-reduce a fusion boundary; the injection-policy passage of the
same page names the two linear layers that take part in the cross-GPU
reduction: the attention output GEMM and the layer output GEMM.

The pages give no formula.  The reading taken (the plain Megatron split) for
W ranks, rank r, heads nh, hidden H, FFN width F, Hl = H / W, Fl = F / W:
  * rank r owns heads r*nh/W .. (r+1)*nh/W - 1: the q, k and v rows of those
    heads in W_qkv / b_qkv, their KV cache, and columns r*Hl .. (r+1)*Hl - 1
    of W_o (the inputs that come from those heads);
  * rank r owns FFN features r*Fl .. (r+1)*Fl - 1: those rows of W_1 / b_1
    and those columns of W_2;
  * LayerNorm parameters are replicated; the biases of the two reduced GEMMs
    (b_o, b_2) and the residuals are added once, by rank 0, before the sum;
  * attention partial:  x1_r = [r == 0](x + b_o) + o_r W_o[:, cols_r]^T
    all-reduce:          x1 = sum_r x1_r
    FFN partial:         y_r = [r == 0](x1 + b_2)
                               + GeLU(LN2(x1) W_1[rows_r]^T + b_1[rows_r]) W_2[:, rows_r]^T
    all-reduce:          y = sum_r y_r.
The sum over ranks equals the unsplit layer (oracle.layer.layer_forward) up
to rounding: attention is per head, GeLU is per feature, and a GEMM whose
input axis is split is the sum of the pieces' GEMMs.
"""
from __future__ import annotations

import numpy as np

from .layer import decode_attention, gelu_tanh, layer_norm, linear


def shard_layer_params(p, heads, tp_size, rank):
    """Rank `rank`'s part of the full layer parameters p (names of
    LAYER_PARAM_NAMES, weights [out][in]).  Shapes: w_qkv [3 Hl][H] (q, k, v
    rows of the rank's heads, in that order), b_qkv [3 Hl], w_o [H][Hl],
    w_fc1 [Fl][H], b_fc1 [Fl], w_fc2 [H][Fl]; LayerNorm parameters, b_o and
    b_fc2 unchanged."""
    H = np.asarray(p["w_qkv"]).shape[1]
    F = np.asarray(p["w_fc1"]).shape[0]
    assert heads % tp_size == 0 and H % tp_size == 0 and F % tp_size == 0
    Hl, Fl = H // tp_size, F // tp_size
    hs = slice(rank * Hl, (rank + 1) * Hl)   # the rank's heads, as feature columns
    fs = slice(rank * Fl, (rank + 1) * Fl)   # the rank's FFN features
    w_qkv = np.asarray(p["w_qkv"])
    b_qkv = np.asarray(p["b_qkv"])
    s = dict(p)
    s["w_qkv"] = np.concatenate([w_qkv[part * H:(part + 1) * H][hs] for part in range(3)], axis=0)
    s["b_qkv"] = np.concatenate([b_qkv[part * H:(part + 1) * H][hs] for part in range(3)], axis=0)
    s["w_o"] = np.asarray(p["w_o"])[:, hs]
    s["w_fc1"] = np.asarray(p["w_fc1"])[fs]
    s["b_fc1"] = np.asarray(p["b_fc1"])[fs]
    s["w_fc2"] = np.asarray(p["w_fc2"])[:, fs]
    return s


def tp_attention_partial(x, s, k_cache, v_cache, past_len, heads_local, rank, eps=1e-5, kv_store=None):
    """Rank's share of x1 (before the first all-reduce) for x [B, T, H].

    s is the rank's shard (shard_layer_params); k_cache / v_cache are the
    rank's float64 caches [B, heads_local, max_len, d], updated in place at
    positions past_len[b] + t (through kv_store, as in layer_forward).
    Returns dict(x1_part [B, T, H], k_new, v_new [B, T, heads_local, d],
    attn [B, T, Hl]).
    """
    x = np.asarray(x, dtype=np.float64)
    B, T, H = x.shape
    Hl = np.asarray(s["w_qkv"]).shape[0] // 3
    d = Hl // heads_local
    h1 = layer_norm(x, s["ln1_g"], s["ln1_b"], eps)
    qkv = linear(h1, s["w_qkv"], s["b_qkv"])
    q = qkv[..., 0:Hl].reshape(B, T, heads_local, d)
    k_new = qkv[..., Hl:2 * Hl].reshape(B, T, heads_local, d)
    v_new = qkv[..., 2 * Hl:3 * Hl].reshape(B, T, heads_local, d)
    store = kv_store if kv_store is not None else (lambda a: a)
    for b in range(B):
        for t in range(T):
            pos = int(past_len[b]) + t
            k_cache[b, :, pos, :] = store(k_new[b, t])
            v_cache[b, :, pos, :] = store(v_new[b, t])
    attn = decode_attention(q, k_cache, v_cache, past_len).reshape(B, T, Hl)
    part = linear(attn, s["w_o"])
    if rank == 0:
        part = part + x + np.asarray(s["b_o"], dtype=np.float64)
    return dict(x1_part=part, k_new=k_new, v_new=v_new, attn=attn)


def tp_ffn_partial(x1, s, rank, eps=1e-5):
    """Rank's share of the layer output (before the second all-reduce), from
    the reduced x1 [..., H].  Returns dict(y_part, g [..., Fl])."""
    x1 = np.asarray(x1, dtype=np.float64)
    h2 = layer_norm(x1, s["ln2_g"], s["ln2_b"], eps)
    g = gelu_tanh(linear(h2, s["w_fc1"], s["b_fc1"]))
    part = linear(g, s["w_fc2"])
    if rank == 0:
        part = part + x1 + np.asarray(s["b_fc2"], dtype=np.float64)
    return dict(y_part=part, g=g)


def tp_layer_forward(x, p, k_caches, v_caches, past_len, heads, tp_size, eps=1e-5, kv_store=None):
    """All ranks of one tensor-sliced layer step, the all-reduces done as
    plain sums in rank order.  k_caches / v_caches: one float64 cache per rank
    [B, heads / tp_size, max_len, d], updated in place.  Returns dict(y, x1,
    x1_parts, y_parts, k_new, v_new (lists per rank))."""
    shards = [shard_layer_params(p, heads, tp_size, r) for r in range(tp_size)]
    att = [tp_attention_partial(x, shards[r], k_caches[r], v_caches[r], past_len, heads // tp_size, r, eps,
                                kv_store) for r in range(tp_size)]
    x1 = att[0]["x1_part"].copy()
    for r in range(1, tp_size):
        x1 = x1 + att[r]["x1_part"]
    ffn = [tp_ffn_partial(x1, shards[r], r, eps) for r in range(tp_size)]
    y = ffn[0]["y_part"].copy()
    for r in range(1, tp_size):
        y = y + ffn[r]["y_part"]
    return dict(y=y, x1=x1, x1_parts=[a["x1_part"] for a in att], y_parts=[f["y_part"] for f in ffn],
                k_new=[a["k_new"] for a in att], v_new=[a["v_new"] for a in att])
