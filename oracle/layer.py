"""Plain float64 CPU oracle of one pre-LN GPT-style transformer layer (decode).

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path imports this module.

Source page, cited below as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU
自适应并行、算子融合推理内核与 MoQ 量化支持".  The attention mask type is a field
of the inference config on the page "DeepSpeed MoE 大规模稀疏模型推理实战指南：
并行切分、PR-MoE 优化与 init_inference 全解析", table "推理配置参数详解"
(``triangular_masking``), cited as [P3].

[P1] §3.2 splits a layer into four fusion regions:
  (1) input LayerNorm + Q, K, V GEMM + bias-add;
  (2) "transform + attention" (the attention GEMMs, read through an implicit
      head-split layout);
  (3) intermediate FF + LayerNorm + bias-add + residual + GeLU;
  (4) bias-add + residual.
This oracle does not fuse anything.  It computes the layer in the plain order
  h1 = LN1(x);  [q|k|v] = h1 W_qkv^T + b_qkv;  append k, v to the cache;
  o  = softmax(q K^T / sqrt(d), causal) V per head;
  x1 = x + o W_o^T + b_o;  h2 = LN2(x1);
  g  = GeLU_tanh(h2 W_1^T + b_1);  y = x1 + g W_2^T + b_2.
The pages give no formula.  The readings taken where they are silent:
  * LayerNorm: biased variance (divide by H), eps = 1e-5, affine after the
    normalisation.
  * Attention scale 1/sqrt(head_dim).
  * GeLU is the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
  * Causal mask ([P3] triangular_masking): new token t of a sequence whose
    cache already holds L positions attends keys 0 .. L+t.
  * Fused QKV weight rows are ordered q, then k, then v; inside each block,
    head i owns rows i*d .. (i+1)*d - 1.
  * Weights are [out][in] row-major (a row is one output feature).
"""
from __future__ import annotations

import numpy as np

LAYER_PARAM_NAMES = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                     "ln2_g", "ln2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def layer_norm(x, gamma, beta, eps=1e-5):
    """LayerNorm over the last axis ([P1] §3.2 regions 1 and 3).

    mean and biased variance over the features, then the affine gamma, beta.
    """
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * _f64(gamma) + _f64(beta)


def linear(x, w, b=None):
    """y = x W^T + b with W stored [out][in] ([P1] §3 intro: the vector-matrix /
    skinny matrix-matrix GEMM that every region is built on)."""
    y = _f64(x) @ _f64(w).T
    if b is not None:
        y = y + _f64(b)
    return y


def gelu_tanh(x):
    """GeLU in its tanh form ([P1] §3.2 region 3 names GeLU; the tanh form is
    the reading taken for every configuration)."""
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def softmax(s, axis=-1):
    """Numerically safe softmax (max subtracted before the exponential)."""
    s = _f64(s)
    m = s.max(axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=axis, keepdims=True)


def decode_attention(q, k_cache, v_cache, past_len):
    """Region 2 of [P1] §3.2: scaled dot-product attention over a KV cache.

    q        [B, T, nh, d]   queries of the T new tokens of each sequence
    k_cache  [B, nh, max_len, d]  keys; positions past_len[b] .. +T-1 already
             hold the new tokens' keys
    v_cache  same layout as k_cache
    past_len [B] positions already cached before this call

    Query t of sequence b attends keys 0 .. past_len[b]+t (causal, [P3]
    triangular_masking), with scores scaled by 1/sqrt(d).
    Returns o [B, T, nh, d].
    """
    q = _f64(q)
    B, T, nh, d = q.shape
    out = np.zeros_like(q)
    scale = 1.0 / np.sqrt(d)
    for b in range(B):
        for t in range(T):
            S = int(past_len[b]) + t + 1
            for h in range(nh):
                K = _f64(k_cache[b, h, :S, :])
                V = _f64(v_cache[b, h, :S, :])
                p = softmax(K @ q[b, t, h] * scale)
                out[b, t, h] = p @ V
    return out


def layer_forward(x, p, k_cache, v_cache, past_len, heads, eps=1e-5, kv_store=None):
    """One pre-LN layer over T new tokens per sequence ([P1] §3.2, regions 1-4).

    x        [B, T, H] layer input (float64 copy of what the device receives)
    p        dict with the arrays named in LAYER_PARAM_NAMES (weights [out][in])
    k_cache, v_cache  float64 [B, nh, max_len, d]; the new keys / values are
             written in place at positions past_len[b] + t
    past_len [B]
    heads    number of attention heads nh (d = H / nh)
    kv_store optional function applied to the new keys and values as they are
             written into the cache (the cache's storage format, e.g. rounding
             to float16 / bfloat16); attention reads the cache, so with T > 1
             the new tokens see each other's stored keys and values.  Default:
             stored exactly.  The returned k_new / v_new are the exact values.

    Returns a dict: y (layer output), h1, q, k_new, v_new [B, T, nh, d],
    attn (o before the output projection, [B, T, H]), x1, h2, g.
    """
    x = _f64(x)
    B, T, H = x.shape
    d = H // heads
    # Region 1: input LayerNorm, fused QKV projection and its bias.
    h1 = layer_norm(x, p["ln1_g"], p["ln1_b"], eps)
    qkv = linear(h1, p["w_qkv"], p["b_qkv"])
    q = qkv[..., 0:H].reshape(B, T, heads, d)
    k_new = qkv[..., H:2 * H].reshape(B, T, heads, d)
    v_new = qkv[..., 2 * H:3 * H].reshape(B, T, heads, d)
    store = kv_store if kv_store is not None else (lambda a: a)
    for b in range(B):
        for t in range(T):
            pos = int(past_len[b]) + t
            k_cache[b, :, pos, :] = store(k_new[b, t])
            v_cache[b, :, pos, :] = store(v_new[b, t])
    # Region 2: attention over the cache (scale, causal mask, softmax, . V).
    attn = decode_attention(q, k_cache, v_cache, past_len).reshape(B, T, H)
    # Region 3 (first half): output projection, bias, residual, next LayerNorm.
    x1 = x + linear(attn, p["w_o"], p["b_o"])
    h2 = layer_norm(x1, p["ln2_g"], p["ln2_b"], eps)
    # Region 3 (second half): FFN up-projection, bias, GeLU.
    g = gelu_tanh(linear(h2, p["w_fc1"], p["b_fc1"]))
    # Region 4: FFN down-projection, bias, residual.
    y = x1 + linear(g, p["w_fc2"], p["b_fc2"])
    return dict(y=y, h1=h1, q=q, k_new=k_new, v_new=v_new, attn=attn,
                x1=x1, h2=h2, g=g)


def stack_forward(x, layers, k_caches, v_caches, past_len, heads, eps=1e-5):
    """A stack of layers: the output of layer l is the input of layer l+1.

    layers / k_caches / v_caches are lists (one entry per layer); the caches are
    float64 and updated in place.  Returns the list of per-layer result dicts.
    """
    outs = []
    h = _f64(x)
    for l, p in enumerate(layers):
        r = layer_forward(h, p, k_caches[l], v_caches[l], past_len, heads, eps)
        outs.append(r)
        h = r["y"]
    return outs
