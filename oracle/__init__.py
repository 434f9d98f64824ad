"""CPU oracle for the fused transformer-layer decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``transformer_layer_gb300``) never imports it, and
this package imports nothing from the product path.

Everything here is plain numpy in float64 with no intermediate rounding: it
states what one pre-LN GPT-style layer computes, region by region, as the page
"DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核与
MoQ 量化支持" describes it (§3 "面向 Transformer 块的定制化推理内核", §3.2
"一个 Transformer 层中的四大融合区域", and §5.2 for the int8 weights).  The
pages print no formula, so each function names the reading it takes.

Modules
-------
layer   LayerNorm, linear, GeLU(tanh), softmax, KV-cache decode attention and
        the whole layer / stack forward.
quant   MoQ-style symmetric per-group int8 quantisation and dequantisation.
moe     the residual-MoE (PR-MoE) FFN block with top-1 routing.
tp      the tensor-sliced (Megatron-style) layer: shards, per-rank partial
        sums and their reduction.
"""
from .layer import (layer_norm, linear, gelu_tanh, softmax, decode_attention,
                    layer_forward, stack_forward, LAYER_PARAM_NAMES)
from .quant import quantize_int8, dequantize_int8, fp16_scale_from_amax
from .moe import ffn, residual_moe_ffn
from .tp import shard_layer_params, tp_attention_partial, tp_ffn_partial, tp_layer_forward

__all__ = [
    "layer_norm", "linear", "gelu_tanh", "softmax", "decode_attention",
    "layer_forward", "stack_forward", "LAYER_PARAM_NAMES",
    "quantize_int8", "dequantize_int8", "fp16_scale_from_amax", "ffn", "residual_moe_ffn",
    "shard_layer_params", "tp_attention_partial", "tp_ffn_partial", "tp_layer_forward",
]
