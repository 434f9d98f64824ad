"""Full-depth stack parity: the 7B-shaped fp16 stack (32 layers, hidden 4096,
512 cached positions) and the 13B-shaped MoQ int8 stack (40 layers, hidden
5120, groups of 64, 1024 cached positions) at batch 1 (streaming kernels) and
batch 16 (tensor-core tiles; ragged cached lengths), decoded for 64 steps
through the graph-replayed stack step, exactly as the benchmark runs them.

At decode steps 1 and 64 the first, a middle and the last layer are checked
teacher-forced against the float64 oracle: the oracle gets that layer's
device input (the output of the same stack's layers before it, recomputed by
a prefix stack on copies of the caches -- the kernels are deterministic, so
it is bit-identical to the activation inside the full step) and the layer's
cache contents before the step; the layer output and the new key / value
rows are compared element by element.  Page: "DeepSpeed Inference 内核优化深度
解析：多 GPU 自适应并行、算子融合推理内核与 MoQ 量化支持", §3.2 (the layer regions; the
token loop calls every layer once per token) and §5.2 (int8 weights).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import DeviceLayer, check_close, new_workspace, to64
from transformer_layer_gb300 import ds, inputs

pytestmark = pytest.mark.gpu

CASES = {
    # name: (layers, hidden, heads, ffn, past, weight dtype, checked layers, batch)
    "7b_f16": (32, 4096, 32, 16384, 512, torch.float16, (0, 15, 31), 1),
    "13b_int8": (40, 5120, 40, 20480, 1024, torch.int8, (0, 19, 39), 1),
    "7b_f16_b16": (32, 4096, 32, 16384, 512, torch.float16, (0, 31), 16),
    "13b_int8_b16": (40, 5120, 40, 20480, 1024, torch.int8, (0, 39), 16),
}
STEPS = 64
CHECK_STEPS = (1, 64)


def _run_prefix(layers, n, x, kc, vc, seq0, max_len, stream):
    """Output of layers [0, n) on copies of their caches (n >= 1)."""
    h = ds.ds_stack_create([l.handle for l in layers[:n]])
    try:
        B = x.shape[0]
        k2 = [k.clone() for k in kc[:n]]
        v2 = [v.clone() for v in vc[:n]]
        seq = seq0.clone()
        nb = ds.ds_stack_workspace_bytes(h, B)
        ws = new_workspace(nb)
        out = torch.empty_like(x)
        # the clones and the workspace are made on torch's current stream:
        # complete before the step reads them on `stream`
        torch.cuda.synchronize()
        ds.ds_stack_decode_step(h, x, out, B, k2, v2, max_len, seq, ws, nb, stream)
        stream.synchronize()
        return out
    finally:
        ds.ds_stack_destroy(h)


@pytest.mark.parametrize("case", sorted(CASES))
def test_full_depth_stack_teacher_forced(case):
    n_layers, H, nh, F, past, wdt, checked, B = CASES[case]
    d, max_len, seed = H // nh, past + STEPS, 1700
    pasts = [past - 5 * b for b in range(B)]  # ragged at batch > 1
    layers = [DeviceLayer(H, nh, F, seed, layer=l, weight_dtype=wdt) for l in range(n_layers)]
    stack = ds.ds_stack_create([l.handle for l in layers])
    try:
        kc, vc = [], []
        for l in range(n_layers):
            k, v = inputs.kv_cache(B, nh, max_len, d, seed, layer=l, device="cuda")
            kc.append(k)
            vc.append(v)
        seq = torch.tensor(pasts, dtype=torch.int32, device="cuda")
        nb = ds.ds_stack_workspace_bytes(stack, B)
        ws = new_workspace(nb)
        stream = torch.cuda.Stream()
        out = torch.empty(B, H, dtype=torch.float16, device="cuda")
        for step in range(1, STEPS + 1):
            x = inputs.hidden(B, 1, H, seed, step=step, device="cuda").reshape(B, H)
            torch.cuda.synchronize()  # (made on torch's current stream; the step runs on `stream`)
            if step in CHECK_STEPS:
                stream.synchronize()
                seq0 = seq.clone()
                cur = seq0.cpu().tolist()
                K = {l: to64(kc[l]) for l in checked}
                V = {l: to64(vc[l]) for l in checked}
                xin = {l: (x if l == 0 else _run_prefix(layers, l, x, kc, vc, seq0, max_len, stream))
                       for l in checked}
                yout = {l: _run_prefix(layers, l + 1, x, kc, vc, seq0, max_len, stream)
                        for l in checked if l + 1 < n_layers}
            ds.ds_stack_decode_step(stack, x, out, B, kc, vc, max_len, seq, ws, nb, stream)
            if step in CHECK_STEPS:
                stream.synchronize()
                yout[n_layers - 1] = out.clone()
                for l in checked:
                    r = oracle.layer_forward(to64(xin[l]).reshape(B, 1, H), layers[l].oracle_params(), K[l], V[l],
                                             cur, nh)
                    check_close(yout[l].reshape(B, 1, H), r["y"], torch.float16, what=f"{case} step {step} layer {l} y")
                    kn = torch.stack([kc[l][b, :, cur[b], :] for b in range(B)])
                    vn = torch.stack([vc[l][b, :, cur[b], :] for b in range(B)])
                    check_close(kn, r["k_new"][:, 0], torch.float16, what=f"{case} step {step} layer {l} k")
                    check_close(vn, r["v_new"][:, 0], torch.float16, what=f"{case} step {step} layer {l} v")
                    layers[l]._oracle = None  # float64 copies of a large layer: release them
        stream.synchronize()
        assert seq.cpu().tolist() == [p + STEPS for p in pasts]
        code, flags = ds.ds_workspace_status(ws)
        assert code == ds.DS_OK and flags == 0
        assert ds.ds_stack_graph_captures(stack) == 1
    finally:
        ds.ds_stack_destroy(stack)
        for l in layers:
            l.close()
