"""GPU parity of the stack decode step (graph replay, device-side seq_len).

Each decode step is checked layer by layer, teacher-forced: the oracle gets
the device's input to that layer and the cache contents the device had before
the step, and its float64 result is compared with the device's layer output
and new cache entries.  Free-running drift of the whole stack is bounded
loosely.  Page: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应
并行、算子融合推理内核与 MoQ 量化支持", §3.2 (layer regions; the stack is the
token-by-token generation loop calling every layer once per token).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import DeviceLayer, cache_store, check_close, new_workspace, to64
from transformer_layer_gb300 import ds, inputs

pytestmark = pytest.mark.gpu


class DeviceStack:
    def __init__(self, n_layers, H, nh, F, B, max_len, past, seed, act=torch.float16, wdt=torch.float16,
                 quant_group=64, mlp_extra_grouping=0):
        self.layers = [DeviceLayer(H, nh, F, seed, layer=l, act_dtype=act, weight_dtype=wdt,
                                   quant_group=quant_group, mlp_extra_grouping=mlp_extra_grouping)
                       for l in range(n_layers)]
        self.handle = ds.ds_stack_create([l.handle for l in self.layers])
        d = H // nh
        self.kc, self.vc = [], []
        for l in range(n_layers):
            k, v = inputs.kv_cache(B, nh, max_len, d, seed, layer=l, dtype=act, device="cuda")
            self.kc.append(k)
            self.vc.append(v)
        self.B, self.H, self.nh, self.max_len = B, H, nh, max_len
        self.seq = torch.tensor(past, dtype=torch.int32, device="cuda")
        self.nbytes = ds.ds_stack_workspace_bytes(self.handle, B)
        self.ws = new_workspace(self.nbytes)
        self.act = act

    def step(self, x, out, stream=None):
        ds.ds_stack_decode_step(self.handle, x, out, self.B, self.kc, self.vc, self.max_len, self.seq,
                                self.ws, self.nbytes, stream)

    def close(self):
        ds.ds_stack_destroy(self.handle)
        for l in self.layers:
            l.close()


def prefix_outputs(S, x, stream):
    """Device input of every layer for one step: run stacks of layers [0..l] on
    copies of the caches and sequence lengths.  The kernels are deterministic,
    so layer l's input inside the full stack is bit-identical to the output of
    the prefix [0..l-1]."""
    outs = []
    for l in range(len(S.layers)):
        h = ds.ds_stack_create([lay.handle for lay in S.layers[:l + 1]])
        try:
            kc = [k.clone() for k in S.kc[:l + 1]]
            vc = [v.clone() for v in S.vc[:l + 1]]
            seq = S.seq.clone()
            nb = ds.ds_stack_workspace_bytes(h, S.B)
            ws = new_workspace(nb)
            o = torch.empty_like(x)
            ds.ds_stack_decode_step(h, x, o, S.B, kc, vc, S.max_len, seq, ws, nb, stream)
            stream.synchronize()
            outs.append(o)
        finally:
            ds.ds_stack_destroy(h)
    return outs


@pytest.mark.parametrize("act,int8,B", [(torch.float16, False, 2), (torch.bfloat16, False, 2),
                                        (torch.float16, True, 2), (torch.bfloat16, True, 3),
                                        (torch.float16, False, 12), (torch.bfloat16, False, 16)])
def test_stack_steps_graph_vs_oracle(act, int8, B):
    """Four graph-replayed decode steps of a 3-layer stack.  Each layer is
    checked against the oracle fed that layer's device input and the device
    cache contents before the step (teacher-forced, layer by layer); the step
    output must equal the last prefix's output bit for bit; the free-running
    drift of the whole stack against the oracle is checked only loosely.  The
    int8 cases take MoQ groups of 128 for w_qkv / w_o and, with the extra MLP
    grouping, 64 for the FFN matrices, so consecutive GEMVs differ in group
    length.  Batch 12 and 16 run the tensor-core tile kernels."""
    n_layers, H, nh, F, max_len = 3, 512, 8, 2048, 40
    quant = {}
    if int8:
        H, nh, quant = 1024, 8, dict(wdt=torch.int8, quant_group=128, mlp_extra_grouping=1)
    past = [(7 + 13 * b) % 30 for b in range(B)]
    S = DeviceStack(n_layers, H, nh, F, B, max_len, past, seed=1100, act=act, **({"wdt": act} | quant))
    stream = torch.cuda.Stream()
    try:
        with torch.cuda.stream(stream):
            for step in range(4):
                x = inputs.hidden(B, 1, H, 1100, step=step, dtype=act, device="cuda").reshape(B, H)
                out = torch.empty_like(x)
                K = [to64(k) for k in S.kc]
                V = [to64(v) for v in S.vc]
                cur = S.seq.cpu().tolist()
                assert cur == [p + step for p in past]
                pre = prefix_outputs(S, x, stream)
                S.step(x, out, stream)
                stream.synchronize()
                assert torch.equal(out, pre[-1])
                params = [l.oracle_params() for l in S.layers]
                for l in range(n_layers):
                    xin = x if l == 0 else pre[l - 1]
                    r = oracle.layer_forward(to64(xin).reshape(B, 1, H), params[l], K[l], V[l], cur, nh)
                    check_close(pre[l].reshape(B, 1, H), r["y"], act, what=f"step {step} layer {l} y")
                    for b in range(B):
                        check_close(S.kc[l][b, :, cur[b], :], r["k_new"][b, 0], act,
                                    what=f"step {step} layer {l} k")
                        check_close(S.vc[l][b, :, cur[b], :], r["v_new"][b, 0], act,
                                    what=f"step {step} layer {l} v")
                free = oracle.stack_forward(to64(x).reshape(B, 1, H), params, K, V, cur, nh)
                drift = float(np.linalg.norm(to64(out) - free[-1]["y"].reshape(B, H)) /
                              np.linalg.norm(free[-1]["y"]))
                assert drift < 1e-2, drift
        assert S.seq.cpu().tolist() == [p + 4 for p in past]
    finally:
        S.close()


def test_graph_replay_matches_direct_and_profile_launches():
    """Graph replay, a direct launch on the legacy stream and profile mode
    (events between the region kernels) run the same chain of deterministic
    region kernels: bit-identical, and profile mode reports per-region times."""
    n_layers, H, nh, F, B, max_len = 2, 256, 4, 1024, 3, 24
    past = [2, 9, 0]
    outs = []
    for mode in ("graph", "legacy", "profile"):
        S = DeviceStack(n_layers, H, nh, F, B, max_len, past, seed=1200)
        try:
            stream = torch.cuda.Stream() if mode != "legacy" else None
            if mode == "profile":
                ds.ds_stack_set_profiling(S.handle, True)
            ys = []
            for step in range(3):
                x = inputs.hidden(B, 1, H, 1200, step=step, device="cuda").reshape(B, H)
                out = torch.empty_like(x)
                torch.cuda.synchronize()
                if mode == "legacy":
                    ds.ds_stack_decode_step(S.handle, x, out, B, S.kc, S.vc, max_len, S.seq, S.ws,
                                            S.nbytes, 0)
                else:
                    S.step(x, out, stream)
                torch.cuda.synchronize()
                ys.append(out.clone())
            if mode == "profile":
                us, n = ds.ds_stack_region_times(S.handle)
                assert n == [3 * n_layers] * 5 and all(u > 0 for u in us)
            assert S.seq.cpu().tolist() == [p + 3 for p in past]
            code, flags = ds.ds_workspace_status(S.ws)
            assert code == ds.DS_OK and flags == 0
            outs.append((torch.stack(ys), torch.stack([k.clone() for k in S.kc])))
        finally:
            S.close()
    assert torch.equal(outs[1][0], outs[0][0])
    assert torch.equal(outs[1][1], outs[0][1])
    assert torch.equal(outs[2][0], outs[0][0])
    assert torch.equal(outs[2][1], outs[0][1])


def test_decode_host_entry_point():
    n_layers, H, nh, F, B, max_len = 2, 256, 4, 1024, 2, 20
    S = DeviceStack(n_layers, H, nh, F, B, max_len, [4, 11], seed=1300)
    S2 = DeviceStack(n_layers, H, nh, F, B, max_len, [4, 11], seed=1300)
    try:
        stream = torch.cuda.Stream()
        x = inputs.hidden(B, 1, H, 1300, device="cuda").reshape(B, H)
        xh = x.cpu().pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        xd, yd = torch.empty_like(x), torch.empty_like(x)
        n0 = ds.ds_launch_count()
        ds.ds_stack_decode_host(S.handle, xh, yh, xd, yd, B, S.kc, S.vc, max_len, S.seq, S.ws, S.nbytes,
                                stream)
        assert ds.ds_launch_count() - n0 == 5 * n_layers   # the region chain, replayed as one graph
        out = torch.empty_like(x)
        S2.step(x, out, stream)
        stream.synchronize()
        assert torch.equal(yh, out.cpu())
    finally:
        S.close()
        S2.close()


@pytest.mark.parametrize("B", [2, 16])
def test_rotating_hidden_buffers_reuse_the_graph(B):
    """A decode loop that rotates its input buffers (three) and output buffers
    (two) keeps one captured graph: the kernel nodes holding x_in / x_out are
    updated in place.  Results are bit-identical to direct launches on the
    legacy stream with the same buffers."""
    n_layers, H, nh, F, max_len = 2, 256, 4, 1024, 24
    past = [(3 + 5 * b) % 17 for b in range(B)]
    ys = {}
    for mode in ("graph", "legacy"):
        S = DeviceStack(n_layers, H, nh, F, B, max_len, past, seed=1400)
        try:
            xs = [inputs.hidden(B, 1, H, 1400, step=i, device="cuda").reshape(B, H) for i in range(3)]
            outs = [torch.empty_like(xs[0]) for _ in range(2)]
            stream = torch.cuda.Stream() if mode == "graph" else None
            got = []
            for step in range(6):
                torch.cuda.synchronize()
                x, out = xs[step % 3], outs[step % 2]
                if mode == "graph":
                    S.step(x, out, stream)
                else:
                    ds.ds_stack_decode_step(S.handle, x, out, B, S.kc, S.vc, max_len, S.seq, S.ws, S.nbytes, 0)
                torch.cuda.synchronize()
                got.append(out.clone())
            if mode == "graph":
                assert ds.ds_stack_graph_captures(S.handle) == 1
            ys[mode] = (torch.stack(got), torch.stack([k.clone() for k in S.kc]))
            assert S.seq.cpu().tolist() == [p + 6 for p in past]
        finally:
            S.close()
    assert torch.equal(ys["graph"][0], ys["legacy"][0])
    assert torch.equal(ys["graph"][1], ys["legacy"][1])


@pytest.mark.parametrize("act,B,T", [(torch.float16, 2, 40), (torch.bfloat16, 1, 96)])
def test_stack_prompt_chunk(act, B, T):
    """ds_stack_forward: a prompt chunk through a 3-layer stack.  Each layer
    is checked against the oracle fed that layer's device input (the output of
    a prefix stack on copies of the caches, bit-identical to the activation
    inside the full stack) and its cache before the chunk; the chunk's keys and
    values land in every layer's cache; past_len is not advanced."""
    n_layers, H, nh, F, max_len = 3, 512, 8, 2048, 200
    past = [11 * (b + 1) for b in range(B)]
    S = DeviceStack(n_layers, H, nh, F, B, max_len, past, seed=1600, act=act, wdt=act)
    try:
        x = inputs.hidden(B, T, H, 1600, dtype=act, device="cuda")
        K = [to64(k) for k in S.kc]
        V = [to64(v) for v in S.vc]
        nb = ds.ds_layer_workspace_bytes(S.layers[0].handle, B, T)
        outs = []
        for n in range(1, n_layers + 1):   # prefixes [0, n); the last is the full stack
            h = ds.ds_stack_create([l.handle for l in S.layers[:n]])
            try:
                kc = [k.clone() for k in S.kc[:n]] if n < n_layers else S.kc
                vc = [v.clone() for v in S.vc[:n]] if n < n_layers else S.vc
                ws = new_workspace(nb)
                o = torch.empty_like(x)
                ds.ds_stack_forward(h, x, o, B, T, kc, vc, max_len, S.seq, ws, nb)
                torch.cuda.synchronize()
                outs.append(o)
            finally:
                ds.ds_stack_destroy(h)
        assert S.seq.cpu().tolist() == past          # not advanced
        for l in range(n_layers):
            xin = x if l == 0 else outs[l - 1]
            r = oracle.layer_forward(to64(xin), S.layers[l].oracle_params(), K[l], V[l], past, nh,
                                     kv_store=cache_store(act))
            check_close(outs[l], r["y"], act, what=f"stack prompt layer {l} y")
            for b in range(B):
                for t in range(T):
                    check_close(S.kc[l][b, :, past[b] + t, :], r["k_new"][b, t], act, what=f"layer {l} k")
                    check_close(S.vc[l][b, :, past[b] + t, :], r["v_new"][b, t], act, what=f"layer {l} v")
    finally:
        S.close()
