"""Tensor-sliced layer on the device: every rank's kernels, against the
unsplit float64 oracle.

Page: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核与
MoQ 量化支持", §3.2 (Megatron-LM style split of the Attn and FF blocks, one
all-reduce after each) and §3.1 (fusion up to each all-reduce boundary).

One GPU plays all W ranks one after the other: each rank's layer is created
over its own shard (sliced on the device by ds_tp_shard_weights) and its own
head slice of the KV caches; the all-reduce between the fused regions, which
a collective library performs across GPUs, is a plain sum of the ranks' fp32
partial buffers here.  No rank's kernel waits on another's.  The output and
every rank's new cache rows must match the unsplit layer of the oracle.
A last test runs the binding's step (tp_layer_forward) with a real NCCL
all-reduce over a one-rank group.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import cache_store, check_close, new_workspace, to64
from transformer_layer_gb300 import ds, inputs

pytestmark = pytest.mark.gpu

SHARD_SHAPES = {"w_qkv": lambda H, F, W: (3 * H // W, H), "b_qkv": lambda H, F, W: (3 * H // W,),
                "w_o": lambda H, F, W: (H, H // W), "w_fc1": lambda H, F, W: (F // W, H),
                "b_fc1": lambda H, F, W: (F // W,), "w_fc2": lambda H, F, W: (H, F // W)}


class TpRanks:
    """W rank layers of one full layer on the current device."""

    def __init__(self, H, nh, F, W, seed, act):
        self.H, self.nh, self.F, self.W, self.act = H, nh, F, W, act
        self.full = inputs.layer_params(H, F, seed, dtype=act, device="cuda")
        self.shards, self.handles = [], []
        for r in range(W):
            sh = dict(self.full)  # replicated: LayerNorm parameters, b_o, b_fc2
            for k, f in SHARD_SHAPES.items():
                sh[k] = torch.empty(f(H, F, W), dtype=act, device="cuda")
            ds.ds_tp_shard_weights(H, nh, F, act, W, r, self.full, sh)
            torch.cuda.synchronize()
            self.shards.append(sh)
            self.handles.append(ds.ds_tp_layer_create(H, nh, F, sh, act, W, r))

    def close(self):
        for h in self.handles:
            ds.ds_tp_layer_destroy(h)


def _step(tp, x, B, T, kcs, vcs, max_len, past, stream):
    """One layer step of all ranks, the all-reduces as sums of the partials."""
    M, H = B * T, tp.H
    nb = max(ds.ds_tp_layer_workspace_bytes(h, B, T) for h in tp.handles)
    ws = [new_workspace(nb) for _ in tp.handles]
    x1p = [torch.empty(M, H, dtype=torch.float32, device="cuda") for _ in tp.handles]
    yp = [torch.empty(M, H, dtype=torch.float32, device="cuda") for _ in tp.handles]
    for r, h in enumerate(tp.handles):
        ds.ds_tp_attention_partial(h, x, x1p[r], B, T, kcs[r], vcs[r], max_len, past, ws[r], nb, stream)
    with torch.cuda.stream(stream):
        x1 = torch.stack(x1p).sum(0)
    for r, h in enumerate(tp.handles):
        ds.ds_tp_ffn_partial(h, x1, yp[r], M, ws[r], nb, stream)
    with torch.cuda.stream(stream):
        y = torch.stack(yp).sum(0)
    out = torch.empty(B, T, H, dtype=tp.act, device="cuda")
    ds.ds_tp_finish(tp.handles[0], y, out, M, stream)
    stream.synchronize()
    for w in ws:
        code, flags = ds.ds_workspace_status(w)
        assert code == ds.DS_OK and flags == 0
    return out, x1, x1p


CASES = [
    # (act, W, H, nh, F, B, T)
    (torch.float16, 2, 1024, 8, 4096, 1, 1),
    (torch.float16, 2, 1024, 8, 4096, 4, 1),
    (torch.float16, 4, 1024, 8, 4096, 3, 5),
    (torch.bfloat16, 2, 1024, 8, 4096, 16, 1),
    (torch.bfloat16, 8, 1024, 16, 2048, 2, 1),
    (torch.float16, 2, 1024, 8, 4096, 2, 32),   # prompt chunk: tiled attention
    (torch.bfloat16, 2, 2048, 16, 8192, 64, 1),
]


@pytest.mark.parametrize("act,W,H,nh,F,B,T", CASES)
def test_tp_ranks_match_unsplit_layer(act, W, H, nh, F, B, T):
    seed, past0 = 900 + W * 7 + B, 40
    max_len = (past0 + 3 * B + T + 15) // 16 * 16
    d = H // nh
    tp = TpRanks(H, nh, F, W, seed, act)
    try:
        K, V = inputs.kv_cache(B, nh, max_len, d, seed, dtype=act, device="cuda")
        nhl = nh // W
        kcs = [K[:, r * nhl:(r + 1) * nhl].contiguous() for r in range(W)]
        vcs = [V[:, r * nhl:(r + 1) * nhl].contiguous() for r in range(W)]
        past = torch.tensor([past0 + 3 * b for b in range(B)], dtype=torch.int32, device="cuda")
        x = inputs.hidden(B, T, H, seed, dtype=act, device="cuda")
        K64, V64 = to64(K), to64(V)
        p64 = {k: to64(v) for k, v in tp.full.items()}
        ref = oracle.layer_forward(to64(x), p64, K64, V64, past.cpu().tolist(), nh, kv_store=cache_store(act))
        out, x1, _ = _step(tp, x, B, T, kcs, vcs, max_len, past, torch.cuda.Stream())
        check_close(x1.reshape(B, T, H), ref["x1"], torch.float32, what="x1")
        check_close(out, ref["y"], act, what="y")
        for r in range(W):
            for b in range(B):
                pos = slice(past0 + 3 * b, past0 + 3 * b + T)
                check_close(kcs[r][b, :, pos, :].permute(1, 0, 2), ref["k_new"][b, :, r * nhl:(r + 1) * nhl], act,
                            what=f"rank {r} k")
                check_close(vcs[r][b, :, pos, :].permute(1, 0, 2), ref["v_new"][b, :, r * nhl:(r + 1) * nhl], act,
                            what=f"rank {r} v")
    finally:
        tp.close()


def test_tp_partials_sum_like_the_oracle_ranks():
    """Each rank's x1 partial against the oracle's partial of the same rank
    (rank 0 carries b_o and the residual, the others only their heads)."""
    act, W, H, nh, F, B = torch.float16, 2, 1024, 8, 4096, 2
    seed, max_len = 31, 64
    tp = TpRanks(H, nh, F, W, seed, act)
    try:
        d, nhl = H // nh, nh // W
        K, V = inputs.kv_cache(B, nh, max_len, d, seed, dtype=act, device="cuda")
        kcs = [K[:, r * nhl:(r + 1) * nhl].contiguous() for r in range(W)]
        vcs = [V[:, r * nhl:(r + 1) * nhl].contiguous() for r in range(W)]
        past = torch.tensor([10, 20], dtype=torch.int32, device="cuda")
        x = inputs.hidden(B, 1, H, seed, dtype=act, device="cuda")
        _, _, x1p = _step(tp, x, B, 1, kcs, vcs, max_len, past, torch.cuda.Stream())
        p64 = {k: to64(v) for k, v in tp.full.items()}
        for r in range(W):
            s = oracle.shard_layer_params(p64, nh, W, r)
            kr, vr = to64(K[:, r * nhl:(r + 1) * nhl]), to64(V[:, r * nhl:(r + 1) * nhl])
            want = oracle.tp_attention_partial(to64(x), s, kr, vr, [10, 20], nhl, r, kv_store=cache_store(act))
            check_close(x1p[r].reshape(B, 1, H), want["x1_part"], torch.float32, what=f"rank {r} x1 partial")
    finally:
        tp.close()


def test_tp_rejects_int8_and_bad_rank():
    full = inputs.layer_params(1024, 4096, 5, dtype=torch.float16, device="cuda")
    with pytest.raises(ds.DSError):
        ds.ds_tp_layer_create(1024, 8, 4096, full, torch.float16, 2, 2)
    cfg = ds._tp_config(1024, 8, 4096, torch.float16, 2, 0)
    cfg.layer.weight_dtype = ds.DS_I8
    w = ds.ds_layer_weights(*[ds._ptr(full.get(n)) for n in ds._WNAMES])
    import ctypes as C
    out = C.c_void_p()
    assert ds.load().ds_tp_layer_create(C.byref(cfg), C.byref(w), C.byref(out)) == ds.DS_ERR_INVALID_ARG


def _nccl_worker(port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        act, H, nh, F, B = torch.float16, 1024, 8, 4096, 3
        tp = TpRanks(H, nh, F, 1, 12, act)
        d = H // nh
        K, V = inputs.kv_cache(B, nh, 64, d, 12, dtype=act, device="cuda")
        past = torch.tensor([5, 9, 13], dtype=torch.int32, device="cuda")
        x = inputs.hidden(B, 1, H, 12, dtype=act, device="cuda")
        ref = oracle.layer_forward(to64(x), {k: to64(v) for k, v in tp.full.items()}, to64(K), to64(V),
                                   [5, 9, 13], nh)
        nb = ds.ds_tp_layer_workspace_bytes(tp.handles[0], B, 1)
        ws = new_workspace(nb)
        x1 = torch.empty(B, H, dtype=torch.float32, device="cuda")
        y = torch.empty(B, H, dtype=torch.float32, device="cuda")
        out = torch.empty(B, 1, H, dtype=act, device="cuda")
        ds.tp_layer_forward(tp.handles[0], x, out, B, 1, K, V, 64, past, ws, nb, x1, y)
        torch.cuda.synchronize()
        check_close(out, ref["y"], act, what="tp_layer_forward y")
        tp.close()
        q.put("ok")
    except Exception as e:  # reported to the parent
        q.put(repr(e))
    finally:
        dist.destroy_process_group()


def test_binding_step_with_nccl_single_rank():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_nccl_worker, args=(port, q))
    p.start()
    msg = q.get(timeout=300)
    p.join(60)
    assert msg == "ok", msg
    assert p.exitcode == 0
