"""The tensor-sliced layer's partition and reduction on CPU ranks (gloo).

Page: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核与
MoQ 量化支持", §3.2 (Megatron-LM style split of the Attn and FF blocks, one
all-reduce after each) and §3.1 (fusion up to each all-reduce boundary).

Two processes joined by a gloo process group play two tensor-parallel ranks.
Each takes its slice of the full layer weights through the library's own
partition (ds_tp_shard_blocks, a host-only call of the C ABI), checks it
against the oracle's independent slicing, computes its partial sums with the
oracle, and sums them with dist.all_reduce at the two boundaries; the result
must be the unsplit layer.  The device kernels of each rank are covered by
the GPU tests; this covers the host-side split and the reduction order.
"""
import os
import shutil
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from transformer_layer_gb300 import build, ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
H, NH, F, L = 256, 4, 512, 7


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        if not os.path.exists(build.LIB):
            pytest.skip("no nvcc and no prebuilt library")
    else:
        build.build()
    return ds.load()


def _full_params(seed):
    rng = np.random.default_rng(seed)
    return {"ln1_g": 1 + 0.1 * rng.standard_normal(H), "ln1_b": 0.1 * rng.standard_normal(H),
            "w_qkv": 0.05 * rng.standard_normal((3 * H, H)), "b_qkv": 0.1 * rng.standard_normal(3 * H),
            "w_o": 0.05 * rng.standard_normal((H, H)), "b_o": rng.standard_normal(H),
            "ln2_g": 1 + 0.1 * rng.standard_normal(H), "ln2_b": 0.1 * rng.standard_normal(H),
            "w_fc1": 0.05 * rng.standard_normal((F, H)), "b_fc1": 0.1 * rng.standard_normal(F),
            "w_fc2": 0.05 * rng.standard_normal((H, F)), "b_fc2": rng.standard_normal(H)}


def _inputs(seed, B, T):
    rng = np.random.default_rng(seed + 1)
    d = H // NH
    return (rng.standard_normal((B, T, H)), rng.standard_normal((B, NH, L, d)),
            rng.standard_normal((B, NH, L, d)))


def _apply_blocks(full, blocks, tp):
    """The rank's matrices built from the library's block list."""
    shape = {"w_qkv": (3 * H // tp, H), "b_qkv": (3 * H // tp, 1), "w_o": (H, H // tp),
             "w_fc1": (F // tp, H), "b_fc1": (F // tp, 1), "w_fc2": (H, F // tp)}
    out = {k: np.full(s, np.nan) for k, s in shape.items()}
    for b in blocks:
        name = ds.TP_MATRIX_NAMES[b["matrix"]]
        src = full[name].reshape(-1, b["src_cols"])
        out[name][b["dst_row"]:b["dst_row"] + b["rows"], :] = \
            src[b["src_row"]:b["src_row"] + b["rows"], b["src_col"]:b["src_col"] + b["cols"]]
    return {k: (v[:, 0] if k.startswith("b_") else v) for k, v in out.items()}


def _worker(rank, world, port, seed, B, T, q):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        full = _full_params(seed)
        x, K, V = _inputs(seed, B, T)
        blocks = ds.ds_tp_shard_blocks(H, NH, F, torch.float16, world, rank)
        mine = _apply_blocks(full, blocks, world)
        ref_shard = oracle.shard_layer_params(full, NH, world, rank)
        for k, v in mine.items():
            assert not np.isnan(v).any(), k           # every element of the shard written
            np.testing.assert_array_equal(v, ref_shard[k], err_msg=k)
        shard = dict(full)
        shard.update(mine)
        nhl = NH // world
        kr = K[:, rank * nhl:(rank + 1) * nhl].copy()
        vr = V[:, rank * nhl:(rank + 1) * nhl].copy()
        past = [3 + b for b in range(B)]
        a = oracle.tp_attention_partial(x, shard, kr, vr, past, nhl, rank)
        x1 = torch.from_numpy(a["x1_part"].copy())
        dist.all_reduce(x1, op=dist.ReduceOp.SUM)
        f = oracle.tp_ffn_partial(x1.numpy(), shard, rank)
        y = torch.from_numpy(f["y_part"].copy())
        dist.all_reduce(y, op=dist.ReduceOp.SUM)
        q.put((rank, x1.numpy(), y.numpy(), kr, vr))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("B,T", [(1, 1), (2, 2)])
def test_two_ranks_reduce_to_the_unsplit_layer(lib, B, T):
    import oracle
    world, seed = 2, 77 + B
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, seed, B, T, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, x1, y, kr, vr = q.get(timeout=180)
        got[r] = (x1, y, kr, vr)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    full = _full_params(seed)
    x, K, V = _inputs(seed, B, T)
    ref = oracle.layer_forward(x, full, K, V, [3 + b for b in range(B)], NH)
    nhl = NH // world
    for r in range(world):
        x1, y, kr, vr = got[r]
        np.testing.assert_allclose(x1, ref["x1"], rtol=0, atol=1e-11)   # the same sum on every rank
        np.testing.assert_allclose(y, ref["y"], rtol=0, atol=1e-11)
        np.testing.assert_allclose(kr, K[:, r * nhl:(r + 1) * nhl], rtol=0, atol=1e-12)
        np.testing.assert_allclose(vr, V[:, r * nhl:(r + 1) * nhl], rtol=0, atol=1e-12)


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_blocks_cover_every_weight_once(lib, tp):
    """Over all ranks, the library's blocks read every element of each sliced
    full matrix exactly once, and within a rank they fill its matrices
    exactly once."""
    Hh, nh, Ff = 1024, 8, 4096
    full_shape = {"w_qkv": (3 * Hh, Hh), "b_qkv": (3 * Hh, 1), "w_o": (Hh, Hh), "w_fc1": (Ff, Hh),
                  "b_fc1": (Ff, 1), "w_fc2": (Hh, Ff)}
    seen = {k: np.zeros(s, np.int32) for k, s in full_shape.items()}
    for r in range(tp):
        blocks = ds.ds_tp_shard_blocks(Hh, nh, Ff, torch.bfloat16, tp, r)
        assert len(blocks) == 10
        filled = {}
        for b in blocks:
            name = ds.TP_MATRIX_NAMES[b["matrix"]]
            assert b["src_cols"] == full_shape[name][1]
            seen[name][b["src_row"]:b["src_row"] + b["rows"], b["src_col"]:b["src_col"] + b["cols"]] += 1
            f = filled.setdefault(name, {})
            for row in range(b["dst_row"], b["dst_row"] + b["rows"]):
                f[row] = f.get(row, 0) + 1
        for name, f in filled.items():
            rows = full_shape[name][0] // tp if name in ("w_qkv", "b_qkv", "w_fc1", "b_fc1") else full_shape[name][0]
            assert sorted(f) == list(range(rows)) and set(f.values()) == {1}, name
    for name, s in seen.items():
        assert s.min() == 1 and s.max() == 1, name


def test_invalid_splits_are_refused(lib):
    with pytest.raises(ds.DSError):
        ds.ds_tp_shard_blocks(1024, 8, 4096, torch.float16, 3, 0)    # 3 does not divide 8 heads
    with pytest.raises(ds.DSError):
        ds.ds_tp_shard_blocks(1024, 8, 4096, torch.float16, 2, 2)    # rank out of range
    with pytest.raises(ds.DSError):
        ds.ds_tp_shard_blocks(1024, 16, 4096, torch.float16, 16, 0)  # H / 16 = 64 is not a multiple of 128
