"""GPU parity of one layer forward (all four fusion regions) against the oracle.

Cases span several 16-row tiles and K slices, ragged cache lengths across
batch rows, several new tokens per sequence (the causal mask inside the new
tokens), the empty cache (past_len = 0), batch rows 1..64 (one to eight MMA
column tiles) and the three weight formats.  Page: "DeepSpeed Inference 内核优化
深度解析：多 GPU 自适应并行、算子融合推理内核与 MoQ 量化支持", §3.2 and §5.2.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import DeviceLayer, cache_store, check_close, new_workspace, to64
from transformer_layer_gb300 import ds, inputs

pytestmark = pytest.mark.gpu


def run_layer(L, B, T, past, max_len, seed=7):
    H, nh = L.hidden, L.heads
    d = H // nh
    kc, vc = inputs.kv_cache(B, nh, max_len, d, seed, dtype=L.act_dtype, device="cuda")
    x = inputs.hidden(B, T, H, seed, dtype=L.act_dtype, device="cuda")
    K0, V0 = to64(kc), to64(vc)
    kc0, vc0 = kc.clone(), vc.clone()
    past_t = torch.tensor(past, dtype=torch.int32, device="cuda")
    out = torch.full_like(x, float("nan"))
    nbytes = ds.ds_layer_workspace_bytes(L.handle, B, T)
    ws = new_workspace(nbytes)
    ds.ds_layer_forward(L.handle, x, out, B, T, kc, vc, max_len, past_t, ws, nbytes)
    torch.cuda.synchronize()
    code, flags = ds.ds_workspace_status(ws)
    assert code == ds.DS_OK and flags == 0
    # the device cache stores the new keys / values in the activation dtype
    # before attention reads them: the oracle stores them the same way
    r = oracle.layer_forward(to64(x), L.oracle_params(), K0, V0, past, nh, kv_store=cache_store(L.act_dtype))
    return dict(out=out, kc=kc, vc=vc, kc0=kc0, vc0=vc0, ref=r, ws=ws, nbytes=nbytes, x=x,
                past_t=past_t)


def check_layer(L, res, B, T, past, what):
    dt = L.act_dtype
    check_close(res["out"].reshape(B, T, -1), res["ref"]["y"], dt, what=what + " y")
    kc, vc = res["kc"], res["vc"]
    newmask = torch.zeros(kc.shape[:3], dtype=torch.bool, device=kc.device)
    for b in range(B):
        for t in range(T):
            pos = past[b] + t
            check_close(kc[b, :, pos, :], res["ref"]["k_new"][b, t], dt, what=f"{what} k[{b},{t}]")
            check_close(vc[b, :, pos, :], res["ref"]["v_new"][b, t], dt, what=f"{what} v[{b},{t}]")
            newmask[b, :, pos] = True
    # every other cache position is untouched, bit for bit
    assert torch.equal(kc[~newmask], res["kc0"][~newmask])
    assert torch.equal(vc[~newmask], res["vc0"][~newmask])


@pytest.mark.parametrize("B,T,past", [
    (1, 1, [32]),          # the single-layer workload: H=256, 4 heads, 32 cached
    (1, 1, [0]),           # empty cache: attention over the new token only
    (3, 1, [5, 31, 0]),    # ragged cache lengths
    (2, 3, [4, 17]),       # three new tokens: causal mask among them
    (8, 1, list(range(0, 40, 5))),
    (16, 1, [(7 * i) % 40 for i in range(16)]),
    (5, 8, [1, 9, 3, 30, 12]),   # 40 rows: four column tiles of the MMA
    (64, 1, [(11 * i) % 45 for i in range(64)]),
])
def test_layer256_f16(B, T, past):
    L = DeviceLayer(256, 4, 1024, seed=1000)
    try:
        res = run_layer(L, B, T, past, max_len=48)
        check_layer(L, res, B, T, past, f"f16 B={B} T={T}")
    finally:
        L.close()


@pytest.mark.parametrize("B,T,past", [(1, 1, [32]), (4, 2, [3, 0, 21, 8]), (24, 1, [(5 * i) % 40 for i in range(24)])])
def test_layer256_bf16(B, T, past):
    L = DeviceLayer(256, 4, 1024, seed=1001, act_dtype=torch.bfloat16, weight_dtype=torch.bfloat16)
    try:
        res = run_layer(L, B, T, past, max_len=48)
        check_layer(L, res, B, T, past, f"bf16 B={B} T={T}")
    finally:
        L.close()


@pytest.mark.parametrize("act", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("B,T,past", [(1, 1, [40]), (6, 1, [0, 3, 9, 27, 33, 12]), (16, 1, [(3 * i) % 41 for i in range(16)])])
def test_layer512_int8(act, B, T, past):
    L = DeviceLayer(512, 4, 1024, seed=1002, act_dtype=act, weight_dtype=torch.int8)
    try:
        for k in ("w_qkv", "w_o", "w_fc1", "w_fc2"):     # codes and scales bit-exact
            q, s = oracle.quantize_int8(L.p[k].cpu().numpy(), 64)
            assert np.array_equal(L.codes[k].cpu().numpy(), q)
            assert np.array_equal(L.scales[k].cpu().numpy().view(np.uint16), s.view(np.uint16))
        res = run_layer(L, B, T, past, max_len=48)
        check_layer(L, res, B, T, past, f"int8/{act} B={B}")
    finally:
        L.close()


@pytest.mark.parametrize("H,nh,F,B", [(2560, 20, 10240, 1), (4096, 32, 16384, 1), (4096, 32, 16384, 4)])
def test_full_width_layer_f16(H, nh, F, B):
    """One layer at the full widths of the GPT-Neo-2.7B- and 7B-shaped stacks
    (many K slices and split-K fix-ups), every output element checked."""
    L = DeviceLayer(H, nh, F, seed=1003)
    try:
        past = [128 + 97 * b for b in range(B)]
        res = run_layer(L, B, 1, past, max_len=640)
        check_layer(L, res, B, 1, past, f"H={H} B={B}")
    finally:
        L.close()


@pytest.mark.parametrize("act,B", [(torch.float16, 2), (torch.float16, 8), (torch.float16, 16),
                                   (torch.float16, 32), (torch.float16, 64), (torch.bfloat16, 1),
                                   (torch.bfloat16, 8), (torch.bfloat16, 64)])
def test_skinny_gemm_sweep_layer(act, B):
    """The batch-row sweep on one 4096-hidden layer (QKV, O-proj, FFN-up and
    FFN-down with their fused epilogues): one to eight MMA column tiles, fp16
    and bf16 (hi/lo operand split), every output element checked."""
    H, nh, F = 4096, 32, 16384
    L = DeviceLayer(H, nh, F, seed=1004, act_dtype=act, weight_dtype=act)
    try:
        past = [16 + (37 * b) % 600 for b in range(B)]
        res = run_layer(L, B, 1, past, max_len=640, seed=11)
        check_layer(L, res, B, 1, past, f"sweep {act} B={B}")
    finally:
        L.close()


@pytest.mark.parametrize("act,B", [(torch.float16, 9), (torch.float16, 32), (torch.float16, 64),
                                   (torch.float16, 150), (torch.bfloat16, 32)])
def test_int8_layer_many_rows(act, B):
    """MoQ int8 weights at 9..150 batch rows: with fp16 activations the
    tensor-core tile kernels, whose converter warps dequantise each stage of
    codes to fp16 in tensor memory (several token tiles at 150 rows); with
    bf16 activations the streaming GEMV kernels (up to 39 rows)."""
    H, nh, F = 1024, 8, 4096
    L = DeviceLayer(H, nh, F, seed=1011, act_dtype=act, weight_dtype=torch.int8)
    try:
        past = [(17 * b) % 90 for b in range(B)]
        res = run_layer(L, B, 1, past, max_len=100, seed=15)
        check_layer(L, res, B, 1, past, f"int8 {act} B={B}")
    finally:
        L.close()


@pytest.mark.parametrize("act,H,nh,F", [(torch.float16, 5120, 40, 20480), (torch.bfloat16, 5120, 40, 20480),
                                        (torch.float16, 2560, 20, 10240)])
def test_uneven_k_slices(act, H, nh, F):
    """Tile GEMMs whose K slices run as one cluster per weight tile, slices
    of unequal length: at 16 batch rows the 40 weight tiles of hidden 5120
    take 3 slices each (O-proj 40 chunks, FFN-down 160), so that O-proj and
    FFN-down fill 120 SMs rather than 80.  (The 20 tiles of hidden 2560 would
    take 7, but clusters of 7 do not all fit on the GPU at once: they keep
    4.)  Every output element checked."""
    L = DeviceLayer(H, nh, F, seed=1013, act_dtype=act, weight_dtype=act)
    try:
        B = 16
        past = [(29 * b) % 200 for b in range(B)]
        res = run_layer(L, B, 1, past, max_len=256, seed=17)
        check_layer(L, res, B, 1, past, f"uneven {act} H={H}")
    finally:
        L.close()


@pytest.mark.parametrize("B", [1, 16])
def test_int8_13b_shaped_layer(B):
    """A 13B-shaped layer (hidden 5120, 40 heads, FFN 20480) with MoQ int8
    group-64 weights quantised on the device, 1024 cached positions, batch 1
    and 16: codes and scales bit-exact, layer output within tolerance."""
    H, nh, F = 5120, 40, 20480
    L = DeviceLayer(H, nh, F, seed=1005, weight_dtype=torch.int8)
    try:
        q, sc = oracle.quantize_int8(L.p["w_o"].cpu().numpy(), 64)
        assert np.array_equal(L.codes["w_o"].cpu().numpy(), q)
        assert np.array_equal(L.scales["w_o"].cpu().numpy().view(np.uint16), sc.view(np.uint16))
        past = [1024 - 3 * b for b in range(B)]
        res = run_layer(L, B, 1, past, max_len=1088, seed=12)
        check_layer(L, res, B, 1, past, f"int8 13B B={B}")
    finally:
        L.close()


@pytest.mark.parametrize("extra", [0, 1])
@pytest.mark.parametrize("group,act,B", [(128, torch.float16, 1), (128, torch.bfloat16, 6),
                                         (128, torch.float16, 16)])
def test_int8_group_lengths(group, act, B, extra):
    """MoQ groupings other than 64 along K: groups of 128 codes in every matrix,
    or (extra MLP grouping) 128 in w_qkv / w_o and twice as many groups, of 64,
    in w_fc1 / w_fc2.  Device codes and scales bit-exact with the oracle's
    quantiser at each matrix's group length, and the layer within tolerance of
    the oracle using its own q * s."""
    H, nh, F = 1024, 8, 4096
    L = DeviceLayer(H, nh, F, seed=1006, act_dtype=act, weight_dtype=torch.int8, quant_group=group,
                    mlp_extra_grouping=extra)
    try:
        for k in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
            q, s = L.oracle_quantized(k)
            assert s.shape[1] == L.p[k].shape[1] // (group // 2 if extra and k in ("w_fc1", "w_fc2") else group)
            assert np.array_equal(L.codes[k].cpu().numpy(), q)
            assert np.array_equal(L.scales[k].cpu().numpy().view(np.uint16), s.view(np.uint16))
        past = [40 + 11 * b for b in range(B)]
        res = run_layer(L, B, 1, past, max_len=256, seed=13)
        check_layer(L, res, B, 1, past, f"int8 g{group} extra {extra} {act} B={B}")
    finally:
        L.close()


@pytest.mark.parametrize("act", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("B,T", [(9, 1), (16, 1), (40, 1), (64, 1), (10, 10), (2, 128), (3, 100)])
def test_tile_path_layer(act, B, T):
    """Above 8 rows (B * T) fp16 / bf16 layers run the tensor-core tile
    kernels: decode batches that are not a multiple of 16, prompt chunks of up
    to 128 new tokens per sequence (causal mask among them), ragged cache
    lengths, several token tiles for 300 rows.  Every element against the
    oracle."""
    H, nh, F = 1024, 8, 4096
    L = DeviceLayer(H, nh, F, seed=1010, act_dtype=act, weight_dtype=act)
    try:
        past = [(29 * b) % 60 for b in range(B)]
        res = run_layer(L, B, T, past, max_len=200, seed=14)
        check_layer(L, res, B, T, past, f"tile {act} B={B} T={T}")
    finally:
        L.close()


@pytest.mark.parametrize("act,B,T,past", [(torch.float16, 2, 128, [0, 333]), (torch.float16, 1, 512, [77]),
                                          (torch.bfloat16, 1, 128, [50]), (torch.bfloat16, 3, 64, [5, 0, 130])])
def test_prompt_chunk_layer_4096(act, B, T, past):
    """A prompt chunk of 64..512 new tokens per sequence through one
    4096-hidden layer (tensor-core tiles for the GEMMs, tiled flash attention
    with the causal mask over the cache and the chunk), ragged cache lengths;
    every output element and every new cache row against the oracle."""
    H, nh, F = 4096, 32, 16384
    L = DeviceLayer(H, nh, F, seed=1012, act_dtype=act, weight_dtype=act)
    try:
        res = run_layer(L, B, T, past, max_len=max(past) + T + 16, seed=16)
        check_layer(L, res, B, T, past, f"prompt {act} B={B} T={T}")
    finally:
        L.close()


@pytest.mark.parametrize("act", [torch.float16, torch.bfloat16])
def test_prompt_chunk_many_tiles(act):
    """A chunk with more output tiles than SMs in every GEMM (4 sequences x 512
    new tokens, hidden 2048, FFN 8192: 384 to 1024 tiles), so that CTAs take
    several whole tiles handed out round-robin; every output element and every
    new cache row against the oracle."""
    H, nh, F, B, T = 2048, 16, 8192, 4, 512
    L = DeviceLayer(H, nh, F, seed=1014, act_dtype=act, weight_dtype=act)
    try:
        past = [0, 17, 100, 3]
        res = run_layer(L, B, T, past, max_len=max(past) + T + 8, seed=18)
        check_layer(L, res, B, T, past, f"many tiles {act}")
    finally:
        L.close()


@pytest.mark.parametrize("B,T,group,extra", [(2, 24, 64, 0), (1, 256, 64, 0), (2, 100, 128, 1)])
def test_prompt_chunk_int8(B, T, group, extra):
    """Prompt chunks with MoQ int8 weights (int8 tile kernels: 48 to 256 rows,
    groups of 64, or 128 with the FFN in groups of 64) and the tiled flash
    attention."""
    L = DeviceLayer(1024, 8, 4096, seed=1013, weight_dtype=torch.int8, quant_group=group,
                    mlp_extra_grouping=extra)
    try:
        past = [9, 40][:B]
        res = run_layer(L, B, T, past, max_len=max(past) + T + 8, seed=17)
        check_layer(L, res, B, T, past, f"int8 prompt B={B} T={T} g{group}")
    finally:
        L.close()


def test_quantizer_group32_bit_exact():
    """ds_quantize_int8 with groups of 32 (the layer takes 64 and 128): codes
    and scales bit-exact with the oracle's quantiser."""
    w = inputs.layer_params(1024, 4096, 1007, device="cuda")["w_fc1"]
    q = torch.empty(w.shape, dtype=torch.int8, device="cuda")
    s = torch.empty((w.shape[0], w.shape[1] // 32), dtype=torch.float16, device="cuda")
    ds.ds_quantize_int8(w, q, s, group=32)
    torch.cuda.synchronize()
    q0, s0 = oracle.quantize_int8(w.cpu().numpy(), 32)
    assert np.array_equal(q.cpu().numpy(), q0)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), s0.view(np.uint16))


def test_zero_weight_layer_is_identity():
    L = DeviceLayer(256, 4, 1024, seed=5)
    try:
        for k in list(L.dev):
            L.dev[k].zero_()
        B, T = 2, 1
        res = run_layer(L, B, T, [3, 7], max_len=16)
        assert torch.equal(res["out"], res["x"])
    finally:
        L.close()


def test_cache_overflow_is_flagged_not_written():
    L = DeviceLayer(256, 4, 1024, seed=6)
    try:
        B, T, max_len = 2, 2, 16
        kc, vc = inputs.kv_cache(B, 4, max_len, 64, 1, device="cuda")
        kc0 = kc.clone()
        x = inputs.hidden(B, T, 256, 1, device="cuda")
        out = torch.empty_like(x)
        past = torch.tensor([3, 15], dtype=torch.int32, device="cuda")   # 15 + 2 > 16
        nbytes = ds.ds_layer_workspace_bytes(L.handle, B, T)
        ws = new_workspace(nbytes)
        ds.ds_layer_forward(L.handle, x, out, B, T, kc, vc, max_len, past, ws, nbytes)
        torch.cuda.synchronize()
        code, flags = ds.ds_workspace_status(ws)
        assert code == ds.DS_ERR_DEVICE and flags & ds.DS_DEVFLAG_CACHE_OVERFLOW
        assert torch.equal(kc[1, :, :15], kc0[1, :, :15])       # nothing before the slot changed
        code, flags = ds.ds_workspace_status(ws)                 # the flag was cleared
        assert code == ds.DS_OK and flags == 0
    finally:
        L.close()


def test_bad_arguments_rejected_before_launch():
    L = DeviceLayer(256, 4, 1024, seed=7)
    try:
        x = torch.zeros(1, 1, 256, dtype=torch.float16, device="cuda")
        out = torch.empty_like(x)
        kc = torch.zeros(1, 4, 8, 64, dtype=torch.float16, device="cuda")
        past = torch.zeros(1, dtype=torch.int32, device="cuda")
        nbytes = ds.ds_layer_workspace_bytes(L.handle, 1, 1)
        ws = new_workspace(nbytes)
        n0 = ds.ds_launch_count()
        with pytest.raises(ds.DSError) as e:
            ds.ds_layer_forward(L.handle, x, out, 1, 1, kc, kc, 8, past, ws, nbytes - 256)
        assert e.value.code == ds.DS_ERR_WORKSPACE
        with pytest.raises(ds.DSError) as e:
            ds.ds_layer_forward(L.handle, x, x, 1, 1, kc, kc, 8, past, ws, nbytes)
        assert e.value.code == ds.DS_ERR_INVALID_ARG
        with pytest.raises(ds.DSError) as e:
            ds.ds_layer_forward(L.handle, x, out, 4097, 1, kc, kc, 8, past, ws, nbytes)
        assert e.value.code == ds.DS_ERR_UNSUPPORTED
        assert ds.ds_launch_count() == n0
    finally:
        L.close()


def test_bounded_wait_runs_out_and_is_reported():
    """A device wait that nothing satisfies gives up after its budget, records
    DS_DEVFLAG_WAIT_TIMEOUT in the workspace status word (read and cleared by
    ds_workspace_status) and returns; the context then still runs a layer."""
    L = DeviceLayer(256, 4, 1024, seed=9)
    try:
        nbytes = ds.ds_layer_workspace_bytes(L.handle, 1, 1)
        ws = new_workspace(nbytes)
        ds.ds_selftest_wait_timeout(ws, 2000)   # 2 ms budget
        code, flags = ds.ds_workspace_status(ws)
        assert code == ds.DS_ERR_DEVICE and flags == ds.DS_DEVFLAG_WAIT_TIMEOUT
        code, flags = ds.ds_workspace_status(ws)
        assert code == ds.DS_OK and flags == 0
        res = run_layer(L, 1, 1, [5], max_len=16)
        check_layer(L, res, 1, 1, [5], "after the timeout")
    finally:
        L.close()


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second GPU to make current")
def test_forward_on_another_current_device_is_rejected():
    """A layer's kernels run on the device it was created on; a call made with
    another device current is refused before any launch."""
    L = DeviceLayer(256, 4, 1024, seed=8)
    try:
        x = torch.zeros(1, 1, 256, dtype=torch.float16, device="cuda:0")
        out = torch.empty_like(x)
        kc = torch.zeros(1, 4, 8, 64, dtype=torch.float16, device="cuda:0")
        past = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        nbytes = ds.ds_layer_workspace_bytes(L.handle, 1, 1)
        ws = new_workspace(nbytes, device="cuda:0")
        n0 = ds.ds_launch_count()
        with torch.cuda.device(1):
            with pytest.raises(ds.DSError) as e:
                ds.ds_layer_forward(L.handle, x, out, 1, 1, kc, kc.clone(), 8, past, ws, nbytes,
                                    stream=torch.cuda.current_stream(0))
            assert e.value.code == ds.DS_ERR_INVALID_ARG
        assert ds.ds_launch_count() == n0
    finally:
        L.close()
