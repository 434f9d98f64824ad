"""GPU parity of the residual-MoE (PR-MoE) FFN block against the oracle.

Page: "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE 优化与
init_inference 全解析", section "用 PR-MoE 结构进一步提速并降低推理成本" (the
formula is the reading documented in oracle/moe.py and include/ds_layer.h).

The expert of every row is an integer decided by floating point: it must equal
the oracle's argmax, except where the oracle's top two logits are within the
rounding of the device's operands (then either is valid, and the oracle is
evaluated at the device's choice).  Outputs are compared element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_close, new_workspace, to64
from transformer_layer_gb300 import ds, inputs

pytestmark = pytest.mark.gpu

_IDS = {"ln2_g": 50, "ln2_b": 51, "w_gate": 52, "w_fc1": 53, "b_fc1": 54, "w_fc2": 55, "b_fc2": 56,
        "we_fc1": 57, "be_fc1": 58, "we_fc2": 59, "be_fc2": 60}


def moe_params(H, F, E, seed, dtype):
    shapes = {"ln2_g": (H,), "ln2_b": (H,), "w_gate": (E, H), "w_fc1": (F, H), "b_fc1": (F,), "w_fc2": (H, F),
              "b_fc2": (H,), "we_fc1": (E, F, H), "be_fc1": (E, F), "we_fc2": (E, H, F), "be_fc2": (E, H)}
    out = {}
    for k, sh in shapes.items():
        mean, std = (1.0, 0.1) if k == "ln2_g" else (0.0, 0.1 if k == "ln2_b" else (0.01 if k.startswith("b") else 0.02))
        out[k] = inputs.normal(sh, mean, std, seed, _IDS[k], dtype, "cuda")
    return out


@pytest.mark.parametrize("act,H,F,E,rows", [(torch.float16, 512, 1024, 8, 1), (torch.float16, 512, 1024, 8, 5),
                                            (torch.bfloat16, 512, 1024, 8, 16), (torch.float16, 4096, 16384, 4, 2)])
def test_residual_moe_ffn_vs_oracle(act, H, F, E, rows):
    p = moe_params(H, F, E, 1800, act)
    moe = ds.ds_moe_ffn_create(H, F, E, p, act)
    try:
        x = inputs.hidden(rows, 1, H, 1800, dtype=act, device="cuda").reshape(rows, H)
        y = torch.full_like(x, float("nan"))
        ex = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        nb = ds.ds_moe_ffn_workspace_bytes(moe, rows)
        ws = new_workspace(nb)
        n0 = ds.ds_launch_count()
        ds.ds_moe_ffn_forward(moe, x, y, rows, ex, ws, nb)
        torch.cuda.synchronize()
        code, flags = ds.ds_workspace_status(ws)
        assert code == ds.DS_OK and flags == 0
        p64 = {k: to64(v) for k, v in p.items()}
        r = oracle.residual_moe_ffn(to64(x), p64)
        dev_e = ex.cpu().numpy()
        lg = r["logits"]
        for row in range(rows):
            order = np.argsort(-lg[row], kind="stable")
            gap = lg[row, order[0]] - lg[row, order[1]] if E > 1 else np.inf
            if gap > 2e-3:
                assert dev_e[row] == r["expert"][row], (row, dev_e[row], r["expert"][row], gap)
            else:
                assert dev_e[row] in (order[0], order[1]), (row, dev_e[row], order[:2])
        ref = oracle.residual_moe_ffn(to64(x), p64, experts=dev_e)
        check_close(y, ref["y"], act, what=f"moe {act} H={H} rows={rows}")
        # a second call on the same workspace gives the same bytes (deterministic, counters self-reset)
        y2 = torch.empty_like(y)
        ds.ds_moe_ffn_forward(moe, x, y2, rows, None, ws, nb)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
    finally:
        ds.ds_moe_ffn_destroy(moe)


def test_moe_rejects_bad_arguments_before_launch():
    H, F, E = 512, 1024, 4
    p = moe_params(H, F, E, 1801, torch.float16)
    moe = ds.ds_moe_ffn_create(H, F, E, p, torch.float16)
    try:
        x = torch.zeros(2, H, dtype=torch.float16, device="cuda")
        nb = ds.ds_moe_ffn_workspace_bytes(moe, 2)
        ws = new_workspace(nb)
        n0 = ds.ds_launch_count()
        with pytest.raises(ds.DSError) as e:
            ds.ds_moe_ffn_forward(moe, x, x, 2, None, ws, nb)      # aliasing
        assert e.value.code == ds.DS_ERR_INVALID_ARG
        with pytest.raises(ds.DSError) as e:
            ds.ds_moe_ffn_forward(moe, x, torch.empty_like(x), 2, None, ws, nb - 256)
        assert e.value.code == ds.DS_ERR_WORKSPACE
        assert ds.ds_launch_count() == n0
    finally:
        ds.ds_moe_ffn_destroy(moe)
