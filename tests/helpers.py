"""Helpers shared by the GPU parity tests (not collected as tests).

The device side is driven only through the C-ABI binding
(transformer_layer_gb300.ds); the expected values come only from the CPU oracle
(oracle/), fed the same input bytes.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from transformer_layer_gb300 import ds, inputs

# Parity bar for fp16 / bf16 layer outputs: max-abs <= 2e-2 per element
# (relaxed to one unit in the last place of the output dtype where a single
# rounding of the stored value already exceeds 2e-2) and relative L2 <= 2e-3.
MAX_ABS = 2e-2
REL_L2 = 2e-3


def ulp(ref: np.ndarray, dtype) -> np.ndarray:
    mant = 10 if dtype == torch.float16 else 7
    a = np.maximum(np.abs(ref), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def check_close(gpu, ref, dtype, max_abs=MAX_ABS, rel_l2=REL_L2, what=""):
    g = gpu.detach().double().cpu().numpy() if torch.is_tensor(gpu) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    tol = np.maximum(max_abs, ulp(r, dtype))
    worst = float((err / tol).max()) if err.size else 0.0
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    assert np.all(err <= tol), f"{what}: max-abs {err.max():.3e} (worst err/tol {worst:.2f})"
    assert rel <= rel_l2, f"{what}: rel-L2 {rel:.3e} > {rel_l2}"
    return float(err.max()), rel


def to64(t):
    return t.detach().double().cpu().numpy()


def cache_store(dtype):
    """The KV cache's storage rounding for the oracle (round to nearest even
    into the cache dtype, float16 or bfloat16)."""
    def store(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).double().numpy()
    return store


class DeviceLayer:
    """One layer's device weights + library handle (int8 weights quantised on
    the device with ds_quantize_int8 when weight_dtype is torch.int8).

    int8 group lengths along K: ``quant_group`` for w_qkv and w_o; with
    ``mlp_extra_grouping`` the FFN matrices w_fc1 and w_fc2 are split into
    twice as many groups (quant_group / 2)."""

    def __init__(self, hidden, heads, ffn, seed, layer=0, act_dtype=torch.float16,
                 weight_dtype=torch.float16, device="cuda", quant_group=64, mlp_extra_grouping=0):
        self.hidden, self.heads, self.ffn = hidden, heads, ffn
        self.quant_group, self.mlp_extra_grouping = quant_group, mlp_extra_grouping
        self.groups = {k: (quant_group // 2 if mlp_extra_grouping and k in ("w_fc1", "w_fc2") else quant_group)
                       for k in ("w_qkv", "w_o", "w_fc1", "w_fc2")}
        self.act_dtype, self.weight_dtype = act_dtype, weight_dtype
        src_dtype = torch.float16 if weight_dtype == torch.int8 else act_dtype
        self.p = inputs.layer_params(hidden, ffn, seed, layer, dtype=src_dtype, device=device)
        if act_dtype != src_dtype:
            for k in ("ln1_g", "ln1_b", "b_qkv", "b_o", "ln2_g", "ln2_b", "b_fc1", "b_fc2"):
                self.p[k] = self.p[k].to(act_dtype)
        self.dev = dict(self.p)
        self.codes, self.scales = {}, {}
        if weight_dtype == torch.int8:
            for k, sk in (("w_qkv", "s_qkv"), ("w_o", "s_o"), ("w_fc1", "s_fc1"), ("w_fc2", "s_fc2")):
                w, grp = self.p[k], self.groups[k]
                q = torch.empty(w.shape, dtype=torch.int8, device=device)
                s = torch.empty((w.shape[0], w.shape[1] // grp), dtype=torch.float16, device=device)
                ds.ds_quantize_int8(w, q, s, group=grp)
                self.dev[k] = q
                self.dev[sk] = s
                self.codes[k], self.scales[k] = q, s
        torch.cuda.synchronize()
        self.handle = ds.ds_layer_create(hidden, heads, ffn, self.dev, act_dtype, weight_dtype,
                                         quant_group=quant_group, mlp_extra_grouping=mlp_extra_grouping)
        self._oracle = None

    def oracle_quantized(self, k):
        """The oracle's own (codes, scales) of int8 matrix k, quantised from the
        same float16 weights the device quantiser read."""
        return oracle.quantize_int8(self.p[k].cpu().numpy(), self.groups[k])

    def oracle_params(self):
        """float64 parameters for the oracle: the float16 / bf16 values the device
        uses, and for int8 weights q * s from the oracle's own quantiser (never
        the device's codes)."""
        if self._oracle is None:
            out = {}
            for k, v in self.p.items():
                if self.weight_dtype == torch.int8 and k in self.groups:
                    q, s = self.oracle_quantized(k)
                    out[k] = oracle.dequantize_int8(q, s, self.groups[k])
                else:
                    out[k] = to64(v)
            self._oracle = out
        return self._oracle

    def close(self):
        ds.ds_layer_destroy(self.handle)


def new_workspace(nbytes, device="cuda"):
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    ds.ds_workspace_init(ws, ws.numel())
    return ws
