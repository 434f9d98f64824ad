"""Pins of the tensor-sliced layer oracle (oracle.tp) against the unsplit
layer oracle and closed forms.

Page: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核与
MoQ 量化支持", §3.2 (Attn and FF blocks split across GPUs in the Megatron-LM
manner, one all-reduce after each) and §3.1 (fusion up to each all-reduce
boundary).  The unsplit layer oracle is pinned on its own (test_oracle_pins);
here the split is held to the identity that defines it: the sum over ranks of
the partial results is the unsplit layer.
"""
import numpy as np
import pytest

import oracle


def _params(rng, H, F, zero=()):
    def w(name, *sh):
        return np.zeros(sh) if name in zero else rng.standard_normal(sh) * 0.2
    return {"ln1_g": 1 + 0.1 * rng.standard_normal(H), "ln1_b": 0.1 * rng.standard_normal(H),
            "w_qkv": w("w_qkv", 3 * H, H), "b_qkv": 0.1 * rng.standard_normal(3 * H),
            "w_o": w("w_o", H, H), "b_o": rng.standard_normal(H),
            "ln2_g": 1 + 0.1 * rng.standard_normal(H), "ln2_b": 0.1 * rng.standard_normal(H),
            "w_fc1": w("w_fc1", F, H), "b_fc1": 0.1 * rng.standard_normal(F),
            "w_fc2": w("w_fc2", H, F), "b_fc2": rng.standard_normal(H)}


def _caches(rng, B, nh, L, d):
    return rng.standard_normal((B, nh, L, d)), rng.standard_normal((B, nh, L, d))


def _split_caches(K, tp):
    nh = K.shape[1]
    step = nh // tp
    return [K[:, r * step:(r + 1) * step].copy() for r in range(tp)]


@pytest.mark.parametrize("tp", [1, 2, 4])
@pytest.mark.parametrize("B,T", [(1, 1), (2, 3)])
def test_sum_over_ranks_is_the_unsplit_layer(tp, B, T):
    rng = np.random.default_rng(100 + 10 * tp + B)
    H, nh, F, L = 16, 4, 24, 9
    d = H // nh
    p = _params(rng, H, F)
    K, V = _caches(rng, B, nh, L, d)
    past = [4, 2][:B]
    x = rng.standard_normal((B, T, H))
    ref_k, ref_v = K.copy(), V.copy()
    ref = oracle.layer_forward(x, p, ref_k, ref_v, past, nh)
    ks, vs = _split_caches(K, tp), _split_caches(V, tp)
    got = oracle.tp_layer_forward(x, p, ks, vs, past, nh, tp)
    np.testing.assert_allclose(got["x1"], ref["x1"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["y"], ref["y"], rtol=0, atol=1e-12)
    # every rank's cache holds exactly its heads of the unsplit cache
    for r in range(tp):
        np.testing.assert_array_equal(ks[r], ref_k[:, r * nh // tp:(r + 1) * nh // tp])
        np.testing.assert_array_equal(vs[r], ref_v[:, r * nh // tp:(r + 1) * nh // tp])
        np.testing.assert_allclose(got["k_new"][r], ref["k_new"][:, :, r * nh // tp:(r + 1) * nh // tp],
                                   rtol=0, atol=1e-13)


def test_bias_and_residual_are_added_once():
    """W_o = 0 and W_2 = 0: x1 = x + b_o and y = x1 + b_2 exactly, all of it on
    rank 0; the other ranks' partial sums are exactly zero (adding the bias or
    the residual on every rank would give x + W b_o)."""
    rng = np.random.default_rng(7)
    H, nh, F, L, tp = 16, 4, 32, 5, 4
    p = _params(rng, H, F, zero=("w_o", "w_fc2"))
    K, V = _caches(rng, 1, nh, L, H // nh)
    x = rng.standard_normal((1, 1, H))
    got = oracle.tp_layer_forward(x, p, _split_caches(K, tp), _split_caches(V, tp), [3], nh, tp)
    np.testing.assert_array_equal(got["x1"], x + p["b_o"])
    np.testing.assert_array_equal(got["y"], x + p["b_o"] + p["b_fc2"])
    for r in range(1, tp):
        assert not np.any(got["x1_parts"][r]) and not np.any(got["y_parts"][r])


def test_single_head_rank_attention_is_that_heads_softmax():
    """One head per rank, a cache of one position plus the new token: the
    attention output of rank r is a two-key softmax mix, written out here by
    hand (w = 1 / (1 + exp(s0 - s1)) on the new value)."""
    rng = np.random.default_rng(11)
    H, nh, F, tp = 8, 2, 16, 2
    d = H // nh
    p = _params(rng, H, F)
    K, V = _caches(rng, 1, nh, 4, d)
    x = rng.standard_normal((1, 1, H))
    for r in range(tp):
        s = oracle.shard_layer_params(p, nh, tp, r)
        kr, vr = K[:, r:r + 1].copy(), V[:, r:r + 1].copy()
        out = oracle.tp_attention_partial(x, s, kr, vr, [1], 1, r)
        h1 = oracle.layer_norm(x[0, 0], p["ln1_g"], p["ln1_b"])
        rows = slice(r * d, (r + 1) * d)
        q = p["w_qkv"][0:H][rows] @ h1 + p["b_qkv"][0:H][rows]
        k = p["w_qkv"][H:2 * H][rows] @ h1 + p["b_qkv"][H:2 * H][rows]
        v = p["w_qkv"][2 * H:][rows] @ h1 + p["b_qkv"][2 * H:][rows]
        s0, s1 = (K[0, r, 0] @ q) / np.sqrt(d), (k @ q) / np.sqrt(d)
        w1 = 1.0 / (1.0 + np.exp(s0 - s1))
        o = (1 - w1) * V[0, r, 0] + w1 * v
        np.testing.assert_allclose(out["attn"][0, 0], o, rtol=0, atol=1e-13)
        want = p["w_o"][:, rows] @ o + ((x[0, 0] + p["b_o"]) if r == 0 else 0.0)
        np.testing.assert_allclose(out["x1_part"][0, 0], want, rtol=0, atol=1e-13)


def test_shard_shapes():
    rng = np.random.default_rng(3)
    H, nh, F, tp = 32, 8, 64, 4
    p = _params(rng, H, F)
    for r in range(tp):
        s = oracle.shard_layer_params(p, nh, tp, r)
        assert s["w_qkv"].shape == (3 * H // tp, H) and s["b_qkv"].shape == (3 * H // tp,)
        assert s["w_o"].shape == (H, H // tp)
        assert s["w_fc1"].shape == (F // tp, H) and s["b_fc1"].shape == (F // tp,)
        assert s["w_fc2"].shape == (H, F // tp)
        for k in ("ln1_g", "ln1_b", "b_o", "ln2_g", "ln2_b", "b_fc2"):
            assert s[k] is p[k]
