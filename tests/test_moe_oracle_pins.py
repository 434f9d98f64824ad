"""Pins of the residual-MoE oracle (oracle.moe) against closed forms.

Page: "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE 优化与
init_inference 全解析", section "用 PR-MoE 结构进一步提速并降低推理成本" (residual
MoE; the formula is the reading documented in oracle/moe.py).
"""
import math

import numpy as np

import oracle


def _params(rng, H, F, E, zero_weights=False):
    def w(*sh):
        return np.zeros(sh) if zero_weights else rng.standard_normal(sh) * 0.3
    return {"ln2_g": 1.0 + 0.1 * rng.standard_normal(H), "ln2_b": 0.1 * rng.standard_normal(H),
            "w_gate": w(E, H), "w_fc1": w(F, H), "b_fc1": rng.standard_normal(F), "w_fc2": w(H, F),
            "b_fc2": rng.standard_normal(H), "we_fc1": w(E, F, H), "be_fc1": rng.standard_normal((E, F)),
            "we_fc2": w(E, H, F), "be_fc2": rng.standard_normal((E, H))}


def test_zero_gate_picks_expert_0_with_weight_1_over_E():
    """All logits 0: softmax 1/E each, the tie resolves to expert 0; with
    bias-only FFNs, y = x + b2 + b2_expert0 / E exactly."""
    rng = np.random.default_rng(41)
    H, F, E = 8, 12, 5
    p = _params(rng, H, F, E, zero_weights=True)
    x = rng.standard_normal((3, H))
    r = oracle.residual_moe_ffn(x, p)
    assert list(r["expert"]) == [0, 0, 0]
    np.testing.assert_allclose(r["weight"], 1.0 / E, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["y"], x + p["b_fc2"] + p["be_fc2"][0] / E, rtol=0, atol=1e-14)


def test_gate_weight_at_known_logits():
    """Gate rows that give logits [0, ln 2, 0] for this row: expert 1, weight
    2 / (1 + 2 + 1) = 1/2 exactly; bias-only FFNs make y = x + b2 + be2[1] / 2."""
    rng = np.random.default_rng(42)
    H, F, E = 8, 12, 3
    p = _params(rng, H, F, E, zero_weights=True)
    x = rng.standard_normal((1, H))
    h = oracle.layer_norm(x, p["ln2_g"], p["ln2_b"])[0]
    p["w_gate"][1] = math.log(2.0) * h / (h @ h)
    r = oracle.residual_moe_ffn(x, p)
    assert r["expert"][0] == 1
    np.testing.assert_allclose(r["logits"][0], [0.0, math.log(2.0), 0.0], rtol=0, atol=1e-14)
    assert abs(r["weight"][0] - 0.5) < 1e-15
    np.testing.assert_allclose(r["y"], x + p["b_fc2"] + 0.5 * p["be_fc2"][1], rtol=0, atol=1e-14)


def test_dominant_gate_row_chooses_its_expert():
    rng = np.random.default_rng(43)
    H, F, E = 16, 8, 6
    p = _params(rng, H, F, E)
    x = rng.standard_normal((4, H))
    h = oracle.layer_norm(x, p["ln2_g"], p["ln2_b"])
    for target in range(E):
        q = dict(p)
        q["w_gate"] = p["w_gate"].copy() * 1e-3
        q["w_gate"][target] = 50.0 * h.sum(axis=0) / np.linalg.norm(h.sum(axis=0)) ** 2 + 0.0
        # rows whose h aligns with the mean direction pick `target`
        r = oracle.residual_moe_ffn(x, q)
        for row in range(4):
            lg = r["logits"][row]
            assert r["expert"][row] == int(np.argmax(lg))
            assert lg[r["expert"][row]] >= lg.max()


def test_single_expert_reduces_to_two_ffns():
    """E = 1: the gate weight is 1, so y = x + MLP(h) + Expert_0(h), built here
    from the layer oracle's pinned pieces (LayerNorm, linear, GeLU)."""
    rng = np.random.default_rng(44)
    H, F, E = 8, 16, 1
    p = _params(rng, H, F, E)
    x = rng.standard_normal((2, H))
    r = oracle.residual_moe_ffn(x, p)
    h = oracle.layer_norm(x, p["ln2_g"], p["ln2_b"])
    want = (x + oracle.linear(oracle.gelu_tanh(oracle.linear(h, p["w_fc1"], p["b_fc1"])), p["w_fc2"], p["b_fc2"])
            + oracle.linear(oracle.gelu_tanh(oracle.linear(h, p["we_fc1"][0], p["be_fc1"][0])), p["we_fc2"][0],
                            p["be_fc2"][0]))
    np.testing.assert_allclose(r["weight"], 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["y"], want, rtol=0, atol=1e-12)


def test_rows_are_independent():
    """Each row routes on its own gate logits: running rows one by one gives
    the same experts and outputs."""
    rng = np.random.default_rng(45)
    H, F, E = 8, 8, 4
    p = _params(rng, H, F, E)
    x = rng.standard_normal((5, H))
    r = oracle.residual_moe_ffn(x, p)
    for row in range(5):
        r1 = oracle.residual_moe_ffn(x[row:row + 1], p)
        assert r1["expert"][0] == r["expert"][row]
        np.testing.assert_allclose(r1["y"][0], r["y"][row], rtol=0, atol=1e-13)
