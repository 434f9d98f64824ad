"""Byte accounting behind bench.py's roofline figures (CPU only).

The roofline fraction divides algorithmic bytes by time, so these counts are
checked against sums written out here parameter by parameter, and against
each other: the per-kernel figures must add up to the per-layer figure.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _params(H, F):
    """Parameter counts of one pre-LN layer: (matrix weights, vector entries)."""
    mats = 3 * H * H + H * H + F * H + H * F          # w_qkv, w_o, w_fc1, w_fc2
    vecs = 3 * H + H + F + H + 4 * H                  # four biases, two LN gamma/beta pairs
    return mats, vecs


@pytest.mark.parametrize("H,F", [(4096, 16384), (2560, 10240), (5120, 20480), (256, 1024)])
def test_layer_bytes_fp16(H, F):
    mats, vecs = _params(H, F)
    assert bench.layer_bytes(H, F, 2.0) == 2 * mats + 2 * vecs


def test_7b_stack_weight_bytes():
    # 32 layers of hidden 4096 / FFN 16384 in fp16: 12.888 GB of parameters
    assert bench.layer_bytes(4096, 16384, 2.0) * 32 == pytest.approx(12.888e9, rel=1e-3)


def test_7b_step_bytes_batch1():
    # weights + K/V rows read at S = 513 .. 576 keys, averaged over one pass of 64 positions
    H, L, past = 4096, 32, 512
    kv = sum(L * 2 * (past + 1 + i) * H * 2 + L * 2 * H * 2 for i in range(64)) / 64
    want = bench.layer_bytes(H, 16384, 2.0) * L + kv
    assert bench.step_bytes(H, 16384, L, 1, past, 64) == pytest.approx(want, rel=1e-12)
    assert want == pytest.approx(13.18e9, rel=2e-3)


def test_int8_bytes_per_matrix_group():
    # one code byte per weight plus one 2-byte fp16 scale per group along K
    H, F = 5120, 20480
    mats, vecs = _params(H, F)
    g64 = bench.layer_bytes(H, F, 1.0 + 2.0 / 64)
    assert g64 == pytest.approx(mats + 2 * mats / 64 + 2 * vecs, rel=1e-12)
    mixed = bench.layer_bytes(H, F, (1.0 + 2.0 / 128, 1.0 + 2.0 / 64))
    att, ffn = 4 * H * H, 2 * F * H
    assert mixed == pytest.approx(att + 2 * att / 128 + ffn + 2 * ffn / 64 + 2 * vecs, rel=1e-12)
    assert g64 * 40 == pytest.approx(12.98e9, rel=1e-3)


@pytest.mark.parametrize("wbytes", [2.0, 1.0 + 2.0 / 64, (1.0 + 2.0 / 128, 1.0 + 2.0 / 64)])
def test_region_bytes_add_up_to_the_layer(wbytes):
    # with no batch rows the four GEMV launches read exactly the layer's parameters
    H, F = 5120, 20480
    r = bench.region_bytes(H, F, 0, 1024, wbytes)
    assert r["attention"] == 0
    total = r["ln_qkv"] + r["oproj_res"] + r["ffn_up"] + r["ffn_down"]
    assert total == pytest.approx(bench.layer_bytes(H, F, wbytes), rel=1e-12)


def test_attention_bytes_are_the_kv_rows():
    # batch 1: K and V rows of S keys (2 bytes each) plus q in and o out (fp32)
    H, past = 4096, 512
    S = past + 1 + 32
    assert bench.region_bytes(H, 16384, 1, past)["attention"] == 2 * S * H * 2 + 2 * H * 4


def test_a_run_with_a_device_flag_reports_nothing(monkeypatch):
    """bench.py reads the workspace status word after its timed, end-to-end and
    profiled steps: a flag (a bounded wait that gave up, a bounds or cache
    check) stops it before any result line; a clean word lets it go on."""
    from transformer_layer_gb300 import ds

    seen = []

    def fake_status(flags):
        def status(ws, stream=None):
            seen.append((ws, stream))
            return (ds.DS_ERR_DEVICE if flags else ds.DS_OK), flags
        return status

    monkeypatch.setattr(ds, "ds_workspace_status", fake_status(0))
    assert bench.check_device("ws", "stream", "the timed decode steps") is None
    monkeypatch.setattr(ds, "ds_workspace_status", fake_status(ds.DS_DEVFLAG_WAIT_TIMEOUT))
    with pytest.raises(SystemExit) as e:
        bench.check_device("ws", "stream", "the timed decode steps")
    assert f"0x{ds.DS_DEVFLAG_WAIT_TIMEOUT:x}" in str(e.value) and "no result" in str(e.value)
    assert seen == [("ws", "stream"), ("ws", "stream")]
