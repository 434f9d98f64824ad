"""The diagnostic build (DS_DEBUG_BOUNDS): device-side bounds checks at the
kernels' global stores and key ranges, which record DS_DEVFLAG_BOUNDS in the
workspace status word and skip the access instead of trapping.  Valid work
must raise no flag and keep parity with the oracle: streaming decode
kernels, tensor-core tiles (fp16, bf16, int8 codes) and decode attention,
each run through libdslayer_debug_bounds.so in a process of its own (the
binding loads one library per process)."""
import os

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(q):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    try:
        import torch
        from transformer_layer_gb300 import build, ds
        ds.load(build.build(debug_bounds=True))
        from helpers import DeviceLayer
        from test_layer_gpu import check_layer, run_layer
        cases = [  # (act, weight, B, T)
            (torch.float16, torch.float16, 2, 1),     # streaming kernels, decode attention
            (torch.bfloat16, torch.bfloat16, 16, 1),  # tiles (bf16 hi/lo), cluster split-K
            (torch.float16, torch.int8, 16, 1),       # int8 tiles
            (torch.float16, torch.float16, 2, 12),    # a short chunk through the decode attention
        ]
        for act, wdt, B, T in cases:
            L = DeviceLayer(1024, 8, 4096, seed=1015, act_dtype=act, weight_dtype=wdt)
            try:
                past = [(13 * b) % 40 for b in range(B)]
                res = run_layer(L, B, T, past, max_len=64, seed=19)  # checks the status word is clear
                check_layer(L, res, B, T, past, f"debug-bounds {act} {wdt} B={B} T={T}")
            finally:
                L.close()
        q.put("ok")
    except BaseException as e:  # reported to the parent
        q.put(repr(e))


def test_debug_bounds_build_raises_no_flag_on_valid_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_worker, args=(q,))
    p.start()
    msg = q.get(timeout=900)
    p.join(120)
    assert msg == "ok", msg
    assert p.exitcode == 0
