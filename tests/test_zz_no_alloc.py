"""The no-allocation layer forward against the workspace forward (GPU).

ds_layer_forward_noalloc serves callers that cannot allocate device memory:
it runs the same kernels on a static workspace inside the library.  Two
calls in a row (the second one reuses the static array left by the first)
must match ds_layer_forward within the parity tolerance used by every other
test; a batch shape whose workspace exceeds the static array is refused.
This file is collected last on purpose.
"""
import pytest
import torch

from helpers import DeviceLayer, check_close, new_workspace
from transformer_layer_gb300 import ds, inputs

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_forward_twice():
    L = DeviceLayer(512, 8, 2048, seed=1500)
    try:
        B, T, max_len = 3, 2, 40
        past = torch.tensor([5, 17, 0], dtype=torch.int32, device="cuda")
        for call in range(2):
            x = inputs.hidden(B, T, 512, 1500, step=call, device="cuda")
            kc, vc = inputs.kv_cache(B, 8, max_len, 64, 1500 + call, device="cuda")
            kc2, vc2 = kc.clone(), vc.clone()
            ref = torch.empty_like(x)
            nbytes = ds.ds_layer_workspace_bytes(L.handle, B, T)
            ws = new_workspace(nbytes)
            ds.ds_layer_forward(L.handle, x, ref, B, T, kc, vc, max_len, past, ws, nbytes)
            out = torch.full_like(x, float("nan"))
            ds.ds_layer_forward_noalloc(L.handle, x, out, B, T, kc2, vc2, max_len, past)
            torch.cuda.synchronize()
            check_close(out, ref.double().cpu().numpy(), torch.float16, what=f"call {call} y")
            check_close(kc2, kc.double().cpu().numpy(), torch.float16, what=f"call {call} k cache")
            check_close(vc2, vc.double().cpu().numpy(), torch.float16, what=f"call {call} v cache")
    finally:
        L.close()


def test_noalloc_refuses_workspace_beyond_static_size():
    L = DeviceLayer(4096, 32, 16384, seed=1501)
    try:
        B, T = 16, 32   # a 512-row prompt chunk
        assert ds.ds_layer_workspace_bytes(L.handle, B, T) > (16 << 20)
        x = torch.zeros(B, T, 4096, dtype=torch.float16, device="cuda")
        kc = torch.zeros(B, 32, T, 128, dtype=torch.float16, device="cuda")
        past = torch.zeros(B, dtype=torch.int32, device="cuda")
        n0 = ds.ds_launch_count()
        with pytest.raises(ds.DSError) as e:
            ds.ds_layer_forward_noalloc(L.handle, x, torch.empty_like(x), B, T, kc, kc.clone(), T, past)
        assert e.value.code == ds.DS_ERR_UNSUPPORTED
        assert ds.ds_launch_count() == n0
    finally:
        L.close()


def test_noalloc_status_reports_a_cache_overflow():
    """The device status flags of the no-allocation path are read back with
    ds_noalloc_status: a row whose cache position is past max_len is not
    written and raises the cache-overflow flag; the flag is cleared once read."""
    L = DeviceLayer(256, 4, 1024, seed=1502)
    try:
        B, T, max_len = 2, 2, 16
        kc, vc = inputs.kv_cache(B, 4, max_len, 64, 1502, device="cuda")
        kc0 = kc.clone()
        x = inputs.hidden(B, T, 256, 1502, device="cuda")
        past = torch.tensor([3, 15], dtype=torch.int32, device="cuda")   # 15 + 2 > 16
        ds.ds_layer_forward_noalloc(L.handle, x, torch.empty_like(x), B, T, kc, vc, max_len, past)
        code, flags = ds.ds_noalloc_status()
        assert code == ds.DS_ERR_DEVICE and flags & ds.DS_DEVFLAG_CACHE_OVERFLOW
        assert torch.equal(kc[1, :, :15], kc0[1, :, :15])
        code, flags = ds.ds_noalloc_status()
        assert code == ds.DS_OK and flags == 0
    finally:
        L.close()
