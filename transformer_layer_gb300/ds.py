"""ctypes binding of libdslayer.so (argument marshalling only).

Every function here forwards to the C entry point of the same name declared
in include/ds_layer.h; tensors are passed as raw device pointers
(``tensor.data_ptr()``) and streams as ``torch.cuda.Stream.cuda_stream``.
Nothing here computes any part of the layer: all of it runs in the library's
CUDA kernels, and a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdslayer.so")
LIB_DEBUG_BOUNDS_PATH = os.path.join(_PKG, "libdslayer_debug_bounds.so")  # diagnostic build

DS_OK, DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED, DS_ERR_CUDA, DS_ERR_WORKSPACE, DS_ERR_DEVICE = range(6)
DS_F16, DS_BF16, DS_I8 = 0, 1, 2
DS_DEVFLAG_CACHE_OVERFLOW = 0x1
DS_DEVFLAG_WAIT_TIMEOUT = 0x2
DS_DEVFLAG_BOUNDS = 0x4

# Every exported symbol of include/ds_layer.h, with (restype, argtypes).
_vp = C.c_void_p
_SIGS = {
    "ds_layer_create": (C.c_int, [_vp, _vp, C.POINTER(_vp)]),
    "ds_layer_destroy": (C.c_int, [_vp]),
    "ds_layer_workspace_bytes": (C.c_size_t, [_vp, C.c_int, C.c_int]),
    "ds_workspace_init": (C.c_int, [_vp, C.c_size_t, _vp]),
    "ds_layer_forward": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, _vp, _vp, C.c_int, _vp, _vp,
                                   C.c_size_t, _vp]),
    "ds_layer_forward_noalloc": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, _vp, _vp, C.c_int, _vp, _vp]),
    "ds_noalloc_status": (C.c_int, [C.POINTER(C.c_uint32), _vp]),
    "ds_stack_create": (C.c_int, [C.POINTER(_vp), C.c_int, C.POINTER(_vp)]),
    "ds_stack_destroy": (C.c_int, [_vp]),
    "ds_stack_workspace_bytes": (C.c_size_t, [_vp, C.c_int]),
    "ds_stack_decode_step": (C.c_int, [_vp, _vp, _vp, C.c_int, C.POINTER(_vp), C.POINTER(_vp),
                                       C.c_int, _vp, _vp, C.c_size_t, _vp]),
    "ds_stack_forward": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, C.POINTER(_vp), C.POINTER(_vp), C.c_int, _vp,
                                   _vp, C.c_size_t, _vp]),
    "ds_stack_decode_host": (C.c_int, [_vp, _vp, _vp, _vp, _vp, C.c_int, C.POINTER(_vp),
                                       C.POINTER(_vp), C.c_int, _vp, _vp, C.c_size_t, _vp]),
    "ds_stack_set_profiling": (C.c_int, [_vp, C.c_int]),
    "ds_stack_region_times": (C.c_int, [_vp, C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "ds_stack_graph_captures": (C.c_uint64, [_vp]),
    "ds_quantize_int8": (C.c_int, [_vp, C.c_int, C.c_int, C.c_int, _vp, _vp, _vp]),
    "ds_workspace_status": (C.c_int, [_vp, C.POINTER(C.c_uint32), _vp]),
    "ds_moe_ffn_create": (C.c_int, [_vp, _vp, C.POINTER(_vp)]),
    "ds_moe_ffn_destroy": (C.c_int, [_vp]),
    "ds_moe_ffn_workspace_bytes": (C.c_size_t, [_vp, C.c_int]),
    "ds_moe_ffn_forward": (C.c_int, [_vp, _vp, _vp, C.c_int, _vp, _vp, C.c_size_t, _vp]),
    "ds_selftest_wait_timeout": (C.c_int, [_vp, C.c_uint32, _vp]),
    "ds_tp_shard_blocks": (C.c_int, [_vp, _vp, C.c_int]),
    "ds_tp_shard_weights": (C.c_int, [_vp, _vp, _vp, _vp]),
    "ds_tp_layer_create": (C.c_int, [_vp, _vp, C.POINTER(_vp)]),
    "ds_tp_layer_destroy": (C.c_int, [_vp]),
    "ds_tp_layer_workspace_bytes": (C.c_size_t, [_vp, C.c_int, C.c_int]),
    "ds_tp_attention_partial": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, _vp, _vp, C.c_int, _vp, _vp,
                                          C.c_size_t, _vp]),
    "ds_tp_ffn_partial": (C.c_int, [_vp, _vp, _vp, C.c_int, _vp, C.c_size_t, _vp]),
    "ds_tp_finish": (C.c_int, [_vp, _vp, _vp, C.c_int, _vp]),
    "ds_launch_count": (C.c_uint64, []),
    "ds_status_string": (C.c_char_p, [C.c_int]),
    "ds_last_error": (C.c_char_p, []),
}
EXPORTED = tuple(_SIGS)


class ds_layer_config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("heads", C.c_int), ("ffn", C.c_int), ("ln_eps", C.c_float),
                ("act_dtype", C.c_int), ("weight_dtype", C.c_int), ("quant_group", C.c_int),
                ("mlp_extra_grouping", C.c_int)]


_WNAMES = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_fc1", "b_fc1",
           "w_fc2", "b_fc2", "s_qkv", "s_o", "s_fc1", "s_fc2")


class ds_layer_weights(C.Structure):
    _fields_ = [(n, _vp) for n in _WNAMES]


class ds_moe_config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("ffn", C.c_int), ("experts", C.c_int), ("ln_eps", C.c_float),
                ("act_dtype", C.c_int)]


_MOE_WNAMES = ("ln2_g", "ln2_b", "w_gate", "w_fc1", "b_fc1", "w_fc2", "b_fc2", "we_fc1", "be_fc1", "we_fc2",
               "be_fc2")


class ds_moe_weights(C.Structure):
    _fields_ = [(n, _vp) for n in _MOE_WNAMES]


class ds_tp_config(C.Structure):
    _fields_ = [("layer", ds_layer_config), ("tp_size", C.c_int), ("tp_rank", C.c_int)]


DS_TP_W_QKV, DS_TP_B_QKV, DS_TP_W_O, DS_TP_W_FC1, DS_TP_B_FC1, DS_TP_W_FC2 = range(6)
TP_MATRIX_NAMES = ("w_qkv", "b_qkv", "w_o", "w_fc1", "b_fc1", "w_fc2")


class ds_tp_block(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("matrix", "src_row", "src_col", "rows", "cols", "src_cols", "dst_row")]


class DSError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        lib = _lib
        name = lib.ds_status_string(code).decode() if lib else str(code)
        detail = lib.ds_last_error().decode() if lib else ""
        super().__init__(f"{where}: {name}: {detail}")


_lib = None


def load(path: str = LIB_PATH):
    """Loads the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} not found: build it with transformer_layer_gb300.build.build()")
    lib = C.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(code, where):
    if code != DS_OK:
        raise DSError(code, where)


def _ptr(t):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr() if hasattr(t, "data_ptr") else int(t))


def _stream(s):
    if s is None:
        import torch
        s = torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream if hasattr(s, "cuda_stream") else int(s))


def _dtype_code(dt):
    import torch
    return {torch.float16: DS_F16, torch.bfloat16: DS_BF16, torch.int8: DS_I8}[dt]


# ---------------------------------------------------------------- thin wrappers
def ds_layer_create(hidden, heads, ffn, weights: dict, act_dtype, weight_dtype, ln_eps=1e-5,
                    quant_group=64, mlp_extra_grouping=0):
    """weights: dict of device tensors keyed like ds_layer_weights' fields."""
    lib = load()
    cfg = ds_layer_config(hidden, heads, ffn, ln_eps, _dtype_code(act_dtype),
                          _dtype_code(weight_dtype), quant_group, int(mlp_extra_grouping))
    w = ds_layer_weights(*[_ptr(weights.get(n)) for n in _WNAMES])
    out = C.c_void_p()
    _check(lib.ds_layer_create(C.byref(cfg), C.byref(w), C.byref(out)), "ds_layer_create")
    return out


def ds_layer_destroy(layer):
    _check(load().ds_layer_destroy(layer), "ds_layer_destroy")


def ds_layer_workspace_bytes(layer, batch, new_tokens):
    return int(load().ds_layer_workspace_bytes(layer, batch, new_tokens))


def ds_workspace_init(ws, nbytes, stream=None):
    _check(load().ds_workspace_init(_ptr(ws), nbytes, _stream(stream)), "ds_workspace_init")


def ds_layer_forward(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len, ws,
                     ws_bytes, stream=None):
    _check(load().ds_layer_forward(layer, _ptr(x_in), _ptr(x_out), batch, new_tokens, _ptr(k_cache),
                                   _ptr(v_cache), max_len, _ptr(past_len), _ptr(ws), ws_bytes,
                                   _stream(stream)), "ds_layer_forward")


def ds_layer_forward_noalloc(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len,
                             stream=None):
    """The layer forward on the library's static workspace (no allocation)."""
    _check(load().ds_layer_forward_noalloc(layer, _ptr(x_in), _ptr(x_out), batch, new_tokens, _ptr(k_cache),
                                           _ptr(v_cache), max_len, _ptr(past_len), _stream(stream)),
           "ds_layer_forward_noalloc")


def ds_noalloc_status(stream=None):
    """Returns (status_code, flags) of the last no-allocation forward on the
    current device and clears its status word."""
    flags = C.c_uint32(0)
    code = load().ds_noalloc_status(C.byref(flags), _stream(stream))
    if code not in (DS_OK, DS_ERR_DEVICE):
        raise DSError(code, "ds_noalloc_status")
    return code, int(flags.value)


def ds_stack_create(layers):
    arr = (C.c_void_p * len(layers))(*[l.value if isinstance(l, C.c_void_p) else l for l in layers])
    out = C.c_void_p()
    _check(load().ds_stack_create(arr, len(layers), C.byref(out)), "ds_stack_create")
    return out


def ds_stack_destroy(stack):
    _check(load().ds_stack_destroy(stack), "ds_stack_destroy")


def ds_stack_workspace_bytes(stack, batch):
    return int(load().ds_stack_workspace_bytes(stack, batch))


def _ptr_array(ts):
    return (C.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def ds_stack_decode_step(stack, x_in, x_out, batch, k_caches, v_caches, max_len, seq_len, ws, ws_bytes,
                         stream=None):
    _check(load().ds_stack_decode_step(stack, _ptr(x_in), _ptr(x_out), batch, _ptr_array(k_caches),
                                       _ptr_array(v_caches), max_len, _ptr(seq_len), _ptr(ws), ws_bytes,
                                       _stream(stream)), "ds_stack_decode_step")


def ds_stack_forward(stack, x_in, x_out, batch, new_tokens, k_caches, v_caches, max_len, past_len, ws, ws_bytes,
                     stream=None):
    _check(load().ds_stack_forward(stack, _ptr(x_in), _ptr(x_out), batch, new_tokens, _ptr_array(k_caches),
                                   _ptr_array(v_caches), max_len, _ptr(past_len), _ptr(ws), ws_bytes,
                                   _stream(stream)), "ds_stack_forward")


def ds_stack_decode_host(stack, x_host, y_host, x_dev_in, x_dev_out, batch, k_caches, v_caches, max_len,
                         seq_len, ws, ws_bytes, stream=None):
    _check(load().ds_stack_decode_host(stack, _ptr(x_host), _ptr(y_host), _ptr(x_dev_in), _ptr(x_dev_out),
                                       batch, _ptr_array(k_caches), _ptr_array(v_caches), max_len,
                                       _ptr(seq_len), _ptr(ws), ws_bytes, _stream(stream)),
           "ds_stack_decode_host")


def ds_stack_set_profiling(stack, enabled):
    _check(load().ds_stack_set_profiling(stack, 1 if enabled else 0), "ds_stack_set_profiling")


def ds_stack_region_times(stack):
    """Returns (us[5], launches[5]) averaged since the last call."""
    us = (C.c_float * 5)()
    n = (C.c_int * 5)()
    _check(load().ds_stack_region_times(stack, us, n), "ds_stack_region_times")
    return list(us), list(n)


def ds_stack_graph_captures(stack):
    return int(load().ds_stack_graph_captures(stack))


def ds_quantize_int8(w_f16, codes, scales, group=64, stream=None):
    n, k = w_f16.shape
    _check(load().ds_quantize_int8(_ptr(w_f16), n, k, group, _ptr(codes), _ptr(scales), _stream(stream)),
           "ds_quantize_int8")


def ds_workspace_status(ws, stream=None):
    """Returns (status_code, flags) and clears the device status word."""
    flags = C.c_uint32(0)
    code = load().ds_workspace_status(_ptr(ws), C.byref(flags), _stream(stream))
    if code not in (DS_OK, DS_ERR_DEVICE):
        raise DSError(code, "ds_workspace_status")
    return code, int(flags.value)


def ds_selftest_wait_timeout(ws, budget_us, stream=None):
    _check(load().ds_selftest_wait_timeout(_ptr(ws), budget_us, _stream(stream)), "ds_selftest_wait_timeout")


def ds_moe_ffn_create(hidden, ffn, experts, weights: dict, act_dtype, ln_eps=1e-5):
    """weights: dict of device tensors keyed like ds_moe_weights' fields."""
    cfg = ds_moe_config(hidden, ffn, experts, ln_eps, _dtype_code(act_dtype))
    w = ds_moe_weights(*[_ptr(weights.get(n)) for n in _MOE_WNAMES])
    out = C.c_void_p()
    _check(load().ds_moe_ffn_create(C.byref(cfg), C.byref(w), C.byref(out)), "ds_moe_ffn_create")
    return out


def ds_moe_ffn_destroy(moe):
    _check(load().ds_moe_ffn_destroy(moe), "ds_moe_ffn_destroy")


def ds_moe_ffn_workspace_bytes(moe, rows):
    return int(load().ds_moe_ffn_workspace_bytes(moe, rows))


def ds_moe_ffn_forward(moe, x_in, x_out, rows, expert_out, ws, ws_bytes, stream=None):
    _check(load().ds_moe_ffn_forward(moe, _ptr(x_in), _ptr(x_out), rows, _ptr(expert_out), _ptr(ws), ws_bytes,
                                     _stream(stream)), "ds_moe_ffn_forward")


def _tp_config(hidden, heads, ffn, act_dtype, tp_size, tp_rank, ln_eps=1e-5):
    code = _dtype_code(act_dtype)
    return ds_tp_config(ds_layer_config(hidden, heads, ffn, ln_eps, code, code, 64, 0), tp_size, tp_rank)


def ds_tp_shard_blocks(hidden, heads, ffn, act_dtype, tp_size, tp_rank, ln_eps=1e-5):
    """The rank's blocks of the full matrices, as dicts of ds_tp_block's fields
    (host-only call: no device is needed)."""
    cfg = _tp_config(hidden, heads, ffn, act_dtype, tp_size, tp_rank, ln_eps)
    out = (ds_tp_block * 16)()
    n = load().ds_tp_shard_blocks(C.byref(cfg), out, 16)
    if n < 0:
        raise DSError(DS_ERR_INVALID_ARG, "ds_tp_shard_blocks")
    return [{f: getattr(out[i], f) for f, _ in ds_tp_block._fields_} for i in range(n)]


def ds_tp_shard_weights(hidden, heads, ffn, act_dtype, tp_size, tp_rank, full: dict, shard: dict, stream=None):
    """Copies the rank's slices of `full` into the buffers of `shard` (dicts
    keyed like ds_layer_weights' fields)."""
    cfg = _tp_config(hidden, heads, ffn, act_dtype, tp_size, tp_rank)
    wf = ds_layer_weights(*[_ptr(full.get(n)) for n in _WNAMES])
    ws = ds_layer_weights(*[_ptr(shard.get(n)) for n in _WNAMES])
    _check(load().ds_tp_shard_weights(C.byref(cfg), C.byref(wf), C.byref(ws), _stream(stream)),
           "ds_tp_shard_weights")


def ds_tp_layer_create(hidden, heads, ffn, weights: dict, act_dtype, tp_size, tp_rank, ln_eps=1e-5):
    """weights: the rank's device tensors keyed like ds_layer_weights' fields."""
    cfg = _tp_config(hidden, heads, ffn, act_dtype, tp_size, tp_rank, ln_eps)
    w = ds_layer_weights(*[_ptr(weights.get(n)) for n in _WNAMES])
    out = C.c_void_p()
    _check(load().ds_tp_layer_create(C.byref(cfg), C.byref(w), C.byref(out)), "ds_tp_layer_create")
    return out


def ds_tp_layer_destroy(layer):
    _check(load().ds_tp_layer_destroy(layer), "ds_tp_layer_destroy")


def ds_tp_layer_workspace_bytes(layer, batch, new_tokens):
    return int(load().ds_tp_layer_workspace_bytes(layer, batch, new_tokens))


def ds_tp_attention_partial(layer, x_in, x1_part, batch, new_tokens, k_cache, v_cache, max_len, past_len, ws,
                            ws_bytes, stream=None):
    _check(load().ds_tp_attention_partial(layer, _ptr(x_in), _ptr(x1_part), batch, new_tokens, _ptr(k_cache),
                                          _ptr(v_cache), max_len, _ptr(past_len), _ptr(ws), ws_bytes,
                                          _stream(stream)), "ds_tp_attention_partial")


def ds_tp_ffn_partial(layer, x1, y_part, rows, ws, ws_bytes, stream=None):
    _check(load().ds_tp_ffn_partial(layer, _ptr(x1), _ptr(y_part), rows, _ptr(ws), ws_bytes, _stream(stream)),
           "ds_tp_ffn_partial")


def ds_tp_finish(layer, y, x_out, rows, stream=None):
    _check(load().ds_tp_finish(layer, _ptr(y), _ptr(x_out), rows, _stream(stream)), "ds_tp_finish")


def tp_layer_forward(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len, ws, ws_bytes,
                     x1, y, group=None, stream=None):
    """One tensor-sliced layer step of this rank: the three library calls with
    a sum all-reduce of the fp32 buffers x1 and y [rows][H] (caller-owned
    device tensors) between them, over torch.distributed's `group` (NCCL on
    GPUs).  The collective runs on torch's current stream, so `stream` must be
    that stream (or None)."""
    import torch
    import torch.distributed as dist
    if stream is not None and stream != torch.cuda.current_stream():
        raise ValueError("tp_layer_forward runs on torch's current stream")
    rows = batch * new_tokens
    ds_tp_attention_partial(layer, x_in, x1, batch, new_tokens, k_cache, v_cache, max_len, past_len, ws, ws_bytes)
    dist.all_reduce(x1, op=dist.ReduceOp.SUM, group=group)
    ds_tp_ffn_partial(layer, x1, y, rows, ws, ws_bytes)
    dist.all_reduce(y, op=dist.ReduceOp.SUM, group=group)
    ds_tp_finish(layer, y, x_out, rows)


def ds_launch_count():
    return int(load().ds_launch_count())


def ds_status_string(code):
    return load().ds_status_string(code).decode()


def ds_last_error():
    return load().ds_last_error().decode()
