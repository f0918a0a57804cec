"""ctypes binding of libtpffn.so (include/tpffn.h), same names as the C ABI.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Pointers may be given as integers, as objects with ``data_ptr()``
(PyTorch tensors) or as None; streams as integers, as objects with a
``cuda_stream`` attribute, or None (the legacy stream).  Importing this module
fails loudly if the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtpffn.so")

TP_OK, TP_ERR_INVALID, TP_ERR_UNSUPPORTED, TP_ERR_CUDA, TP_ERR_TIMEOUT, TP_ERR_ALIGN = range(6)
TP_ACT_NONE, TP_ACT_GELU_TANH, TP_ACT_SWIGLU = 0, 1, 2
TP_F32, TP_BF16 = 0, 1
TP_PACK_COLUMNS, TP_PACK_ROWS = 0, 1
TP_SUM_STANDALONE, TP_SUM_FUSED, TP_FLAG_SYNC, TP_FLAG_TIMING, TP_SUM_OVERLAP = 0, 1, 2, 4, 8
TP_FLAG_DEBUG_SKIP_LOAD = 1 << 16

ABI_FUNCTIONS = (
    "tp_ffn_plan_create", "tp_attn_out_plan_create", "tp_ffn_plan_destroy", "tp_ffn_plan_info",
    "tp_ffn_packed_bytes", "tp_ffn_saved_bytes", "tp_ffn_workspace_bytes", "tp_ffn_shard_columns",
    "tp_ffn_shard_rows", "tp_ffn_unshard_columns", "tp_ffn_unshard_rows", "tp_ffn_fwd", "tp_ffn_bwd",
    "tp_ffn_last_device_error", "tp_ffn_status_string", "tp_ffn_kernel_times", "tp_ffn_last_launch_count",
    "tp_ffn_fwd_static_scratch", "tp_ffn_seq_parallel_workspace_bytes", "tp_ffn_fwd_seq_parallel",
    "tp_ffn_bwd_seq_parallel",
    "tp_attn_plan_create", "tp_attn_plan_destroy", "tp_attn_plan_info", "tp_attn_packed_bytes",
    "tp_attn_shard_weights", "tp_attn_unshard_weights", "tp_attn_saved_bytes", "tp_attn_saved_offsets",
    "tp_attn_workspace_bytes", "tp_attn_fwd", "tp_attn_bwd", "tp_attn_core_fwd", "tp_attn_core_bwd",
    "tp_attn_kernel_times", "tp_attn_last_launch_count",
)
TPFFN_STATIC_SCRATCH_BYTES = 32 << 20


class TPFFNError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {tp_ffn_status_string(status)} ({status})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run megatron_tensor_transformer_w1_gb300.build.build() "
                      "(there is no CPU or library fallback)")

_lib = ctypes.CDLL(LIB_PATH)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGS = {
    "tp_ffn_plan_create": (_INT, [ctypes.POINTER(_P), _I64, _I64, _INT, _INT, _INT]),
    "tp_attn_out_plan_create": (_INT, [ctypes.POINTER(_P), _I64, _INT, _INT, _I64, _INT, _INT]),
    "tp_ffn_plan_destroy": (None, [_P]),
    "tp_ffn_plan_info": (_INT, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_INT),
                                ctypes.POINTER(_INT), ctypes.POINTER(_INT), ctypes.POINTER(_I64),
                                ctypes.POINTER(_I64)]),
    "tp_ffn_packed_bytes": (_SZ, [_P, _INT]),
    "tp_ffn_saved_bytes": (_SZ, [_P, _I64]),
    "tp_ffn_workspace_bytes": (_SZ, [_P, _I64, _INT]),
    "tp_ffn_shard_columns": (_INT, [_P, _P, _P, _P, _P]),
    "tp_ffn_shard_rows": (_INT, [_P, _P, _P, _P]),
    "tp_ffn_unshard_columns": (_INT, [_P, _P, _P, _P, _P]),
    "tp_ffn_unshard_rows": (_INT, [_P, _P, _P, _P]),
    "tp_ffn_fwd": (_INT, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_ffn_bwd": (_INT, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_ffn_last_device_error": (_INT, [_P, _P, _P]),
    "tp_ffn_status_string": (ctypes.c_char_p, [_INT]),
    "tp_ffn_kernel_times": (_INT, [_P, _INT, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]),
    "tp_ffn_last_launch_count": (_INT, [_P]),
    "tp_ffn_fwd_static_scratch": (_INT, [_P, _I64, _P, _P, _P, _P, _P, _P, _P]),
    "tp_ffn_seq_parallel_workspace_bytes": (_SZ, [_P, _I64, _INT]),
    "tp_ffn_fwd_seq_parallel": (_INT, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_ffn_bwd_seq_parallel": (_INT, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_attn_plan_create": (_INT, [ctypes.POINTER(_P), _I64, _INT, _INT, _I64, _INT, _INT, _INT]),
    "tp_attn_plan_destroy": (None, [_P]),
    "tp_attn_plan_info": (_INT, [_P] + [ctypes.POINTER(_I64)] * 4),
    "tp_attn_packed_bytes": (_SZ, [_P, _INT]),
    "tp_attn_shard_weights": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "tp_attn_unshard_weights": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "tp_attn_saved_bytes": (_SZ, [_P, _I64, _I64]),
    "tp_attn_saved_offsets": (_INT, [_P, _I64, _I64] + [ctypes.POINTER(_SZ)] * 3),
    "tp_attn_workspace_bytes": (_SZ, [_P, _I64, _I64, _INT]),
    "tp_attn_fwd": (_INT, [_P, _I64, _I64, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_attn_bwd": (_INT, [_P, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_attn_core_fwd": (_INT, [_P, _I64, _I64, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_attn_core_bwd": (_INT, [_P, _I64, _I64, _P, _P, _P, _P, _P, _P, _SZ, _INT, _P]),
    "tp_attn_kernel_times": (_INT, [_P, _INT, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]),
    "tp_attn_last_launch_count": (_INT, [_P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------- raw ABI calls
def tp_ffn_status_string(status):
    return _lib.tp_ffn_status_string(int(status)).decode()


def tp_ffn_plan_create(d, d_ff, T_p, act, dtype):
    """Returns (status, plan handle or None)."""
    h = _P()
    rc = _lib.tp_ffn_plan_create(ctypes.byref(h), d, d_ff, T_p, act, dtype)
    return rc, (h.value if rc == TP_OK else None)


def tp_attn_out_plan_create(d_model, n_heads, n_kv_heads, head_dim, T_p, dtype):
    h = _P()
    rc = _lib.tp_attn_out_plan_create(ctypes.byref(h), d_model, n_heads, n_kv_heads, head_dim, T_p, dtype)
    return rc, (h.value if rc == TP_OK else None)


def tp_ffn_plan_destroy(plan):
    _lib.tp_ffn_plan_destroy(plan)


def tp_ffn_plan_info(plan):
    d, d_ff, s, s_pad = _I64(), _I64(), _I64(), _I64()
    T_p, act, dtype = _INT(), _INT(), _INT()
    rc = _lib.tp_ffn_plan_info(plan, ctypes.byref(d), ctypes.byref(d_ff), ctypes.byref(T_p), ctypes.byref(act),
                               ctypes.byref(dtype), ctypes.byref(s), ctypes.byref(s_pad))
    if rc != TP_OK:
        raise TPFFNError(rc, "tp_ffn_plan_info")
    return dict(d=d.value, d_ff=d_ff.value, T_p=T_p.value, act=act.value, dtype=dtype.value, s=s.value,
                s_pad=s_pad.value)


def tp_ffn_packed_bytes(plan, which):
    return _lib.tp_ffn_packed_bytes(plan, which)


def tp_ffn_saved_bytes(plan, n_tokens):
    return _lib.tp_ffn_saved_bytes(plan, n_tokens)


def tp_ffn_workspace_bytes(plan, n_tokens, flags=0):
    return _lib.tp_ffn_workspace_bytes(plan, n_tokens, flags)


def tp_ffn_shard_columns(plan, W1, W3, packed, stream=None):
    return _lib.tp_ffn_shard_columns(plan, _ptr(W1), _ptr(W3), _ptr(packed), _stream(stream))


def tp_ffn_shard_rows(plan, W2, packed, stream=None):
    return _lib.tp_ffn_shard_rows(plan, _ptr(W2), _ptr(packed), _stream(stream))


def tp_ffn_unshard_columns(plan, packed, W1, W3, stream=None):
    return _lib.tp_ffn_unshard_columns(plan, _ptr(packed), _ptr(W1), _ptr(W3), _stream(stream))


def tp_ffn_unshard_rows(plan, packed, W2, stream=None):
    return _lib.tp_ffn_unshard_rows(plan, _ptr(packed), _ptr(W2), _stream(stream))


def tp_ffn_fwd(plan, n_tokens, x, w13p, w2p, b1, b2, y, partials, saved, workspace, workspace_bytes, flags=0,
               stream=None):
    return _lib.tp_ffn_fwd(plan, n_tokens, _ptr(x), _ptr(w13p), _ptr(w2p), _ptr(b1), _ptr(b2), _ptr(y),
                           _ptr(partials), _ptr(saved), _ptr(workspace), workspace_bytes, flags, _stream(stream))


def tp_ffn_bwd(plan, n_tokens, x, w13p, w2p, saved, dy, dx, dx_partials, dw13p, dw2p, db1, db2, workspace,
               workspace_bytes, flags=0, stream=None):
    return _lib.tp_ffn_bwd(plan, n_tokens, _ptr(x), _ptr(w13p), _ptr(w2p), _ptr(saved), _ptr(dy), _ptr(dx),
                           _ptr(dx_partials), _ptr(dw13p), _ptr(dw2p), _ptr(db1), _ptr(db2), _ptr(workspace),
                           workspace_bytes, flags, _stream(stream))


def tp_ffn_last_device_error(plan, workspace, stream=None):
    return _lib.tp_ffn_last_device_error(plan, _ptr(workspace), _stream(stream))


def tp_ffn_kernel_times(plan, max_records=64):
    names = (ctypes.c_char_p * max_records)()
    ms = (ctypes.c_float * max_records)()
    n = _lib.tp_ffn_kernel_times(plan, max_records, names, ms)
    return [(names[i].decode(), ms[i]) for i in range(min(n, max_records))]


def tp_ffn_last_launch_count(plan):
    return _lib.tp_ffn_last_launch_count(plan)


def tp_ffn_fwd_static_scratch(plan, n_tokens, x, w13p, w2p, b1, b2, y, stream=None):
    """Forward pass that allocates no device memory (scratch in the library's
    static array of TPFFN_STATIC_SCRATCH_BYTES); for callers that may not
    allocate.  See include/tpffn.h for its limit and sharing rules."""
    return _lib.tp_ffn_fwd_static_scratch(plan, n_tokens, _ptr(x), _ptr(w13p), _ptr(w2p), _ptr(b1), _ptr(b2),
                                          _ptr(y), _stream(stream))


def _ptr_array(items):
    """A host array of device pointers (None -> NULL) for the slice arguments."""
    if items is None:
        return None
    arr = (ctypes.c_void_p * len(items))(*[_ptr(a) for a in items])
    return ctypes.cast(arr, ctypes.c_void_p), arr  # keep `arr` alive with the call


def tp_ffn_seq_parallel_workspace_bytes(plan, n_tokens, flags=0):
    return _lib.tp_ffn_seq_parallel_workspace_bytes(plan, n_tokens, flags)


def tp_ffn_fwd_seq_parallel(plan, n_tokens, x_slices, w13p, w2p, b1, b2, y_slices, saved, workspace,
                            workspace_bytes, flags=0, stream=None):
    xs, ys = _ptr_array(x_slices), _ptr_array(y_slices)
    return _lib.tp_ffn_fwd_seq_parallel(plan, n_tokens, xs and xs[0], _ptr(w13p), _ptr(w2p), _ptr(b1), _ptr(b2),
                                        ys and ys[0], _ptr(saved), _ptr(workspace), workspace_bytes, flags,
                                        _stream(stream))


def tp_ffn_bwd_seq_parallel(plan, n_tokens, x_slices, w13p, w2p, saved, dy_slices, dx_slices, dw13p, dw2p, db1, db2,
                            workspace, workspace_bytes, flags=0, stream=None):
    xs, dys, dxs = _ptr_array(x_slices), _ptr_array(dy_slices), _ptr_array(dx_slices)
    return _lib.tp_ffn_bwd_seq_parallel(plan, n_tokens, xs and xs[0], _ptr(w13p), _ptr(w2p), _ptr(saved),
                                        dys and dys[0], dxs and dxs[0], _ptr(dw13p), _ptr(dw2p), _ptr(db1), _ptr(db2),
                                        _ptr(workspace), workspace_bytes, flags, _stream(stream))


# ------------------------------------------------------------ attention sublayer
def tp_attn_plan_create(d_model, n_heads, n_kv_heads, head_dim, T_p, causal, dtype):
    """Returns (status, plan handle or None)."""
    h = _P()
    rc = _lib.tp_attn_plan_create(ctypes.byref(h), d_model, n_heads, n_kv_heads, head_dim, T_p, int(causal), dtype)
    return rc, (h.value if rc == TP_OK else None)


def tp_attn_plan_destroy(plan):
    _lib.tp_attn_plan_destroy(plan)


def tp_attn_plan_info(plan):
    vals = [_I64() for _ in range(4)]
    rc = _lib.tp_attn_plan_info(plan, *[ctypes.byref(v) for v in vals])
    if rc != TP_OK:
        raise TPFFNError(rc, "tp_attn_plan_info")
    return dict(zip(("qkv_width", "slice", "sq", "sk"), (v.value for v in vals)))


def tp_attn_packed_bytes(plan, which):
    return _lib.tp_attn_packed_bytes(plan, which)


def tp_attn_shard_weights(plan, Wq, Wk, Wv, Wo, wqkv, wo_packed, stream=None):
    return _lib.tp_attn_shard_weights(plan, _ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(Wo), _ptr(wqkv), _ptr(wo_packed),
                                      _stream(stream))


def tp_attn_unshard_weights(plan, wqkv, wo_packed, Wq, Wk, Wv, Wo, stream=None):
    return _lib.tp_attn_unshard_weights(plan, _ptr(wqkv), _ptr(wo_packed), _ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(Wo),
                                        _stream(stream))


def tp_attn_saved_bytes(plan, B, S):
    return _lib.tp_attn_saved_bytes(plan, B, S)


def tp_attn_saved_offsets(plan, B, S):
    vals = [_SZ() for _ in range(3)]
    rc = _lib.tp_attn_saved_offsets(plan, B, S, *[ctypes.byref(v) for v in vals])
    if rc != TP_OK:
        raise TPFFNError(rc, "tp_attn_saved_offsets")
    return dict(zip(("qkv", "c", "lse"), (v.value for v in vals)))


def tp_attn_workspace_bytes(plan, B, S, flags=0):
    return _lib.tp_attn_workspace_bytes(plan, B, S, flags)


def tp_attn_fwd(plan, B, S, x, wqkv, wo_packed, y, saved, workspace, workspace_bytes, flags=0, stream=None):
    return _lib.tp_attn_fwd(plan, B, S, _ptr(x), _ptr(wqkv), _ptr(wo_packed), _ptr(y), _ptr(saved), _ptr(workspace),
                            workspace_bytes, flags, _stream(stream))


def tp_attn_bwd(plan, B, S, x, wqkv, wo_packed, saved, dy, dx, dwqkv, dwo_packed, workspace, workspace_bytes,
                flags=0, stream=None):
    return _lib.tp_attn_bwd(plan, B, S, _ptr(x), _ptr(wqkv), _ptr(wo_packed), _ptr(saved), _ptr(dy), _ptr(dx),
                            _ptr(dwqkv), _ptr(dwo_packed), _ptr(workspace), workspace_bytes, flags, _stream(stream))


def tp_attn_core_fwd(plan, B, S, qkv, o, lse, workspace, workspace_bytes, flags=0, stream=None):
    return _lib.tp_attn_core_fwd(plan, B, S, _ptr(qkv), _ptr(o), _ptr(lse), _ptr(workspace), workspace_bytes, flags,
                                 _stream(stream))


def tp_attn_core_bwd(plan, B, S, qkv, o, lse, dO, dqkv, workspace, workspace_bytes, flags=0, stream=None):
    return _lib.tp_attn_core_bwd(plan, B, S, _ptr(qkv), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dqkv), _ptr(workspace),
                                 workspace_bytes, flags, _stream(stream))


def tp_attn_kernel_times(plan, max_records=64):
    names = (ctypes.c_char_p * max_records)()
    ms = (ctypes.c_float * max_records)()
    n = _lib.tp_attn_kernel_times(plan, max_records, names, ms)
    return [(names[i].decode(), ms[i]) for i in range(min(n, max_records))]


def tp_attn_last_launch_count(plan):
    return _lib.tp_attn_last_launch_count(plan)


def check(status, where=""):
    if status != TP_OK:
        raise TPFFNError(status, where)
