"""A thin convenience layer over the C ABI: PyTorch allocates the device
buffers and supplies the stream; every computation is a libtpffn.so call.

    ffn = TensorParallelFFN(d=4096, d_ff=14336, T_p=8, act="swiglu", dtype="bf16")
    w13p, w2p = ffn.pack(W1, W2, W3)
    y, saved = ffn.forward(x, w13p, w2p)
    grads = ffn.backward(x, w13p, w2p, saved, dy)
"""
from __future__ import annotations

import torch

from . import tpffn as abi

_ACTS = {"none": abi.TP_ACT_NONE, "gelu_tanh": abi.TP_ACT_GELU_TANH, "swiglu": abi.TP_ACT_SWIGLU}
_DTYPES = {"f32": (abi.TP_F32, torch.float32), "bf16": (abi.TP_BF16, torch.bfloat16)}


class TensorParallelFFN:
    """All T_p shards of one tensor-parallel FFN (or W_O projection) on one GPU."""

    def __init__(self, d, d_ff, T_p, act="gelu_tanh", dtype="bf16", device="cuda", n_heads=None,
                 n_kv_heads=None, head_dim=None):
        self.act_name = act
        self.dtype_code, self.torch_dtype = _DTYPES[dtype]
        self.device = torch.device(device)
        if act == "none" and n_heads is not None:
            rc, h = abi.tp_attn_out_plan_create(d, n_heads, n_kv_heads or n_heads, head_dim, T_p, self.dtype_code)
        else:
            rc, h = abi.tp_ffn_plan_create(d, d_ff, T_p, _ACTS[act], self.dtype_code)
        abi.check(rc, "plan_create")
        self.plan = h
        self.info = abi.tp_ffn_plan_info(h)
        self.d, self.d_ff, self.T_p = self.info["d"], self.info["d_ff"], self.info["T_p"]
        self._ws = None

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan:
            abi.tp_ffn_plan_destroy(plan)
            self.plan = None

    # ------------------------------------------------------------ buffers
    def _bytes(self, nbytes):
        return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=self.device)

    def workspace(self, n_tokens, flags=0):
        need = abi.tp_ffn_workspace_bytes(self.plan, n_tokens, flags)
        if self._ws is None or self._ws.numel() < need:
            self._ws = self._bytes(need)
        return self._ws

    def _stream(self):
        return torch.cuda.current_stream(self.device)

    # ------------------------------------------------------------ packing
    def pack(self, W1, W2, W3=None):
        st = self._stream()
        w13p = None
        if self.act_name != "none":
            w13p = self._bytes(abi.tp_ffn_packed_bytes(self.plan, abi.TP_PACK_COLUMNS))
            abi.check(abi.tp_ffn_shard_columns(self.plan, W1, W3, w13p, st), "shard_columns")
        w2p = self._bytes(abi.tp_ffn_packed_bytes(self.plan, abi.TP_PACK_ROWS))
        abi.check(abi.tp_ffn_shard_rows(self.plan, W2, w2p, st), "shard_rows")
        return w13p, w2p

    def unpack_columns(self, w13p):
        st = self._stream()
        W1 = torch.empty(self.d_ff, self.d, dtype=self.torch_dtype, device=self.device)
        W3 = torch.empty_like(W1) if self.act_name == "swiglu" else None
        abi.check(abi.tp_ffn_unshard_columns(self.plan, w13p, W1, W3, st), "unshard_columns")
        return W1, W3

    def unpack_rows(self, w2p):
        st = self._stream()
        W2 = torch.empty(self.d, self.d_ff, dtype=self.torch_dtype, device=self.device)
        abi.check(abi.tp_ffn_unshard_rows(self.plan, w2p, W2, st), "unshard_rows")
        return W2

    # ------------------------------------------------------------ passes
    def forward(self, x, w13p, w2p, b1=None, b2=None, save=True, fused=False, want_partials=False, flags=0,
                overlap=False):
        n = x.shape[0]
        flags |= abi.TP_SUM_FUSED if fused else 0
        flags |= abi.TP_SUM_OVERLAP if overlap else 0
        st = self._stream()
        y = torch.empty(n, self.d, dtype=self.torch_dtype, device=self.device)
        saved = self._bytes(abi.tp_ffn_saved_bytes(self.plan, n)) if save and self.act_name != "none" else None
        part = torch.empty(self.T_p, n, self.d, dtype=torch.float32, device=self.device) if want_partials else None
        ws = self.workspace(n, flags)
        abi.check(abi.tp_ffn_fwd(self.plan, n, x, w13p, w2p, b1, b2, y, part, saved, ws, ws.numel(), flags, st),
                  "fwd")
        return y, saved, part

    def backward(self, x, w13p, w2p, saved, dy, fused=False, want_partials=False, bias=False, flags=0,
                 overlap=False):
        n = dy.shape[0]
        flags |= abi.TP_SUM_FUSED if fused else 0
        flags |= abi.TP_SUM_OVERLAP if overlap else 0
        st = self._stream()
        d_in = self.d_ff if self.act_name == "none" else self.d
        dx = torch.empty(n, d_in, dtype=self.torch_dtype, device=self.device)
        part = torch.empty(self.T_p, n, self.d, dtype=torch.float32, device=self.device) if want_partials else None
        dw13p = None
        if self.act_name != "none":
            dw13p = self._bytes(abi.tp_ffn_packed_bytes(self.plan, abi.TP_PACK_COLUMNS))
        dw2p = self._bytes(abi.tp_ffn_packed_bytes(self.plan, abi.TP_PACK_ROWS))
        db1 = torch.empty(self.d_ff, dtype=self.torch_dtype, device=self.device) if bias and self.act_name == "gelu_tanh" else None
        db2 = torch.empty(self.d, dtype=self.torch_dtype, device=self.device) if bias else None
        ws = self.workspace(n, flags)
        abi.check(abi.tp_ffn_bwd(self.plan, n, x, w13p, w2p, saved, dy, dx, part, dw13p, dw2p, db1, db2, ws,
                                 ws.numel(), flags, st), "bwd")
        return dict(dx=dx, dx_partials=part, dw13p=dw13p, dw2p=dw2p, db1=db1, db2=db2)
