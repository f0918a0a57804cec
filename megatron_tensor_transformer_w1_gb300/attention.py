"""Head-sharded attention sublayer over the C ABI (tp_attn_* of include/tpffn.h).

PyTorch allocates the device buffers and supplies the stream; every step runs
in libtpffn.so ("7.9 Tensor and pipeline parallelism (TP, PP)", §2.2
"Attention, sharded").

    attn = TensorParallelAttention(d=3072, n_heads=24, n_kv_heads=24, head_dim=128, T_p=8)
    wqkv, wo = attn.pack(Wq, Wk, Wv, Wo)
    y, saved = attn.forward(x, B, S, wqkv, wo)
    g = attn.backward(x, B, S, wqkv, wo, saved, dy)   # dx, dwqkv, dwo
"""
from __future__ import annotations

import torch

from . import tpffn as abi


class TensorParallelAttention:
    """All T_p shards of one attention sublayer on one GPU (bf16, head_dim 128)."""

    def __init__(self, d, n_heads, n_kv_heads, head_dim, T_p, causal=True, device="cuda"):
        rc, h = abi.tp_attn_plan_create(d, n_heads, n_kv_heads, head_dim, T_p, causal, abi.TP_BF16)
        abi.check(rc, "tp_attn_plan_create")
        self.plan = h
        self.d, self.H, self.Hkv, self.hd, self.T_p = d, n_heads, n_kv_heads, head_dim, T_p
        self.causal = bool(causal)
        self.device = torch.device(device)
        self.info = abi.tp_attn_plan_info(h)
        self._ws = None

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan:
            abi.tp_attn_plan_destroy(plan)
            self.plan = None

    def _bytes(self, nbytes):
        return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=self.device)

    def _stream(self):
        return torch.cuda.current_stream(self.device)

    def workspace(self, B, S, flags=0):
        need = abi.tp_attn_workspace_bytes(self.plan, B, S, flags)
        if self._ws is None or self._ws.numel() < need:
            self._ws = self._bytes(need)
        return self._ws

    # ------------------------------------------------------------ weights
    def pack(self, Wq, Wk, Wv, Wo):
        wqkv = self._bytes(abi.tp_attn_packed_bytes(self.plan, abi.TP_PACK_COLUMNS))
        wo = self._bytes(abi.tp_attn_packed_bytes(self.plan, abi.TP_PACK_ROWS))
        abi.check(abi.tp_attn_shard_weights(self.plan, Wq, Wk, Wv, Wo, wqkv, wo, self._stream()), "shard_weights")
        return wqkv, wo

    def unpack(self, wqkv, wo):
        bf = dict(dtype=torch.bfloat16, device=self.device)
        Wq = torch.empty(self.H * self.hd, self.d, **bf)
        Wk = torch.empty(self.Hkv * self.hd, self.d, **bf)
        Wv = torch.empty_like(Wk)
        Wo = torch.empty(self.d, self.H * self.hd, **bf)
        abi.check(abi.tp_attn_unshard_weights(self.plan, wqkv, wo, Wq, Wk, Wv, Wo, self._stream()),
                  "unshard_weights")
        return Wq, Wk, Wv, Wo

    # ------------------------------------------------------------ passes
    def saved_views(self, saved, B, S):
        """(qkv [B*S, qkv_width], c [B*S, H*hd], lse [B*H, S_pad]) views of `saved`."""
        off = abi.tp_attn_saved_offsets(self.plan, B, S)
        n, W, nq = B * S, self.info["qkv_width"], self.H * self.hd
        s_pad = (S + 127) // 128 * 128
        qkv = saved[off["qkv"]:off["qkv"] + n * W * 2].view(torch.bfloat16).view(n, W)
        c = saved[off["c"]:off["c"] + n * nq * 2].view(torch.bfloat16).view(n, nq)
        lse = saved[off["lse"]:off["lse"] + B * self.H * s_pad * 4].view(torch.float32).view(B * self.H, s_pad)
        return qkv, c, lse

    def forward(self, x, B, S, wqkv, wo, fused=False, overlap=False, flags=0):
        flags |= (abi.TP_SUM_FUSED if fused else 0) | (abi.TP_SUM_OVERLAP if overlap else 0)
        y = torch.empty(B * S, self.d, dtype=torch.bfloat16, device=self.device)
        saved = self._bytes(abi.tp_attn_saved_bytes(self.plan, B, S))
        ws = self.workspace(B, S, flags)
        abi.check(abi.tp_attn_fwd(self.plan, B, S, x, wqkv, wo, y, saved, ws, ws.numel(), flags, self._stream()),
                  "tp_attn_fwd")
        return y, saved

    def backward(self, x, B, S, wqkv, wo, saved, dy, fused=False, overlap=False, flags=0):
        flags |= (abi.TP_SUM_FUSED if fused else 0) | (abi.TP_SUM_OVERLAP if overlap else 0)
        dx = torch.empty(B * S, self.d, dtype=torch.bfloat16, device=self.device)
        dwqkv = self._bytes(abi.tp_attn_packed_bytes(self.plan, abi.TP_PACK_COLUMNS))
        dwo = self._bytes(abi.tp_attn_packed_bytes(self.plan, abi.TP_PACK_ROWS))
        ws = self.workspace(B, S, flags)
        abi.check(abi.tp_attn_bwd(self.plan, B, S, x, wqkv, wo, saved, dy, dx, dwqkv, dwo, ws, ws.numel(), flags,
                                  self._stream()), "tp_attn_bwd")
        return dict(dx=dx, dwqkv=dwqkv, dwo=dwo)

    def core_forward(self, qkv, B, S, flags=0):
        o = torch.empty(B * S, self.H * self.hd, dtype=torch.bfloat16, device=self.device)
        lse = torch.empty(B * self.H, (S + 127) // 128 * 128, dtype=torch.float32, device=self.device)
        ws = self.workspace(B, S, flags)
        abi.check(abi.tp_attn_core_fwd(self.plan, B, S, qkv, o, lse, ws, ws.numel(), flags, self._stream()),
                  "tp_attn_core_fwd")
        return o, lse

    def core_backward(self, qkv, o, lse, dO, B, S, flags=0):
        dqkv = torch.empty_like(qkv)
        ws = self.workspace(B, S, flags)
        abi.check(abi.tp_attn_core_bwd(self.plan, B, S, qkv, o, lse, dO, dqkv, ws, ws.numel(), flags,
                                       self._stream()), "tp_attn_core_bwd")
        return dqkv
