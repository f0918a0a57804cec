"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the method: it only draws normal variates
from numpy's PCG64 generator (one independent stream per tensor, spawned from
one SeedSequence per workload) and rounds them to the workload's storage type
with PyTorch's own conversion (round-to-nearest-even).  Both sides then read
the very same rounded values: the CUDA library as bf16/fp32 device tensors,
the oracle as their exact float64 widenings.

Workloads (tokens N, model width d, hidden width d_ff, shards T_p):

=============================  =====  ====  =====  ===  =========  =====
name                           N      d     d_ff   T_p  act        dtype
=============================  =====  ====  =====  ===  =========  =====
tiny_gelu_fp32                 8      64    256    2    gelu_tanh  f32
gpt2_small_gelu_bf16           4096   768   3072   4    gelu_tanh  bf16 (+ biases)
llama3_8b_swiglu_bf16          8192   4096  14336  8    swiglu     bf16
megatron_8p3b_gelu_bf16        8192   3072  12288  8    gelu_tanh  bf16
megatron_8p3b_attn_out_bf16    8192   3072  3072   8    none       bf16 (24 heads x 128)
llama3_70b_decode_swiglu_bf16  32     8192  28672  8    swiglu     bf16 (forward only)
=============================  =====  ====  =====  ===  =========  =====

Value distributions: activations x (or the concatenated head outputs c) and
the upstream gradient dy are N(0, 1); weights are N(0, 1/fan_in) (W1, W3:
fan_in d; W2: fan_in d_ff), except the GPT-2-small workload, whose weights
are N(0, 0.02^2) and biases N(0, 0.01^2).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

BASE_SEED = 20260000


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    d: int
    d_ff: int
    T_p: int
    act: str             # "gelu_tanh" | "swiglu" | "none"
    dtype: str           # "f32" | "bf16"
    bias: bool = False
    fwd_only: bool = False
    w_std: float | None = None   # fixed weight std (else 1/sqrt(fan_in))
    b_std: float = 0.0
    seed_index: int = 0
    n_heads: int = 0     # act "none": heads feeding the projection
    n_kv_heads: int = 0
    head_dim: int = 0
    x_std: float = 1.0   # std of x (activation-tail cases scale it up)

    @property
    def s(self):
        return self.d_ff // self.T_p

    @property
    def d_in(self):
        return self.d_ff if self.act == "none" else self.d

    def fwd_flops(self):
        mult = {"gelu_tanh": 4, "swiglu": 6, "none": 2}[self.act]
        return mult * self.N * self.d * self.d_ff

    def bwd_flops(self):
        return 2 * self.fwd_flops()

    def weight_bytes(self):
        esz = 4 if self.dtype == "f32" else 2
        n_mats = {"gelu_tanh": 2, "swiglu": 3, "none": 1}[self.act]
        return n_mats * self.d * self.d_ff * esz

    def replace(self, **kw):
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_gelu_fp32", 8, 64, 256, 2, "gelu_tanh", "f32", seed_index=1),
        Workload("gpt2_small_gelu_bf16", 4096, 768, 3072, 4, "gelu_tanh", "bf16", bias=True,
                 w_std=0.02, b_std=0.01, seed_index=2),
        Workload("llama3_8b_swiglu_bf16", 8192, 4096, 14336, 8, "swiglu", "bf16", seed_index=3),
        Workload("megatron_8p3b_gelu_bf16", 8192, 3072, 12288, 8, "gelu_tanh", "bf16", seed_index=4),
        Workload("megatron_8p3b_attn_out_bf16", 8192, 3072, 3072, 8, "none", "bf16",
                 seed_index=5, n_heads=24, n_kv_heads=24, head_dim=128),
        Workload("llama3_70b_decode_swiglu_bf16", 32, 8192, 28672, 8, "swiglu", "bf16",
                 fwd_only=True, seed_index=6),
    ]
}


def _torch_dtype(dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _draw(rng, shape, std, dtype):
    """N(0, std^2) values rounded to the storage dtype (torch RNE cast)."""
    if dtype == "f32":
        a = rng.standard_normal(shape, dtype=np.float64) * std
        return torch.from_numpy(a).to(torch.float32)
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


_ORDER = ("x", "W1", "W3", "W2", "b1", "b2", "dy")


def make_inputs(w: Workload, seed: int | None = None):
    """Host tensors of the workload's storage dtype.

    Keys: x [N, d_in], W1, W3 [d_ff, d] (W3 for SwiGLU only), W2 [d, d_ff],
    b1 [d_ff], b2 [d] (biased workloads only), dy [N, d] (not forward-only).
    Missing tensors are None.
    """
    seed = BASE_SEED + w.seed_index if seed is None else seed
    streams = np.random.SeedSequence(seed).spawn(len(_ORDER))
    rng = {k: np.random.Generator(np.random.PCG64(s)) for k, s in zip(_ORDER, streams)}
    dt = w.dtype
    out = dict.fromkeys(_ORDER)
    out["x"] = _draw(rng["x"], (w.N, w.d_in), w.x_std, dt)
    if w.act != "none":
        std1 = w.w_std if w.w_std is not None else 1.0 / np.sqrt(w.d)
        out["W1"] = _draw(rng["W1"], (w.d_ff, w.d), std1, dt)
        if w.act == "swiglu":
            out["W3"] = _draw(rng["W3"], (w.d_ff, w.d), std1, dt)
    std2 = w.w_std if w.w_std is not None else 1.0 / np.sqrt(w.d_ff)
    out["W2"] = _draw(rng["W2"], (w.d, w.d_ff), std2, dt)
    if w.bias:
        out["b1"] = _draw(rng["b1"], (w.d_ff,), w.b_std, dt)
        out["b2"] = _draw(rng["b2"], (w.d,), w.b_std, dt)
    if not w.fwd_only:
        out["dy"] = _draw(rng["dy"], (w.N, w.d), 1.0, dt)
    return out


def small_case(N, d, d_ff, T_p, act, dtype="bf16", bias=False, seed=7, fwd_only=False, x_std=1.0, b_std=None):
    """A small workload of the same value distributions (for full-oracle parity).
    x_std > 1 (or a large b_std) drives the pre-activations into the tails of
    the activation functions."""
    tag = "" if x_std == 1.0 and b_std is None else f"_xs{x_std:g}" + ("" if b_std is None else f"_bs{b_std:g}")
    return Workload(f"small_{act}_{dtype}_{N}x{d}x{d_ff}_tp{T_p}{tag}", N, d, d_ff, T_p, act, dtype,
                    bias=bias, fwd_only=fwd_only, w_std=(0.05 if bias else None),
                    b_std=(b_std if b_std is not None else 0.02) if bias else 0.0, seed_index=seed, x_std=x_std)


@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Head-sharded attention sublayer: B sequences of S tokens, model width d,
    H query heads and Hkv key/value heads of width hd, T_p shards."""
    name: str
    B: int
    S: int
    d: int
    H: int
    Hkv: int
    hd: int
    T_p: int
    causal: bool = True
    dtype: str = "bf16"
    seed_index: int = 0

    @property
    def N(self):
        return self.B * self.S

    def proj_flops(self):
        """Q/K/V and output projections, forward."""
        return 2 * self.N * self.d * (2 * self.H * self.hd + 2 * self.Hkv * self.hd)

    def core_flops(self):
        """q k^T and p v of every head, forward, counting only the visible
        (causal: lower-triangle incl. diagonal) score entries."""
        pairs = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return 4 * self.B * self.H * pairs * self.hd

    def fwd_flops(self):
        return self.proj_flops() + self.core_flops()

    def bwd_flops(self):
        """Projections: 2x forward; core: dV, dP, dS-K, dS-Q = 2.5x forward
        (recomputing the scores is not counted)."""
        return 2 * self.proj_flops() + 5 * self.core_flops() // 2

    def replace(self, **kw):
        return dataclasses.replace(self, **kw)


ATTN_WORKLOADS = {
    w.name: w for w in [
        AttnWorkload("megatron_8p3b_attention_bf16", 8, 1024, 3072, 24, 24, 128, 8, seed_index=7),
        AttnWorkload("llama3_8b_attention_bf16", 1, 8192, 4096, 32, 8, 128, 8, seed_index=8),
    ]
}

_ATTN_ORDER = ("x", "Wq", "Wk", "Wv", "Wo", "dy")


def make_attention_inputs(w: AttnWorkload, seed: int | None = None):
    """Host tensors of an attention workload: x [N, d] and dy [N, d] ~ N(0, 1);
    Wq [H*hd, d], Wk, Wv [Hkv*hd, d] ~ N(0, 1/d); Wo [d, H*hd] ~ N(0, 1/(H*hd))."""
    seed = BASE_SEED + w.seed_index if seed is None else seed
    streams = np.random.SeedSequence(seed).spawn(len(_ATTN_ORDER))
    rng = {k: np.random.Generator(np.random.PCG64(s)) for k, s in zip(_ATTN_ORDER, streams)}
    dt = w.dtype
    nq, nk = w.H * w.hd, w.Hkv * w.hd
    return dict(
        x=_draw(rng["x"], (w.N, w.d), 1.0, dt),
        Wq=_draw(rng["Wq"], (nq, w.d), 1.0 / np.sqrt(w.d), dt),
        Wk=_draw(rng["Wk"], (nk, w.d), 1.0 / np.sqrt(w.d), dt),
        Wv=_draw(rng["Wv"], (nk, w.d), 1.0 / np.sqrt(w.d), dt),
        Wo=_draw(rng["Wo"], (w.d, nq), 1.0 / np.sqrt(nq), dt),
        dy=_draw(rng["dy"], (w.N, w.d), 1.0, dt),
    )


def make_core_inputs(B, S, H, Hkv, hd, seed, q_scale=1.0):
    """bf16 host tensors q [B*S, H*hd] ~ N(0, q_scale^2), k, v [B*S, Hkv*hd] and
    dO [B*S, H*hd] ~ N(0, 1) for the attention core alone (q_scale > 1 sharpens
    the softmax)."""
    streams = np.random.SeedSequence(BASE_SEED + 1000 + seed).spawn(4)
    rng = [np.random.Generator(np.random.PCG64(s)) for s in streams]
    n = B * S
    return dict(q=_draw(rng[0], (n, H * hd), q_scale, "bf16"), k=_draw(rng[1], (n, Hkv * hd), 1.0, "bf16"),
                v=_draw(rng[2], (n, Hkv * hd), 1.0, "bf16"), dO=_draw(rng[3], (n, H * hd), 1.0, "bf16"))


def to_f64(t):
    """Exact float64 widening of a host tensor (None passes through)."""
    if t is None:
        return None
    return t.to(torch.float64).numpy()
