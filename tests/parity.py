"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare.

Tolerances (written here once, used by every parity test):
  * bf16 outputs (y, dx, weight and bias gradients) against the oracle in the
    workloads' stated precision ("bf16 weights/activations, fp32 accumulate":
    the oracle rounds the stored activations h, z / a, g and dz / da, dg to
    bf16 and computes everything else in float64):
        max |gpu - ref| <= 1e-2 * (|ref| + 1)
    y and dx are also held to the same bound against the pure float64 chain.
    Weight gradients are not: they sum the rounding noise of the stored bf16
    activations over all tokens (sigma ~ sqrt(N) * |dy| * |h| * 2^-9 / sqrt(3)),
    which exceeds 1e-2 * (|ref| + 1) for small entries at any N in the hundreds
  * fp32 outputs and fp32 shard partials:
        max |gpu - ref| <= 1e-4 * (|ref| + 1)  (+ the rounding allowance below)
  * rounding allowance for partials of bf16 workloads: the partials are sums
    over the bf16-stored hidden activations.  The oracle reproduces that
    storage (round_bf16=True), but a rounding decision whose pre-rounding
    value lies within float noise of a bf16 midpoint may legitimately go
    either way on the GPU (fp32 accumulation) and in the oracle (float64).
    For exactly those terms the allowance adds one bf16 ulp (two for a
    derivative whose own input was such a case) times the weight it
    multiplies; every other term is held to the plain 1e-4 bound.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from synth import to_f64

BF16_REL = 1e-2
F32_REL = 1e-4
NOISE_REL = 2.0 ** -17     # relative float noise treated as "at the midpoint"


def bf16_ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def near_midpoint(pre, scale):
    """True where `pre` lies within float noise of a bf16 rounding midpoint."""
    u = bf16_ulp(pre)
    q = pre / u
    dist = np.abs((q - np.floor(q)) - 0.5) * u
    return dist <= NOISE_REL * (np.abs(pre) + scale)


def check(got, ref, rel, what, extra=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    tol = rel * (np.abs(ref) + 1.0)
    if extra is not None:
        tol = tol + extra
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - tol, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements beyond tolerance; "
                             f"worst at {i}: gpu={got[i]!r} ref={ref[i]!r} tol={tol[i]:.3e}")


# ------------------------------------------------------------------ GPU side
def run_gpu_tensors(w, inp, fused=False, want_partials=True, backward=True):
    """Runs pack + forward (+ backward) of workload `w` on cuda:0 through the
    C ABI; returns the device tensors (gradients unpacked to [out, in]) and
    the number of kernels the forward call launched."""
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi

    dev = torch.device("cuda", 0)
    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    if w.act == "none":
        ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, "none", w.dtype, device=dev, n_heads=w.n_heads,
                                n_kv_heads=w.n_kv_heads, head_dim=w.head_dim)
    else:
        ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, w.dtype, device=dev)
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    partials = want_partials and not fused
    y, saved, part = ffn.forward(g["x"], w13p, w2p, b1=g["b1"], b2=g["b2"], save=backward, fused=fused,
                                 want_partials=partials)
    n_fwd = abi.tp_ffn_last_launch_count(ffn.plan)
    out = dict(y=y, partials=part)
    if backward and g["dy"] is not None:
        gr = ffn.backward(g["x"], w13p, w2p, saved, g["dy"], fused=fused,
                          want_partials=partials and w.act != "none", bias=w.bias)
        out.update(dx=gr["dx"], dx_partials=gr["dx_partials"], db1=gr["db1"], db2=gr["db2"])
        if w.act != "none":
            out["dW1"], out["dW3"] = ffn.unpack_columns(gr["dw13p"])
        out["dW2"] = ffn.unpack_rows(gr["dw2p"])
    torch.cuda.synchronize()
    return out, n_fwd


def run_gpu(w, inp, fused=False, want_partials=True, backward=True):
    """run_gpu_tensors, converted to float64 numpy (small workloads)."""
    out, n_fwd = run_gpu_tensors(w, inp, fused, want_partials, backward)
    assert n_fwd >= 1, "the forward pass launched no kernel of libtpffn.so"
    res = {k: (None if v is None else v.to(torch.float64).cpu().numpy()) for k, v in out.items()}
    res["_raw"] = {k: (None if v is None else v.cpu()) for k, v in out.items()}
    return res


# --------------------------------------------------------------- oracle side
def oracle_problem(w, inp, round_bf16=False):
    f = {k: to_f64(v) for k, v in inp.items()}
    return oracle.FFN(f["x"], f["W2"], w.T_p, w.act, W1=f["W1"], W3=f["W3"], b1=f["b1"], b2=f["b2"],
                      round_bf16=round_bf16), f


def partial_allowance(w, f, dump, rows, which):
    """Per-element allowance for the fp32 partials of bf16 workloads.

    which == "y" : y^(t)[n, c]  = sum_{j in t} h[n, j]  W2[c, j]
    which == "dx": dx^(t)[n, k] = sum_{j in t} dz[n, j] W1[j, k] (+ dg W3)
    Returns [T_p, n_rows, d].
    """
    T, s = w.T_p, w.s
    if w.dtype != "bf16" or w.act == "none":
        return 0.0
    if which == "y":
        pre = dump["h_pre"]
        amb = near_midpoint(pre, np.sqrt(np.mean(pre ** 2)))
        weight = np.where(amb, bf16_ulp(pre), 0.0)
        out = np.zeros((T, len(rows), w.d))
        for t in range(T):
            sl = slice(t * s, (t + 1) * s)
            out[t] = weight[:, sl] @ np.abs(f["W2"][:, sl]).T
        return out
    # backward: dz (or da) and dg; an ambiguous saved input (z, a or g) may
    # move the derivative by about one ulp of its own, so allow two there
    zp, dzp = dump["z_pre"], dump["dz_pre"]
    amb_in = near_midpoint(zp, np.sqrt(np.mean(zp ** 2)))
    if w.act == "swiglu":
        gp = dump["g_pre"]
        amb_in |= near_midpoint(gp, np.sqrt(np.mean(gp ** 2)))
    amb_dz = near_midpoint(dzp, np.sqrt(np.mean(dzp ** 2)))
    wz = np.where(amb_in, 2.0, np.where(amb_dz, 1.0, 0.0)) * bf16_ulp(dzp)
    out = np.zeros((T, len(rows), w.d))
    for t in range(T):
        sl = slice(t * s, (t + 1) * s)
        out[t] = wz[:, sl] @ np.abs(f["W1"][sl])
    if w.act == "swiglu":
        dgp = dump["dg_pre"]
        amb_dg = near_midpoint(dgp, np.sqrt(np.mean(dgp ** 2)))
        wg = np.where(amb_in, 2.0, np.where(amb_dg, 1.0, 0.0)) * bf16_ulp(dgp)
        for t in range(T):
            sl = slice(t * s, (t + 1) * s)
            out[t] += wg[:, sl] @ np.abs(f["W3"][sl])
    return out
