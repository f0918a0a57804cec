"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare.

Tolerances (written here once, used by every parity test):
  * bf16 outputs (y, dx, weight and bias gradients) against the oracle in the
    workloads' stated precision ("bf16 weights/activations, fp32 accumulate":
    the oracle rounds the stored activations h, z / a, g and dz / da, dg to
    bf16 and computes everything else in float64):
        max |gpu - ref| <= 1e-2 * (|ref| + 1)
    y and dx are also held to the same bound against the pure float64 chain,
    widened by six standard deviations of the noise that storing the hidden
    activations in bf16 adds to their sums (chain_noise): over a hidden width
    of thousands that noise alone can reach 1e-2 * (|ref| + 1) for an
    occasional element.  Weight gradients are not held against the chain at
    all: they sum the rounding noise of the stored bf16
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
# Accumulation error of the fp32 tensor-core GEMM, measured on GB300 against
# exact sums of bf16 products for K = 256 .. 16384: the largest error seen was
# about 5.6e-9 * K * ||p||_2 (p = the K products).  The model below, 2^-26 * K
# * ||p||_2, is 2.7 times that.  EVAL_ERR and EVAL_ERR_D cover the fp32
# evaluation of the activation functions in the kernels (GELU in logistic
# form with the SFU's ex2 / rcp, SwiGLU's logistic with expf and an IEEE
# division): relative errors of at most 2^-19 for the values h, silu(a) and
# 2^-15 for the derivative factors gelu', silu' -- the bounds that
# tests/test_gpu_activation_accuracy.py holds the kernels to (measured at
# most 9.3e-7 and 1.4e-5).
ACC_ERR = 2.0 ** -26
EVAL_ERR = 2.0 ** -19
EVAL_ERR_D = 2.0 ** -15
# bounds of activation derivatives used to propagate the errors
GELU_D1, GELU_D2, SILU_D1, SILU_D2 = 1.13, 1.0, 1.1, 0.5


def bf16_ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def near_midpoint(pre, err):
    """True where the value `pre` lies within `err` of a bf16 rounding midpoint,
    i.e. where a value that far off could round to the other neighbour."""
    u = bf16_ulp(pre)
    q = pre / u
    dist = np.abs((q - np.floor(q)) - 0.5) * u
    return dist <= err


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


def chain_noise(w, f, dump):
    """Bound on how far a correct bf16-storage result may lie from the pure
    float64 chain: the kernel and the rounded oracle both store h, z / a, g and
    dz / da, dg in bf16.  A stored value x carries a rounding error of at most
    u |x| (u = 2^-8, bf16's unit roundoff), taken as uniform (sigma u |x| /
    sqrt 3).  y sums d_ff values h_j W2[:, j], each rounded once; dx sums the
    dz_j W1[j] (and dg_j W3[j]), each carrying its own rounding and, through
    g and silu'(a) or gelu'(z), that of the forward values it is formed from:
    three roundings.  The bound is six standard deviations of the sum, per
    element.  Returns dict(y, dx) shaped like y and dx, or None where no
    activation is stored in bf16."""
    if w.dtype != "bf16" or w.act == "none":
        return None
    sigma_u = 2.0 ** -8 / np.sqrt(3.0)
    h, dz, dg = dump["h_pre"], dump["dz_pre"], dump["dg_pre"]
    var_y = (h * h) @ (f["W2"] * f["W2"]).T
    var_dx = (dz * dz) @ (f["W1"] * f["W1"])
    if w.act == "swiglu":
        var_dx = var_dx + (dg * dg) @ (f["W3"] * f["W3"])
    return dict(y=6.0 * sigma_u * np.sqrt(var_y), dx=6.0 * sigma_u * np.sqrt(3.0 * var_dx))


# ------------------------------------------------------------------ GPU side
def run_gpu_tensors(w, inp, fused=False, want_partials=True, backward=True, overlap=False):
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
                                 want_partials=partials, overlap=overlap)
    n_fwd = abi.tp_ffn_last_launch_count(ffn.plan)
    out = dict(y=y, partials=part)
    if backward and g["dy"] is not None:
        gr = ffn.backward(g["x"], w13p, w2p, saved, g["dy"], fused=fused,
                          want_partials=partials and w.act != "none", bias=w.bias,
                          overlap=overlap and w.act != "none")
        out.update(dx=gr["dx"], dx_partials=gr["dx_partials"], db1=gr["db1"], db2=gr["db2"])
        if w.act != "none":
            out["dW1"], out["dW3"] = ffn.unpack_columns(gr["dw13p"])
        out["dW2"] = ffn.unpack_rows(gr["dw2p"])
    torch.cuda.synchronize()
    return out, n_fwd


def run_gpu(w, inp, fused=False, want_partials=True, backward=True, overlap=False):
    """run_gpu_tensors, converted to float64 numpy (small workloads)."""
    out, n_fwd = run_gpu_tensors(w, inp, fused, want_partials, backward, overlap)
    # the error-word reset and at least one compute kernel of libtpffn.so
    assert n_fwd >= 2, "the forward pass launched no compute kernel of libtpffn.so"
    res = {k: (None if v is None else v.to(torch.float64).cpu().numpy()) for k, v in out.items()}
    res["_raw"] = {k: (None if v is None else v.cpu()) for k, v in out.items()}
    return res


# --------------------------------------------------------------- oracle side
def oracle_problem(w, inp, round_bf16=False):
    f = {k: to_f64(v) for k, v in inp.items()}
    return oracle.FFN(f["x"], f["W2"], w.T_p, w.act, W1=f["W1"], W3=f["W3"], b1=f["b1"], b2=f["b2"],
                      round_bf16=round_bf16), f


def rounding_weights(w, dump):
    """Per (token, hidden unit) allowance weights of the stored bf16
    activations: for each stored value whose rounding may legitimately differ
    between the GPU (fp32 accumulation) and the oracle (float64), the largest
    change that difference can make to it; zero elsewhere.
    Returns dict(H=..., DZ=..., DG=...) of arrays shaped like the dump."""
    if w.dtype != "bf16" or w.act == "none":
        return None
    K = w.d  # the up GEMM and dh both contract over d
    z, g, h = dump["z_pre"], dump["g_pre"], dump["h_pre"]
    dh, dz, dg = dump["dh"], dump["dz_pre"], dump["dg_pre"]
    tz, tg, tdh = ACC_ERR * K * dump["nz"], ACC_ERR * K * dump["ng"], ACC_ERR * K * dump["ndh"]
    if w.act == "gelu_tanh":
        dh_err = GELU_D1 * tz + EVAL_ERR * np.abs(h)
        amb_z = near_midpoint(z, tz)
        dz_err = tdh * np.abs(np.divide(dz, dh, out=np.zeros_like(dz), where=dh != 0)) + EVAL_ERR_D * np.abs(dz)
        amb_dz = near_midpoint(dz, dz_err)
        DZ = np.where(amb_z, np.abs(dh) * GELU_D2 * bf16_ulp(z), 0.0) + np.where(amb_z | amb_dz, bf16_ulp(dz), 0.0)
        DG = np.zeros_like(dz)
    else:
        silu_a = np.divide(h, g, out=np.abs(z), where=g != 0)
        dh_err = np.abs(g) * SILU_D1 * tz + np.abs(silu_a) * tg + EVAL_ERR * np.abs(h)
        amb_a, amb_g = near_midpoint(z, tz), near_midpoint(g, tg)
        da_err = tdh * np.abs(np.divide(dz, dh, out=np.zeros_like(dz), where=dh != 0)) + EVAL_ERR_D * np.abs(dz)
        dg_err = tdh * np.abs(np.divide(dg, dh, out=np.zeros_like(dg), where=dh != 0)) + EVAL_ERR * np.abs(dg)
        amb_da, amb_dg = near_midpoint(dz, da_err), near_midpoint(dg, dg_err)
        gs = np.abs(g) * (1 + 2.0 ** -8)
        DZ = (np.where(amb_a, np.abs(dh) * gs * SILU_D2 * bf16_ulp(z), 0.0)
              + np.where(amb_g, np.abs(dh) * SILU_D1 * bf16_ulp(g), 0.0)
              + np.where(amb_a | amb_g | amb_da, bf16_ulp(dz), 0.0))
        DG = (np.where(amb_a, np.abs(dh) * SILU_D1 * bf16_ulp(z), 0.0)
              + np.where(amb_a | amb_dg, bf16_ulp(dg), 0.0))
    H = np.where(near_midpoint(h, dh_err), bf16_ulp(h), 0.0)
    return dict(H=H, DZ=DZ, DG=DG)


def allowance_rows(w, f, wts):
    """Allowances of the row outputs for the dumped token rows:
    partials y^(t), y, dx partials, dx; each [T_p, n, d] or [n, d]."""
    T, s = w.T_p, w.s
    out = {}
    py = np.stack([wts["H"][:, t * s:(t + 1) * s] @ np.abs(f["W2"][:, t * s:(t + 1) * s]).T for t in range(T)])
    out["partials"], out["y"] = py, py.sum(0)
    if "DZ" in wts and f.get("dy") is not None:
        pdx = np.stack([wts["DZ"][:, t * s:(t + 1) * s] @ np.abs(f["W1"][t * s:(t + 1) * s])
                        + (wts["DG"][:, t * s:(t + 1) * s] @ np.abs(f["W3"][t * s:(t + 1) * s])
                           if w.act == "swiglu" else 0.0) for t in range(T)])
        out["dx_partials"], out["dx"] = pdx, pdx.sum(0)
    return out


def allowance_wgrad(w, f, wts_cols, ks, cs):
    """Allowances of weight/bias-gradient entries at hidden units `js` (the
    columns of wts_cols, dumped over ALL tokens), inputs ks, outputs cs."""
    out = {"dW2": np.abs(f["dy"][:, cs]).T @ wts_cols["H"]}
    if ks is not None:
        ax = np.abs(f["x"][:, ks])
        out["dW1"] = wts_cols["DZ"].T @ ax
        out["dW3"] = wts_cols["DG"].T @ ax
    out["db1"] = wts_cols["DZ"].sum(0)
    return out
