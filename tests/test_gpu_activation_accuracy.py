"""Accuracy of the activation functions the kernels evaluate, measured end to
end through the C ABI against the oracle's float64 functions.

With an fp32 plan, T_p = 1, d = d_ff = 64 and identity weights (W1 = W2 = I,
and W3 = I for SwiGLU) every GEMM sum holds a single nonzero term, so the
outputs are exactly what the epilogues compute from x:
    GELU:   y = gelu(x),             dx = dy gelu'(x)
    SwiGLU: y = silu(x) x,           dx = dy (x silu'(x) + silu(x))
(the SwiGLU dx is the fp32 sum of the two epilogue outputs da and dg).  x runs
over [-40, 40] in steps of 2^-6.  The bounds are the kernels' stated
evaluation errors (tp_act.cuh) with a factor-two margin: 2^-19 relative for
the activation values, relative to max(|value|, 1e-3), and 2^-15 for the
derivatives, relative to max(|value|, 1e-2) -- a derivative formed from two
cancelling terms near its zero crossing keeps an absolute error of a few
fp32 ulps of those terms.
The same functions serve the bf16 tensor-core epilogues, whose rounding
allowance in tests/parity.py assumes these bounds.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

VAL_BOUND, DER_BOUND = 2.0 ** -19, 2.0 ** -15


def _identity_case(act):
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    d = 64
    z = torch.arange(-40 * 64, 40 * 64 + 64, dtype=torch.float64) / 64.0  # 2^-6 steps, exact in fp32
    z = z[: (z.numel() // d) * d].reshape(-1, d)
    x = z.to(torch.float32).to(dev)
    eye = torch.eye(d, dtype=torch.float32, device=dev)
    ffn = TensorParallelFFN(d, d, 1, act, "f32", device=dev)
    w13p, w2p = ffn.pack(eye, eye, eye if act == "swiglu" else None)
    y, saved, _ = ffn.forward(x, w13p, w2p)
    dy = torch.ones_like(x)
    dx = ffn.backward(x, w13p, w2p, saved, dy)["dx"]
    torch.cuda.synchronize()
    return z.numpy().ravel(), y.double().cpu().numpy().ravel(), dx.double().cpu().numpy().ravel()


def _check(got, ref, bound, what, floor=1e-3):
    err = np.abs(got - ref)
    tol = bound * np.maximum(np.abs(ref), floor)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} beyond {bound:.2e}; worst relative "
                           f"{np.max(err / np.maximum(np.abs(ref), floor)):.3e}")


def test_gelu_and_derivative_accuracy():
    z, y, dx = _identity_case("gelu_tanh")
    _check(y, np.array([oracle.gelu_tanh(v) for v in z]), VAL_BOUND, "gelu")
    _check(dx, np.array([oracle.gelu_tanh_grad(v) for v in z]), DER_BOUND, "gelu'", floor=1e-2)


def test_swiglu_and_derivative_accuracy():
    z, y, dx = _identity_case("swiglu")
    silu = np.array([oracle.silu(v) for v in z])
    dsilu = np.array([oracle.silu_grad(v) for v in z])
    _check(y, silu * z, VAL_BOUND, "silu(x) x")
    # dx = da + dg: each term within its own bound, then one fp32 addition
    err = np.abs(dx - (z * dsilu + silu))
    tol = DER_BOUND * np.maximum(np.abs(z * dsilu), 1e-2) + VAL_BOUND * np.maximum(np.abs(silu), 1e-3) \
        + 2.0 ** -24 * np.abs(dx)
    assert np.all(err <= tol), f"swiglu dx: {int((err > tol).sum())} beyond the bound"
