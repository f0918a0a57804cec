"""The forward pass that allocates no device memory.

tp_ffn_fwd_static_scratch is for callers that may not call cudaMalloc while
they run the layer: a serving engine that reserves all its device memory at
start-up, or a plugin inside a framework that owns the allocator.  It keeps
its scratch in one static device array shared by every call.  This test runs
it twice in a row on different inputs (the array keeps the first call's
contents) and compares each result with the ordinary tp_ffn_fwd, within the
bf16 tolerance the parity tests use.  The file sorts last so that a run that
stops at the first failure has already run every other test.
"""
import pytest
import torch

from synth import make_inputs, small_case
from tests.parity import BF16_REL, check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act,bias", [("swiglu", False), ("gelu_tanh", True)])
def test_static_scratch_forward_matches_tp_ffn_fwd(act, bias):
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN

    dev = torch.device("cuda", 0)
    w = small_case(48, 1024, 4096, 8, act, bias=bias, seed=901)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, act, "bf16", device=dev)
    st = torch.cuda.current_stream(dev)
    for call, seed in enumerate((901, 902)):  # two calls in a row
        inp = make_inputs(w, seed=seed)
        g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
        y_ref, _, _ = ffn.forward(g["x"], w13p, w2p, b1=g["b1"], b2=g["b2"], save=False)
        y = torch.full_like(y_ref, float("nan"))
        rc = abi.tp_ffn_fwd_static_scratch(ffn.plan, w.N, g["x"], w13p, w2p, g["b1"], g["b2"], y, st)
        assert rc == abi.TP_OK, abi.tp_ffn_status_string(rc)
        torch.cuda.synchronize(dev)
        check(y.double().cpu().numpy(), y_ref.double().cpu().numpy(), BF16_REL,
              f"static-scratch forward, call {call + 1}")
    # sizes beyond the static array are refused before any work is enqueued
    n_big = 1
    while abi.tp_ffn_workspace_bytes(ffn.plan, n_big, abi.TP_SUM_STANDALONE) <= abi.TPFFN_STATIC_SCRATCH_BYTES:
        n_big *= 2
    x_big = torch.empty(n_big, w.d, dtype=torch.bfloat16, device=dev)
    y_big = torch.empty_like(x_big)
    rc = abi.tp_ffn_fwd_static_scratch(ffn.plan, n_big, x_big, w13p, w2p, None, None, y_big, st)
    assert rc == abi.TP_ERR_UNSUPPORTED
