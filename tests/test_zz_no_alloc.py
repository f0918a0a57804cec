"""The forward pass that allocates no device memory.

tp_ffn_fwd_static_scratch is for callers that may not call cudaMalloc while
they run the layer: a serving engine that reserves all its device memory at
start-up, or a plugin inside a framework that owns the allocator.  It keeps
its scratch in one static device array shared by every call.

This test makes the set-up call (n_tokens = 0) first, as such a caller would
at start-up, then runs the entry point twice in a row on different inputs
(the array keeps the first call's contents) for three shapes: a SwiGLU and a
biased GELU forward, and a 17-token SwiGLU forward whose up GEMM is split in
two K parts (the parts live in the static array too).  Each result must equal
the ordinary tp_ffn_fwd with the standalone shard-sum bit for bit: both run
the same kernels on the same inputs.  The device's free memory must not
change across a static-scratch call.  The file sorts last so that a run that
stops at the first failure has already run every other test.
"""
import pytest
import torch

from synth import make_inputs, small_case

pytestmark = pytest.mark.gpu

CASES = [small_case(48, 1024, 4096, 8, "swiglu", seed=901),
         small_case(48, 1024, 4096, 8, "gelu_tanh", bias=True, seed=903),
         small_case(17, 2048, 3072, 3, "swiglu", seed=905)]   # decode-sized: K split in two parts


def _kernel_names(abi, plan):
    return [name for name, _ in abi.tp_ffn_kernel_times(plan, 1000)]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_static_scratch_forward_equals_tp_ffn_fwd(w):
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    st = torch.cuda.current_stream(dev)
    # start-up: the static array becomes resident on this device
    assert abi.tp_ffn_fwd_static_scratch(ffn.plan, 0, None, None, None, None, None, None, st) == abi.TP_OK
    for call, seed in enumerate((w.seed_index, w.seed_index + 1)):  # two calls in a row
        inp = make_inputs(w, seed=seed)
        g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
        y_ref, _, _ = ffn.forward(g["x"], w13p, w2p, b1=g["b1"], b2=g["b2"], save=False,
                                  flags=abi.TP_FLAG_TIMING)
        names = _kernel_names(abi, ffn.plan)
        if w.N <= 32:
            assert "swiglu_combine" in names, names  # the K split is taken on this GPU
        y = torch.full_like(y_ref, float("nan"))
        torch.cuda.synchronize(dev)
        free0, _ = torch.cuda.mem_get_info(dev)
        rc = abi.tp_ffn_fwd_static_scratch(ffn.plan, w.N, g["x"], w13p, w2p, g["b1"], g["b2"], y, st)
        torch.cuda.synchronize(dev)
        free1, _ = torch.cuda.mem_get_info(dev)
        assert rc == abi.TP_OK, abi.tp_ffn_status_string(rc)
        assert free1 == free0, f"call {call + 1}: device free memory changed by {free0 - free1} bytes"
        # the timed kernels plus the untimed one that clears the device error word
        assert abi.tp_ffn_last_launch_count(ffn.plan) == len(names) + 1
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), f"call {call + 1}: not bit-identical"
    # sizes beyond the static array are refused before any work is enqueued
    n_big = 1
    while abi.tp_ffn_workspace_bytes(ffn.plan, n_big, abi.TP_SUM_STANDALONE) <= abi.TPFFN_STATIC_SCRATCH_BYTES:
        n_big *= 2
    x_big = torch.empty(n_big, w.d, dtype=torch.bfloat16, device=dev)
    y_big = torch.empty_like(x_big)
    rc = abi.tp_ffn_fwd_static_scratch(ffn.plan, n_big, x_big, w13p, w2p, None, None, y_big, st)
    assert rc == abi.TP_ERR_UNSUPPORTED
