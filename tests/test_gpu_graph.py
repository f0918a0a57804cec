"""The forward and backward calls replayed from a CUDA graph.

Small token batches are launch-bound: a caller captures tp_ffn_fwd and
tp_ffn_bwd once (after one ordinary call on the device) and replays the
graph.  Every call enqueues only stream work -- a memset of the workspace
header and kernel launches, with programmatic dependent launches between
them -- so the replay must give exactly the eager call's bits, also when
replayed twice in a row, for the training shapes (both sum modes) and for a
decode-sized SwiGLU forward whose up GEMM is split in two K parts, and for
a backward whose weight-gradient GEMMs run in K parts with their ordered
part sums and the merged bias column sums.
"""
import pytest
import torch

from synth import make_inputs, small_case

pytestmark = pytest.mark.gpu

CASES = [small_case(333, 264, 600, 3, "swiglu", seed=801),
         small_case(300, 256, 768, 4, "gelu_tanh", bias=True, seed=802),
         small_case(17, 2048, 3072, 3, "swiglu", seed=803, fwd_only=True),
         small_case(2100, 256, 1024, 4, "gelu_tanh", bias=True, seed=804)]  # weight gradients in K parts


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.uint8)


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_graph_replay_is_bit_identical_to_eager(w, fused):
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    flags = abi.TP_SUM_FUSED if fused else 0
    n = w.N
    ws = ffn.workspace(n, flags)
    saved = None if w.fwd_only else torch.empty(abi.tp_ffn_saved_bytes(ffn.plan, n), dtype=torch.uint8,
                                                device=dev)
    y = torch.empty(n, w.d, dtype=torch.bfloat16, device=dev)
    dx = torch.empty_like(y)
    dw13p, dw2p = torch.empty_like(w13p), torch.empty_like(w2p)
    db1 = torch.empty(w.d_ff, dtype=torch.bfloat16, device=dev) if w.bias else None
    db2 = torch.empty(w.d, dtype=torch.bfloat16, device=dev) if w.bias else None
    outs = [y] if w.fwd_only else [y, dx, dw13p, dw2p] + ([db1, db2] if w.bias else [])

    def step():
        st = torch.cuda.current_stream(dev)
        abi.check(abi.tp_ffn_fwd(ffn.plan, n, g["x"], w13p, w2p, g["b1"], g["b2"], y, None, saved, ws, ws.numel(),
                                 flags, st), "fwd")
        if not w.fwd_only:
            abi.check(abi.tp_ffn_bwd(ffn.plan, n, g["x"], w13p, w2p, saved, g["dy"], dx, None, dw13p, dw2p, db1,
                                     db2, ws, ws.numel(), flags, st), "bwd")

    step()  # the eager call (it also sets the kernels' launch attributes on this device)
    torch.cuda.synchronize(dev)
    eager = [o.clone() for o in outs]
    for o in outs:
        o.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for replay in range(2):
        for o in outs:
            o.fill_(7)
        graph.replay()
        torch.cuda.synchronize(dev)
        for i, (a, b) in enumerate(zip(eager, outs)):
            assert torch.equal(_bits(a), _bits(b)), f"replay {replay + 1}: output {i} differs from the eager call"
    assert abi.tp_ffn_last_device_error(ffn.plan, ws, torch.cuda.current_stream(dev)) == abi.TP_OK
