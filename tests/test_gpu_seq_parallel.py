"""Sequence-parallel forms (all-gather before the column-sharded GEMM,
reduce-scatter after the row-sharded GEMM; "7.9 Tensor and pipeline
parallelism (TP, PP)", §2.5).  Each virtual rank's token slice lives in its
own buffer.  The results must be bit-identical to the ordinary path on the
concatenated tensors, and match the oracle."""
import numpy as np
import pytest
import torch

from synth import Workload, make_inputs, small_case
from tests.parity import (BF16_REL, allowance_rows, check, oracle_problem, rounding_weights)

pytestmark = pytest.mark.gpu

CASES = [small_case(336, 264, 600, 3, "swiglu", seed=701),
         small_case(512, 192, 768, 4, "gelu_tanh", bias=True, seed=702),
         small_case(512, 256, 2048, 4, "gelu_tanh", bias=True, seed=704),  # fused: last wave in 4 K parts
         Workload("attn_out_sp_300x256_h6x64_tp3", 300, 256, 384, 3, "none", "bf16", seed_index=703,
                  n_heads=6, n_kv_heads=6, head_dim=64)]


@pytest.mark.parametrize("fused", [False, True], ids=["reduce_scatter", "fused_then_scatter"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_sequence_parallel_matches_tensor_parallel_bitwise_and_oracle(w, fused):
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    inp = make_inputs(w)
    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    if w.act == "none":
        ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, "none", "bf16", device=dev, n_heads=w.n_heads,
                                n_kv_heads=w.n_kv_heads, head_dim=w.head_dim)
    else:
        ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    st = torch.cuda.current_stream(dev)
    flags = abi.TP_SUM_FUSED if fused else 0
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    # the ordinary path
    y_ref, saved, _ = ffn.forward(g["x"], w13p, w2p, b1=g["b1"], b2=g["b2"], fused=fused)
    gr = ffn.backward(g["x"], w13p, w2p, saved, g["dy"], fused=fused, bias=w.bias)
    # per-rank slices in separate buffers
    T, ns = w.T_p, w.N // w.T_p
    xs = [g["x"][t * ns:(t + 1) * ns].clone() for t in range(T)]
    dys = [g["dy"][t * ns:(t + 1) * ns].clone() for t in range(T)]
    ys = [torch.full((ns, w.d), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(T)]
    dxs = [torch.full((ns, w.d_in), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(T)]
    ws = torch.empty(abi.tp_ffn_seq_parallel_workspace_bytes(ffn.plan, w.N, flags), dtype=torch.uint8, device=dev)
    saved_sp = None if saved is None else torch.empty_like(saved)
    rc = abi.tp_ffn_fwd_seq_parallel(ffn.plan, w.N, xs, w13p, w2p, g["b1"], g["b2"], ys, saved_sp, ws, ws.numel(),
                                     flags, st)
    assert rc == abi.TP_OK, abi.tp_ffn_status_string(rc)
    dw13p = None if w13p is None else torch.empty_like(w13p)
    dw2p = torch.empty_like(w2p)
    db1 = torch.empty_like(gr["db1"]) if gr["db1"] is not None else None
    db2 = torch.empty_like(gr["db2"]) if gr["db2"] is not None else None
    rc = abi.tp_ffn_bwd_seq_parallel(ffn.plan, w.N, xs, w13p, w2p, saved_sp, dys, dxs, dw13p, dw2p, db1, db2, ws,
                                     ws.numel(), flags, st)
    assert rc == abi.TP_OK, abi.tp_ffn_status_string(rc)
    torch.cuda.synchronize(dev)
    y_sp, dx_sp = torch.cat(ys), torch.cat(dxs)
    as_bytes = lambda t: t.contiguous().view(torch.uint8)
    assert torch.equal(as_bytes(y_sp), as_bytes(y_ref))
    assert torch.equal(as_bytes(dx_sp), as_bytes(gr["dx"]))
    assert torch.equal(as_bytes(dw2p), as_bytes(gr["dw2p"]))
    if dw13p is not None:
        assert torch.equal(as_bytes(dw13p), as_bytes(gr["dw13p"]))
    for a, b in ((db1, gr["db1"]), (db2, gr["db2"])):
        if a is not None:
            assert torch.equal(as_bytes(a), as_bytes(b))
    rb, f = oracle_problem(w, inp, round_bf16=True)
    wts = rounding_weights(w, rb.hidden_dump(f["dy"])) if w.act != "none" else None
    A = allowance_rows(w, f, wts) if wts is not None else {}
    check(y_sp.double().cpu().numpy(), rb.forward_sharded()["y"], BF16_REL, f"{w.name} SP y", A.get("y"))
    check(dx_sp.double().cpu().numpy(), rb.backward_rows(f["dy"])["dx"], BF16_REL, f"{w.name} SP dx", A.get("dx"))


def test_sequence_parallel_rejects_ragged_token_counts():
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    rc, plan = abi.tp_ffn_plan_create(64, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_BF16)
    try:
        A = 1 << 20
        ws = abi.tp_ffn_seq_parallel_workspace_bytes(plan, 9, 0)
        assert abi.tp_ffn_fwd_seq_parallel(plan, 9, [A, A], A, A, None, None, [A, A], None, A, ws, 0) == \
            abi.TP_ERR_INVALID  # 9 tokens over 2 ranks
    finally:
        abi.tp_ffn_plan_destroy(plan)
