"""Full-size parity of the attention core on sampled rows.

The two attention workloads timed by bench.py -- the Megatron 8.3B block
(8 sequences of 1024 tokens, 24 heads of 128) and the Llama-3-8B attention
(one sequence of 8192 tokens, 32 query and 8 key/value heads) -- run through
tp_attn_core_fwd / tp_attn_core_bwd, the kernels and launch configuration of
the sublayer ("7.9 Tensor and pipeline parallelism (TP, PP)", §2.2), on
seeded synthetic q, k, v, dO of the workloads' shapes.  The oracle computes
sampled rows one by one (orc_attn_core_sample): output rows, log-sum-exp and
dq rows of sampled queries, dk and dv rows of sampled keys -- first and last
rows, tile edges and interior rows.  Tolerance as in test_gpu_attention: bf16
values within 1e-2 (|ref| + 1) plus 3x the rounding allowance, lse within
1e-4 (|ref| + 1).  For the 8192-token sequence the sampled keys lie in its
last quarter: a key's gradient needs the softmax statistics of every later
query, and the earlier keys' cost grows with S^2.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import ATTN_WORKLOADS, make_core_inputs, to_f64
from tests.parity import check
from tests.test_gpu_attention import ALLOW_FACTOR, BF16_REL, F32_REL, HD, U, pack_qkv, unpack_qkv

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLES = {
    "megatron_8p3b_attention_bf16": dict(
        rows=[(0, 0, 0), (7, 23, 1023), (3, 11, 127), (3, 11, 128), (5, 7, 511), (2, 17, 900), (6, 2, 64),
              (1, 20, 333)],
        kv_rows=[(0, 0, 0), (7, 23, 1023), (4, 5, 128), (1, 12, 640), (6, 19, 127)]),
    "llama3_8b_attention_bf16": dict(
        rows=[(0, 0, 0), (0, 31, 8191), (0, 5, 4095), (0, 17, 128), (0, 9, 6000), (0, 26, 127), (0, 3, 2048)],
        kv_rows=[(0, 0, 8191), (0, 7, 6144), (0, 3, 7000), (0, 5, 8064)]),
}


@pytest.mark.parametrize("name", sorted(SAMPLES))
def test_attention_core_fullsize_sampled(name):
    w = ATTN_WORKLOADS[name]
    B, S, H, Hkv, T = w.B, w.S, w.H, w.Hkv, w.T_p
    inp = make_core_inputs(B, S, H, Hkv, HD, seed=w.seed_index)
    from megatron_tensor_transformer_w1_gb300.attention import TensorParallelAttention
    attn = TensorParallelAttention(d=w.d, n_heads=H, n_kv_heads=Hkv, head_dim=HD, T_p=T, causal=w.causal)
    qkv = pack_qkv(inp["q"], inp["k"], inp["v"], H, Hkv, T).cuda()
    o, lse = attn.core_forward(qkv, B, S)
    dqkv = attn.core_backward(qkv, o, lse, inp["dO"].cuda(), B, S)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu().double().numpy()
    dq, dk, dv = unpack_qkv(dqkv.cpu(), H, Hkv, T)
    del qkv, dqkv

    core = oracle.AttentionCore(B, S, H, Hkv, HD, causal=w.causal)
    smp = core.sample(*(to_f64(inp[n]) for n in ("q", "k", "v", "dO")), U, SAMPLES[name]["rows"],
                      SAMPLES[name]["kv_rows"])
    rb = lambda x: np.vectorize(oracle.round_bf16)(x)  # the stored outputs are bf16
    for s, (b, h, i) in enumerate(SAMPLES[name]["rows"]):
        r, cols = b * S + i, slice(h * HD, (h + 1) * HD)
        check(to_f64(o[r, cols]), rb(smp["o"][s]), BF16_REL, f"o[{b},{h},{i}]", ALLOW_FACTOR * smp["a_o"][s])
        check(lse[b * H + h, i] * math.log(2.0), smp["lse"][s], F32_REL, f"lse[{b},{h},{i}]")
        check(to_f64(dq[r, cols]), rb(smp["dq"][s]), BF16_REL, f"dq[{b},{h},{i}]", ALLOW_FACTOR * smp["a_dq"][s])
    for s, (b, hk, j) in enumerate(SAMPLES[name]["kv_rows"]):
        r, cols = b * S + j, slice(hk * HD, (hk + 1) * HD)
        check(to_f64(dk[r, cols]), rb(smp["dk"][s]), BF16_REL, f"dk[{b},{hk},{j}]", ALLOW_FACTOR * smp["a_dk"][s])
        check(to_f64(dv[r, cols]), rb(smp["dv"][s]), BF16_REL, f"dv[{b},{hk},{j}]", ALLOW_FACTOR * smp["a_dv"][s])
