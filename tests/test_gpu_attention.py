"""GPU parity of the head-sharded attention sublayer against the float64 oracle.

The attention core (tp_attn_core_fwd / tp_attn_core_bwd) and the whole
sublayer (tp_attn_fwd / tp_attn_bwd: column-sharded Q/K/V, per-head attention,
row-sharded W_O with the ordered shard-sum, and the backward with the ordered
dx sum) of "7.9 Tensor and pipeline parallelism (TP, PP)", §2.2 "Attention,
sharded" run through the C ABI on seeded synthetic inputs; the oracle takes the
same bf16 values widened to float64 and rounds to bf16 where the library
stores (q, k, v, head outputs, dO, dq, dk, dv).

Tolerance: every bf16 output within 1e-2 (|ref| + 1) plus 3x its rounding
allowance elementwise, and in relative RMS within 1e-2 (a systematic error --
a wrong scale, a dropped term -- shows up there even where the elementwise
bound is loose); the fp32 log-sum-exp within 1e-4 (|ref| + 1).  The RMS bound
is taken against max(RMS(ref), 1e-3).  The allowance (the oracle's
orc_attn_core_allowance, then propagated through the projections as a
root-sum-square) is how far a computation that rounds P, dS and every stored
tensor to bf16, and forms D_i = dO_i . o_i from the stored o, may stray from
the exact values by rounding alone: a weight gradient sums that noise over
every token, so 1e-2 (|ref| + 1) alone does not bound it.  Shapes span several 128-row tiles with
ragged tails, GQA groups, causal and full masks, a one-token sequence, and
sharp softmaxes that exercise the lazy rescale of the running maximum.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import AttnWorkload, make_attention_inputs, make_core_inputs, to_f64
from tests.parity import check

pytestmark = pytest.mark.gpu

HD = 128
BF16_REL = 1e-2
F32_REL = 1e-4
RMS_REL = 1e-2
U = 2.0 ** -8        # one bf16 unit, relative
ALLOW_FACTOR = 3.0


def _attn_mod():
    from megatron_tensor_transformer_w1_gb300.attention import TensorParallelAttention
    return TensorParallelAttention


def pack_qkv(q, k, v, H, Hkv, T):
    """Host copy of the library's packed q/k/v column order: shard slices of
    [query heads | key heads | value heads]."""
    hq, hk = H // T * HD, Hkv // T * HD
    parts = []
    for t in range(T):
        parts += [q[:, t * hq:(t + 1) * hq], k[:, t * hk:(t + 1) * hk], v[:, t * hk:(t + 1) * hk]]
    return torch.cat(parts, 1).contiguous()


def unpack_qkv(qkv, H, Hkv, T):
    hq, hk = H // T * HD, Hkv // T * HD
    sl = hq + 2 * hk
    q = torch.cat([qkv[:, t * sl:t * sl + hq] for t in range(T)], 1)
    k = torch.cat([qkv[:, t * sl + hq:t * sl + hq + hk] for t in range(T)], 1)
    v = torch.cat([qkv[:, t * sl + hq + hk:(t + 1) * sl] for t in range(T)], 1)
    return q, k, v


def rms_check(got, ref, what, rel=RMS_REL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.sqrt(np.mean((got - ref) ** 2))
    # floor: a reference that vanishes exactly (one visible key: softmax
    # gradients are 0) leaves only rounding noise, which the elementwise
    # bound already covers
    den = max(np.sqrt(np.mean(ref ** 2)), 1e-3)
    assert num <= rel * den, f"{what}: relative RMS error {num / den:.3e} > {rel}"


def both(got, ref, what, allow=None):
    check(got, ref, BF16_REL, what, None if allow is None else ALLOW_FACTOR * allow)
    rms_check(got, ref, what)


def rss_matmul(a, b):
    """Root-sum-square propagation of per-element errors a through a product
    with b: sqrt(a^2 @ b^2)."""
    return np.sqrt(np.square(a) @ np.square(b))


CORE_CASES = [  # B, S, H, Hkv, T_p, causal, q_scale
    (2, 200, 4, 2, 2, True, 1.0),
    (1, 300, 2, 2, 1, False, 1.0),
    (3, 64, 4, 1, 1, True, 1.0),
    (1, 1, 2, 2, 2, True, 1.0),
    (2, 128, 8, 4, 4, True, 1.0),
    (1, 129, 4, 4, 4, False, 1.0),
    (2, 384, 2, 2, 1, True, 4.0),
    (1, 520, 4, 2, 2, False, 3.0),
    (1, 257, 16, 2, 2, True, 1.0),   # GQA groups of 8, a one-row tail tile
    (3, 97, 2, 1, 1, False, 2.0),    # T_p 1, ragged non-causal
    (2, 2, 4, 4, 2, True, 1.0),      # two tokens
    (1, 640, 2, 2, 2, True, 1.0),    # odd number of 128-row tiles (5)
    (2, 768, 16, 4, 4, True, 1.0),   # 192 work items: CTAs take a second item (item-to-item hand-over)
]


def _core_sweep(n=6, seed=20261203):
    """Seeded random attention-core shapes: sequence lengths across tile
    boundaries, GQA groups of 1 to 4, T_p dividing the key/value heads,
    causal or not, and sharper or flatter softmaxes."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        Hkv = int(rng.choice([1, 2, 4]))
        G = int(rng.choice([1, 2, 4]))
        T = int(rng.choice([t for t in (1, 2, 4) if Hkv % t == 0]))
        out.append((int(rng.integers(1, 4)), int(rng.integers(1, 600)), Hkv * G, Hkv, T, bool(rng.integers(0, 2)),
                    float(rng.choice([0.5, 1.0, 2.0, 3.0]))))
    return out


CORE_CASES = CORE_CASES + _core_sweep()


@pytest.mark.parametrize("case", CORE_CASES, ids=lambda c: "B%d_S%d_H%d_kv%d_tp%d_%s_q%g" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full", c[6]))
def test_attention_core_matches_oracle(case):
    B, S, H, Hkv, T, causal, qs = case
    inp = make_core_inputs(B, S, H, Hkv, HD, seed=sum(case[:5]), q_scale=qs)
    attn = _attn_mod()(d=128, n_heads=H, n_kv_heads=Hkv, head_dim=HD, T_p=T, causal=causal)
    qkv = pack_qkv(inp["q"], inp["k"], inp["v"], H, Hkv, T).cuda()
    o, lse = attn.core_forward(qkv, B, S)
    dqkv = attn.core_backward(qkv, o, lse, inp["dO"].cuda(), B, S)
    torch.cuda.synchronize()

    core = oracle.AttentionCore(B, S, H, Hkv, HD, causal=causal, round_bf16=True)
    q64, k64, v64, dO64 = (to_f64(inp[n]) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = core.forward(q64, k64, v64)
    a_o, a_dq, a_dk, a_dv = core.allowance(q64, k64, v64, dO64, U)
    both(to_f64(o.cpu()), o_ref, "o", a_o)
    lse_nat = lse.cpu().double().numpy()[:, :S].reshape(B, H, S) * math.log(2.0)
    check(lse_nat, lse_ref, F32_REL, "lse")
    dq_ref, dk_ref, dv_ref = core.backward(q64, k64, v64, dO64)
    dq, dk, dv = unpack_qkv(dqkv.cpu(), H, Hkv, T)
    both(to_f64(dq), dq_ref, "dq", a_dq)
    both(to_f64(dk), dk_ref, "dk", a_dk)
    both(to_f64(dv), dv_ref, "dv", a_dv)


def test_attention_forward_lazy_rescale_path():
    """Keys whose scale grows along the sequence make each row's running
    maximum (per 64-key half of a 128-key block, in log2 units) rise by more
    than 2^8 after its first block, so the forward's lazy rescale of its O
    accumulators runs; checked on the inputs before the comparison."""
    B, S, H, Hkv, T = 1, 512, 2, 2, 1
    inp = make_core_inputs(B, S, H, Hkv, HD, seed=77, q_scale=2.0)
    ramp = torch.from_numpy(1.0 + 3.0 * np.arange(S, dtype=np.float64) / S).to(torch.float32)[:, None]
    inp["k"] = (inp["k"].to(torch.float32) * ramp).to(torch.bfloat16)
    q64, k64, v64, dO64 = (to_f64(inp[n]) for n in ("q", "k", "v", "dO"))
    scale_log2 = math.log2(math.e) / math.sqrt(HD)
    rises = 0
    for hh in range(H):
        sc = q64[:, hh * HD:(hh + 1) * HD] @ k64[:, hh * HD:(hh + 1) * HD].T * scale_log2  # [S, S]
        for half in range(2):
            blk = np.stack([sc[:, j * 128 + half * 64:j * 128 + half * 64 + 64].max(1) for j in range(S // 128)], 1)
            rises += int((np.maximum.accumulate(blk, 1)[:, 1:] > blk[:, :1] + 8.0).any(1).sum())
    assert rises > 0, "the inputs do not exercise the lazy rescale"
    attn = _attn_mod()(d=128, n_heads=H, n_kv_heads=Hkv, head_dim=HD, T_p=T, causal=False)
    qkv = pack_qkv(inp["q"], inp["k"], inp["v"], H, Hkv, T).cuda()
    o, lse = attn.core_forward(qkv, B, S)
    torch.cuda.synchronize()
    core = oracle.AttentionCore(B, S, H, Hkv, HD, causal=False, round_bf16=True)
    o_ref, lse_ref = core.forward(q64, k64, v64)
    a_o, _, _, _ = core.allowance(q64, k64, v64, dO64, U)
    both(to_f64(o.cpu()), o_ref, "o", a_o)
    lse_nat = lse.cpu().double().numpy()[:, :S].reshape(B, H, S) * math.log(2.0)
    check(lse_nat, lse_ref, F32_REL, "lse")


SUB_CASES = [  # B, S, d, H, Hkv, T_p, causal, fused
    (2, 160, 256, 4, 2, 2, True, False),
    (2, 160, 256, 4, 2, 2, True, True),
    (1, 200, 384, 8, 8, 4, False, False),
    (3, 70, 128, 4, 4, 4, True, True),
    (1, 130, 256, 16, 2, 2, True, False),  # GQA groups of 8
    (2, 256, 1024, 8, 8, 4, True, True),  # Q/K/V projection (24 tiles) and W_O forward (8) split into K parts
]


def _run_sublayer(w, inp, fused):
    attn = _attn_mod()(d=w.d, n_heads=w.H, n_kv_heads=w.Hkv, head_dim=HD, T_p=w.T_p, causal=w.causal)
    dev = {k: v.cuda() for k, v in inp.items()}
    wqkv, wo = attn.pack(dev["Wq"], dev["Wk"], dev["Wv"], dev["Wo"])
    y, saved = attn.forward(dev["x"], w.B, w.S, wqkv, wo, fused=fused)
    _, c, _ = attn.saved_views(saved, w.B, w.S)
    g = attn.backward(dev["x"], w.B, w.S, wqkv, wo, saved, dev["dy"], fused=fused)
    dWq, dWk, dWv, dWo = attn.unpack(g["dwqkv"], g["dwo"])
    torch.cuda.synchronize()
    return dict(y=y.cpu(), c=c.cpu(), dx=g["dx"].cpu(), dWq=dWq.cpu(), dWk=dWk.cpu(), dWv=dWv.cpu(),
                dWo=dWo.cpu())


@pytest.mark.parametrize("case", SUB_CASES, ids=lambda c: "B%d_S%d_d%d_H%d_kv%d_tp%d_%s_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full", "fused" if c[7] else "standalone"))
def test_attention_sublayer_matches_oracle(case):
    B, S, d, H, Hkv, T, causal, fused = case
    w = AttnWorkload("small_attention", B, S, d, H, Hkv, HD, T, causal=causal, seed_index=900 + sum(case[:6]))
    inp = make_attention_inputs(w)
    got = _run_sublayer(w, inp, fused)
    A = oracle.Attention(to_f64(inp["x"]), to_f64(inp["Wq"]), to_f64(inp["Wk"]), to_f64(inp["Wv"]),
                         to_f64(inp["Wo"]), B, S, H, Hkv, HD, T, causal=causal, round_bf16=True)
    c_ref, y_ref = A.forward()
    dy64 = to_f64(inp["dy"])
    ref = A.backward(dy64)
    # rounding allowances: the core's, propagated through the projections
    mid = A.intermediates(dy64)
    core = oracle.AttentionCore(B, S, H, Hkv, HD, causal=causal, round_bf16=True)
    a_o, a_dq, a_dk, a_dv = core.allowance(mid["q"], mid["k"], mid["v"], mid["dO"], U)
    x64, Wq, Wk, Wv, Wo = (to_f64(inp[n]) for n in ("x", "Wq", "Wk", "Wv", "Wo"))
    allow = dict(
        y=rss_matmul(a_o, Wo.T) + U * np.abs(y_ref),
        dx=np.sqrt(rss_matmul(a_dq, Wq) ** 2 + rss_matmul(a_dk, Wk) ** 2 + rss_matmul(a_dv, Wv) ** 2)
        + U * np.abs(ref["dx"]),
        dWq=rss_matmul(a_dq.T, x64) + U * np.abs(ref["dWq"]),
        dWk=rss_matmul(a_dk.T, x64) + U * np.abs(ref["dWk"]),
        dWv=rss_matmul(a_dv.T, x64) + U * np.abs(ref["dWv"]),
        dWo=rss_matmul(dy64.T, a_o) + U * np.abs(ref["dWo"]),
    )
    both(to_f64(got["c"]), c_ref, "c (head outputs)", a_o)
    both(to_f64(got["y"]), y_ref, "y", allow["y"])
    both(to_f64(got["dx"]), ref["dx"], "dx", allow["dx"])
    for n in ("dWq", "dWk", "dWv", "dWo"):
        both(to_f64(got[n]), ref[n], n, allow[n])


def test_attention_weight_packing_round_trips_bit_exact():
    w = AttnWorkload("pack", 1, 8, 256, 8, 4, HD, 4)
    inp = make_attention_inputs(w)
    attn = _attn_mod()(d=w.d, n_heads=w.H, n_kv_heads=w.Hkv, head_dim=HD, T_p=w.T_p)
    dev = {k: v.cuda() for k, v in inp.items()}
    wqkv, wo = attn.pack(dev["Wq"], dev["Wk"], dev["Wv"], dev["Wo"])
    back = attn.unpack(wqkv, wo)
    for name, t in zip(("Wq", "Wk", "Wv", "Wo"), back):
        assert torch.equal(t.cpu(), inp[name]), name
    # the packed q/k/v rows follow the documented shard-slice order
    packed = wqkv.view(torch.bfloat16).view(-1, w.d).cpu()
    assert torch.equal(packed, pack_qkv(inp["Wq"].T, inp["Wk"].T, inp["Wv"].T, w.H, w.Hkv, w.T_p).T)


def test_attention_sublayer_is_bitwise_deterministic():
    w = AttnWorkload("det", 2, 192, 256, 4, 2, HD, 2, seed_index=950)
    inp = make_attention_inputs(w)
    a = _run_sublayer(w, inp, fused=False)
    b = _run_sublayer(w, inp, fused=False)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_attention_empty_batch_is_a_no_op():
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    attn = _attn_mod()(d=128, n_heads=2, n_kv_heads=2, head_dim=HD, T_p=1)
    ws = attn.workspace(0, 0)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = abi.tp_attn_fwd(attn.plan, 0, 5, dummy, dummy, dummy, dummy, dummy, ws, ws.numel(), 0)
    assert rc == abi.TP_OK
    assert abi.tp_attn_last_launch_count(attn.plan) == 0
