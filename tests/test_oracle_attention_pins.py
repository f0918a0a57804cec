"""Pins of the float64 attention oracle to facts outside itself (CPU only).

The head-sharded attention sublayer ("7.9 Tensor and pipeline parallelism
(TP, PP)", §2.2 "Attention, sharded"; the GQA divisibility rule of "S17 Tensor &
Pipeline Parallelism", "Attention shards by head, and GQA caps the degree") is
tied to:

* PyTorch's own scaled dot-product attention and linear layers in float64, with
  autograd for every gradient (a library routine written independently);
* closed forms: all-zero queries give uniform weights, so each output is the
  mean of the visible values and the log-sum-exp is log(#visible keys); a
  one-token sequence returns its value;
* exact invariants: a shift of every key by one vector leaves the output
  unchanged (softmax is shift invariant), so the key gradients of a head sum to
  zero over its keys; the sharded sum is independent of T_p;
* central finite differences of a scalar loss;
* the rounding points of the bf16 mode.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

CORE_CASES = [  # B, S, H, Hkv, hd, causal
    (2, 7, 4, 2, 8, True),
    (1, 9, 3, 3, 4, False),
    (2, 5, 4, 1, 6, True),
]


def _core_inputs(B, S, H, Hkv, hd, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B * S, H * hd))
    k = rng.standard_normal((B * S, Hkv * hd))
    v = rng.standard_normal((B * S, Hkv * hd))
    dO = rng.standard_normal((B * S, H * hd))
    return q, k, v, dO


def _heads(a, B, S, nh, hd, grad=False):
    """[B*S, nh*hd] -> torch [B, nh, S, hd]."""
    t = torch.tensor(a, dtype=torch.float64).view(B, S, nh, hd).transpose(1, 2)
    return t.detach().requires_grad_(grad)


def _flat(t):
    B, nh, S, hd = t.shape
    return t.transpose(1, 2).reshape(B * S, nh * hd)


def _torch_core(q, k, v, B, S, H, Hkv, hd, causal):
    """Library attention: GQA by repeating each key/value head for its group."""
    Q, K, V = _heads(q, B, S, H, hd, True), _heads(k, B, S, Hkv, hd, True), _heads(v, B, S, Hkv, hd, True)
    G = H // Hkv
    O = F.scaled_dot_product_attention(Q, K.repeat_interleave(G, 1), V.repeat_interleave(G, 1),
                                       is_causal=causal)
    return Q, K, V, O


# ------------------------------------------------------------------ core
@pytest.mark.parametrize("case", CORE_CASES)
def test_attn_core_matches_torch_sdpa_and_autograd(case):
    B, S, H, Hkv, hd, causal = case
    q, k, v, dO = _core_inputs(B, S, H, Hkv, hd, seed=1)
    C = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal)
    o, lse = C.forward(q, k, v)
    Q, K, V, O = _torch_core(q, k, v, B, S, H, Hkv, hd, causal)
    np.testing.assert_allclose(o, _flat(O).detach().numpy(), rtol=0, atol=1e-12)
    # log-sum-exp of the scaled scores, from the library's logsumexp
    s = (Q @ K.repeat_interleave(H // Hkv, 1).transpose(-1, -2)) / math.sqrt(hd)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).detach().numpy(), rtol=0, atol=1e-12)
    _flat(O).backward(torch.tensor(dO))
    dq, dk, dv = C.backward(q, k, v, dO)
    np.testing.assert_allclose(dq, _flat(Q.grad).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, _flat(K.grad).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, _flat(V.grad).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_attn_core_zero_queries_give_visible_means(causal):
    B, S, H, Hkv, hd = 2, 6, 4, 2, 3
    _, k, v, _ = _core_inputs(B, S, H, Hkv, hd, seed=2)
    q = np.zeros((B * S, H * hd))
    o, lse = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal).forward(q, k, v)
    G = H // Hkv
    for b in range(B):
        for h in range(H):
            vh = v[b * S:(b + 1) * S, (h // G) * hd:(h // G + 1) * hd]
            for i in range(S):
                n = i + 1 if causal else S
                np.testing.assert_allclose(o[b * S + i, h * hd:(h + 1) * hd], vh[:n].mean(0), rtol=0, atol=1e-14)
                assert abs(lse[b, h, i] - math.log(n)) < 1e-14


def test_attn_core_single_token_returns_value():
    B, S, H, Hkv, hd = 3, 1, 2, 2, 5
    q, k, v, _ = _core_inputs(B, S, H, Hkv, hd, seed=3)
    o, _ = oracle.AttentionCore(B, S, H, Hkv, hd, causal=True).forward(q, k, v)
    np.testing.assert_array_equal(o, v)


@pytest.mark.parametrize("case", CORE_CASES)
def test_attn_core_key_shift_invariance_and_zero_key_gradient_sum(case):
    B, S, H, Hkv, hd, causal = case
    q, k, v, dO = _core_inputs(B, S, H, Hkv, hd, seed=4)
    C = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal)
    o, _ = C.forward(q, k, v)
    w = np.random.default_rng(5).standard_normal(Hkv * hd)
    o2, _ = C.forward(q, k + w[None, :], v)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    _, dk, _ = C.backward(q, k, v, dO)
    sums = dk.reshape(B, S, Hkv * hd).sum(1)
    np.testing.assert_allclose(sums, 0.0, rtol=0, atol=1e-12)


def test_attn_core_central_finite_differences():
    B, S, H, Hkv, hd, causal = 1, 5, 2, 1, 3, True
    q, k, v, dO = _core_inputs(B, S, H, Hkv, hd, seed=6)
    C = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal)
    grads = dict(zip("qkv", C.backward(q, k, v, dO)))
    arrays = dict(q=q, k=k, v=v)
    eps = 1e-6
    rng = np.random.default_rng(7)
    for name in "qkv":
        a = arrays[name]
        for _ in range(6):
            idx = (int(rng.integers(a.shape[0])), int(rng.integers(a.shape[1])))
            loss = []
            for sgn in (1, -1):
                b = {n: x.copy() for n, x in arrays.items()}
                b[name][idx] += sgn * eps
                loss.append((C.forward(b["q"], b["k"], b["v"])[0] * dO).sum())
            fd = (loss[0] - loss[1]) / (2 * eps)
            assert abs(fd - grads[name][idx]) < 1e-7 * (1 + abs(fd)), (name, idx, fd, grads[name][idx])


def test_attn_core_bf16_mode_rounds_only_its_outputs():
    B, S, H, Hkv, hd, causal = 2, 6, 4, 2, 8, True
    q, k, v, dO = (oracle_round(a) for a in _core_inputs(B, S, H, Hkv, hd, seed=8))
    exact = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal)
    rounded = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal, round_bf16=True)
    o, lse = exact.forward(q, k, v)
    ob, lseb = rounded.forward(q, k, v)
    np.testing.assert_array_equal(ob, oracle_round(o))
    np.testing.assert_array_equal(lseb, lse)
    for g, gb in zip(exact.backward(q, k, v, dO), rounded.backward(q, k, v, dO)):
        np.testing.assert_array_equal(gb, oracle_round(g))


def oracle_round(a):
    return np.vectorize(oracle.round_bf16)(np.asarray(a, dtype=np.float64))


# ------------------------------------------------------------------ sublayer
def _sublayer(B, S, d, H, Hkv, hd, T_p, causal=True, seed=0, round_bf16=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B * S, d))
    Wq = rng.standard_normal((H * hd, d)) / math.sqrt(d)
    Wk = rng.standard_normal((Hkv * hd, d)) / math.sqrt(d)
    Wv = rng.standard_normal((Hkv * hd, d)) / math.sqrt(d)
    Wo = rng.standard_normal((d, H * hd)) / math.sqrt(H * hd)
    dy = rng.standard_normal((B * S, d))
    A = oracle.Attention(x, Wq, Wk, Wv, Wo, B, S, H, Hkv, hd, T_p, causal=causal, round_bf16=round_bf16)
    return A, dict(x=x, Wq=Wq, Wk=Wk, Wv=Wv, Wo=Wo, dy=dy)


SUB_CASES = [  # B, S, d, H, Hkv, hd, T_p, causal
    (2, 6, 12, 4, 2, 4, 2, True),
    (1, 7, 10, 6, 6, 3, 3, False),
    (2, 5, 8, 8, 4, 2, 4, True),
]


@pytest.mark.parametrize("case", SUB_CASES)
def test_attn_sublayer_matches_torch_linear_sdpa_and_autograd(case):
    B, S, d, H, Hkv, hd, T_p, causal = case
    A, w = _sublayer(B, S, d, H, Hkv, hd, T_p, causal, seed=11)
    c, y = A.forward()
    t = {n: torch.tensor(a, dtype=torch.float64, requires_grad=True) for n, a in w.items() if n != "dy"}
    Q = F.linear(t["x"], t["Wq"]).view(B, S, H, hd).transpose(1, 2)
    K = F.linear(t["x"], t["Wk"]).view(B, S, Hkv, hd).transpose(1, 2)
    V = F.linear(t["x"], t["Wv"]).view(B, S, Hkv, hd).transpose(1, 2)
    G = H // Hkv
    O = F.scaled_dot_product_attention(Q, K.repeat_interleave(G, 1), V.repeat_interleave(G, 1), is_causal=causal)
    cy = O.transpose(1, 2).reshape(B * S, H * hd)
    Y = F.linear(cy, t["Wo"])
    np.testing.assert_allclose(c, cy.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(y, Y.detach().numpy(), rtol=0, atol=1e-12)
    Y.backward(torch.tensor(w["dy"]))
    g = A.backward(w["dy"])
    np.testing.assert_allclose(g["dx"], t["x"].grad.numpy(), rtol=0, atol=1e-11)
    for n in ("Wq", "Wk", "Wv", "Wo"):
        np.testing.assert_allclose(g["d" + n], t[n].grad.numpy(), rtol=0, atol=1e-11)


def test_attn_sublayer_independent_of_shard_count():
    B, S, d, H, Hkv, hd = 2, 5, 8, 8, 4, 3
    ref = None
    for T_p in (1, 2, 4):
        A, w = _sublayer(B, S, d, H, Hkv, hd, T_p, True, seed=12)
        c, y = A.forward()
        g = A.backward(w["dy"])
        if ref is None:
            ref = (c, y, g)
            continue
        np.testing.assert_array_equal(c, ref[0])
        np.testing.assert_allclose(y, ref[1], rtol=0, atol=1e-13)
        np.testing.assert_allclose(g["dx"], ref[2]["dx"], rtol=0, atol=1e-13)
        for n in ("dWq", "dWk", "dWv", "dWo"):
            np.testing.assert_array_equal(g[n], ref[2][n])


def test_attn_sublayer_finite_differences_of_x():
    B, S, d, H, Hkv, hd, T_p = 1, 4, 6, 4, 2, 2, 2
    A, w = _sublayer(B, S, d, H, Hkv, hd, T_p, True, seed=13)
    dx = A.backward(w["dy"])["dx"]
    eps = 1e-6
    for idx in [(0, 0), (1, 3), (3, 5), (2, 1)]:
        loss = []
        for sgn in (1, -1):
            x = w["x"].copy()
            x[idx] += sgn * eps
            B2 = oracle.Attention(x, w["Wq"], w["Wk"], w["Wv"], w["Wo"], B, S, H, Hkv, hd, T_p)
            loss.append((B2.forward()[1] * w["dy"]).sum())
        fd = (loss[0] - loss[1]) / (2 * eps)
        assert abs(fd - dx[idx]) < 1e-7 * (1 + abs(fd))


def test_attn_sublayer_bf16_mode_stores_bf16_head_outputs():
    A, w = _sublayer(2, 6, 12, 4, 2, 4, 2, True, seed=14, round_bf16=True)
    c, _ = A.forward()
    np.testing.assert_array_equal(c, oracle_round(c))
    E, _ = _sublayer(2, 6, 12, 4, 2, 4, 2, True, seed=14)
    ce, ye = E.forward()
    _, yb = A.forward()
    # storage rounding only: relative deviations of the order of 2^-8
    assert np.abs(c - ce).max() < 2 ** -6 * (np.abs(ce).max() + 1)
    assert np.abs(yb - ye).max() < 2 ** -5 * (np.abs(ye).max() + 1)


def test_attn_gqa_divisibility_golden():
    """Rule of "S17 Tensor & Pipeline Parallelism": T_p must divide the query
    and the key/value heads (the golden file lists the cases and verdicts)."""
    cases = json.load(open(os.path.join(GOLDEN, "gqa_divisibility.json")))["cases"]
    for case in cases:
        H, Hkv, T_p, ok = case["n_heads"], case["n_kv_heads"], case["T_p"], case["valid"]
        hd, d, B, S = 2, 4, 1, 2
        x = np.zeros((B * S, d))
        args = (x, np.zeros((H * hd, d)), np.zeros((Hkv * hd, d)), np.zeros((Hkv * hd, d)),
                np.zeros((d, H * hd)), B, S, H, Hkv, hd, T_p)
        if ok:
            oracle.Attention(*args)
        else:
            with pytest.raises(ValueError):
                oracle.Attention(*args)


# ------------------------------------------------------------------ tolerance model
def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _emulate_bf16_core(q, k, v, dO, B, S, H, Hkv, hd, causal):
    """A bf16 attention core written with numpy: unnormalised probabilities
    rounded before p v, o rounded, D from the rounded o, dS rounded before its
    products, every output rounded (the rounding points the allowance models)."""
    G = H // Hkv
    sc = 1 / math.sqrt(hd)
    o, dq = np.zeros_like(q), np.zeros_like(q)
    dk, dv = np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        rows = slice(b * S, (b + 1) * S)
        for h in range(H):
            hk = h // G
            Q, K, V = q[rows, h * hd:(h + 1) * hd], k[rows, hk * hd:(hk + 1) * hd], v[rows, hk * hd:(hk + 1) * hd]
            s = (Q @ K.T) * sc
            if causal:
                s = np.where(np.tril(np.ones((S, S))) > 0, s, -np.inf)
            e = np.exp(s - s.max(1, keepdims=True))
            l = e.sum(1, keepdims=True)
            ob = _bf16((_bf16(e) @ V) / l)
            o[rows, h * hd:(h + 1) * hd] = ob
            P = e / l
            g = dO[rows, h * hd:(h + 1) * hd]
            dS = _bf16(P * (g @ V.T - (g * ob).sum(1, keepdims=True)) * sc)
            dq[rows, h * hd:(h + 1) * hd] = dS @ K
            dk[rows, hk * hd:(hk + 1) * hd] += dS.T @ Q
            dv[rows, hk * hd:(hk + 1) * hd] += _bf16(P).T @ g
    return o, _bf16(dq), _bf16(dk), _bf16(dv)


@pytest.mark.parametrize("case", [(2, 40, 4, 2, 16, True, 1.0), (1, 64, 2, 2, 32, False, 4.0)])
def test_attn_allowance_bounds_a_bf16_computation(case):
    """The rounding allowance used by the GPU parity tests bounds how far a
    bf16 computation of the same steps strays from the exact result (here a
    numpy emulation of those rounding points), with the factor those tests
    use; and it is not vacuous: it stays within 10% of the values' RMS."""
    B, S, H, Hkv, hd, causal, qs = case
    rng = np.random.default_rng(21)
    q = _bf16(rng.standard_normal((B * S, H * hd)) * qs)
    k, v = (_bf16(rng.standard_normal((B * S, Hkv * hd))) for _ in range(2))
    dO = _bf16(rng.standard_normal((B * S, H * hd)))
    C = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal, round_bf16=True)
    o, _ = C.forward(q, k, v)
    exact = (o,) + C.backward(q, k, v, dO)
    allow = C.allowance(q, k, v, dO, 2.0 ** -8)
    emul = _emulate_bf16_core(q, k, v, dO, B, S, H, Hkv, hd, causal)
    for name, e, r, a in zip(("o", "dq", "dk", "dv"), emul, exact, allow):
        assert np.all(np.abs(e - r) <= 1e-2 * (np.abs(r) + 1) + 3 * a), name
        assert np.sqrt(np.mean(a ** 2)) < 0.1 * np.sqrt(np.mean(r ** 2)), name


@pytest.mark.parametrize("causal", [True, False])
def test_attn_sampled_rows_equal_full_computation(causal):
    """The sampled-row function (used at full sizes) returns exactly what the
    full core, backward and allowance give at the same positions."""
    B, S, H, Hkv, hd = 2, 21, 4, 2, 8
    q, k, v, dO = _core_inputs(B, S, H, Hkv, hd, seed=31)
    C = oracle.AttentionCore(B, S, H, Hkv, hd, causal=causal)
    u = 2.0 ** -8
    o, lse = C.forward(q, k, v)
    dq, dk, dv = C.backward(q, k, v, dO)
    a_o, a_dq, a_dk, a_dv = C.allowance(q, k, v, dO, u)
    rows = [(0, 0, 0), (1, 3, 20), (0, 2, 7), (1, 1, 13)]
    kv_rows = [(0, 0, 0), (1, 1, 20), (1, 0, 5), (0, 1, 11)]
    smp = C.sample(q, k, v, dO, u, rows, kv_rows)
    for s, (b, h, i) in enumerate(rows):
        sl = (b * S + i, slice(h * hd, (h + 1) * hd))
        np.testing.assert_allclose(smp["o"][s], o[sl], rtol=0, atol=1e-13)
        np.testing.assert_allclose(smp["dq"][s], dq[sl], rtol=0, atol=1e-13)
        np.testing.assert_allclose(smp["a_o"][s], a_o[sl], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(smp["a_dq"][s], a_dq[sl], rtol=1e-10, atol=1e-15)
        assert abs(smp["lse"][s] - lse[b, h, i]) < 1e-13
    for s, (b, hk, j) in enumerate(kv_rows):
        sl = (b * S + j, slice(hk * hd, (hk + 1) * hd))
        np.testing.assert_allclose(smp["dk"][s], dk[sl], rtol=0, atol=1e-13)
        np.testing.assert_allclose(smp["dv"][s], dv[sl], rtol=0, atol=1e-13)
        np.testing.assert_allclose(smp["a_dk"][s], a_dk[sl], rtol=1e-10, atol=1e-15)
        np.testing.assert_allclose(smp["a_dv"][s], a_dv[sl], rtol=1e-10, atol=1e-15)
