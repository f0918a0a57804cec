"""Pins of the float64 oracle to facts outside itself (CPU only).

Each test ties one part of the oracle to something it does not compute itself:
a library routine (PyTorch float64 ops and autograd), a closed form or exact
identity, central finite differences, an independent brute-force writing in
pure Python, or the invariants the pages state for the sharded FFN
("7.9 Tensor and pipeline parallelism (TP, PP)", §2.1; "S17 Tensor & Pipeline
Parallelism", "Run it locally": the sharded forward equals the unsharded one
at TP1 through TP11).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bruteforce
from synth import make_inputs, small_case, to_f64, WORKLOADS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_problem(N, d, d_ff, T_p, act, bias=False, seed=0, round_bf16=False, lib=None):
    rng = np.random.default_rng(seed)
    d_in = d_ff if act == "none" else d
    x = rng.standard_normal((N, d_in))
    W1 = rng.standard_normal((d_ff, d)) / math.sqrt(d) if act != "none" else None
    W3 = rng.standard_normal((d_ff, d)) / math.sqrt(d) if act == "swiglu" else None
    W2 = rng.standard_normal((d, d_ff)) / math.sqrt(d_ff)
    b1 = rng.standard_normal(d_ff) * 0.1 if bias and act not in ("swiglu", "none") else None
    b2 = rng.standard_normal(d) * 0.1 if bias else None
    dy = rng.standard_normal((N, d))
    P = oracle.FFN(x, W2, T_p, act, W1=W1, W3=W3, b1=b1, b2=b2, round_bf16=round_bf16, lib=lib)
    return P, dict(x=x, W1=W1, W3=W3, W2=W2, b1=b1, b2=b2, dy=dy)


def _torch_ffn(t, act):
    """Dense FFN written with PyTorch library ops (float64)."""
    x = t["x"]
    if act == "none":
        h = x
    elif act == "swiglu":
        h = F.silu(F.linear(x, t["W1"])) * F.linear(x, t["W3"])
    else:
        z = F.linear(x, t["W1"], t.get("b1"))
        h = F.gelu(z, approximate="tanh") if act == "gelu_tanh" else z
    return F.linear(h, t["W2"], t.get("b2"))


def _tt(a, grad=False):
    if a is None:
        return None
    return torch.tensor(a, dtype=torch.float64, requires_grad=grad)


# ------------------------------------------------------------------ scalars
U = np.concatenate([np.linspace(-12, 12, 481), [0.0, 1e-8, -1e-8, 3.5, -7.25, 40.0, -40.0]])


def test_activations_match_torch_library():
    u = torch.tensor(U, dtype=torch.float64)
    g_ref = F.gelu(u, approximate="tanh").numpy()
    s_ref = F.silu(u).numpy()
    g = np.array([oracle.gelu_tanh(v) for v in U])
    s = np.array([oracle.silu(v) for v in U])
    # 1 + tanh(.) cancels for u << 0, so both evaluations carry an absolute
    # error of a few |u| * 2^-52 there; elsewhere they agree to ~1e-14 relative
    np.testing.assert_allclose(g, g_ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(s, s_ref, rtol=1e-14, atol=1e-14)


def test_activation_identities():
    assert oracle.gelu_tanh(0.0) == 0.0 and oracle.silu(0.0) == 0.0
    for v in U:
        # gelu(u) - gelu(-u) = u and silu(u) - silu(-u) = u, exactly in reals
        assert abs(oracle.gelu_tanh(v) - oracle.gelu_tanh(-v) - v) <= 1e-14 * (1 + abs(v))
        assert abs(oracle.silu(v) - oracle.silu(-v) - v) <= 1e-14 * (1 + abs(v))
    # large-|u| limits: sigma(u)/u -> 1 for u -> +inf, sigma(u) -> 0 for u -> -inf
    assert abs(oracle.gelu_tanh(40.0) / 40.0 - 1) < 1e-15
    assert abs(oracle.silu(40.0) / 40.0 - 1) < 1e-15
    assert abs(oracle.gelu_tanh(-40.0)) < 1e-30 and abs(oracle.silu(-40.0)) < 1e-15
    # the tanh form approximates the exact erf GELU to better than 5e-4 everywhere
    for v in U:
        exact = 0.5 * v * (1 + math.erf(v / math.sqrt(2)))
        assert abs(oracle.gelu_tanh(v) - exact) < 5e-4


def test_activation_derivatives_autograd_and_fd():
    u = torch.tensor(U, dtype=torch.float64, requires_grad=True)
    (gg,) = torch.autograd.grad(F.gelu(u, approximate="tanh").sum(), u)
    (sg,) = torch.autograd.grad(F.silu(u).sum(), u)
    gd = np.array([oracle.gelu_tanh_grad(v) for v in U])
    sd = np.array([oracle.silu_grad(v) for v in U])
    # same cancellation for u << 0 as in the values: absolute 1e-13 there
    np.testing.assert_allclose(gd, gg.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sd, sg.numpy(), rtol=1e-13, atol=1e-13)
    hstep = 1e-5
    for v in U[::7]:
        fd = (oracle.gelu_tanh(v + hstep) - oracle.gelu_tanh(v - hstep)) / (2 * hstep)
        assert abs(fd - oracle.gelu_tanh_grad(v)) < 1e-8
        fd = (oracle.silu(v + hstep) - oracle.silu(v - hstep)) / (2 * hstep)
        assert abs(fd - oracle.silu_grad(v)) < 1e-8


def test_round_bf16_matches_torch_and_ties():
    rng = np.random.default_rng(3)
    # float32-representable inputs: PyTorch rounds float32 -> bf16 (RNE), and
    # the oracle rounds the same value directly; no double rounding can occur
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        [1e-40, -3e-39, 3.3e38, -3.39e38]]).astype(np.float32).astype(np.float64)
    ref = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(a) for a in v])
    np.testing.assert_array_equal(got, ref)
    # ties go to the even significand
    assert oracle.round_bf16(1 + 2.0 ** -8) == 1.0
    assert oracle.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert oracle.round_bf16(-(1 + 2.0 ** -8)) == -1.0
    assert oracle.round_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert oracle.round_bf16(0.0) == 0.0


# ------------------------------------------------------------ dense forms
@pytest.mark.parametrize("act,bias", [("gelu_tanh", False), ("gelu_tanh", True), ("swiglu", False),
                                      ("none", True), ("identity", True)])
def test_dense_forward_matches_torch_library(act, bias):
    P, a = _rand_problem(7, 24, 40, 4, act, bias=bias, seed=11)
    t = {k: _tt(v) for k, v in a.items() if v is not None}
    ref = _torch_ffn(t, act).numpy()
    np.testing.assert_allclose(P.forward_dense(), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(P.forward_sharded()["y"], ref, rtol=1e-12, atol=1e-12)


def test_linear_special_case_reassociated():
    """sigma = identity, no bias: y = x (W2 W1)^T, multiplied the other way round."""
    P, a = _rand_problem(9, 16, 48, 3, "identity", seed=5)
    ref = a["x"] @ (a["W2"] @ a["W1"]).T
    np.testing.assert_allclose(P.forward_sharded()["y"], ref, rtol=1e-12, atol=1e-12)
    # and the backward: dx = dy (W2 W1), dW1 = (dy W2)^T x, dW2 = dy^T (x W1^T)
    g = P.backward_full(a["dy"])
    np.testing.assert_allclose(g["dx"], a["dy"] @ (a["W2"] @ a["W1"]), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW1"], (a["dy"] @ a["W2"]).T @ a["x"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW2"], a["dy"].T @ (a["x"] @ a["W1"].T), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act,bias", [("gelu_tanh", True), ("swiglu", False), ("none", False)])
def test_backward_matches_torch_autograd(act, bias):
    P, a = _rand_problem(6, 16, 24, 3, act, bias=bias, seed=13)
    t = {k: _tt(v, grad=(k != "dy")) for k, v in a.items() if v is not None}
    y = _torch_ffn(t, act)
    y.backward(t["dy"])
    g = P.backward_full(a["dy"])
    np.testing.assert_allclose(g["dx"], t["x"].grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dW2"], t["W2"].grad.numpy(), rtol=1e-12, atol=1e-12)
    if act != "none":
        np.testing.assert_allclose(g["dW1"], t["W1"].grad.numpy(), rtol=1e-12, atol=1e-12)
    if act == "swiglu":
        np.testing.assert_allclose(g["dW3"], t["W3"].grad.numpy(), rtol=1e-12, atol=1e-12)
    if bias:
        np.testing.assert_allclose(g["db2"], t["b2"].grad.numpy(), rtol=1e-12, atol=1e-12)
        if "b1" in t:
            np.testing.assert_allclose(g["db1"], t["b1"].grad.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_backward_central_finite_differences(act):
    """dL/dtheta for L = sum(dy * y), against central differences of the forward."""
    P, a = _rand_problem(4, 8, 12, 2, act, bias=(act == "gelu_tanh"), seed=17)
    g = P.backward_full(a["dy"])
    eps = 1e-6

    def loss(**over):
        kw = {k: over.get(k, a[k]) for k in ("x", "W1", "W3", "W2", "b1", "b2")}
        Q = oracle.FFN(kw["x"], kw["W2"], 2, act, W1=kw["W1"], W3=kw["W3"], b1=kw["b1"], b2=kw["b2"])
        return float((Q.forward_dense() * a["dy"]).sum())

    checks = [("x", (1, 3), g["dx"][1, 3]), ("W1", (5, 2), g["dW1"][5, 2]),
              ("W2", (3, 7), g["dW2"][3, 7])]
    if act == "swiglu":
        checks.append(("W3", (9, 4), g["dW3"][9, 4]))
    else:
        checks.append(("b1", (6,), g["db1"][6]))
    for name, idx, analytic in checks:
        plus, minus = a[name].copy(), a[name].copy()
        plus[idx] += eps
        minus[idx] -= eps
        fd = (loss(**{name: plus}) - loss(**{name: minus})) / (2 * eps)
        assert abs(fd - analytic) <= 1e-6 * max(1.0, abs(analytic)), (name, fd, analytic)


# --------------------------------------------------------- sharding pins
def test_shard_sum_equals_dense_tp1_to_tp11():
    """Sum of the shard partials equals the unsharded output at TP1..TP11."""
    spec = json.load(open(os.path.join(GOLDEN, "tp_degrees.json")))
    for T_p in spec["tp_degrees"]:
        for act in ("gelu_tanh", "swiglu"):
            P, a = _rand_problem(5, 12, 6 * T_p, T_p, act, bias=(act == "gelu_tanh"), seed=T_p)
            dense = P.forward_dense()
            sh = P.forward_sharded()
            np.testing.assert_allclose(sh["partials"].sum(0) + (a["b2"] if a["b2"] is not None else 0),
                                       sh["y"], rtol=0, atol=1e-13)
            assert np.all(np.abs(sh["y"] - dense) <= 1e-12 * (np.abs(dense) + 1)), T_p
            if T_p == 1:
                assert np.array_equal(sh["y"], dense)  # same summation order: bitwise
            # backward mirror: the dx shard-sum equals the unsharded dx
            dxs = P.backward_rows(a["dy"])
            dxd = P.backward_dense_dx(a["dy"])
            assert np.all(np.abs(dxs["dx"] - dxd) <= 1e-12 * (np.abs(dxd) + 1)), T_p
            np.testing.assert_allclose(dxs["dx_partials"].sum(0), dxs["dx"], rtol=0, atol=1e-13)


def test_activation_commutes_with_column_split():
    P, a = _rand_problem(6, 10, 32, 4, "gelu_tanh", bias=True, seed=23)
    h_shards = P.forward_sharded()["h"]
    z = torch.tensor(a["x"]) @ torch.tensor(a["W1"]).T + torch.tensor(a["b1"])
    np.testing.assert_allclose(h_shards, F.gelu(z, approximate="tanh").numpy(), rtol=1e-13, atol=1e-15)


def test_row_split_of_first_matrix_does_not_commute():
    """Splitting W1 along its input dimension needs the sum before sigma."""
    P, a = _rand_problem(6, 16, 32, 4, "gelu_tanh", seed=29)
    bad = P.forward_rowsplit_bad()
    good = P.forward_dense()
    assert np.max(np.abs(bad - good)) > 1e-2
    # with a linear sigma the row split is exact: the non-linearity is the reason
    L, _ = _rand_problem(6, 16, 32, 4, "identity", seed=29)
    np.testing.assert_allclose(L.forward_rowsplit_bad(), L.forward_dense(), rtol=1e-12, atol=1e-12)


def test_bruteforce_python_agrees_on_tiny_workload():
    w = WORKLOADS["tiny_gelu_fp32"]
    inp = make_inputs(w)
    f = {k: to_f64(v) for k, v in inp.items()}
    for act in ("gelu_tanh", "swiglu", "none"):
        x = f["x"] if act != "none" else np.random.default_rng(1).standard_normal((w.N, w.d_ff))
        W3 = f["W1"][::-1].copy() if act == "swiglu" else None
        P = oracle.FFN(x, f["W2"], w.T_p, act, W1=f["W1"], W3=W3)
        y_bf, part_bf = bruteforce.ffn_sharded_forward(x.tolist(), f["W1"].tolist(),
                                                       None if W3 is None else W3.tolist(), None,
                                                       f["W2"].tolist(), None, w.T_p, act)
        sh = P.forward_sharded()
        np.testing.assert_allclose(sh["y"], np.array(y_bf), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(sh["partials"], np.array(part_bf), rtol=1e-13, atol=1e-13)


def test_sampled_functions_equal_full_computation():
    w = small_case(37, 24, 60, 3, "gelu_tanh", dtype="bf16", bias=True, seed=31)
    inp = make_inputs(w)
    f = {k: to_f64(v) for k, v in inp.items()}
    P = oracle.FFN(f["x"], f["W2"], w.T_p, "gelu_tanh", W1=f["W1"], b1=f["b1"], b2=f["b2"],
                   round_bf16=True)
    full = P.forward_sharded()
    rows = np.array([36, 0, 17, 5])
    sub = P.forward_sharded(rows)
    np.testing.assert_array_equal(sub["y"], full["y"][rows])
    np.testing.assert_array_equal(sub["partials"], full["partials"][:, rows])
    g = P.backward_full(f["dy"])
    gs = P.backward_rows(f["dy"], rows)
    np.testing.assert_array_equal(gs["dx"], g["dx"][rows])
    js, ks, cs = np.array([59, 3, 20]), np.array([0, 23]), np.array([7, 1])
    e = P.wgrad_entries(f["dy"], js, ks, cs)
    np.testing.assert_array_equal(e["dW1"], g["dW1"][np.ix_(js, ks)])
    np.testing.assert_array_equal(e["dW2"], g["dW2"][np.ix_(cs, js)])
    np.testing.assert_array_equal(e["db1"], g["db1"][js])
    np.testing.assert_array_equal(e["db2"], g["db2"][cs])


def test_bf16_mode_rounds_only_stored_activations():
    w = small_case(9, 16, 32, 2, "swiglu", dtype="bf16", seed=41)
    inp = make_inputs(w)
    f = {k: to_f64(v) for k, v in inp.items()}
    P = oracle.FFN(f["x"], f["W2"], 2, "swiglu", W1=f["W1"], W3=f["W3"], round_bf16=True)
    E = oracle.FFN(f["x"], f["W2"], 2, "swiglu", W1=f["W1"], W3=f["W3"], round_bf16=False)
    sp, se = P.forward_sharded(), E.forward_sharded()
    rb = torch.tensor(sp["h"]).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(sp["h"], rb)           # h is bf16-representable
    np.testing.assert_allclose(sp["h"], se["h"], rtol=2.0 ** -8, atol=1e-30)  # within half an ulp
    # the partial is the exact float64 product of the rounded h with W2
    s = w.s
    for t in range(2):
        ref = sp["h"][:, t * s:(t + 1) * s] @ f["W2"][:, t * s:(t + 1) * s].T
        np.testing.assert_allclose(sp["partials"][t], ref, rtol=1e-12, atol=1e-13)


def test_hidden_dump_rounds_to_stored_values():
    """The pre-rounding dump rounds (RNE, bf16) to exactly the stored values,
    equals them in float64 mode, its dh is W2^T dy, its norms are those of the
    products, and a column subset equals the same columns of the full dump."""
    for act in ("gelu_tanh", "swiglu"):
        w = small_case(11, 16, 48, 3, act, dtype="bf16", bias=(act == "gelu_tanh"), seed=43)
        f = {k: to_f64(v) for k, v in make_inputs(w).items()}
        kw = dict(W1=f["W1"], W3=f["W3"], b1=f["b1"], b2=f["b2"])
        for rb in (False, True):
            P = oracle.FFN(f["x"], f["W2"], 3, act, round_bf16=rb, **kw)
            dump = P.hidden_dump(f["dy"])
            sh = P.forward_sharded()
            # the oracle's own bf16 rounding (pinned above against PyTorch); a
            # float64 -> float32 -> bf16 cast would round twice
            R = np.vectorize(oracle.round_bf16) if rb else (lambda a: a)
            np.testing.assert_array_equal(R(dump["h_pre"]), sh["h"])
            if act == "swiglu":
                np.testing.assert_array_equal(R(dump["z_pre"]), sh["ag_saved"][:, 0])
                np.testing.assert_array_equal(R(dump["g_pre"]), sh["ag_saved"][:, 1])
                np.testing.assert_allclose(dump["ng"], np.sqrt((f["x"] ** 2) @ (f["W3"] ** 2).T), rtol=1e-12)
            else:
                np.testing.assert_array_equal(R(dump["z_pre"]), sh["z_saved"])
            np.testing.assert_allclose(dump["dh"], f["dy"] @ f["W2"], rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(dump["nz"], np.sqrt((f["x"] ** 2) @ (f["W1"] ** 2).T), rtol=1e-12)
            np.testing.assert_allclose(dump["ndh"], np.sqrt((f["dy"] ** 2) @ (f["W2"] ** 2)), rtol=1e-12)
            js = np.arange(w.d_ff)
            e = P.wgrad_entries(f["dy"], js)
            if act == "gelu_tanh":  # db1 = sum over tokens of the stored dz
                np.testing.assert_allclose(R(dump["dz_pre"]).sum(0), e["db1"], rtol=1e-12, atol=1e-12)
            sub = P.hidden_dump(f["dy"], rows=[3, 0], cols=[47, 5, 20])
            for k in dump:
                np.testing.assert_array_equal(sub[k], dump[k][np.ix_([3, 0], [47, 5, 20])])


def test_chain_noise_bounds_bf16_storage_and_is_not_vacuous():
    """The widening that the GPU parity tests give the comparison of y and dx
    with the pure float64 chain (tests.parity.chain_noise) covers what bf16
    storage of the hidden activations does to them: the rounded oracle stays
    within 1e-2 (|ref| + 1) plus that bound of the float64 chain, for both
    activations and a hidden width in the thousands; and the bound is of the
    size of that noise, not a blanket pass: measured in the bound's standard
    deviation (bound / 6), the rounded oracle's distances have a root mean
    square between 0.1 and 1 (about 0.75 for y, whose h is rounded once)."""
    from tests.parity import chain_noise
    for act, (N, d, d_ff, T) in (("swiglu", (96, 64, 2048, 4)), ("gelu_tanh", (96, 64, 4096, 4))):
        w = small_case(N, d, d_ff, T, act, dtype="bf16", seed=47)
        f = {k: to_f64(v) for k, v in make_inputs(w).items()}
        kw = dict(W1=f["W1"], W3=f["W3"], b1=f["b1"], b2=f["b2"])
        P = oracle.FFN(f["x"], f["W2"], T, act, round_bf16=True, **kw)
        E = oracle.FFN(f["x"], f["W2"], T, act, round_bf16=False, **kw)
        C = chain_noise(w, f, E.hidden_dump(f["dy"]))
        got = dict(y=P.forward_sharded()["y"], dx=P.backward_rows(f["dy"])["dx"])
        ref = dict(y=E.forward_sharded()["y"], dx=E.backward_rows(f["dy"])["dx"])
        for k in ("y", "dx"):
            err = np.abs(got[k] - ref[k])
            assert np.all(err <= 1e-2 * (np.abs(ref[k]) + 1.0) + C[k]), (act, k)
            z = np.sqrt(np.mean((err / (C[k] / 6.0)) ** 2))
            assert 0.1 < z < 1.0, (act, k, z)
