"""Parity at the full workload sizes, in the launch configuration the
benchmark times: seeded token rows of y, dx and the shard partials, and seeded
entries of every weight and bias gradient, each computed one by one by the
float64 oracle.  Tolerances: see tests/parity.py."""
import functools

import numpy as np
import pytest
import torch

from synth import WORKLOADS, make_inputs
from tests.parity import (BF16_REL, F32_REL, allowance_rows, allowance_wgrad, check, oracle_problem,
                          rounding_weights, run_gpu_tensors)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FULL = ["gpt2_small_gelu_bf16", "llama3_8b_swiglu_bf16", "megatron_8p3b_gelu_bf16",
        "megatron_8p3b_attn_out_bf16", "llama3_70b_decode_swiglu_bf16"]


def _samples(w):
    """Seeded sample positions: 64 token rows (both ends included) of y, dx
    and the partials; 64 hidden units (both ends of the first and last shard
    and the two units either side of every interior shard boundary) by 64
    inputs and 64 outputs, i.e. 4096 entries of each of dW1, dW3 and dW2."""
    rng = np.random.default_rng(9000 + w.seed_index)
    n_rows = min(w.N, 64)
    rows = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, n_rows - 2, replace=False)]))
    s = w.s
    edges = [0, w.d_ff - 1] + [e for t in range(1, w.T_p) for e in (t * s - 1, t * s)]
    rest = np.setdiff1d(np.arange(w.d_ff), edges)
    js = np.unique(np.concatenate([edges, rng.choice(rest, 64 - len(edges), replace=False)]))
    ks = np.unique(np.concatenate([[0, w.d - 1], rng.choice(np.arange(1, w.d - 1), 62, replace=False)]))
    cs = np.unique(np.concatenate([[0, w.d - 1], rng.choice(np.arange(1, w.d - 1), 62, replace=False)]))
    return rows, js, ks, cs


@functools.lru_cache(maxsize=1)
def _reference(name):
    """Oracle values at the sampled positions (cached across the two sum modes)."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    rows, js, ks, cs = _samples(w)
    exact, f = oracle_problem(w, inp, round_bf16=False)
    rb, _ = oracle_problem(w, inp, round_bf16=True)
    ref = dict(rows=rows, js=js, ks=ks, cs=cs)
    ref["y_exact"] = exact.forward_sharded(rows)["y"]
    fs = rb.forward_sharded(rows)
    ref["y"], ref["partials"] = fs["y"], fs["partials"]
    A, W = {}, {}
    if w.act != "none":
        A = allowance_rows(w, f, rounding_weights(w, rb.hidden_dump(f["dy"], rows)))
        if not w.fwd_only:
            W = allowance_wgrad(w, f, rounding_weights(w, rb.hidden_dump(f["dy"], None, js)), ks, cs)
    ref["A"], ref["W"] = A, W
    if not w.fwd_only:
        ref["dx_exact"] = exact.backward_rows(f["dy"], rows)["dx"]
        br = rb.backward_rows(f["dy"], rows)
        ref["dx"], ref["dx_partials"] = br["dx"], br["dx_partials"]
        ref.update(rb.wgrad_entries(f["dy"], js, ks, cs))
    return w, inp, ref


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name, fused):
    w, inp, ref = _reference(name)
    out, n_fwd = run_gpu_tensors(w, inp, fused=fused, backward=not w.fwd_only)
    assert n_fwd >= 2  # the error-word reset and the compute kernels
    rows, js, ks, cs = (torch.as_tensor(ref[k]).cuda() for k in ("rows", "js", "ks", "cs"))
    get = lambda t: t.to(torch.float64).cpu().numpy()
    A, W = ref["A"], ref["W"]
    check(get(out["y"][rows]), ref["y"], BF16_REL, f"{name} y rows", A.get("y"))
    check(get(out["y"][rows]), ref["y_exact"], BF16_REL, f"{name} y rows vs float64 chain")
    if out["partials"] is not None:
        check(get(out["partials"][:, rows]), ref["partials"], F32_REL, f"{name} partials rows", A.get("partials"))
    if w.fwd_only:
        return
    check(get(out["dx"][rows]), ref["dx"], BF16_REL, f"{name} dx rows", A.get("dx"))
    check(get(out["dx"][rows]), ref["dx_exact"], BF16_REL, f"{name} dx rows vs float64 chain")
    if out["dx_partials"] is not None:
        check(get(out["dx_partials"][:, rows]), ref["dx_partials"], F32_REL, f"{name} dx partials rows",
              A.get("dx_partials"))
    check(get(out["dW2"][cs][:, js]), ref["dW2"], BF16_REL, f"{name} dW2 entries", W.get("dW2"))
    if w.act != "none":
        check(get(out["dW1"][js][:, ks]), ref["dW1"], BF16_REL, f"{name} dW1 entries", W.get("dW1"))
    if w.act == "swiglu":
        check(get(out["dW3"][js][:, ks]), ref["dW3"], BF16_REL, f"{name} dW3 entries", W.get("dW3"))
    if w.bias:
        check(get(out["db1"][js]), ref["db1"], BF16_REL, f"{name} db1 entries", W.get("db1"))
        check(get(out["db2"][cs]), ref["db2"], BF16_REL, f"{name} db2 entries")


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("name", FULL)
def test_full_size_bitwise_reproducible(name, fused):
    """Two runs of the whole benchmarked step (pack, forward, backward) on the
    same inputs, each with freshly allocated buffers, give the same bits in
    every output: y, the fp32 partials, dx and its partials, every weight and
    bias gradient.  Covers the fused shard K-loop of the persistent pair GEMMs
    under programmatic dependent launch, the standalone ordered sums, the
    ordered column sums of the bias gradients and, for the decode shapes, the
    split up GEMM with its combine kernel."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    a, _ = run_gpu_tensors(w, inp, fused=fused, backward=not w.fwd_only)
    b, _ = run_gpu_tensors(w, inp, fused=fused, backward=not w.fwd_only)
    compared = []
    for k, v in a.items():
        if v is None:
            continue
        assert torch.equal(_bits(v), _bits(b[k])), f"{name}: {k} differs between two runs"
        compared.append(k)
    expect = {"y"} | ({"partials"} if not fused else set())
    if not w.fwd_only:
        expect |= {"dx", "dW2"} | ({"dx_partials"} if not fused and w.act != "none" else set())
    assert expect <= set(compared), (expect, compared)
