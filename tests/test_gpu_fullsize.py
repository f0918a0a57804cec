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
    rng = np.random.default_rng(9000 + w.seed_index)
    n_rows = min(w.N, 40)
    rows = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, n_rows - 2, replace=False)]))
    # hidden units: include both ends of every shard
    s = w.s
    js = np.unique(np.concatenate([[0, s - 1, w.d_ff - 1, (w.T_p - 1) * s], rng.choice(w.d_ff, 12, replace=False)]))
    ks = np.unique(np.concatenate([[0, w.d - 1], rng.choice(w.d, 14, replace=False)]))
    cs = np.unique(np.concatenate([[0, w.d - 1], rng.choice(w.d, 14, replace=False)]))
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
    assert n_fwd >= 1
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
