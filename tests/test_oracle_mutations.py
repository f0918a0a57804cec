"""Planted mistakes: each plausible error in the oracle must fail some pin.

The mistake is planted in a temporary copy of the oracle's C source, compiled
on the CPU and swapped in for the real library while the pins of
test_oracle_pins run.  Nothing here touches a GPU.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import tests.test_oracle_attention_pins as apins
import tests.test_oracle_pins as pins

_SRC = os.path.join(os.path.dirname(oracle.__file__), "tpffn_oracle.c")

MUTATIONS = {
    "drop_b2": ("if (P->b2) acc += P->b2[c];", "if (P->b2) acc += 0.0 * P->b2[c];"),
    "gelu_constant": ("0.5 * u * (1.0 + tanh(c * (u + 0.044715 * u * u * u)))",
                      "0.5 * u * (1.0 + tanh(c * (u + 0.04715 * u * u * u)))"),
    "silu_grad_sign": ("return sg * (1.0 + u * (1.0 - sg));", "return sg * (1.0 - u * (1.0 - sg));"),
    "wrong_w2_shard": ("acc += P->W2[c * dff + t * s + jj] * ht[jj];",
                       "acc += P->W2[c * dff + ((t + 1) % T) * s + jj] * ht[jj];"),
    "b2_per_shard": ("for (int t = 0; t < T; ++t) acc += part[(int64_t)t * d + c];\n      if (P->b2)",
                     "for (int t = 0; t < T; ++t) acc += part[(int64_t)t * d + c] + (P->b2 ? P->b2[c] : 0.0);\n      if (P->b2)"),
    "ties_to_odd": ("(fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0", "(fmod(lo, 2.0) == 0.0) ? lo + 1.0 : lo"),
    "dW1_uses_h": ("acc1 += dzcol[n] * P->x[n * d + k];", "acc1 += hcol[n] * P->x[n * d + k];"),
    "dg_uses_grad": ("v1 = dh * orc_silu(as);", "v1 = dh * orc_silu_grad(as);"),
    "gelu_grad_drops_term": ("return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th * th) * dinner;",
                             "return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th) * dinner;"),
    "dx_skips_last_shard": ("for (int t = 0; t < T; ++t) acc += part[(int64_t)t * d + k];",
                            "for (int t = 0; t + 1 < T; ++t) acc += part[(int64_t)t * d + k];"),
    # attention sublayer
    "attn_kv_head_modulo": ("const int64_t hk = h / (C->H / C->Hkv);", "const int64_t hk = h % C->Hkv;"),
    "attn_scale_without_sqrt": ("const double scale = 1.0 / sqrt((double)hd);", "const double scale = 1.0 / (double)hd;"),
    "attn_causal_sees_next_key": ("const int64_t jmax = C->causal ? i : S - 1;",
                                  "const int64_t jmax = C->causal ? (i + 1 < S ? i + 1 : i) : S - 1;"),
    "attn_drops_rowdot": ("ds[j] = p[j] * (ds[j] - rowdot) * scale;", "ds[j] = p[j] * ds[j] * scale;"),
    "attn_dv_uses_dS": ("av += P[row * S + j] * dO[(b * S + i) * nq + h * hd + jd];",
                        "av += dS[row * S + j] * dO[(b * S + i) * nq + h * hd + jd];"),
    "attn_wo_shard_rotated": ("part += A->Wo[o * nq + jj] * c_out[r * nq + jj];",
                              "part += A->Wo[o * nq + (jj + s) % nq] * c_out[r * nq + jj];"),
    "attn_dx_skips_v": ("part += dv[r * nk + c2] * A->Wv[c2 * d + kk];", "part += 0.0 * dv[r * nk + c2];"),
    "attn_lse_drops_max": ("return m + log(sum);", "return log(sum);"),
}


def _pin_calls():
    calls = [pins.test_activations_match_torch_library, pins.test_activation_identities,
             pins.test_activation_derivatives_autograd_and_fd, pins.test_round_bf16_matches_torch_and_ties,
             pins.test_linear_special_case_reassociated, pins.test_shard_sum_equals_dense_tp1_to_tp11,
             pins.test_activation_commutes_with_column_split, pins.test_bruteforce_python_agrees_on_tiny_workload,
             pins.test_bf16_mode_rounds_only_stored_activations]
    for act, bias in [("gelu_tanh", True), ("swiglu", False), ("none", True)]:
        calls.append(lambda a=act, b=bias: pins.test_dense_forward_matches_torch_library(a, b))
    for act, bias in [("gelu_tanh", True), ("swiglu", False), ("none", False)]:
        calls.append(lambda a=act, b=bias: pins.test_backward_matches_torch_autograd(a, b))
    for act in ("gelu_tanh", "swiglu"):
        calls.append(lambda a=act: pins.test_backward_central_finite_differences(a))
    for case in apins.CORE_CASES:
        calls.append(lambda c=case: apins.test_attn_core_matches_torch_sdpa_and_autograd(c))
        calls.append(lambda c=case: apins.test_attn_core_key_shift_invariance_and_zero_key_gradient_sum(c))
    for case in apins.SUB_CASES:
        calls.append(lambda c=case: apins.test_attn_sublayer_matches_torch_linear_sdpa_and_autograd(c))
    calls += [lambda: apins.test_attn_core_zero_queries_give_visible_means(True),
              apins.test_attn_core_single_token_returns_value, apins.test_attn_core_central_finite_differences,
              apins.test_attn_core_bf16_mode_rounds_only_its_outputs,
              apins.test_attn_sublayer_independent_of_shard_count,
              apins.test_attn_sublayer_finite_differences_of_x]
    return calls


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    before, after = MUTATIONS[name]
    src = open(_SRC).read()
    assert src.count(before) >= 1, "mutation anchor not found: " + name
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mut.c")
        so = os.path.join(tmp, "libmut.so")
        open(c, "w").write(src.replace(before, after))
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", c, "-o", so, "-lm"])
        monkeypatch.setattr(oracle, "_lib", oracle.load_library(so))
        failed = []
        for call in _pin_calls():
            try:
                call()
            except AssertionError:
                failed.append(getattr(call, "__name__", "lambda"))
        assert failed, f"planted mistake {name!r} passed every pin"
