"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Small and ragged shapes are compared element by element with the full
oracle; the full-size workloads (GPT-2 small, Llama-3-8B, Megatron-8.3B FFN
and W_O, Llama-3-70B decode) on seeded token rows and weight-gradient entries
that the oracle computes one by one.  Tolerances: see tests/parity.py.
"""
import numpy as np
import pytest
import torch

from synth import WORKLOADS, Workload, make_inputs, small_case
from tests.parity import (BF16_REL, F32_REL, allowance_rows, allowance_wgrad, chain_noise, check,
                          oracle_problem, rounding_weights, run_gpu)

pytestmark = pytest.mark.gpu


def _full_compare(w, fused):
    """Every output against the oracle in the workload's stated precision
    (bf16-stored activations for bf16 workloads), plus y and dx against the
    pure float64 chain."""
    inp = make_inputs(w)
    got = run_gpu(w, inp, fused=fused, backward=not w.fwd_only)
    bf = w.dtype == "bf16"
    rel = BF16_REL if bf else F32_REL
    exact, f = oracle_problem(w, inp, round_bf16=False)
    rb, _ = oracle_problem(w, inp, round_bf16=bf)
    wts, C = None, {}
    if bf and w.act != "none":
        dump = exact.hidden_dump(f["dy"])
        wts = rounding_weights(w, rb.hidden_dump(f["dy"]))
        C = chain_noise(w, f, dump)
    A = allowance_rows(w, f, wts) if wts is not None else {}
    W = allowance_wgrad(w, f, wts, np.arange(w.d), np.arange(w.d)) if wts is not None and not w.fwd_only else {}
    sh = rb.forward_sharded()
    check(got["y"], sh["y"], rel, f"{w.name} y", A.get("y"))
    check(got["y"], exact.forward_sharded()["y"], rel, f"{w.name} y vs float64 chain", C.get("y"))
    if got["partials"] is not None:
        check(got["partials"], sh["partials"], F32_REL, f"{w.name} partials", A.get("partials"))
    if w.fwd_only:
        return
    g = rb.backward_full(f["dy"])
    check(got["dx"], g["dx"], rel, f"{w.name} dx", A.get("dx"))
    check(got["dx"], exact.backward_rows(f["dy"])["dx"], rel, f"{w.name} dx vs float64 chain", C.get("dx"))
    check(got["dW2"], g["dW2"], rel, f"{w.name} dW2", W.get("dW2"))
    if w.act != "none":
        check(got["dW1"], g["dW1"], rel, f"{w.name} dW1", W.get("dW1"))
    if w.act == "swiglu":
        check(got["dW3"], g["dW3"], rel, f"{w.name} dW3", W.get("dW3"))
    if w.bias:
        check(got["db2"], g["db2"], rel, f"{w.name} db2")
        if w.act == "gelu_tanh":
            check(got["db1"], g["db1"], rel, f"{w.name} db1", W.get("db1"))
    if got["dx_partials"] is not None:
        check(got["dx_partials"], g["dx_partials"], F32_REL, f"{w.name} dx partials", A.get("dx_partials"))


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
def test_tiny_fp32_workload(fused):
    _full_compare(WORKLOADS["tiny_gelu_fp32"], fused)


SMALL = [
    # ragged on every axis: 333 tokens (M tail), d = 264 (K tail), s = 200
    small_case(333, 264, 600, 3, "gelu_tanh", bias=True, seed=101),
    small_case(333, 264, 600, 3, "swiglu", seed=102),          # s = 200 -> padded to 256
    small_case(200, 256, 768, 4, "swiglu", seed=103),          # two 128-blocks per shard
    small_case(130, 128, 264, 11, "gelu_tanh", seed=104),      # TP11, s = 24
    small_case(257, 192, 384, 1, "gelu_tanh", bias=True, seed=105),  # TP1 = dense
    small_case(1, 64, 256, 2, "swiglu", seed=106),             # a single token
    small_case(300, 136, 96, 2, "gelu_tanh", bias=True, seed=107),   # s = 48 < one tile
    small_case(520, 192, 900, 3, "swiglu", seed=108),          # s = 300 -> 384: the second N tile half empty
    small_case(32, 256, 1536, 4, "swiglu", seed=109),          # decode-sized: 32-row A tiles
    small_case(17, 200, 600, 3, "swiglu", seed=110),           # decode-sized, ragged: 17 of 32 rows
    small_case(17, 2048, 3072, 3, "swiglu", seed=112),         # decode-sized up GEMM split in two K parts
    small_case(1, 2048, 3072, 3, "swiglu", seed=113),          # one token through the K split
]
# The K split is taken when it spreads the up GEMM's weight tiles over clearly
# more SMs: with 3 x 8 = 24 tiles it doubles the SMs in use on any GPU of up to
# several hundred SMs, so these two cases exercise it on every GB300.
KSPLIT = [w for w in SMALL if w.N <= 32 and w.d >= 2048]


@pytest.mark.parametrize("w", KSPLIT, ids=[w.name for w in KSPLIT])
def test_decode_ksplit_is_taken(w):
    """The decode-sized cases above really run the split up GEMM and the
    SwiGLU combine kernel (the launch records name it)."""
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    g = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    for fused in (False, True):
        ffn.forward(g["x"], w13p, w2p, fused=fused, flags=abi.TP_FLAG_TIMING)
        names = [n for n, _ in abi.tp_ffn_kernel_times(ffn.plan, 1000)]
        assert names[:2] == ["up_swiglu", "swiglu_combine"], names


# Pre-activations driven into the tails of the activation functions: x ~
# N(0, 16^2) puts z (or a and g) at |z| up to ~70 on both signs, where tanh
# saturates, the z^3 term dominates and gelu', silu' are formed from
# cancelling terms; a large b1 holds a hidden unit's z deep in one tail for
# every token; x ~ N(0, 48^2) takes |a| past 88, where e^-a overflows in fp32.
# Every output of both sum modes is compared element by element.
TAILS = [
    small_case(300, 256, 768, 3, "gelu_tanh", seed=701, x_std=16.0),
    small_case(300, 256, 768, 3, "gelu_tanh", bias=True, seed=702, b_std=16.0),
    small_case(300, 256, 768, 3, "swiglu", seed=703, x_std=16.0),
    small_case(300, 256, 768, 3, "swiglu", seed=704, x_std=48.0),
    small_case(17, 2048, 3072, 3, "swiglu", seed=705, x_std=16.0),       # through the decode K split
    small_case(40, 64, 256, 2, "gelu_tanh", dtype="f32", seed=706, x_std=16.0),   # the fp32 (SIMT) path
]


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", TAILS, ids=[w.name for w in TAILS])
def test_activation_tails_against_full_oracle(w, fused):
    _full_compare(w, fused)


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_bf16_against_full_oracle(w, fused):
    _full_compare(w, fused)


# Up to 256 pair tiles per GEMM (2048 tokens, d 512, d_ff 4096, T_p 4): the
# two-CTA clusters of the persistent GEMM take several tiles in turn, so the
# second tensor-memory accumulator, its empty / full hand-over and the
# backward epilogue's look-ahead copy into the next tile are all compared
# element by element (the other small cases fit one tile per cluster).
MANY_TILES = small_case(2048, 512, 4096, 4, "swiglu", seed=111)


def test_many_tiles_per_cluster_against_full_oracle():
    _full_compare(MANY_TILES, True)


# Weight-gradient GEMMs with few output tiles split their K (token) axis in
# two fp32 parts, summed in part order: 2100 tokens = 33 K blocks of 64 (17 +
# 16, the last one ragged); M = 264 leaves the second 256-row tile pair
# nearly empty; GELU with biases and SwiGLU both split both weight GEMMs.
WGRAD_SPLIT = [small_case(2100, 256, 1024, 4, "gelu_tanh", bias=True, seed=114),
               small_case(2500, 264, 600, 3, "swiglu", seed=115)]


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", WGRAD_SPLIT, ids=[w.name for w in WGRAD_SPLIT])
def test_wgrad_ksplit_against_full_oracle(w, fused):
    _full_compare(w, fused)


@pytest.mark.parametrize("w", WGRAD_SPLIT + [MANY_TILES], ids=[w.name for w in WGRAD_SPLIT + [MANY_TILES]])
def test_wgrad_ksplit_is_taken(w):
    """The cases above run their weight-gradient GEMMs as K parts: the launch
    records name the part sums right after each split GEMM."""
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    g = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    _, saved, _ = ffn.forward(g["x"], w13p, w2p, g["b1"], g["b2"], fused=True)
    ffn.backward(g["x"], w13p, w2p, saved, g["dy"], fused=True, bias=w.bias, flags=abi.TP_FLAG_TIMING)
    names = [n for n, _ in abi.tp_ffn_kernel_times(ffn.plan, 1000)]
    wg1 = "wgrad_w13" if w.act == "swiglu" else "wgrad_w1"
    assert "wgrad_w2" in names and names[names.index("wgrad_w2") + 1] == "wgrad_w2_ksum", names
    if w is not MANY_TILES:  # 64 tiles of 2048 x 512 already fill the SM pairs
        assert names[names.index(wg1) + 1] == wg1 + "_ksum", names


# Fused-sum forwards whose output tiles leave the last wave of SM pairs at
# most half full run those tiles as K parts (fp32), summed in part order by a
# fix-up kernel: 6 tiles of 4 parts (GELU with biases, ragged rows), 6 tiles
# of 3 unequal parts (9, 9 and 10 of 28 K blocks) and 9 tiles of 3 parts
# (SwiGLU, ragged rows and d).
TAIL_SPLIT = [small_case(700, 512, 2048, 2, "gelu_tanh", bias=True, seed=116),
              small_case(700, 512, 1792, 7, "gelu_tanh", bias=True, seed=118),
              small_case(600, 760, 1536, 4, "swiglu", seed=117)]
# The up GEMMs take the same split (the fix-up adds b1 and applies GELU, or
# forms silu(a) g, and writes h and the saved activations): 18 GELU tiles and
# 36 SwiGLU tiles (ragged rows, d and hidden units) of 2 parts here, and the
# down GEMMs' 12 tiles 3 parts.
TAIL_SPLIT_UP = [small_case(600, 1024, 1536, 3, "gelu_tanh", bias=True, seed=121),
                 small_case(530, 1000, 1500, 3, "swiglu", seed=122)]


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", TAIL_SPLIT_UP, ids=[w.name for w in TAIL_SPLIT_UP])
def test_tail_split_up_against_full_oracle(w, fused):
    _full_compare(w, fused)


@pytest.mark.parametrize("w", TAIL_SPLIT, ids=[w.name for w in TAIL_SPLIT])
def test_tail_split_against_full_oracle(w):
    _full_compare(w, True)


@pytest.mark.parametrize("w", TAIL_SPLIT_UP, ids=[w.name for w in TAIL_SPLIT_UP])
def test_tail_split_up_is_taken(w):
    """Both GEMMs of the cases above split their last wave: the fix-up
    follows each in the launch records."""
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    g = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    ffn.forward(g["x"], w13p, w2p, g["b1"], g["b2"], fused=True, flags=abi.TP_FLAG_TIMING)
    names = [n for n, _ in abi.tp_ffn_kernel_times(ffn.plan, 1000)]
    up = "up_gelu" if w.act == "gelu_tanh" else "up_swiglu"
    assert names == [up, "tail_fixup", "down_fused_sum", "tail_fixup"], names


@pytest.mark.parametrize("w", TAIL_SPLIT + [MANY_TILES], ids=[w.name for w in TAIL_SPLIT + [MANY_TILES]])
def test_tail_split_is_taken(w):
    """The fused forward's down GEMM of the cases above splits its last wave:
    the launch records name the fix-up right after it."""
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    dev = torch.device("cuda", 0)
    g = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(w).items()}
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, w.act, "bf16", device=dev)
    w13p, w2p = ffn.pack(g["W1"], g["W2"], g["W3"])
    ffn.forward(g["x"], w13p, w2p, g["b1"], g["b2"], fused=True, flags=abi.TP_FLAG_TIMING)
    names = [n for n, _ in abi.tp_ffn_kernel_times(ffn.plan, 1000)]
    assert names[names.index("down_fused_sum") + 1:] == ["tail_fixup"], names


def _sweep_cases(n=10, seed=20261202):
    """Seeded random shapes across both kernel paths (token counts of at most
    32, under 256 and above), both activations, biases on or off, ragged
    d and hidden widths (multiples of 8), and T_p from 1 to 8."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        N = int(rng.choice([rng.integers(1, 33), rng.integers(33, 256), rng.integers(256, 700)]))
        d = 8 * int(rng.integers(1, 41))
        T = int(rng.choice([1, 2, 3, 4, 5, 8]))
        s = 8 * int(rng.integers(1, 41))
        act = "swiglu" if i % 2 else "gelu_tanh"
        bias = act == "gelu_tanh" and bool(rng.integers(0, 2))
        out.append(small_case(N, d, s * T, T, act, bias=bias, seed=300 + i))
    return out


SWEEP = _sweep_cases()


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", SWEEP, ids=[w.name for w in SWEEP])
def test_seeded_shape_sweep_against_full_oracle(w, fused):
    _full_compare(w, fused)


def _attn_case(N, d_model, n_heads, head_dim, T_p, seed):
    return Workload(f"attn_out_{N}x{d_model}_h{n_heads}x{head_dim}_tp{T_p}", N, d_model, n_heads * head_dim, T_p,
                    "none", "bf16", seed_index=seed, n_heads=n_heads, n_kv_heads=n_heads, head_dim=head_dim)


ATTN = [_attn_case(200, 256, 6, 64, 3, 201), _attn_case(77, 136, 8, 16, 4, 202)]


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("w", ATTN, ids=[w.name for w in ATTN])
def test_attention_out_projection_against_full_oracle(w, fused):
    _full_compare(w, fused)


def test_empty_token_batch_is_a_no_op():
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    rc, plan = abi.tp_ffn_plan_create(64, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_BF16)
    assert rc == abi.TP_OK
    try:
        assert abi.tp_ffn_fwd(plan, 0, None, None, None, None, None, None, None, None, None, 0, 0) == abi.TP_OK
        assert abi.tp_ffn_last_launch_count(plan) == 0
        assert abi.tp_ffn_bwd(plan, 0, *([None] * 12), 0, 0) == abi.TP_OK
    finally:
        abi.tp_ffn_plan_destroy(plan)


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_pack_layout_and_roundtrip_bit_exact(act):
    """Packing is byte work: compare bit for bit with the layout of tpffn.h."""
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    w = small_case(8, 72, 3 * 200, 3, act, seed=301)
    inp = make_inputs(w)
    dev = torch.device("cuda", 0)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, act, "bf16", device=dev)
    W1, W2 = inp["W1"].to(dev), inp["W2"].to(dev)
    W3 = inp["W3"].to(dev) if act == "swiglu" else None
    w13p, w2p = ffn.pack(W1, W2, W3)
    s, sp, d, T = ffn.info["s"], ffn.info["s_pad"], w.d, w.T_p
    cols = w13p.view(torch.bfloat16).cpu().view(torch.int16)
    rows = w2p.view(torch.bfloat16).cpu().view(torch.int16).reshape(T, d, sp)
    W1i, W2i = inp["W1"].view(torch.int16), inp["W2"].view(torch.int16)
    for t in range(T):
        assert torch.equal(rows[t, :, :s], W2i[:, t * s:(t + 1) * s])
        assert not rows[t, :, s:].any()
    if act == "swiglu":
        W3i = inp["W3"].view(torch.int16)
        c = cols.reshape(T, sp // 128, 2, 128, d)
        for t in range(T):
            for j in range(sp):
                blk, r = divmod(j, 128)
                if j < s:
                    assert torch.equal(c[t, blk, 0, r], W1i[t * s + j])
                    assert torch.equal(c[t, blk, 1, r], W3i[t * s + j])
                else:
                    assert not c[t, blk, :, r].any()
    else:
        c = cols.reshape(T, sp, d)
        for t in range(T):
            assert torch.equal(c[t, :s], W1i[t * s:(t + 1) * s])
    U1, U3 = ffn.unpack_columns(w13p)
    assert torch.equal(U1.cpu().view(torch.int16), W1i)
    if act == "swiglu":
        assert torch.equal(U3.cpu().view(torch.int16), inp["W3"].view(torch.int16))
    assert torch.equal(ffn.unpack_rows(w2p).cpu().view(torch.int16), W2i)


@pytest.mark.parametrize("fused", [False, True], ids=["standalone", "fused"])
@pytest.mark.parametrize("case", ["ragged", "tail_split"])
def test_bitwise_reproducible_run_to_run(fused, case):
    # tail_split: both forward GEMMs sum their last wave's K parts in a fix-up
    w = small_case(333, 264, 600, 3, "swiglu", seed=401) if case == "ragged" else TAIL_SPLIT_UP[1]
    inp = make_inputs(w)
    a = run_gpu(w, inp, fused=fused)["_raw"]
    b = run_gpu(w, inp, fused=fused)["_raw"]
    for k, v in a.items():
        if v is not None:
            assert torch.equal(v.view(torch.uint8) if v.dtype != torch.float32 else v.view(torch.int32),
                               b[k].view(torch.uint8) if v.dtype != torch.float32 else b[k].view(torch.int32)), k


def test_bounded_wait_expires_and_context_survives():
    """The test hook makes the first GEMM's producer skip a load; the waiting
    MMA and epilogue warps give up after their time limit, the call reports
    TP_ERR_TIMEOUT, and the next call on the same context is correct."""
    from megatron_tensor_transformer_w1_gb300 import tpffn as abi
    from megatron_tensor_transformer_w1_gb300.ffn import TensorParallelFFN
    w = small_case(64, 128, 256, 2, "gelu_tanh", seed=501)
    inp = make_inputs(w)
    dev = torch.device("cuda", 0)
    ffn = TensorParallelFFN(w.d, w.d_ff, w.T_p, "gelu_tanh", "bf16", device=dev)
    g = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    w13p, w2p = ffn.pack(g["W1"], g["W2"])
    y = torch.empty(w.N, w.d, dtype=torch.bfloat16, device=dev)
    ws = ffn.workspace(w.N)
    rc = abi.tp_ffn_fwd(ffn.plan, w.N, g["x"], w13p, w2p, None, None, y, None, None, ws, ws.numel(),
                        abi.TP_FLAG_SYNC | abi.TP_FLAG_DEBUG_SKIP_LOAD, torch.cuda.current_stream())
    assert rc == abi.TP_ERR_TIMEOUT
    assert abi.tp_ffn_last_device_error(ffn.plan, ws, torch.cuda.current_stream()) == abi.TP_ERR_TIMEOUT
    rc = abi.tp_ffn_fwd(ffn.plan, w.N, g["x"], w13p, w2p, None, None, y, None, None, ws, ws.numel(),
                        abi.TP_FLAG_SYNC, torch.cuda.current_stream())
    assert rc == abi.TP_OK
    rb, _ = oracle_problem(w, inp, round_bf16=True)
    check(y.double().cpu().numpy(), rb.forward_sharded()["y"], BF16_REL, "y after timeout")


OVERLAP = [small_case(700, 264, 600, 3, "swiglu", seed=601),             # 3 token chunks of 256 (+ a ragged one)
           small_case(1300, 192, 768, 4, "gelu_tanh", bias=True, seed=602),
           _attn_case(600, 256, 6, 64, 3, 603)]


@pytest.mark.parametrize("w", OVERLAP, ids=[w.name for w in OVERLAP])
def test_overlapped_shard_sum_matches_oracle_and_is_bit_identical(w):
    """TP_SUM_OVERLAP: the chunked GEMM + second-stream sum gives exactly the
    standalone path's bits, and matches the oracle."""
    inp = make_inputs(w)
    ov = run_gpu(w, inp, overlap=True)["_raw"]
    st = run_gpu(w, inp, overlap=False)["_raw"]
    for k in ("y", "partials", "dx", "dx_partials"):
        if st.get(k) is not None:
            assert torch.equal(ov[k].view(torch.uint8), st[k].view(torch.uint8)), k
    _full_compare_overlap(w, inp)


def _full_compare_overlap(w, inp):
    got = run_gpu(w, inp, overlap=True)
    rb, f = oracle_problem(w, inp, round_bf16=True)
    wts = rounding_weights(w, rb.hidden_dump(f["dy"])) if w.act != "none" else None
    A = allowance_rows(w, f, wts) if wts is not None else {}
    check(got["y"], rb.forward_sharded()["y"], BF16_REL, f"{w.name} overlap y", A.get("y"))
    check(got["dx"], rb.backward_rows(f["dy"])["dx"], BF16_REL, f"{w.name} overlap dx", A.get("dx"))
