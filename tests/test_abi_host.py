"""Host-side checks of the C ABI (no GPU needed): the library loads and exports
every function include/tpffn.h declares, and argument validation returns the
documented status codes before any device work is enqueued."""
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpffn.h")


@pytest.fixture(scope="module")
def abi():
    from megatron_tensor_transformer_w1_gb300 import build
    build.build()
    from megatron_tensor_transformer_w1_gb300 import tpffn
    return tpffn


def test_library_exports_every_declared_symbol(abi):
    declared = set(re.findall(r"TPFFN_API\s+[\w\s\*]+?\b(tp_\w+)\s*\(", open(HEADER).read()))
    assert declared == set(abi.ABI_FUNCTIONS), declared ^ set(abi.ABI_FUNCTIONS)
    for name in declared:
        assert hasattr(abi._lib, name), name


def test_plan_validation(abi):
    ok = abi.TP_OK
    assert abi.tp_ffn_plan_create(4096, 14336, 8, abi.TP_ACT_SWIGLU, abi.TP_BF16)[0] == ok
    assert abi.tp_ffn_plan_create(64, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_F32)[0] == ok
    assert abi.tp_ffn_plan_create(64, 250, 3, abi.TP_ACT_GELU_TANH, abi.TP_BF16)[0] == abi.TP_ERR_INVALID
    assert abi.tp_ffn_plan_create(0, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_BF16)[0] == abi.TP_ERR_INVALID
    assert abi.tp_ffn_plan_create(64, 256, 0, abi.TP_ACT_GELU_TANH, abi.TP_BF16)[0] == abi.TP_ERR_INVALID
    assert abi.tp_ffn_plan_create(64, 256, 2, 7, abi.TP_BF16)[0] == abi.TP_ERR_INVALID
    assert abi.tp_ffn_plan_create(64, 256, 2, abi.TP_ACT_GELU_TANH, 9)[0] == abi.TP_ERR_INVALID
    # the 16-byte row rule of the tensor-memory-access unit (bf16 only)
    assert abi.tp_ffn_plan_create(66, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_BF16)[0] == abi.TP_ERR_UNSUPPORTED
    assert abi.tp_ffn_plan_create(66, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_F32)[0] == ok


def test_gqa_divisibility_golden(abi):
    spec = json.load(open(os.path.join(ROOT, "tests", "golden", "gqa_divisibility.json")))
    for c in spec["cases"]:
        rc, plan = abi.tp_attn_out_plan_create(3072, c["n_heads"], c["n_kv_heads"], 128, c["T_p"], abi.TP_BF16)
        assert (rc == abi.TP_OK) == c["valid"], c
        if plan:
            info = abi.tp_ffn_plan_info(plan)
            assert info["act"] == abi.TP_ACT_NONE and info["d_ff"] == c["n_heads"] * 128
            abi.tp_ffn_plan_destroy(plan)


@pytest.mark.parametrize("act,mats", [("gelu", 1), ("swiglu", 2)])
def test_per_shard_weight_bytes_are_one_over_tp(abi, act, mats):
    """'7.9 Tensor and pipeline parallelism (TP, PP)', §2.3: per-device weights
    are 1/T_p of the original (exactly, when no shard needs padding)."""
    a = abi.TP_ACT_SWIGLU if act == "swiglu" else abi.TP_ACT_GELU_TANH
    for T in (1, 2, 4, 8):
        rc, p = abi.tp_ffn_plan_create(4096, 14336, T, a, abi.TP_BF16)
        assert rc == abi.TP_OK
        cols = abi.tp_ffn_packed_bytes(p, abi.TP_PACK_COLUMNS)
        rows = abi.tp_ffn_packed_bytes(p, abi.TP_PACK_ROWS)
        assert cols == mats * 14336 * 4096 * 2 and rows == 14336 * 4096 * 2
        assert cols % T == 0 and rows % T == 0  # each shard holds exactly 1/T_p
        abi.tp_ffn_plan_destroy(p)


def test_call_validation_without_device_work(abi):
    rc, p = abi.tp_ffn_plan_create(64, 256, 2, abi.TP_ACT_GELU_TANH, abi.TP_BF16)
    assert rc == abi.TP_OK
    try:
        n = 16
        ws_need = abi.tp_ffn_workspace_bytes(p, n, 0)
        assert ws_need > 0 and abi.tp_ffn_saved_bytes(p, n) > 0
        A = 1 << 20  # a 16-byte-aligned address; never dereferenced on these paths
        fwd = lambda **kw: abi.tp_ffn_fwd(p, kw.get("n", n), kw.get("x", A), kw.get("w13p", A), kw.get("w2p", A),
                                          kw.get("b1"), None, kw.get("y", A), kw.get("partials"), None,
                                          kw.get("ws", A), kw.get("wsb", ws_need), kw.get("flags", 0))
        assert fwd(x=None) == abi.TP_ERR_INVALID
        assert fwd(w13p=None) == abi.TP_ERR_INVALID
        assert fwd(y=None) == abi.TP_ERR_INVALID
        assert fwd(ws=None) == abi.TP_ERR_INVALID
        assert fwd(n=-1) == abi.TP_ERR_INVALID
        assert fwd(partials=A, flags=abi.TP_SUM_FUSED) == abi.TP_ERR_INVALID
        assert fwd(wsb=ws_need - 1) == abi.TP_ERR_INVALID
        assert fwd(x=A + 2) == abi.TP_ERR_ALIGN
        assert fwd(ws=A + 8) == abi.TP_ERR_ALIGN
        assert abi.tp_ffn_bwd(p, n, A, A, A, None, A, A, None, A, A, None, None, A, ws_need, 0) == \
            abi.TP_ERR_INVALID  # saved is required for an activation
        assert abi.tp_ffn_shard_columns(p, None, None, A) == abi.TP_ERR_INVALID
        assert abi.tp_ffn_shard_rows(p, A, None) == abi.TP_ERR_INVALID
        assert abi.tp_ffn_last_device_error(None, A) == abi.TP_ERR_INVALID
        assert abi.tp_ffn_kernel_times(None) == []
    finally:
        abi.tp_ffn_plan_destroy(p)
    rc, s = abi.tp_ffn_plan_create(64, 256, 2, abi.TP_ACT_SWIGLU, abi.TP_BF16)
    try:
        A = 1 << 20
        ws = abi.tp_ffn_workspace_bytes(s, 8, 0)
        # biases of the first matrix are supported for the GELU form only
        assert abi.tp_ffn_fwd(s, 8, A, A, A, A, None, A, None, None, A, ws, 0) == abi.TP_ERR_UNSUPPORTED
        assert abi.tp_ffn_shard_columns(s, A, None, A) == abi.TP_ERR_INVALID  # W3 missing
    finally:
        abi.tp_ffn_plan_destroy(s)


def test_status_strings(abi):
    for code in range(6):
        assert abi.tp_ffn_status_string(code).startswith("TP_")
    assert abi.tp_ffn_status_string(99) == "unknown status"


def test_static_scratch_limit_and_decode_split_workspace(abi):
    """The header's example: for the Llama-3-70B-shaped decode FFN the static
    scratch serves up to 76 tokens and refuses more.  Decode-sized SwiGLU
    calls (at most 32 tokens) also hold two fp32 K parts of the up GEMM
    (T_p x n x 2 s_pad floats each) in their workspace, and still fit."""
    rc, plan = abi.tp_ffn_plan_create(8192, 28672, 8, abi.TP_ACT_SWIGLU, abi.TP_BF16)
    assert rc == abi.TP_OK
    try:
        ws = lambda n: abi.tp_ffn_workspace_bytes(plan, n, abi.TP_SUM_STANDALONE)
        lim = abi.TPFFN_STATIC_SCRATCH_BYTES
        assert all(ws(n) <= lim for n in range(1, 77))
        assert ws(77) > lim
        parts = 2 * 8 * 32 * (2 * 3584) * 4
        # at 32 tokens the parts are there; at 33 (no split) they are not
        assert ws(32) - ws(33) * 32 / 33 > 0.9 * parts
    finally:
        abi.tp_ffn_plan_destroy(plan)
