"""float64 CPU oracle for the Megatron tensor-parallel FFN sublayer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It
shares no code with the CUDA library under ``megatron_tensor_transformer_w1_gb300``
and never imports it.

The arithmetic lives in ``tpffn_oracle.c`` (plain loops, float64); this module
only compiles it with gcc on first use and marshals numpy arrays.  The forms it
computes are stated in that file's header:

* the dense FFN and its explicitly column/row-sharded form with the rank-ordered
  shard-sum ("7.9 Tensor and pipeline parallelism (TP, PP)", §2.1 "The FFN,
  sharded"; SwiGLU per "S17 Tensor & Pipeline Parallelism", listing "the
  megatron pattern");
* the backward by the chain rule, with the dx shard-sum (the f operator of §2.1);
* the row-parallel attention output projection (§2.2 "Attention, sharded"),
  as activation NONE;
* the whole head-sharded attention sublayer of §2.2 (column-sharded Q/K/V with
  the GQA divisibility rule of "S17 Tensor & Pipeline Parallelism", the scaled
  dot-product attention of each head, the row-sharded W_O with the ordered
  shard-sum) and its backward, and the attention core alone (``AttentionCore``).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tpffn_oracle.c")
_LIB = os.path.join(_HERE, f"liboracle-{platform.machine()}.so")
_lock = threading.Lock()
_lib = None

ACT_NONE = 0
ACT_GELU_TANH = 1
ACT_SWIGLU = 2
ACT_IDENTITY = 3  # oracle-only: sigma = identity, for the linear special case

ACT_BY_NAME = {"none": ACT_NONE, "gelu_tanh": ACT_GELU_TANH, "swiglu": ACT_SWIGLU,
               "identity": ACT_IDENTITY}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over independent outputs only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Ffn(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("d", ctypes.c_int64), ("d_ff", ctypes.c_int64),
                ("T_p", ctypes.c_int), ("act", ctypes.c_int), ("round_bf16", ctypes.c_int),
                ("x", ctypes.c_void_p), ("W1", ctypes.c_void_p), ("W3", ctypes.c_void_p),
                ("b1", ctypes.c_void_p), ("W2", ctypes.c_void_p), ("b2", ctypes.c_void_p)]


def load_library(path):
    """Load an oracle shared object (the default one, or a test's variant)."""
    lib = ctypes.CDLL(path)
    for name in ("orc_gelu_tanh", "orc_gelu_tanh_grad", "orc_silu", "orc_silu_grad",
                         "orc_round_bf16", "orc_sigmoid"):
        f = getattr(lib, name)
        f.restype = ctypes.c_double
        f.argtypes = [ctypes.c_double]
    lib.orc_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f64(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int64)


class FFN:
    """One FFN problem: the float64 values the oracle computes with.

    x  : [N, d] (act "none": [N, d_ff], the concatenated head outputs)
    W1, W3 : [d_ff, d]   W2 : [d, d_ff]   b1 : [d_ff]   b2 : [d]
    round_bf16 : round the stored activations to bf16 (see tpffn_oracle.c).
    """

    def __init__(self, x, W2, T_p, act, W1=None, W3=None, b1=None, b2=None, round_bf16=False,
                 lib=None):
        self._lib = lib
        self.act = ACT_BY_NAME[act] if isinstance(act, str) else int(act)
        self.x = _f64(x)
        self.W1, self.W3, self.W2 = _f64(W1), _f64(W3), _f64(W2)
        self.b1, self.b2 = _f64(b1), _f64(b2)
        self.N = self.x.shape[0]
        self.d = self.W2.shape[0]
        self.d_ff = self.W2.shape[1]
        self.T_p = int(T_p)
        if self.d_ff % self.T_p:
            raise ValueError("d_ff must be divisible by T_p")
        if self.act == ACT_NONE:
            assert self.x.shape == (self.N, self.d_ff)
        else:
            assert self.x.shape == (self.N, self.d) and self.W1.shape == (self.d_ff, self.d)
        if self.act == ACT_SWIGLU:
            assert self.W3 is not None and self.W3.shape == (self.d_ff, self.d)
        self.round_bf16 = bool(round_bf16)
        self._s = _Ffn(self.N, self.d, self.d_ff, self.T_p, self.act, int(self.round_bf16),
                       _ptr(self.x), _ptr(self.W1), _ptr(self.W3), _ptr(self.b1),
                       _ptr(self.W2), _ptr(self.b2))

    def lib(self):
        return self._lib if self._lib is not None else _load()

    @property
    def d_in(self):
        return self.d_ff if self.act == ACT_NONE else self.d

    def _rows(self, rows):
        if rows is None:
            return self.N, None
        rows = _i64(rows)
        assert rows.min() >= 0 and rows.max() < self.N
        return len(rows), rows

    # ------------------------------------------------------------- forward
    def forward_dense(self, rows=None, want_h=False):
        lib = self.lib()
        n, r = self._rows(rows)
        y = np.zeros((n, self.d))
        h = np.zeros((n, self.d_ff)) if want_h else None
        lib.orc_ffn_forward_dense(ctypes.byref(self._s), ctypes.c_int64(n), _ptr(r), _ptr(y), _ptr(h))
        return (y, h) if want_h else y

    def forward_sharded(self, rows=None):
        """Returns dict(y, partials [T_p, n, d], h [n, d_ff], z_saved, ag_saved)."""
        lib = self.lib()
        n, r = self._rows(rows)
        y = np.zeros((n, self.d))
        part = np.zeros((self.T_p, n, self.d))
        h = np.zeros((n, self.d_ff))
        z = np.zeros((n, self.d_ff))
        ag = np.zeros((n, 2, self.d_ff))
        lib.orc_ffn_forward_sharded(ctypes.byref(self._s), ctypes.c_int64(n), _ptr(r),
                                    _ptr(part), _ptr(y), _ptr(h), _ptr(z), _ptr(ag))
        return dict(y=y, partials=part, h=h, z_saved=z, ag_saved=ag)

    def forward_rowsplit_bad(self):
        lib = self.lib()
        y = np.zeros((self.N, self.d))
        lib.orc_ffn_forward_rowsplit_bad(ctypes.byref(self._s), _ptr(y))
        return y

    # ------------------------------------------------------------ backward
    def backward_rows(self, dy, rows=None):
        """Returns dict(dx [n, d_in], dx_partials [T_p, n, d] (not for NONE))."""
        lib = self.lib()
        dy = _f64(dy)
        assert dy.shape == (self.N, self.d)
        n, r = self._rows(rows)
        dx = np.zeros((n, self.d_in))
        part = None if self.act == ACT_NONE else np.zeros((self.T_p, n, self.d))
        lib.orc_ffn_backward_rows(ctypes.byref(self._s), _ptr(dy), ctypes.c_int64(n), _ptr(r),
                                  _ptr(part), _ptr(dx))
        return dict(dx=dx, dx_partials=part)

    def backward_dense_dx(self, dy):
        lib = self.lib()
        dy = _f64(dy)
        dx = np.zeros((self.N, self.d))
        lib.orc_ffn_backward_dense_dx(ctypes.byref(self._s), _ptr(dy), _ptr(dx))
        return dx

    def wgrad_entries(self, dy, js, ks=None, cs=None):
        """Gradient entries: dW1[js][:, ks], dW3[js][:, ks], dW2[cs][:, js],
        db1[js], db2[cs].  ks is ignored for act NONE."""
        lib = self.lib()
        dy = _f64(dy)
        js = _i64(js)
        ks = _i64(ks if ks is not None else np.zeros(0))
        cs = _i64(cs if cs is not None else np.zeros(0))
        nj, nk, nc = len(js), len(ks), len(cs)
        out = dict(dW1=np.zeros((nj, nk)), dW3=np.zeros((nj, nk)), dW2=np.zeros((nc, nj)),
                   db1=np.zeros(nj), db2=np.zeros(nc))
        lib.orc_ffn_wgrad_entries(ctypes.byref(self._s), _ptr(dy),
                                  ctypes.c_int64(nj), _ptr(js), ctypes.c_int64(nk), _ptr(ks),
                                  ctypes.c_int64(nc), _ptr(cs),
                                  _ptr(out["dW1"]), _ptr(out["dW3"]), _ptr(out["dW2"]),
                                  _ptr(out["db1"]), _ptr(out["db2"]))
        return out

    DUMP_PLANES = ("h_pre", "z_pre", "g_pre", "dh", "dz_pre", "dg_pre", "nz", "ng", "ndh")

    def hidden_dump(self, dy=None, rows=None, cols=None):
        """Stored hidden quantities at (rows x cols) before bf16 rounding, with
        the exact dh and the L2 norms of the producing dot products; a dict of
        [n_rows, n_cols] arrays keyed by DUMP_PLANES (see tpffn_oracle.c)."""
        lib = self.lib()
        n, r = self._rows(rows)
        if cols is None:
            nc, c = self.d_ff, None
        else:
            c = _i64(cols)
            nc = len(c)
        out = np.zeros((len(self.DUMP_PLANES), n, nc))
        dyp = None
        if dy is not None:
            dyp = _f64(dy)
            assert dyp.shape == (self.N, self.d)
        lib.orc_ffn_hidden_dump(ctypes.byref(self._s), _ptr(dyp), ctypes.c_int64(n), _ptr(r),
                                ctypes.c_int64(nc), _ptr(c), _ptr(out))
        return dict(zip(self.DUMP_PLANES, out))

    def backward_full(self, dy):
        """All gradients in full (small problems only)."""
        js = np.arange(self.d_ff)
        ks = np.arange(self.d) if self.act != ACT_NONE else None
        cs = np.arange(self.d)
        w = self.wgrad_entries(dy, js, ks, cs)
        b = self.backward_rows(dy)
        w.update(b)
        return w


class _AttnCore(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("S", ctypes.c_int64), ("H", ctypes.c_int64),
                ("Hkv", ctypes.c_int64), ("hd", ctypes.c_int64), ("causal", ctypes.c_int),
                ("round_bf16", ctypes.c_int)]


class _Attn(ctypes.Structure):
    _fields_ = [("core", _AttnCore), ("d", ctypes.c_int64), ("T_p", ctypes.c_int),
                ("x", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("Wk", ctypes.c_void_p),
                ("Wv", ctypes.c_void_p), ("Wo", ctypes.c_void_p)]


class AttentionCore:
    """Scaled dot-product attention of B sequences of S tokens, H query heads
    of width hd reading Hkv key/value heads (query head h reads h // (H/Hkv)).

    q, o : [B*S, H*hd]   k, v : [B*S, Hkv*hd]   (token rows, head columns)
    """

    def __init__(self, B, S, H, Hkv, hd, causal=True, round_bf16=False, lib=None):
        if H % Hkv:
            raise ValueError("H must be a multiple of Hkv")
        self.B, self.S, self.H, self.Hkv, self.hd = int(B), int(S), int(H), int(Hkv), int(hd)
        self.causal, self.round_bf16 = bool(causal), bool(round_bf16)
        self._lib = lib
        self._s = _AttnCore(self.B, self.S, self.H, self.Hkv, self.hd, int(self.causal), int(self.round_bf16))

    def lib(self):
        return self._lib if self._lib is not None else _load()

    def forward(self, q, k, v):
        """Returns (o [B*S, H*hd], lse [B, H, S])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        n = self.B * self.S
        assert q.shape == (n, self.H * self.hd) and k.shape == v.shape == (n, self.Hkv * self.hd)
        o = np.empty((n, self.H * self.hd))
        lse = np.empty((self.B, self.H, self.S))
        self.lib().orc_attn_core_fwd(ctypes.byref(self._s), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse))
        return o, lse

    def backward(self, q, k, v, dO):
        """Returns (dq, dk, dv)."""
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        self.lib().orc_attn_core_bwd(ctypes.byref(self._s), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq),
                                     _ptr(dk), _ptr(dv))
        return dq, dk, dv

    def allowance(self, q, k, v, dO, u):
        """Per-element rounding allowances (a_o, a_dq, a_dk, a_dv) of a bf16
        computation of this core; see orc_attn_core_allowance."""
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        out = [np.empty_like(q), np.empty_like(q), np.empty_like(k), np.empty_like(v)]
        self.lib().orc_attn_core_allowance(ctypes.byref(self._s), _ptr(q), _ptr(k), _ptr(v), _ptr(dO),
                                           ctypes.c_double(u), *[_ptr(a) for a in out])
        return tuple(out)


def _attn_core_sample(core, q, k, v, dO, u, rows, kv_rows):
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    kv_rows = np.asarray(kv_rows, dtype=np.int64).reshape(-1, 3)
    nr, nkv, hd = len(rows), len(kv_rows), core.hd
    rb, rh, ri = (np.ascontiguousarray(rows[:, c]) for c in range(3))
    kb, kh, kj = (np.ascontiguousarray(kv_rows[:, c]) for c in range(3))
    out = {n: np.zeros((nr, hd)) for n in ("o", "dq", "a_o", "a_dq")}
    out["lse"] = np.zeros(nr)
    out.update({n: np.zeros((nkv, hd)) for n in ("dk", "dv", "a_dk", "a_dv")})
    core.lib().orc_attn_core_sample(ctypes.byref(core._s), _ptr(q), _ptr(k), _ptr(v), _ptr(dO), ctypes.c_double(u),
                                    ctypes.c_int64(nr), _ptr(rb), _ptr(rh), _ptr(ri), _ptr(out["o"]),
                                    _ptr(out["lse"]), _ptr(out["dq"]), _ptr(out["a_o"]), _ptr(out["a_dq"]),
                                    ctypes.c_int64(nkv), _ptr(kb), _ptr(kh), _ptr(kj), _ptr(out["dk"]),
                                    _ptr(out["dv"]), _ptr(out["a_dk"]), _ptr(out["a_dv"]))
    return out


AttentionCore.sample = lambda self, q, k, v, dO, u, rows, kv_rows: _attn_core_sample(self, q, k, v, dO, u, rows,
                                                                                      kv_rows)
AttentionCore.sample.__doc__ = """Sampled rows: rows = [(b, h, i)] give o, lse, dq (+ a_o, a_dq);
kv_rows = [(b, hk, j)] give dk, dv (+ a_dk, a_dv).  Unrounded values."""


class Attention:
    """The head-sharded attention sublayer of one problem.

    x : [B*S, d]   Wq : [H*hd, d]   Wk, Wv : [Hkv*hd, d]   Wo : [d, H*hd]
    Shard t owns query heads [t*H/T_p, (t+1)*H/T_p) and key/value heads
    [t*Hkv/T_p, (t+1)*Hkv/T_p); both counts must divide by T_p.
    """

    def __init__(self, x, Wq, Wk, Wv, Wo, B, S, H, Hkv, hd, T_p, causal=True, round_bf16=False, lib=None):
        if H % T_p or Hkv % T_p:
            raise ValueError("the tensor-parallel degree must divide the query and the key/value heads")
        self.core = AttentionCore(B, S, H, Hkv, hd, causal, round_bf16, lib)
        self.x, self.Wq, self.Wk, self.Wv, self.Wo = _f64(x), _f64(Wq), _f64(Wk), _f64(Wv), _f64(Wo)
        self.d = self.x.shape[1]
        self.T_p = int(T_p)
        assert self.x.shape[0] == B * S
        assert self.Wq.shape == (H * hd, self.d) and self.Wk.shape == self.Wv.shape == (Hkv * hd, self.d)
        assert self.Wo.shape == (self.d, H * hd)
        self._s = _Attn(self.core._s, self.d, self.T_p, _ptr(self.x), _ptr(self.Wq), _ptr(self.Wk),
                        _ptr(self.Wv), _ptr(self.Wo))

    def forward(self):
        """Returns (c [B*S, H*hd] head outputs, y [B*S, d])."""
        n = self.x.shape[0]
        c = np.empty((n, self.Wo.shape[1]))
        y = np.empty((n, self.d))
        self.core.lib().orc_attn_forward(ctypes.byref(self._s), _ptr(c), _ptr(y))
        return c, y

    def intermediates(self, dy):
        """The stored intermediates: dict q, k, v, c (head outputs), dO."""
        dy = _f64(dy)
        n = self.x.shape[0]
        nq, nk = self.Wq.shape[0], self.Wk.shape[0]
        out = dict(q=np.empty((n, nq)), k=np.empty((n, nk)), v=np.empty((n, nk)), c=np.empty((n, nq)),
                   dO=np.empty((n, nq)))
        self.core.lib().orc_attn_intermediates(ctypes.byref(self._s), _ptr(dy),
                                               *[_ptr(out[m]) for m in ("q", "k", "v", "c", "dO")])
        return out

    def backward(self, dy):
        """Returns dict dx, dWq, dWk, dWv, dWo."""
        dy = _f64(dy)
        assert dy.shape == (self.x.shape[0], self.d)
        out = dict(dx=np.empty_like(self.x), dWq=np.empty_like(self.Wq), dWk=np.empty_like(self.Wk),
                   dWv=np.empty_like(self.Wv), dWo=np.empty_like(self.Wo))
        self.core.lib().orc_attn_backward(ctypes.byref(self._s), _ptr(dy), _ptr(out["dx"]), _ptr(out["dWq"]),
                                          _ptr(out["dWk"]), _ptr(out["dWv"]), _ptr(out["dWo"]))
        return out


# -------------------------------------------------------------- scalar API
def gelu_tanh(u):
    return _load().orc_gelu_tanh(float(u))


def gelu_tanh_grad(u):
    return _load().orc_gelu_tanh_grad(float(u))


def silu(u):
    return _load().orc_silu(float(u))


def silu_grad(u):
    return _load().orc_silu_grad(float(u))


def round_bf16(u):
    return _load().orc_round_bf16(float(u))


def num_threads():
    return _load().orc_num_threads()
