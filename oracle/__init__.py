"""fp64 CPU oracle for the Gated DeltaNet prompt-prefill path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``gated_deltanet_linear_pre_gb300``) and never calls it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision, built
with gcc); this module widens inputs to float64 exactly, composes the stages
in the order the method defines them and loops over the sequences of a packed
variable-length batch.  ``chunked.py`` holds a second, chunk-wise formulation
of the recurrence that the tests check against the token-sequential one.

Stage definitions (the pages time these stages but never print the
equations; see the comments in ``gdn_oracle.c`` for the passages each one is
consistent with):

  pre   conv (4 taps, carried 3-token history) -> SiLU -> L2-normalise each
        q/k head -> lam = -exp(A_log) * softplus(a + dt_bias), g = exp(lam),
        beta = sigmoid(b)
  scan  per value head h (key head h // (hv/hk)), per token:
        S <- g S;  u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q / sqrt(dk)
  post  y = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c with gcc (OpenMP over heads, no fast-math, no FMA
    contraction) into oracle/_build/libgdn_oracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-Wall", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # GDN_ORACLE_LIB lets the mutation tests load a deliberately broken
            # copy of the oracle to show that the pins catch it
            lib = ctypes.CDLL(os.environ.get("GDN_ORACLE_LIB") or build())
            lib.gdn_oracle_sigmoid.restype = ctypes.c_double
            lib.gdn_oracle_sigmoid.argtypes = [ctypes.c_double]
            lib.gdn_oracle_silu_scalar.restype = ctypes.c_double
            lib.gdn_oracle_silu_scalar.argtypes = [ctypes.c_double]
            lib.gdn_oracle_softplus.restype = ctypes.c_double
            lib.gdn_oracle_softplus.argtypes = [ctypes.c_double]
            lib.gdn_oracle_conv.argtypes = [_I64, _I64, _D, _D, _D, _D, _D]
            lib.gdn_oracle_silu.argtypes = [_I64, _D, _D]
            lib.gdn_oracle_l2norm.argtypes = [_I64, _I64, ctypes.c_double, _D, _D]
            lib.gdn_oracle_gates.argtypes = [_I64, _I64, _D, _D, _D, _D, _D, _D, _D]
            lib.gdn_oracle_scan.argtypes = [_I64, _I64, _I64, _I64, _I64, _D, _D, _D, _D, _D, _D,
                                            ctypes.POINTER(ctypes.c_int32), _I64, _D, _D]
            lib.gdn_oracle_post.argtypes = [_I64, _I64, ctypes.c_double, _D, _D, _D, _D]
            lib.gdn_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle's scan uses."""
    return int(_load().gdn_oracle_max_threads())


def _f64(x) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array."""
    return np.ascontiguousarray(np.asarray(x), dtype=np.float64)


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


# ---- scalar activations ---------------------------------------------------
def sigmoid(x: float) -> float:
    return float(_load().gdn_oracle_sigmoid(float(x)))


def silu_scalar(x: float) -> float:
    return float(_load().gdn_oracle_silu_scalar(float(x)))


def softplus(x: float) -> float:
    return float(_load().gdn_oracle_softplus(float(x)))


# ---- stages ---------------------------------------------------------------
def conv(x, w, hist):
    """Causal width-4 depthwise conv.  x [T, C], w [C, 4], hist [C, 3] (oldest
    first) -> (y [T, C], hist_out [C, 3])."""
    x, w, hist = _f64(x), _f64(w), _f64(hist)
    T, C = x.shape
    assert w.shape == (C, 4) and hist.shape == (C, 3)
    y = np.empty((T, C))
    hist_out = np.empty((C, 3))
    _load().gdn_oracle_conv(T, C, _p(x), _p(w), _p(hist), _p(y), _p(hist_out))
    return y, hist_out


def silu(x):
    x = _f64(x)
    out = np.empty_like(x)
    _load().gdn_oracle_silu(x.size, _p(x), _p(out))
    return out


def l2norm(x, eps: float):
    """Normalise each row of the last axis: x / sqrt(sum(x^2) + eps)."""
    x = _f64(x)
    d = x.shape[-1]
    out = np.empty_like(x)
    _load().gdn_oracle_l2norm(x.size // d, d, float(eps), _p(x), _p(out))
    return out


def gates(a, b, A_log, dt_bias):
    """a, b [T, hv]; A_log, dt_bias [hv] -> (g, lam, beta), each [T, hv]."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    T, hv = a.shape
    g, lam, beta = np.empty((T, hv)), np.empty((T, hv)), np.empty((T, hv))
    _load().gdn_oracle_gates(T, hv, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(g), _p(lam), _p(beta))
    return g, lam, beta


def scan(q, k, v, g, beta, S0, heads=None):
    """Token-sequential recurrence for one sequence.

    q, k [T, hk, dk]; v [T, hv, dv]; g, beta [T, hv]; S0 [hv, dk, dv]
    -> (o [T, hv, dv], S_out [hv, dk, dv]).  With ``heads`` only those value
    heads are computed; the rest of o / S_out is NaN.
    """
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    T, hk, dk = q.shape
    _, hv, dv = v.shape
    assert k.shape == q.shape and g.shape == (T, hv) and beta.shape == (T, hv)
    assert S0.shape == (hv, dk, dv) and hv % hk == 0
    o = np.full((T, hv, dv), np.nan)
    S_out = np.full((hv, dk, dv), np.nan)
    if heads is None:
        hp, nh = None, 0
    else:
        harr = np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
        assert harr.min() >= 0 and harr.max() < hv
        hp, nh = harr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), harr.size
    _load().gdn_oracle_scan(T, hk, hv, dk, dv, _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0),
                            hp, nh, _p(o), _p(S_out))
    return o, S_out


def post(o, z, gamma, eps: float):
    """o, z [..., dv]; gamma [dv] -> y [..., dv] (fp64)."""
    o, z, gamma = _f64(o), _f64(z), _f64(gamma)
    dv = o.shape[-1]
    assert z.shape == o.shape and gamma.shape == (dv,)
    y = np.empty_like(o)
    _load().gdn_oracle_post(o.size // dv, dv, float(eps), _p(o), _p(z), _p(gamma), _p(y))
    return y


def pre(qkv, conv_w, hist, a, b, A_log, dt_bias, hk, hv, dk, dv, eps):
    """Stage 1 for ONE sequence.  qkv [T, C] with channels q | k | v."""
    T = qkv.shape[0]
    yc, hist_out = conv(qkv, conv_w, hist)
    s = silu(yc)
    q = s[:, : hk * dk].reshape(T, hk, dk)
    k = s[:, hk * dk: 2 * hk * dk].reshape(T, hk, dk)
    v = s[:, 2 * hk * dk:].reshape(T, hv, dv)
    qn = l2norm(q, eps)
    kn = l2norm(k, eps)
    g, lam, beta = gates(a, b, A_log, dt_bias)
    return dict(q=qn, k=kn, v=v, g=g, lam=lam, beta=beta, hist_out=hist_out, conv=yc)


def layer(inp, eps: float = 1e-6, heads=None, hk=16, hv=48, dk=128, dv=128):
    """Whole layer over a packed batch.

    ``inp`` has the fields of ``gated_deltanet_linear_pre_gb300.inputs.LayerInputs``
    (numpy arrays).  Returns a dict with fp64 ``y`` [T, hv, dv], ``hist_out``
    [n_seq, C, 3], ``S_out`` [n_seq, hv, dk, dv] and the stage tensors
    ``q, k`` [T, hk, dk], ``v, o`` [T, hv, dv], ``g, lam, beta`` [T, hv].
    With ``heads`` only the listed value heads go through scan and post (the
    rest is NaN); pre is always complete.
    """
    cu = np.asarray(inp.cu_seqlens, dtype=np.int64)
    n_seq = cu.size - 1
    T = int(cu[-1])
    C = inp.qkv.shape[1]
    out = dict(
        q=np.empty((T, hk, dk)), k=np.empty((T, hk, dk)), v=np.empty((T, hv, dv)),
        g=np.empty((T, hv)), lam=np.empty((T, hv)), beta=np.empty((T, hv)),
        o=np.full((T, hv, dv), np.nan), y=np.full((T, hv, dv), np.nan),
        hist_out=np.empty((n_seq, C, 3)), S_out=np.full((n_seq, hv, dk, dv), np.nan),
    )
    for s in range(n_seq):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        sl = slice(t0, t1)
        p = pre(inp.qkv[sl], inp.conv_w, inp.hist[s], inp.a[sl], inp.b[sl], inp.A_log,
                inp.dt_bias, hk, hv, dk, dv, eps)
        for key in ("q", "k", "v", "g", "lam", "beta"):
            out[key][sl] = p[key]
        out["hist_out"][s] = p["hist_out"]
        o, S_out = scan(p["q"], p["k"], p["v"], p["g"], p["beta"], inp.S0[s], heads=heads)
        out["o"][sl] = o
        out["S_out"][s] = S_out
    hsel = slice(None) if heads is None else np.asarray(heads)
    out["y"][:, hsel] = post(out["o"][:, hsel], inp.z[:, hsel], inp.gamma, eps)
    return out
