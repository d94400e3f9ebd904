"""ctypes marshalling for the fp64 oracle (test infrastructure only).

The arithmetic lives in ``bam_oracle.cpp``; nothing here computes any part
of the method.  ``build()`` compiles the C++ source with g++ into
``oracle/_build/libbam_oracle.so``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bam_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libbam_oracle.so")
_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle (plain g++, no fast-math, no FMA contraction: each
    expression rounds as written, the same on x86-64 and aarch64) if missing
    or stale."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(__file__))  # source or flags changed
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i = ctypes.c_int
            d = ctypes.c_double
            lib.bam_oracle_bias.restype = d
            lib.bam_oracle_bias.argtypes = [d, d, d, d, d, i]
            lib.bam_oracle_bias_grad.restype = None
            lib.bam_oracle_bias_grad.argtypes = [d, d, d, d, d, i, dp]
            lib.bam_oracle_fwd.restype = i
            lib.bam_oracle_fwd.argtypes = [dp, dp, dp, i, i, i, i, dp, dp, dp, dp, d, i, i, i,
                                           dp, dp, i]
            lib.bam_oracle_fwd_rows.restype = i
            lib.bam_oracle_fwd_rows.argtypes = [dp, dp, dp, i, i, i, i, dp, dp, dp, dp, d, i,
                                                i, i, ip, ctypes.c_int64, dp, dp, i]
            lib.bam_oracle_decode.restype = i
            lib.bam_oracle_decode.argtypes = [dp, dp, dp, i, i, i, i, dp, dp, dp, dp, d, i, i,
                                              dp, dp, i]
            lib.bam_oracle_bwd.restype = i
            lib.bam_oracle_bwd.argtypes = [dp, dp, dp, dp, i, i, i, i, dp, dp, dp, dp, d, i,
                                           i, i, dp, dp, dp, dp, dp, dp, dp, dp, dp, i]
            _lib = lib
    return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _head_params(H, alpha, beta, mu, s):
    alpha = _f64(alpha).reshape(H)
    beta = _f64(beta).reshape(H)
    mu = _f64(mu).reshape(H)
    s = _f64(np.ones(H) if s is None else s).reshape(H)
    return alpha, beta, mu, s


# prior: 0 for b = -(u/alpha)^beta with the eps clamp; 1 for the theta prior
# b = -exp(theta_alpha) (|d - mu| + eps)^theta_beta, mu = 2 sinh(theta_mu), in
# which case (alpha, beta, mu) carry (theta_alpha, theta_beta, theta_mu) and
# the gradients are with respect to those.
PRIOR_ALPHA = 0
PRIOR_THETA = 1


def bias(d: float, alpha: float, beta: float, mu: float, eps: float = 1e-5,
         prior: int = PRIOR_ALPHA) -> float:
    return _load().bam_oracle_bias(float(d), float(alpha), float(beta), float(mu), float(eps),
                                   int(prior))


def bias_grad(d, alpha, beta, mu, eps=1e-5, prior=PRIOR_ALPHA) -> np.ndarray:
    out = np.zeros(3, dtype=np.float64)
    _load().bam_oracle_bias_grad(float(d), float(alpha), float(beta), float(mu), float(eps),
                                 int(prior), _dp(out))
    return out


def fwd(q, k, v, alpha, beta, mu, s=None, eps=1e-5, causal=True, ssmax=False, nthreads=0,
        prior=PRIOR_ALPHA):
    """q, k, v: [B,H,T,D] -> (o [B,H,T,D], lse [B,H,T]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    a, b, m, sc = _head_params(H, alpha, beta, mu, s)
    o = np.empty_like(q)
    lse = np.empty((B, H, T), dtype=np.float64)
    rc = _load().bam_oracle_fwd(_dp(q), _dp(k), _dp(v), B, H, T, D, _dp(a), _dp(b), _dp(m),
                                _dp(sc), float(eps), int(bool(causal)), int(bool(ssmax)),
                                int(prior), _dp(o), _dp(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle fwd: bad sizes")
    return o, lse


def fwd_rows(q, k, v, rows, alpha, beta, mu, s=None, eps=1e-5, causal=True, ssmax=False,
             nthreads=0, prior=PRIOR_ALPHA):
    """Selected rows (flat index (b*H+h)*T+i) -> (o [n,D], lse [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, D = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    a, b, m, sc = _head_params(H, alpha, beta, mu, s)
    o = np.empty((rows.size, D), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    rc = _load().bam_oracle_fwd_rows(
        _dp(q), _dp(k), _dp(v), B, H, T, D, _dp(a), _dp(b), _dp(m), _dp(sc), float(eps),
        int(bool(causal)), int(bool(ssmax)), int(prior),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.size, _dp(o), _dp(lse),
        int(nthreads))
    if rc != 0:
        raise ValueError("oracle fwd_rows: bad sizes")
    return o, lse


def decode(q, kc, vc, alpha, beta, mu, s=None, eps=1e-5, ssmax=False, nthreads=0,
           prior=PRIOR_ALPHA):
    """q [B,H,D], kc/vc [B,H,Tkv,D] -> (o [B,H,D], lse [B,H])."""
    q, kc, vc = _f64(q), _f64(kc), _f64(vc)
    B, H, Tkv, D = kc.shape
    assert q.shape == (B, H, D) and vc.shape == kc.shape
    a, b, m, sc = _head_params(H, alpha, beta, mu, s)
    o = np.empty((B, H, D), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    rc = _load().bam_oracle_decode(_dp(q), _dp(kc), _dp(vc), B, H, Tkv, D, _dp(a), _dp(b),
                                   _dp(m), _dp(sc), float(eps), int(bool(ssmax)), int(prior),
                                   _dp(o), _dp(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode: bad sizes")
    return o, lse


def bwd(q, k, v, dO, alpha, beta, mu, s=None, eps=1e-5, causal=True, ssmax=False,
        nthreads=0, prior=PRIOR_ALPHA):
    """Gradients of sum(O * dO).

    Returns a dict with dq, dk, dv [B,H,T,D], dalpha, dbeta, dmu, ds [H],
    absg [4,H] (sum of |per-element term| of each scalar gradient) and absp
    [4,H] (sum of P (|dP| + |Delta|) |X|: the magnitudes before the
    cancellation inside dS, which set the fp32 noise of any evaluation).
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, T, D = q.shape
    a, b, m, sc = _head_params(H, alpha, beta, mu, s)
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    g = [np.empty(H, dtype=np.float64) for _ in range(4)]
    absg = np.empty((4, H), dtype=np.float64)
    absp = np.empty((4, H), dtype=np.float64)
    rc = _load().bam_oracle_bwd(_dp(q), _dp(k), _dp(v), _dp(dO), B, H, T, D, _dp(a), _dp(b),
                                _dp(m), _dp(sc), float(eps), int(bool(causal)),
                                int(bool(ssmax)), int(prior), _dp(dq), _dp(dk), _dp(dv),
                                _dp(g[0]),
                                _dp(g[1]), _dp(g[2]), _dp(g[3]), _dp(absg), _dp(absp),
                                int(nthreads))
    if rc != 0:
        raise ValueError("oracle bwd: bad sizes")
    return {"dq": dq, "dk": dk, "dv": dv, "dalpha": g[0], "dbeta": g[1], "dmu": g[2],
            "ds": g[3], "absg": absg, "absp": absp}
