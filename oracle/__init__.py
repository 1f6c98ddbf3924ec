"""fp64 CPU oracle for Kimi Delta Attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never imports, links or calls it, and it shares no code with the
CUDA path.

The arithmetic lives in ``kda_oracle.c`` (the explicit token-by-token
recurrence, its prologue and its reverse mode; that file's header cites the
pages it follows).  This module compiles it with the host C compiler and
marshals numpy float64 arrays through ctypes.

Parity status: the recurrence, the L2 norm, sigmoid(beta), state I/O,
packed documents, grouped key heads, the backward pass and the short
convolution + SiLU prologue are pinned by the tests in
``tests/test_oracle_pins.py``.  The gate formulas
``g = lower_bound * sigmoid(exp(a_log) * (g_raw + dt_bias))`` and, for the
unbounded gate, ``g = -exp(a_log) * softplus(g_raw + dt_bias)``, and the
L2-norm epsilon (1e-6) are readings of pages that print none of them, and so is the
gated output norm's formula (``gated_norm_fwd``: RMS norm with a weight, gated by a sigmoid):
parity unpinned for those choices (the tests pin only their limits and
special values, and the gradients through them by finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libkda_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_gate_value.restype = ctypes.c_double
            lib.oracle_gate_value.argtypes = [ctypes.c_double] * 4 + [ctypes.c_int]
            lib.oracle_recurrence.restype = ctypes.c_int
            lib.oracle_recurrence.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                              _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_double, _dp, _dp]
            common = [ctypes.c_int] * 7 + [_ip] + [_dp] * 7 + [ctypes.c_double, ctypes.c_double, ctypes.c_int, _dp]
            lib.oracle_kda_fwd.restype = ctypes.c_int
            lib.oracle_kda_fwd.argtypes = common + [_dp, _dp, ctypes.c_int]
            lib.oracle_kda_bwd.restype = ctypes.c_int
            lib.oracle_kda_bwd.argtypes = common + [_dp, _dp] + [_dp] * 8 + [ctypes.c_int]
            conv = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int, _dp, _dp, _dp]
            lib.oracle_short_conv_fwd.restype = ctypes.c_int
            lib.oracle_short_conv_fwd.argtypes = conv + [_dp]
            lib.oracle_short_conv_bwd.restype = ctypes.c_int
            lib.oracle_short_conv_bwd.argtypes = conv + [_dp, _dp, _dp, _dp]
            gn = [ctypes.c_int64, ctypes.c_int, _dp, _dp, _dp, ctypes.c_double]
            lib.oracle_gated_norm_fwd.restype = ctypes.c_int
            lib.oracle_gated_norm_fwd.argtypes = gn + [_dp]
            lib.oracle_gated_norm_bwd.restype = ctypes.c_int
            lib.oracle_gated_norm_bwd.argtypes = gn + [_dp, _dp, _dp, _dp]
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(_dp)


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None, None
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    return cu, cu.ctypes.data_as(_ip)


def default_threads() -> int:
    return os.cpu_count() or 1


GATES = {"lower_bounded": 0, "softplus": 1}


def _gate_kind(gate):
    if gate not in GATES:
        raise ValueError(f"gate must be one of {sorted(GATES)}, got {gate!r}")
    return GATES[gate]


def gate(g_raw, a_log, dt_bias, lower_bound, kind="lower_bounded"):
    """Log-decay g of one gate element (scalar inputs).

    kind "lower_bounded": g = lower_bound * sigmoid(exp(a_log) * (g_raw + dt_bias));
    kind "softplus": g = -exp(a_log) * softplus(g_raw + dt_bias) (lower_bound unused).
    """
    return _load().oracle_gate_value(float(g_raw), float(a_log), float(dt_bias), float(lower_bound),
                                     _gate_kind(kind))


def recurrence(q_hat, k_hat, v, g, beta, scale, S0=None):
    """Token loop with the prologue bypassed, one segment and one head.

    q_hat, k_hat, g: [L, K]; v: [L, V]; beta: [L]; S0: [K, V] or None.
    ``g`` is the log-decay (alpha = exp(g)).  Returns (out [L, V], S_T [K, V]).
    """
    q_hat, k_hat, v, g, beta, S0 = map(_f64, (q_hat, k_hat, v, g, beta, S0))
    L, K = q_hat.shape
    V = v.shape[1]
    out = np.zeros((L, V))
    ST = np.zeros((K, V))
    rc = _load().oracle_recurrence(L, K, V, _ptr(q_hat), _ptr(k_hat), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(S0), float(scale), _ptr(out), _ptr(ST))
    if rc:
        raise MemoryError("oracle_recurrence failed")
    return out, ST


def kda_fwd(q, k, v, g_raw, beta_raw, a_log, dt_bias, *, scale, lower_bound, gate="lower_bounded",
            cu_seqlens=None, initial_state=None, output_final_state=True, nthreads=0):
    """Full forward.  q, k: [B, T, Hk, K]; g_raw: [B, T, H, K]; v: [B, T, H, V]; beta_raw: [B, T, H].

    H counts value heads, Hk key heads (H a multiple of Hk; value head h reads key head
    h // (H // Hk)).  With ``cu_seqlens`` (B must be 1) every segment is its own recurrence.
    ``gate`` selects the gate activation (see :func:`gate`).
    Returns (out [B, T, H, V], final_state [N, H, K, V] or None).
    """
    q, k, v, g_raw, beta_raw, a_log, dt_bias, S0 = map(
        _f64, (q, k, v, g_raw, beta_raw, a_log, dt_bias, initial_state))
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    if H % Hk:
        raise ValueError("value heads must be a multiple of key heads")
    cu, cu_p = _cu(cu_seqlens)
    N = (len(cu) - 1) if cu is not None else B
    out = np.zeros((B, T, H, V))
    fs = np.zeros((N, H, K, V)) if output_final_state else None
    rc = _load().oracle_kda_fwd(B, T, H, Hk, K, V, N, cu_p, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                _ptr(beta_raw), _ptr(a_log), _ptr(dt_bias), float(scale),
                                float(lower_bound), _gate_kind(gate), _ptr(S0), _ptr(out), _ptr(fs), int(nthreads))
    if rc:
        raise MemoryError("oracle_kda_fwd failed")
    return out, fs


def kda_bwd(q, k, v, g_raw, beta_raw, a_log, dt_bias, dout, *, scale, lower_bound, gate="lower_bounded",
            cu_seqlens=None, initial_state=None, dfinal_state=None, nthreads=0):
    """Reverse mode of :func:`kda_fwd`.

    Returns a dict with dq, dk, dv, dg_raw, dbeta_raw, da_log, ddt_bias,
    dinitial_state (always computed, [N, H, K, V]).  dq, dk have the key heads' shape.
    """
    q, k, v, g_raw, beta_raw, a_log, dt_bias, dout, S0, dST = map(
        _f64, (q, k, v, g_raw, beta_raw, a_log, dt_bias, dout, initial_state, dfinal_state))
    B, T, Hk, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    if H % Hk:
        raise ValueError("value heads must be a multiple of key heads")
    cu, cu_p = _cu(cu_seqlens)
    N = (len(cu) - 1) if cu is not None else B
    res = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg_raw=np.zeros_like(g_raw), dbeta_raw=np.zeros_like(beta_raw),
               da_log=np.zeros(H), ddt_bias=np.zeros(H * K), dinitial_state=np.zeros((N, H, K, V)))
    rc = _load().oracle_kda_bwd(B, T, H, Hk, K, V, N, cu_p, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                _ptr(beta_raw), _ptr(a_log), _ptr(dt_bias), float(scale),
                                float(lower_bound), _gate_kind(gate), _ptr(S0), _ptr(dout), _ptr(dST),
                                _ptr(res["dq"]), _ptr(res["dk"]), _ptr(res["dv"]),
                                _ptr(res["dg_raw"]), _ptr(res["dbeta_raw"]), _ptr(res["da_log"]),
                                _ptr(res["ddt_bias"]), _ptr(res["dinitial_state"]), int(nthreads))
    if rc:
        raise MemoryError("oracle_kda_bwd failed")
    return res


def short_conv_fwd(x, weight, bias=None, cu_seqlens=None):
    """Causal depthwise short convolution + SiLU over tokens (the layer's q/k/v prologue).

    x: [B, T, C]; weight: [C, W]; bias: [C] or None.  With ``cu_seqlens`` (B must be 1) every
    segment starts from zero history.  Returns y [B, T, C].
    """
    x, weight, bias = map(_f64, (x, weight, bias))
    B, T, C = x.shape
    W = weight.shape[1]
    cu, cu_p = _cu(cu_seqlens)
    y = np.zeros_like(x)
    _load().oracle_short_conv_fwd(B * T, T, C, W, cu_p, (len(cu) - 1) if cu is not None else 0,
                                  _ptr(x), _ptr(weight), _ptr(bias), _ptr(y))
    return y


def short_conv_bwd(x, weight, bias, dy, cu_seqlens=None):
    """Reverse mode of :func:`short_conv_fwd`: dict(dx [B, T, C], dweight [C, W], dbias [C] or None)."""
    x, weight, bias, dy = map(_f64, (x, weight, bias, dy))
    B, T, C = x.shape
    W = weight.shape[1]
    cu, cu_p = _cu(cu_seqlens)
    dx, dw = np.zeros_like(x), np.zeros_like(weight)
    db = np.zeros(C) if bias is not None else None
    _load().oracle_short_conv_bwd(B * T, T, C, W, cu_p, (len(cu) - 1) if cu is not None else 0,
                                  _ptr(x), _ptr(weight), _ptr(bias), _ptr(dy), _ptr(dx), _ptr(dw), _ptr(db))
    return dict(dx=dx, dweight=dw, dbias=db)


def gated_norm_fwd(o, gate, weight, eps):
    """The output epilogue: y = o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate) over the last axis.

    o, gate: [..., V]; weight: [V].  Returns y like o.
    """
    o, gate, weight = map(_f64, (o, gate, weight))
    V = o.shape[-1]
    y = np.zeros_like(o)
    _load().oracle_gated_norm_fwd(o.size // V, V, _ptr(o), _ptr(gate), _ptr(weight), float(eps), _ptr(y))
    return y


def gated_norm_bwd(o, gate, weight, eps, dy):
    """Reverse mode of :func:`gated_norm_fwd`: dict(do, dgate like o, dweight [V])."""
    o, gate, weight, dy = map(_f64, (o, gate, weight, dy))
    V = o.shape[-1]
    d_o, dg, dw = np.zeros_like(o), np.zeros_like(o), np.zeros(V)
    _load().oracle_gated_norm_bwd(o.size // V, V, _ptr(o), _ptr(gate), _ptr(weight), float(eps), _ptr(dy),
                                  _ptr(d_o), _ptr(dg), _ptr(dw))
    return dict(do=d_o, dgate=dg, dweight=dw)
