"""fp64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import this package.  The product library never loads it, and it shares no
code with the CUDA path.  The arithmetic lives in ``gdn_oracle.c`` (plain C, IEEE double);
this module only marshals numpy arrays through ctypes.

Definitions followed (see the C file's header for the full list):
  * recurrence: model card "Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron", "How It Works";
  * gate g = -exp(A_log) softplus(a + dt_bias): same card, "Correctness Contract";
  * chunked WY/UT form with a direct triangular solve: PR #164 "Fused DeltaNet Direct-Solve
    Follow-Up", "Why This Exists" / "Implementation Details".
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import build as _build

_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


class OracleCfg(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int),
                ("num_k_heads", ctypes.c_int), ("num_v_heads", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("conv_width", ctypes.c_int),
                ("qk_l2norm", ctypes.c_int), ("l2_eps", ctypes.c_double),
                ("scale", ctypes.c_double), ("conv_silu", ctypes.c_int),
                ("gates_precomputed", ctypes.c_int), ("erase", ctypes.c_int)]


def lib():
    global _lib
    if _lib is None:
        # GDN_ORACLE_LIB lets the mutation test load a deliberately broken copy of the oracle
        path = os.environ.get("GDN_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        L.gdn_oracle_softplus.restype = ctypes.c_double
        L.gdn_oracle_softplus.argtypes = [ctypes.c_double]
        L.gdn_oracle_sigmoid.restype = ctypes.c_double
        L.gdn_oracle_sigmoid.argtypes = [ctypes.c_double]
        L.gdn_oracle_gate.restype = ctypes.c_double
        L.gdn_oracle_gate.argtypes = [ctypes.c_double] * 3
        L.gdn_oracle_l2norm.restype = None
        L.gdn_oracle_l2norm.argtypes = [ctypes.c_int, _dp, ctypes.c_double, ctypes.c_double, _dp]
        L.gdn_oracle_conv1d.restype = None
        L.gdn_oracle_conv1d.argtypes = [ctypes.c_int] * 4 + [_dp, _dp, _dp, _dp, ctypes.c_int,
                                                             _dp, _dp]
        L.gdn_oracle_recurrence.restype = None
        L.gdn_oracle_recurrence.argtypes = [ctypes.c_int] * 3 + [_dp] * 5 + [ctypes.c_int, _dp, _dp]
        L.gdn_oracle_chunked.restype = None
        L.gdn_oracle_chunked.argtypes = [ctypes.c_int] * 4 + [_dp] * 5 + [ctypes.c_int, _dp, _dp]
        L.gdn_oracle_unit_lower_inverse.restype = None
        L.gdn_oracle_unit_lower_inverse.argtypes = [ctypes.c_int, _dp, _dp]
        L.gdn_oracle_layer.restype = ctypes.c_int
        L.gdn_oracle_gated_rmsnorm.restype = None
        L.gdn_oracle_gated_rmsnorm.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
                                               ctypes.c_double, _dp]
        L.gdn_oracle_layer.argtypes = [ctypes.POINTER(OracleCfg)] + [_dp] * 13 + [ctypes.c_int]
        _lib = L
    return _lib


def _f64(a) -> np.ndarray:
    """Exact upcast to a C-contiguous float64 array (torch tensors included)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: Optional[np.ndarray]):
    return a.ctypes.data_as(_dp) if a is not None else None


def softplus(x: float) -> float:
    return lib().gdn_oracle_softplus(float(x))


def sigmoid(x: float) -> float:
    return lib().gdn_oracle_sigmoid(float(x))


def gate(a: float, A_log: float, dt_bias: float = 0.0) -> float:
    return lib().gdn_oracle_gate(float(a), float(A_log), float(dt_bias))


def l2norm(x, eps: float = 1e-6, scale: float = 1.0) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    lib().gdn_oracle_l2norm(x.size, _p(x), eps, scale, _p(y))
    return y


def conv1d(x, w, bias=None, state=None, silu: bool = False):
    """x [B,T,C], w [C,W], state [B,W-1,C] -> (y [B,T,C], new_state [B,W-1,C])."""
    x, w = _f64(x), _f64(w)
    B, T, C = x.shape
    W = w.shape[1]
    bias = _f64(bias)
    state = _f64(state)
    y = np.empty_like(x)
    st_out = np.zeros((B, max(W - 1, 0), C))
    lib().gdn_oracle_conv1d(B, T, C, W, _p(x), _p(w), _p(bias), _p(state), int(silu), _p(y),
                            _p(st_out))
    return y, st_out


def recurrence(q, k, v, g, beta, S0, erase: bool = True):
    """One (batch, head) unit, sequential.  q,k [T,dk] (already normalised), v [T,dv],
    g, beta [T], S0 [dv,dk].  Returns (o [T,dv], S_T [dv,dk])."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    S = _f64(S0).copy()
    T, dk = q.shape
    dv = v.shape[1]
    o = np.zeros((T, dv))
    lib().gdn_oracle_recurrence(T, dk, dv, _p(q), _p(k), _p(v), _p(g), _p(beta), int(erase),
                                _p(S), _p(o))
    return o, S


def chunked(q, k, v, g, beta, S0, chunk: int = 64, erase: bool = True):
    """Same as :func:`recurrence` through the chunked WY/UT form (fp64)."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    S = _f64(S0).copy()
    T, dk = q.shape
    dv = v.shape[1]
    o = np.zeros((T, dv))
    lib().gdn_oracle_chunked(T, dk, dv, chunk, _p(q), _p(k), _p(v), _p(g), _p(beta),
                             int(erase), _p(S), _p(o))
    return o, S


def unit_lower_inverse(A) -> np.ndarray:
    A = _f64(A)
    n = A.shape[0]
    T = np.empty_like(A)
    lib().gdn_oracle_unit_lower_inverse(n, _p(A), _p(T))
    return T


@dataclass
class LayerOut:
    out: np.ndarray          # [B,T,Hv,dv]
    state: np.ndarray        # [B,Hv,dv,dk]
    conv_state: Optional[np.ndarray]   # [B,W-1,C_conv]


def gated_rmsnorm(o, z, w, eps: float = 1e-6) -> np.ndarray:
    """Gated RMS norm over the last axis (length n): w * o / sqrt(mean(o^2) + eps) * silu(z)."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    assert o.shape == z.shape and w.shape == (o.shape[-1],)
    n = o.shape[-1]
    rows = o.size // n if n else 0
    y = np.zeros(o.shape)
    lib().gdn_oracle_gated_rmsnorm(int(rows), int(n), _p(np.ascontiguousarray(o)),
                                   _p(np.ascontiguousarray(z)), _p(w), float(eps), _p(y))
    return y


def layer(*, num_k_heads: int, num_v_heads: int, q=None, k=None, v=None, x=None, a, b,
          A_log=None, dt_bias=None, conv_weight=None, conv_bias=None, state=None,
          conv_state=None, scale: float = 1.0, l2_eps: float = 1e-6, qk_l2norm: bool = True,
          conv_silu: bool = True, gates_precomputed: bool = False, erase: bool = True,
          head_dim: int = 128, nthreads: Optional[int] = None) -> LayerOut:
    """The whole gated-delta-net layer hot path (conv -> norm -> gates -> recurrence)."""
    a, b = _f64(a), _f64(b)
    B, T, Hv = a.shape
    Hk = num_k_heads
    assert Hv == num_v_heads
    d = head_dim
    W = 0
    if x is not None:
        x = _f64(x)
        conv_weight = _f64(conv_weight)
        W = conv_weight.shape[1]
        C = x.shape[2]
        cs = (_f64(conv_state).copy() if conv_state is not None
              else np.zeros((B, W - 1, C)))
    else:
        q, k, v = _f64(q), _f64(k), _f64(v)
        cs = None
    S = (_f64(state).copy() if state is not None else np.zeros((B, Hv, d, d)))
    out = np.zeros((B, T, Hv, d))
    cfg = OracleCfg(B, T, Hk, Hv, d, d, W, int(qk_l2norm), float(l2_eps), float(scale),
                    int(conv_silu), int(gates_precomputed), int(erase))
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    A_log_a = _f64(A_log)
    dtb = _f64(dt_bias)
    cb = _f64(conv_bias)
    rc = lib().gdn_oracle_layer(ctypes.byref(cfg), _p(q), _p(k), _p(v), _p(x), _p(a), _p(b),
                                _p(A_log_a), _p(dtb), _p(conv_weight), _p(cb),
                                _p(S), _p(cs), _p(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: invalid layer configuration")
    return LayerOut(out, S, cs)
