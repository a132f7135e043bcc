"""gated_deltanet_linear_13_gb300 -- Python binding of libgdn.so (GB300 / sm_103a).

The gated delta rule (Gated DeltaNet) behind a C ABI (``include/gdn.h``):
``gdn_chunk_prefill``, ``gdn_decode_step``, ``causal_conv1d_update``, ``gdn_state_checkpoint``.
This module only marshals torch tensors into pointers and sizes: every step of the path runs
in the CUDA kernels of ``libgdn.so``.  It checks shapes, dtypes, devices and contiguity
before handing raw pointers to the library (a wrong size would otherwise let a kernel read
past a buffer).  If ``libgdn.so`` is missing the import fails: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")
HEAD_DIM = 128

GDN_OK = 0
GDN_F32, GDN_BF16 = 0, 1
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARGUMENT", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_WORKSPACE", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_TIMEOUT",
                6: "GDN_ERR_DEVICE_INDEX"}

EXPORTED = ("gdn_prefill_workspace_size", "gdn_chunk_prefill", "gdn_decode_step",
            "causal_conv1d_update", "gdn_state_checkpoint", "gdn_chunk_prefill_noalloc",
            "gdn_chunk_prefill_snapshots", "gdn_chunk_prefill_gated", "gdn_decode_step_gated",
            "gdn_prefill_varlen_workspace_size", "gdn_chunk_prefill_varlen", "gdn_decode_multi",
            "gdn_get_device_error", "gdn_status_string", "gdn_version",
            "gdn_selftest_device_timeout", "gdn_chunk_prefill_ex")
NOALLOC_SCRATCH_BYTES = 64 << 20   # GDN_NOALLOC_SCRATCH_BYTES in include/gdn.h


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class GdnDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32),
                ("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("chunk_size", ctypes.c_int32),
                ("conv_width", ctypes.c_int32), ("num_slots", ctypes.c_int32)]


class GdnOpts(ctypes.Structure):
    _fields_ = [("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("qk_l2norm", ctypes.c_int32), ("l2_eps", ctypes.c_float),
                ("scale", ctypes.c_float), ("conv_silu", ctypes.c_int32),
                ("gates_precomputed", ctypes.c_int32)]


class GdnOutGate(ctypes.Structure):
    _fields_ = [("z", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("eps", ctypes.c_float)]


class GdnPrefillExt(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("snap_every", ctypes.c_int32),
                ("snap_state", ctypes.c_void_p), ("snap_conv_state", ctypes.c_void_p),
                ("num_snap_slots", ctypes.c_int32), ("snap_slots", ctypes.c_void_p),
                ("prev_workspace", ctypes.c_void_p)]


_vp = ctypes.c_void_p
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so (raises OSError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"libgdn.so not found at {path}: build it with "
                      "`python -m gated_deltanet_linear_13_gb300.build_lib`")
    L = ctypes.CDLL(path)
    dp, op = ctypes.POINTER(GdnDims), ctypes.POINTER(GdnOpts)
    L.gdn_prefill_workspace_size.restype = ctypes.c_size_t
    L.gdn_prefill_workspace_size.argtypes = [dp, op]
    L.gdn_chunk_prefill.restype = ctypes.c_int
    L.gdn_chunk_prefill.argtypes = [dp, op] + [_vp] * 14 + [ctypes.c_size_t, _vp]
    L.gdn_chunk_prefill_snapshots.restype = ctypes.c_int
    L.gdn_chunk_prefill_snapshots.argtypes = ([dp, op] + [_vp] * 13 +
                                              [ctypes.c_int32, _vp, _vp, ctypes.c_int32, _vp,
                                               _vp, ctypes.c_size_t, _vp])
    gp = ctypes.POINTER(GdnOutGate)
    L.gdn_chunk_prefill_gated.restype = ctypes.c_int
    L.gdn_chunk_prefill_gated.argtypes = [dp, op] + [_vp] * 13 + [gp, _vp, ctypes.c_size_t, _vp]
    L.gdn_chunk_prefill_ex.restype = ctypes.c_int
    L.gdn_chunk_prefill_ex.argtypes = ([dp, op] + [_vp] * 13 +
                                       [ctypes.POINTER(GdnPrefillExt), _vp, ctypes.c_size_t, _vp])
    L.gdn_decode_step_gated.restype = ctypes.c_int
    L.gdn_decode_step_gated.argtypes = [dp, op] + [_vp] * 13 + [gp, _vp]
    L.gdn_prefill_varlen_workspace_size.restype = ctypes.c_size_t
    L.gdn_prefill_varlen_workspace_size.argtypes = [dp, op]
    L.gdn_chunk_prefill_varlen.restype = ctypes.c_int
    L.gdn_chunk_prefill_varlen.argtypes = [dp, op] + [_vp] * 14 + [gp, _vp, ctypes.c_size_t, _vp]
    L.gdn_decode_multi.restype = ctypes.c_int
    L.gdn_decode_multi.argtypes = [dp, op] + [_vp] * 15 + [ctypes.c_int32, _vp, _vp]
    L.gdn_chunk_prefill_noalloc.restype = ctypes.c_int
    L.gdn_chunk_prefill_noalloc.argtypes = [dp, op] + [_vp] * 13 + [_vp]
    L.gdn_decode_step.restype = ctypes.c_int
    L.gdn_decode_step.argtypes = [dp, op] + [_vp] * 13 + [_vp]
    L.causal_conv1d_update.restype = ctypes.c_int
    L.causal_conv1d_update.argtypes = ([ctypes.c_int32] * 4 + [ctypes.c_int] + [_vp] * 4 +
                                       [ctypes.c_int32, _vp, ctypes.c_int32, _vp, _vp])
    L.gdn_state_checkpoint.restype = ctypes.c_int
    L.gdn_state_checkpoint.argtypes = ([ctypes.c_int32, dp, ctypes.c_int] + [_vp] * 4 +
                                       [ctypes.c_int32, _vp, _vp, ctypes.c_int32, _vp])
    L.gdn_get_device_error.restype = ctypes.c_int
    L.gdn_get_device_error.argtypes = [_vp]
    L.gdn_selftest_device_timeout.restype = ctypes.c_int
    L.gdn_selftest_device_timeout.argtypes = [ctypes.c_uint32, _vp]
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_status_string.argtypes = [ctypes.c_int]
    L.gdn_version.restype = ctypes.c_int32
    L.gdn_version.argtypes = []
    _lib = L
    return L


# ---------------------------------------------------------------- marshalling helpers

def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: Optional[torch.Tensor], name: str, shape, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str):
    if status != GDN_OK:
        raise GDNError(status, where)


def _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state, state, state_slots,
                num_slots_hint):
    B, T, Hv = a.shape
    W = 0 if conv_weight is None else conv_weight.shape[1]
    if W > 0:
        Hk = num_k_heads
        C = (2 * Hk + Hv) * HEAD_DIM
        if q.shape != (B, T, C):
            raise ValueError(f"x: shape {tuple(q.shape)}, expected {(B, T, C)}")
    else:
        Hk = q.shape[2]
    num_slots = state.shape[0]
    if state_slots is None and num_slots < B:
        raise ValueError("state has fewer rows than the batch and no state_slots given")
    return B, T, Hk, Hv, W, num_slots


def _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed):
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    in_t = q.dtype
    d = HEAD_DIM
    C = (2 * Hk + Hv) * d
    if W > 0:
        if k is not None or v is not None:
            raise ValueError("with a conv, pass the pre-conv x as q and k = v = None")
        _need(conv_weight, "conv_weight", (C, W), in_t, dev)
        if conv_bias is not None:
            _need(conv_bias, "conv_bias", (C,), in_t, dev)
        if W > 1:
            _need(conv_state, "conv_state", (num_slots, W - 1, C), in_t, dev)
    else:
        _need(q, "q", (B, T, Hk, d), in_t, dev)
        _need(k, "k", (B, T, Hk, d), in_t, dev)
        _need(v, "v", (B, T, Hv, d), in_t, dev)
    gt = torch.float32 if gates_precomputed else in_t
    _need(a, "a", (B, T, Hv), gt, dev)
    _need(b, "b", (B, T, Hv), gt, dev)
    if not gates_precomputed:
        _need(A_log, "A_log", (Hv,), torch.float32, dev)
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", (Hv,), torch.float32, dev)
    _need(state, "state", (num_slots, Hv, d, d), torch.float32, dev)
    if state_slots is not None:
        _need(state_slots, "state_slots", (B,), torch.int32, dev)
    if out.device != dev or not out.is_contiguous() or tuple(out.shape) != (B, T, Hv, d):
        raise ValueError(f"out: expected contiguous {(B, T, Hv, d)} on {dev}")


def _opts(in_dtype, out_dtype, qk_l2norm, eps, scale, conv_silu, gates_precomputed):
    return GdnOpts(in_dtype, out_dtype, int(qk_l2norm), float(eps), float(scale),
                   int(conv_silu), int(gates_precomputed))


# ---------------------------------------------------------------- public API

def gdn_prefill_workspace_size(batch: int, seqlen: int, num_k_heads: int, num_v_heads: int,
                               conv_width: int, in_dtype=torch.bfloat16) -> int:
    L = load_library()
    dims = GdnDims(batch, seqlen, num_k_heads, num_v_heads, HEAD_DIM, 64, conv_width, 0)
    dt = GDN_BF16 if in_dtype == torch.bfloat16 else GDN_F32
    opts = _opts(dt, dt, 1, 1e-6, 1.0, 1, 0)
    return int(L.gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))


def gdn_chunk_prefill(q, k, v, a, b, A_log, dt_bias, state, out, *, num_k_heads=None,
                      conv_weight=None, conv_bias=None, conv_state=None, state_slots=None,
                      scale: float = 1.0, eps: float = 1e-6, qk_l2norm: bool = True,
                      conv_silu: bool = True, gates_precomputed: bool = False,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Chunked prefill (see gdn_chunk_prefill in include/gdn.h).  With a conv, ``q`` is the
    pre-conv x [B,T,C_conv] and ``k = v = None``.  ``state`` (and ``conv_state``) are updated
    in place; ``out`` [B,T,Hv,128] is written.  Returns ``out``."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    dims = GdnDims(B, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    need = int(L.gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = L.gdn_chunk_prefill(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v),
                             _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(conv_weight),
                             _ptr(conv_bias), _ptr(state), _ptr(conv_state), _ptr(state_slots),
                             _ptr(out), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "gdn_chunk_prefill")
    return out


def gdn_chunk_prefill_snapshots(q, k, v, a, b, A_log, dt_bias, state, out, *, snap_every: int,
                                snap_state, snap_slots, snap_conv_state=None, num_k_heads=None,
                                conv_weight=None, conv_bias=None, conv_state=None,
                                state_slots=None, scale: float = 1.0, eps: float = 1e-6,
                                qk_l2norm: bool = True, conv_silu: bool = True,
                                gates_precomputed: bool = False,
                                workspace: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """gdn_chunk_prefill over the whole prompt in one call, recording the state after every
    ``snap_every`` tokens (see gdn_chunk_prefill_snapshots in include/gdn.h): snapshot j of
    row b goes to bank row ``snap_slots[b, j]`` of ``snap_state`` [n, Hv, 128, 128] (and of
    ``snap_conv_state`` [n, W-1, C_conv] with a conv), j < T // snap_every.  Returns ``out``."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    dev = q.device
    n_snap = T // snap_every if snap_every > 0 else 0
    nb = snap_state.shape[0]
    _need(snap_state, "snap_state", (nb, Hv, HEAD_DIM, HEAD_DIM), torch.float32, dev)
    _need(snap_slots, "snap_slots", (B, n_snap), torch.int32, dev)
    if W > 1:
        _need(snap_conv_state, "snap_conv_state", (nb, W - 1, (2 * Hk + Hv) * HEAD_DIM),
              q.dtype, dev)
    dims = GdnDims(B, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    need = int(L.gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = L.gdn_chunk_prefill_snapshots(
        ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
        _ptr(A_log), _ptr(dt_bias), _ptr(conv_weight), _ptr(conv_bias), _ptr(state),
        _ptr(conv_state), _ptr(state_slots), _ptr(out), int(snap_every), _ptr(snap_state),
        _ptr(snap_conv_state), nb, _ptr(snap_slots), _ptr(workspace), ws_bytes,
        _stream(stream))
    _check(st, "gdn_chunk_prefill_snapshots")
    return out


def gdn_chunk_prefill_noalloc(q, k, v, a, b, A_log, dt_bias, state, out, *, num_k_heads=None,
                              conv_weight=None, conv_bias=None, conv_state=None,
                              state_slots=None, scale: float = 1.0, eps: float = 1e-6,
                              qk_l2norm: bool = True, conv_silu: bool = True,
                              gates_precomputed: bool = False, stream=None) -> torch.Tensor:
    """gdn_chunk_prefill without a workspace, for callers that cannot allocate: the library's
    fixed device scratch array (NOALLOC_SCRATCH_BYTES per GPU) holds the call's workspace.  Raises GDNError(GDN_ERR_WORKSPACE) when the call needs more than that.
    Calls that overlap on the GPU share that array and must be serialised."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    dims = GdnDims(B, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    st = L.gdn_chunk_prefill_noalloc(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k),
                                     _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                     _ptr(conv_weight), _ptr(conv_bias), _ptr(state),
                                     _ptr(conv_state), _ptr(state_slots), _ptr(out),
                                     _stream(stream))
    _check(st, "gdn_chunk_prefill_noalloc")
    return out


def gdn_decode_step(q, k, v, a, b, A_log, dt_bias, state, out, *, num_k_heads=None,
                    conv_weight=None, conv_bias=None, conv_state=None, state_slots=None,
                    scale: float = 1.0, eps: float = 1e-6, qk_l2norm: bool = True,
                    conv_silu: bool = True, gates_precomputed: bool = False,
                    stream=None) -> torch.Tensor:
    """One decode step for B sequences (T = 1), fused into one kernel launch."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    if T != 1:
        raise ValueError("gdn_decode_step takes exactly one token per sequence")
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    dims = GdnDims(B, 1, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    st = L.gdn_decode_step(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(conv_weight),
                           _ptr(conv_bias), _ptr(state), _ptr(conv_state), _ptr(state_slots),
                           _ptr(out), _stream(stream))
    _check(st, "gdn_decode_step")
    return out


def _out_gate(gate_z, gate_weight, gate_eps, out, in_dtype) -> GdnOutGate:
    dev = out.device
    _need(gate_z, "gate_z", tuple(out.shape), in_dtype, dev)
    _need(gate_weight, "gate_weight", (HEAD_DIM,), torch.float32, dev)
    return GdnOutGate(_ptr(gate_z), _ptr(gate_weight), float(gate_eps))


def gdn_chunk_prefill_gated(q, k, v, a, b, A_log, dt_bias, state, out, *, gate_z, gate_weight,
                            gate_eps: float = 1e-6, num_k_heads=None, conv_weight=None,
                            conv_bias=None, conv_state=None, state_slots=None,
                            scale: float = 1.0, eps: float = 1e-6, qk_l2norm: bool = True,
                            conv_silu: bool = True, gates_precomputed: bool = False,
                            workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """gdn_chunk_prefill with the gated RMS norm on the output (see gdn_out_gate in
    include/gdn.h): out = gate_weight * o / sqrt(mean(o^2) + gate_eps) * silu(gate_z) per
    (token, value head); gate_z has the shape of out and the input dtype."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    gate = _out_gate(gate_z, gate_weight, gate_eps, out, q.dtype)
    dims = GdnDims(B, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    need = int(L.gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = L.gdn_chunk_prefill_gated(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                   _ptr(conv_weight), _ptr(conv_bias), _ptr(state),
                                   _ptr(conv_state), _ptr(state_slots), _ptr(out),
                                   ctypes.byref(gate), _ptr(workspace), ws_bytes,
                                   _stream(stream))
    _check(st, "gdn_chunk_prefill_gated")
    return out


def gdn_chunk_prefill_ex(q, k, v, a, b, A_log, dt_bias, state, out, *, num_k_heads=None,
                         conv_weight=None, conv_bias=None, conv_state=None, state_slots=None,
                         scale: float = 1.0, eps: float = 1e-6, qk_l2norm: bool = True,
                         conv_silu: bool = True, gates_precomputed: bool = False,
                         gate_z=None, gate_weight=None, gate_eps: float = 1e-6,
                         snap_every: int = 0, snap_state=None, snap_slots=None,
                         snap_conv_state=None, prev_workspace: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """gdn_chunk_prefill with any of its optional parts (see gdn_chunk_prefill_ex in
    include/gdn.h): the gated output norm (``gate_z``, ``gate_weight``), in-call snapshots
    (``snap_every`` > 0, as gdn_chunk_prefill_snapshots), and ``prev_workspace``: the
    workspace of the previous prefill call of the same sequences on this stream, which this
    call continues (its kernels may then start while that call finishes; pass the two
    workspaces alternately).  Returns ``out``."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    dev = q.device
    ext = GdnPrefillExt()
    gate = None
    if gate_z is not None or gate_weight is not None:
        gate = _out_gate(gate_z, gate_weight, gate_eps, out, q.dtype)
        ext.gate = ctypes.cast(ctypes.pointer(gate), ctypes.c_void_p)
    if snap_every:
        n_snap = T // snap_every if snap_every > 0 else 0
        nb = snap_state.shape[0]
        _need(snap_state, "snap_state", (nb, Hv, HEAD_DIM, HEAD_DIM), torch.float32, dev)
        _need(snap_slots, "snap_slots", (B, n_snap), torch.int32, dev)
        if W > 1:
            _need(snap_conv_state, "snap_conv_state", (nb, W - 1, (2 * Hk + Hv) * HEAD_DIM),
                  q.dtype, dev)
        ext.snap_every = int(snap_every)
        ext.snap_state = _ptr(snap_state)
        ext.snap_conv_state = _ptr(snap_conv_state)
        ext.num_snap_slots = nb
        ext.snap_slots = _ptr(snap_slots)
    ext.prev_workspace = _ptr(prev_workspace)
    dims = GdnDims(B, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    need = int(L.gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = L.gdn_chunk_prefill_ex(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                _ptr(conv_weight), _ptr(conv_bias), _ptr(state),
                                _ptr(conv_state), _ptr(state_slots), _ptr(out),
                                ctypes.byref(ext), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "gdn_chunk_prefill_ex")
    return out


def gdn_prefill_varlen_workspace_size(num_seqs: int, total_tokens: int, num_k_heads: int,
                                      num_v_heads: int, conv_width: int,
                                      in_dtype=torch.bfloat16) -> int:
    L = load_library()
    dims = GdnDims(num_seqs, total_tokens, num_k_heads, num_v_heads, HEAD_DIM, 64, conv_width, 0)
    dt = GDN_BF16 if in_dtype == torch.bfloat16 else GDN_F32
    opts = _opts(dt, dt, 1, 1e-6, 1.0, 1, 0)
    return int(L.gdn_prefill_varlen_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))


def gdn_chunk_prefill_varlen(q, k, v, a, b, A_log, dt_bias, state, out, *, cu_seqlens,
                             num_k_heads=None, conv_weight=None, conv_bias=None,
                             conv_state=None, state_slots=None, gate_z=None, gate_weight=None,
                             gate_eps: float = 1e-6, scale: float = 1.0, eps: float = 1e-6,
                             qk_l2norm: bool = True, conv_silu: bool = True,
                             gates_precomputed: bool = False,
                             workspace: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """Prefill of a packed variable-length batch (see gdn_chunk_prefill_varlen in
    include/gdn.h): every tensor has the layout of a one-sequence call over all T packed
    tokens ([1, T, ...]); sequence n is tokens cu_seqlens[n] .. cu_seqlens[n+1] - 1 and uses
    state row state_slots[n] (or n).  Optional gated output norm (gate_z shaped like out)."""
    L = load_library()
    _, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, None, None)
    if a.shape[0] != 1:
        raise ValueError("a packed batch has all its tokens in one row: a must be [1, T, Hv]")
    N = cu_seqlens.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens needs N + 1 >= 1 entries")
    _need(cu_seqlens, "cu_seqlens", (N + 1,), torch.int32, q.device)
    if state_slots is None and num_slots < N:
        raise ValueError("state has fewer rows than sequences and no state_slots given")
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 None, out, 1, T, Hk, Hv, W, num_slots, gates_precomputed)
    if state_slots is not None:
        _need(state_slots, "state_slots", (N,), torch.int32, q.device)
    gate = None
    if gate_z is not None:
        gate = _out_gate(gate_z, gate_weight, gate_eps, out, q.dtype)
    dims = GdnDims(N, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    need = int(L.gdn_prefill_varlen_workspace_size(ctypes.byref(dims), ctypes.byref(opts)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = L.gdn_chunk_prefill_varlen(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k),
                                    _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                    _ptr(conv_weight), _ptr(conv_bias), _ptr(state),
                                    _ptr(conv_state), _ptr(state_slots), _ptr(cu_seqlens),
                                    _ptr(out), None if gate is None else ctypes.byref(gate),
                                    _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "gdn_chunk_prefill_varlen")
    return out


def gdn_decode_multi(q, k, v, a, b, A_log, dt_bias, state, out, *, num_k_heads=None,
                     conv_weight=None, conv_bias=None, conv_state=None, state_slots=None,
                     snap_state=None, snap_conv_state=None, snap_slots=None,
                     scale: float = 1.0, eps: float = 1e-6, qk_l2norm: bool = True,
                     conv_silu: bool = True, gates_precomputed: bool = False,
                     stream=None) -> torch.Tensor:
    """A decode step over T <= 16 tokens per sequence (see gdn_decode_multi in
    include/gdn.h); inputs shaped as for gdn_chunk_prefill with seqlen T.  With snap_slots
    [B, T] the state (and conv state) after every token go to those rows of snap_state
    (snap_conv_state)."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    nb = 0
    if snap_slots is not None:
        dev = q.device
        nb = snap_state.shape[0]
        _need(snap_slots, "snap_slots", (B, T), torch.int32, dev)
        _need(snap_state, "snap_state", (nb, Hv, HEAD_DIM, HEAD_DIM), torch.float32, dev)
        if W > 1:
            _need(snap_conv_state, "snap_conv_state", (nb, W - 1, (2 * Hk + Hv) * HEAD_DIM),
                  q.dtype, dev)
    dims = GdnDims(B, T, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    st = L.gdn_decode_multi(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(conv_weight),
                            _ptr(conv_bias), _ptr(state), _ptr(conv_state), _ptr(state_slots),
                            _ptr(out), _ptr(snap_state), _ptr(snap_conv_state), nb,
                            _ptr(snap_slots), _stream(stream))
    _check(st, "gdn_decode_multi")
    return out


def gdn_decode_step_gated(q, k, v, a, b, A_log, dt_bias, state, out, *, gate_z, gate_weight,
                          gate_eps: float = 1e-6, num_k_heads=None, conv_weight=None,
                          conv_bias=None, conv_state=None, state_slots=None, scale: float = 1.0,
                          eps: float = 1e-6, qk_l2norm: bool = True, conv_silu: bool = True,
                          gates_precomputed: bool = False, stream=None) -> torch.Tensor:
    """gdn_decode_step with the gated RMS norm on the output (gate_z shaped like out)."""
    L = load_library()
    B, T, Hk, Hv, W, num_slots = _layer_dims(q, k, v, a, num_k_heads, conv_weight, conv_state,
                                             state, state_slots, None)
    if T != 1:
        raise ValueError("gdn_decode_step_gated takes exactly one token per sequence")
    _check_layer(q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state, conv_state,
                 state_slots, out, B, T, Hk, Hv, W, num_slots, gates_precomputed)
    gate = _out_gate(gate_z, gate_weight, gate_eps, out, q.dtype)
    dims = GdnDims(B, 1, Hk, Hv, HEAD_DIM, 64, W, num_slots)
    opts = _opts(_dt(q), _dt(out), qk_l2norm, eps, scale, conv_silu, gates_precomputed)
    st = L.gdn_decode_step_gated(ctypes.byref(dims), ctypes.byref(opts), _ptr(q), _ptr(k),
                                 _ptr(v), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                                 _ptr(conv_weight), _ptr(conv_bias), _ptr(state),
                                 _ptr(conv_state), _ptr(state_slots), _ptr(out),
                                 ctypes.byref(gate), _stream(stream))
    _check(st, "gdn_decode_step_gated")
    return out


def causal_conv1d_update(x, weight, conv_state, y, *, bias=None, state_slots=None,
                         silu: bool = True, stream=None) -> torch.Tensor:
    """Standalone causal depthwise conv with carried state: x, y [B,T,C]; weight [C,W];
    conv_state [num_slots, W-1, C] updated in place."""
    L = load_library()
    B, T, C = x.shape
    W = weight.shape[1]
    dev, dt = x.device, x.dtype
    _need(x, "x", (B, T, C), dt, dev)
    _need(y, "y", (B, T, C), dt, dev)
    _need(weight, "weight", (C, W), dt, dev)
    if bias is not None:
        _need(bias, "bias", (C,), dt, dev)
    ns = conv_state.shape[0]
    _need(conv_state, "conv_state", (ns, W - 1, C), dt, dev)
    if state_slots is not None:
        _need(state_slots, "state_slots", (B,), torch.int32, dev)
    st = L.causal_conv1d_update(B, T, C, W, _dt(x), _ptr(x), _ptr(weight), _ptr(bias),
                                _ptr(conv_state), ns, _ptr(state_slots), int(silu), _ptr(y),
                                _stream(stream))
    _check(st, "causal_conv1d_update")
    return y


def gdn_state_checkpoint(op: str, state, conv_state, slot_state, slot_conv_state, rows, slots,
                         *, num_k_heads: int, stream=None) -> None:
    """op 'save' (live rows -> bank slots) or 'restore' (bank slots -> live rows)."""
    L = load_library()
    opc = {"save": 0, "restore": 1}[op]
    ns, Hv, d, _ = state.shape
    nb = slot_state.shape[0]
    dev = state.device
    _need(state, "state", (ns, Hv, d, d), torch.float32, dev)
    _need(slot_state, "slot_state", (nb, Hv, d, d), torch.float32, dev)
    W = 0
    cdt = GDN_BF16
    if conv_state is not None:
        W = conv_state.shape[1] + 1
        C = conv_state.shape[2]
        if C != (2 * num_k_heads + Hv) * d:
            raise ValueError("conv_state channels do not match the head geometry")
        _need(conv_state, "conv_state", (ns, W - 1, C), conv_state.dtype, dev)
        _need(slot_conv_state, "slot_conv_state", (nb, W - 1, C), conv_state.dtype, dev)
        cdt = _dt(conv_state)
    n = rows.shape[0]
    _need(rows, "rows", (n,), torch.int32, dev)
    _need(slots, "slots", (n,), torch.int32, dev)
    dims = GdnDims(ns, 1, num_k_heads, Hv, d, 64, W, ns)
    st = L.gdn_state_checkpoint(opc, ctypes.byref(dims), cdt, _ptr(state), _ptr(conv_state),
                                _ptr(slot_state), _ptr(slot_conv_state), nb, _ptr(rows),
                                _ptr(slots), n, _stream(stream))
    _check(st, "gdn_state_checkpoint")


def gdn_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status code."""
    return int(load_library().gdn_get_device_error(_stream(stream)))


def gdn_selftest_device_timeout(max_iters: int = 1024, stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that nothing ends, on no copy or MMA): the
    next gdn_get_device_error() returns GDN_ERR_DEVICE_TIMEOUT."""
    st = load_library().gdn_selftest_device_timeout(int(max_iters), _stream(stream))
    _check(st, "gdn_selftest_device_timeout")


def gdn_status_string(status: int) -> str:
    return load_library().gdn_status_string(int(status)).decode()
