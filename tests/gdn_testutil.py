"""Shared helpers of the parity tests: run the CUDA path and the fp64 oracle on the same
seeded inputs and compare them with the stated tolerances.

Tolerances (gated-delta-rule targets):
  * bf16 inputs, fp32 state: output cosine >= 0.9999 and max|o - o_ref| / max|o_ref| <= 5e-3
    (outputs scaled to unit range) for the computation; an output stored in bf16 adds its own
    rounding, at most 2^-8 of max|o_ref| at the top of the range, so bf16 outputs are held to
    5e-3 + 2^-8.  Final state: cosine >= 0.9999 and relative Frobenius error <= 5e-3.
  * all-fp32 mode: relative Frobenius error <= 1e-4 for the outputs and the final state.
"""
from __future__ import annotations

import concurrent.futures as cf
import json
import os

import numpy as np
import torch

import oracle

BF16_COS = 0.9999
BF16_MAXREL = 5e-3
BF16_OUT_ROUNDING = 2.0 ** -8
BF16_STATE_RELF = 5e-3
F32_RELF = 1e-4


def _np(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def metrics(x, ref) -> dict:
    x = _np(x).ravel()
    ref = _np(ref).ravel()
    nr = np.linalg.norm(ref)
    nx = np.linalg.norm(x)
    cos = float(x @ ref / (nx * nr)) if nr > 0 and nx > 0 else (1.0 if nr == nx else 0.0)
    scale = np.abs(ref).max() if ref.size else 0.0
    maxrel = float(np.abs(x - ref).max() / scale) if scale > 0 else float(np.abs(x - ref).max())
    relf = float(np.linalg.norm(x - ref) / nr) if nr > 0 else float(np.linalg.norm(x))
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    maxrms = float(np.abs(x - ref).max() / rms) if rms > 0 else 0.0
    return dict(cos=cos, maxrel=maxrel, relf=relf, max_over_rms=maxrms,
                finite=bool(np.isfinite(x).all()))


# ------------------------------------------------------------------ measured figures

def record(case: str, **figures):
    """Print one measured parity figure set (visible with ``pytest -s`` or in a failure report)
    and, when the environment variable GDN_PARITY_LOG names a file, append it there as one
    JSON line, so that a run leaves the worst errors it saw next to its pass/fail verdict."""
    line = {"case": case}
    for k, v in figures.items():
        line[k] = float(v) if isinstance(v, (float, np.floating)) else v
    print("[parity]", json.dumps(line))
    path = os.environ.get("GDN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")


def unit_metrics(x, ref):
    """Per-unit figures of two arrays shaped [U, n] (row u = every element of unit u):
    max|x - ref| / max|ref| (the unit's outputs scaled to unit range), cosine and relative
    Frobenius error, each an array of U values, plus the sums they come from (so that the
    pieces of one unit can be merged, see :func:`merge_units`)."""
    x = _np(x)
    ref = _np(ref)
    U = ref.shape[0]
    x = x.reshape(U, -1)
    ref = ref.reshape(U, -1)
    diff = x - ref
    raw = dict(maxerr=np.abs(diff).max(axis=1), scale=np.abs(ref).max(axis=1),
               xr=(x * ref).sum(axis=1), xx=(x * x).sum(axis=1), rr=(ref * ref).sum(axis=1),
               dd=(diff * diff).sum(axis=1), finite=bool(np.isfinite(x).all()))
    return _figures(raw)


def _figures(raw):
    scale, nr, nx = raw["scale"], np.sqrt(raw["rr"]), np.sqrt(raw["xx"])
    with np.errstate(divide="ignore", invalid="ignore"):
        maxrel = np.where(scale > 0, raw["maxerr"] / scale, raw["maxerr"])
        cos = np.where((nr > 0) & (nx > 0), raw["xr"] / (nx * nr), np.where(nr == nx, 1.0, 0.0))
        relf = np.where(nr > 0, np.sqrt(raw["dd"]) / nr, np.sqrt(raw["dd"]))
    return dict(raw, maxrel=maxrel, cos=cos, relf=relf)


def merge_units(pieces):
    """Merge :func:`unit_metrics` results that cover different elements of the same U units
    (e.g. consecutive segments of tokens) into the figures of the whole units."""
    raw = dict(maxerr=np.max([p["maxerr"] for p in pieces], axis=0),
               scale=np.max([p["scale"] for p in pieces], axis=0),
               finite=all(p["finite"] for p in pieces))
    for k in ("xr", "xx", "rr", "dd"):
        raw[k] = np.sum([p[k] for p in pieces], axis=0)
    return _figures(raw)


def concat_units(pieces):
    """Concatenate :func:`unit_metrics` results of different units into one result."""
    out = {k: np.concatenate([p[k] for p in pieces])
           for k in ("maxerr", "scale", "xr", "xx", "rr", "dd")}
    out["finite"] = all(p["finite"] for p in pieces)
    return _figures(out)


def check_units(parts, case: str, maxrel: float = None, cos: float = BF16_COS,
                relf: float = None):
    """Every unit of a list of :func:`unit_metrics` results against its own bound: worst
    per-unit max|err|/max|ref| <= maxrel, worst cosine >= cos, worst relative Frobenius error
    <= relf (each when given).  The worst figures are recorded (see :func:`record`) before
    anything is asserted."""
    if isinstance(parts, dict):
        parts = [parts]
    m = dict(maxrel=np.concatenate([p["maxrel"] for p in parts]),
             cos=np.concatenate([p["cos"] for p in parts]),
             relf=np.concatenate([p["relf"] for p in parts]),
             finite=all(p["finite"] for p in parts))
    worst = dict(units=int(m["maxrel"].size), maxrel=float(m["maxrel"].max()),
                 cos=float(m["cos"].min()), relf=float(m["relf"].max()),
                 worst_unit=int(m["maxrel"].argmax()))
    record(case, **worst)
    assert m["finite"], f"{case}: non-finite values"
    if maxrel is not None:
        assert worst["maxrel"] <= maxrel, f"{case}: max|err|/max|ref| {worst}"
    if cos is not None:
        assert worst["cos"] >= cos, f"{case}: cosine {worst}"
    if relf is not None:
        assert worst["relf"] <= relf, f"{case}: rel-F {worst}"
    return worst


def assert_units(x, ref, case: str, maxrel: float = None, cos: float = BF16_COS,
                 relf: float = None):
    """:func:`check_units` of two [U, n] arrays (row u = every element of unit u)."""
    return check_units(unit_metrics(x, ref), case, maxrel=maxrel, cos=cos, relf=relf)


def assert_bf16_parity(out, ref, what="out"):
    """`out` may be a torch tensor (its dtype decides whether the bf16 output rounding is
    added to the bound) or an fp32/fp64 array."""
    stored_bf16 = hasattr(out, "dtype") and out.dtype == torch.bfloat16
    bound = BF16_MAXREL + (BF16_OUT_ROUNDING if stored_bf16 else 0.0)
    m = metrics(out, ref)
    assert m["finite"], f"{what}: non-finite values"
    assert m["cos"] >= BF16_COS, f"{what}: cosine {m['cos']:.7f} < {BF16_COS} ({m})"
    assert m["maxrel"] <= bound, f"{what}: max|err|/max|ref| {m['maxrel']:.3e} > {bound} ({m})"
    return m


def assert_state_parity(S, ref, fp32: bool = False, what="state"):
    m = metrics(S, ref)
    assert m["finite"], f"{what}: non-finite values"
    if fp32:
        assert m["relf"] <= F32_RELF, f"{what}: rel-F {m['relf']:.3e} > {F32_RELF}"
    else:
        assert m["cos"] >= BF16_COS, f"{what}: cosine {m['cos']:.7f} ({m})"
        assert m["relf"] <= BF16_STATE_RELF, f"{what}: rel-F {m['relf']:.3e} ({m})"
    return m


def assert_f32_parity(out, ref, what="out"):
    m = metrics(out, ref)
    assert m["finite"], f"{what}: non-finite values"
    assert m["relf"] <= F32_RELF, f"{what}: rel-F {m['relf']:.3e} > {F32_RELF} ({m})"
    return m


# ------------------------------------------------------------------ oracle on selected heads

def head_slice(inp, b: int, h: int, t0: int = 0, t1=None):
    """Inputs of one (batch row, value head) unit as a 1-key-head / 1-value-head layer
    (depthwise conv and GQA make this exact): returns kwargs for ``oracle.layer``."""
    sh = inp.shape
    d, Hk, Hv = sh.head_dim, sh.num_k_heads, sh.num_v_heads
    r = Hv // Hk
    kh = h // r
    t1 = sh.seqlen if t1 is None else t1
    cpu = lambda t: t.detach().to("cpu")
    kw = dict(num_k_heads=1, num_v_heads=1, head_dim=d,
              a=cpu(inp.a[b:b + 1, t0:t1, h:h + 1]), b=cpu(inp.b[b:b + 1, t0:t1, h:h + 1]),
              A_log=cpu(inp.A_log[h:h + 1]), dt_bias=cpu(inp.dt_bias[h:h + 1]),
              state=cpu(inp.state[b:b + 1, h:h + 1]))
    if sh.conv_width > 0:
        idx = torch.cat([torch.arange(kh * d, (kh + 1) * d),
                         torch.arange(Hk * d + kh * d, Hk * d + (kh + 1) * d),
                         torch.arange(2 * Hk * d + h * d, 2 * Hk * d + (h + 1) * d)])
        idx_dev = idx.to(inp.x.device)
        kw["x"] = cpu(inp.x[b:b + 1, t0:t1].index_select(2, idx_dev))
        kw["conv_weight"] = cpu(inp.conv_weight.index_select(0, idx_dev))
        kw["conv_state"] = cpu(inp.conv_state[b:b + 1].index_select(2, idx_dev))
    else:
        kw["q"] = cpu(inp.q[b:b + 1, t0:t1, kh:kh + 1])
        kw["k"] = cpu(inp.k[b:b + 1, t0:t1, kh:kh + 1])
        kw["v"] = cpu(inp.v[b:b + 1, t0:t1, h:h + 1])
    return kw


def kh_slice(inp, b: int, kh: int, t0: int = 0, t1=None, state=None, conv_state=None):
    """Inputs of key head kh of batch row b with its r value heads, as a 1-key-head /
    r-value-head layer (exact: the conv is depthwise and value head h reads key head h / r).
    ``state`` [1, r, d, d] / ``conv_state`` [1, W-1, (2 + r) d] replace the inputs' own."""
    sh = inp.shape
    d, Hk, Hv = sh.head_dim, sh.num_k_heads, sh.num_v_heads
    r = Hv // Hk
    h0 = kh * r
    t1 = sh.seqlen if t1 is None else t1
    cpu = lambda t: t.detach().to("cpu")
    kw = dict(num_k_heads=1, num_v_heads=r, head_dim=d, nthreads=r,
              a=cpu(inp.a[b:b + 1, t0:t1, h0:h0 + r]), b=cpu(inp.b[b:b + 1, t0:t1, h0:h0 + r]),
              A_log=cpu(inp.A_log[h0:h0 + r]), dt_bias=cpu(inp.dt_bias[h0:h0 + r]),
              state=cpu(inp.state[b:b + 1, h0:h0 + r]) if state is None else state)
    if sh.conv_width > 0:
        idx = torch.cat([torch.arange(kh * d, (kh + 1) * d),
                         torch.arange(Hk * d + kh * d, Hk * d + (kh + 1) * d),
                         torch.arange(2 * Hk * d + h0 * d, 2 * Hk * d + (h0 + r) * d)])
        idx_dev = idx.to(inp.x.device)
        kw["x"] = cpu(inp.x[b:b + 1, t0:t1].index_select(2, idx_dev))
        kw["conv_weight"] = cpu(inp.conv_weight.index_select(0, idx_dev))
        kw["conv_state"] = (cpu(inp.conv_state[b:b + 1].index_select(2, idx_dev))
                            if conv_state is None else conv_state)
    else:
        kw["q"] = cpu(inp.q[b:b + 1, t0:t1, kh:kh + 1])
        kw["k"] = cpu(inp.k[b:b + 1, t0:t1, kh:kh + 1])
        kw["v"] = cpu(inp.v[b:b + 1, t0:t1, h0:h0 + r])
    return kw


def oracle_many(jobs, workers: int = None):
    """oracle.layer over a list of keyword sets, several at a time (the C oracle runs outside
    the interpreter lock); results in order."""
    if workers is None:
        workers = max(1, len(os.sched_getaffinity(0)) // 3)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda kw: oracle.layer(**kw), jobs))


def oracle_full(inp, **opts):
    """The oracle over every unit of a (small) workload."""
    kw = dict(num_k_heads=inp.shape.num_k_heads, num_v_heads=inp.shape.num_v_heads,
              head_dim=inp.shape.head_dim, a=inp.a, b=inp.b, A_log=inp.A_log,
              dt_bias=inp.dt_bias, state=inp.state)
    if inp.shape.conv_width > 0:
        kw.update(x=inp.x, conv_weight=inp.conv_weight, conv_state=inp.conv_state)
    else:
        kw.update(q=inp.q, k=inp.k, v=inp.v)
    kw.update(opts)
    return oracle.layer(**kw)


# ------------------------------------------------------------------ CUDA path

def to_device(inp, device="cuda"):
    """Copy every tensor of a GDNInputs to the device (a new GDNInputs-like namespace)."""
    import copy
    out = copy.copy(inp)
    for k, v in inp.__dict__.items():
        if isinstance(v, torch.Tensor):
            setattr(out, k, v.to(device).contiguous())
    return out


def run_prefill(gdn, inp, out_dtype=torch.bfloat16, state_slots=None, **kw):
    """Run gdn_chunk_prefill on device inputs; returns out (the state is updated in place)."""
    sh = inp.shape
    out = torch.empty(sh.batch, sh.seqlen, sh.num_v_heads, sh.head_dim, dtype=out_dtype,
                      device=inp.state.device)
    if sh.conv_width > 0:
        gdn.gdn_chunk_prefill(inp.x, None, None, inp.a, inp.b, inp.A_log, inp.dt_bias, inp.state,
                              out, num_k_heads=sh.num_k_heads, conv_weight=inp.conv_weight,
                              conv_state=inp.conv_state, state_slots=state_slots, **kw)
    else:
        gdn.gdn_chunk_prefill(inp.q, inp.k, inp.v, inp.a, inp.b, inp.A_log, inp.dt_bias,
                              inp.state, out, state_slots=state_slots, **kw)
    return out
