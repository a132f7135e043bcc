"""The gated RMS norm fused into the output (gdn_chunk_prefill_gated, gdn_decode_step_gated)
against the fp64 oracle (the recurrence, then oracle.gated_rmsnorm of its outputs).

Covered: the tensor-core prefill with bf16 and fp32 outputs (ragged tail, GQA, conv), the
27B shape with a skipped batch row, the all-fp32 prefill, and the decode step on both of its
kernels (the per-item cluster kernel at small batch, the streaming kernel at large batch) in
bf16 and fp32.  The gate must leave the recurrent and conv state exactly as the plain call
does.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gdn_testutil
import oracle
from gdn_testutil import assert_f32_parity, oracle_full, to_device

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_13_gb300 as m
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def _gate_inputs(shape, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(*shape, generator=g)
    w = torch.rand(shape[-1], generator=g) + 0.5
    return (z.to(torch.bfloat16) if dtype == "bf16" else z), w


def _prefill(gdn, dev, out, gate=None, state_slots=None):
    sh = dev.shape
    kw = dict(state_slots=state_slots)
    if sh.conv_width > 0:
        args = (dev.x, None, None)
        kw.update(num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight,
                  conv_state=dev.conv_state)
    else:
        args = (dev.q, dev.k, dev.v)
    args = args + (dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state, out)
    if gate is None:
        gdn.gdn_chunk_prefill(*args, **kw)
    else:
        z, w = gate
        gdn.gdn_chunk_prefill_gated(*args, gate_z=z, gate_weight=w, gate_eps=EPS, **kw)


def _assert_norm_of(y, o32, z, w, bf16_out, what):
    """y must be the gated norm of the kernel's own fp32 output o32 (the same o the gated
    call normalises): fp32 arithmetic with the fast exponential, division and reciprocal root
    (relative 1e-5 per element), plus, for a bf16 output, one rounding (2^-9 relative) and a
    SiLU through the hardware tanh, z/2 (1 + tanh(z/2)), whose absolute error (at most about
    2^-11 on tanh) reaches the element as |z|/2 * 2^-11 times the normalised, weighted
    value u = w o / rms(o) (allowed twice over)."""
    ref = oracle.gated_rmsnorm(o32, z, w, EPS)
    u = oracle.gated_rmsnorm(o32, np.full(ref.shape, 60.0), w, EPS) / 60.0   # silu(60) = 60
    zz = np.abs(np.asarray(z.float().numpy(), dtype=np.float64))
    y = np.asarray(y.float().cpu().numpy(), dtype=np.float64)
    err = np.abs(y - ref)
    rel = (2.0 ** -8 if bf16_out else 0.0) + 1e-5
    tol = rel * np.abs(ref) + 1e-6 * np.abs(ref).max()
    if bf16_out:
        tol = tol + 2.0 * 0.5 * zz * 2.0 ** -11 * np.abs(u)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} elements off, worst {(err - tol).max():.3e}"


def _assert_end_to_end(y, o_plain, o_ref, z, w, bf16_out, what):
    """Against the oracle all the way (its recurrence, then its norm), element by element.

    The gated call runs the same recurrence as the plain call (its states are bit-identical)
    and normalises that fp32 output o' = o + e, where e is the recurrence's error, itself held
    to the parity bar by the plain-call tests.  Per token, with delta = max_i |e_i| (measured:
    the plain call's fp32 output against the oracle) and r = sqrt(mean(o^2) + eps) of the
    oracle's vector, |rms(o') - r| <= delta (triangle inequality of the RMS), and
    o'/rms(o') - o/r = e/rms(o') + o (1/rms(o') - 1/r) give, for delta < r,
        |u'_i - u_i| <= delta / (r - delta) * (1 + |o_i| / r),      u = o / r,
    which y = w silu(z) u inherits times |w_i silu(z_i)|.  On top come the norm's own fp32
    arithmetic, the output rounding and the hardware-tanh SiLU (as in _assert_norm_of).  A
    token whose recurrence error reaches half its own rms (delta >= r/2: an output vector far
    smaller than the state's scale, e.g. a query almost orthogonal to the stored keys, where
    the bf16 snapshot of the state costs more than the vector itself) has no useful bound:
    such tokens are counted and must stay below 1% (their gated value is still held to the
    norm of the kernel's own output by _assert_norm_of); the whole-tensor cosine >= 0.9999 is
    held as well."""
    o_ref = np.asarray(o_ref, dtype=np.float64)
    want = oracle.gated_rmsnorm(o_ref, z, w, EPS)
    yy = np.asarray(y.float().cpu().numpy(), dtype=np.float64)
    op = np.asarray(o_plain.float().cpu().numpy(), dtype=np.float64)
    zz = np.asarray(z.float().numpy(), dtype=np.float64)
    ww = np.asarray(w.float().numpy(), dtype=np.float64)
    delta = np.abs(op - o_ref).max(axis=-1, keepdims=True)
    rr = np.sqrt((o_ref ** 2).mean(axis=-1, keepdims=True) + EPS)
    silu = zz / (1.0 + np.exp(-zz))
    lin = np.abs(ww * silu) * delta / np.maximum(rr - delta, 1e-300) * (1.0 + np.abs(o_ref) / rr)
    u = np.abs(ww * o_ref / rr)
    rel = (2.0 ** -8 if bf16_out else 0.0) + 1e-5
    tol = lin + rel * np.abs(want) + 1e-6 * np.abs(want).max()
    if bf16_out:
        tol = tol + 2.0 * 0.5 * np.abs(zz) * 2.0 ** -11 * (u + lin)
    err = np.abs(yy - want)
    m = gdn_testutil.metrics(yy, want)
    ok_tok = np.broadcast_to(delta < 0.5 * rr, err.shape)
    ill = 1.0 - float((delta < 0.5 * rr).mean())
    gdn_testutil.record(what, cos=m["cos"], maxrel=m["maxrel"],
                        worst_err_over_bound=float((err / tol)[ok_tok].max()),
                        ill_conditioned_tokens=ill)
    assert m["finite"], what
    assert ill <= 0.01, f"{what}: {ill:.2%} of the tokens have a recurrence error >= rms / 2"
    bad = (err > tol) & ok_tok
    assert not bad.any(), f"{what}: {bad.sum()} elements off, worst {(err - tol)[bad].max():.3e}"
    assert m["cos"] >= 0.9999, f"{what}: {m}"


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_prefill_tensor_core_path(gdn, out_dtype):
    """bf16 inputs, GQA 1:3, width-4 conv, T = 200 (three full chunks and a ragged tail)."""
    sh = gi.GDNShape(2, 200, 2, 6, conv_width=4)
    inp = gi.make_inputs(sh, seed=6100, dtype="bf16", state="normal")
    z, w = _gate_inputs((2, 200, 6, 128), 1, "bf16")
    ref = oracle_full(inp)
    plain = to_device(inp)
    out_p = torch.empty(2, 200, 6, 128, dtype=torch.float32, device="cuda")
    _prefill(gdn, plain, out_p)
    gated = to_device(inp)
    out_g = torch.empty(2, 200, 6, 128, dtype=out_dtype, device="cuda")
    _prefill(gdn, gated, out_g, gate=(z.cuda(), w.cuda()))
    assert gdn.gdn_get_device_error() == 0
    _assert_norm_of(out_g, out_p.cpu(), z, w, out_dtype == torch.bfloat16, "gated out")
    _assert_end_to_end(out_g, out_p, ref.out, z, w, out_dtype == torch.bfloat16,
                       f"gated prefill B2 T200 ({out_dtype}) vs oracle")
    assert torch.equal(gated.state, plain.state)
    assert torch.equal(gated.conv_state, plain.conv_state)


def test_prefill_27b_shape_skipped_row(gdn):
    """A 512-token call at the 27B shape (16/48 heads); batch row 1 is skipped by
    state_slots and its outputs stay as they were.  Every head of rows 0 and 2 against the
    oracle."""
    sh = gi.GDNShape(3, 512, 16, 48, conv_width=4)
    inp = gi.make_inputs(sh, seed=6200, dtype="bf16", state="normal")
    z, w = _gate_inputs((3, 512, 48, 128), 2, "bf16")
    slots = torch.tensor([2, -1, 0], dtype=torch.int32, device="cuda")
    outs = []
    for gate, dt in ((None, torch.float32), ((z.cuda(), w.cuda()), torch.bfloat16)):
        dev = to_device(inp)
        st = dev.state.clone()
        dev.state[2], dev.state[0] = st[0], st[2]
        cs = dev.conv_state.clone()
        dev.conv_state[2], dev.conv_state[0] = cs[0], cs[2]
        out = torch.full((3, 512, 48, 128), 7.0, dtype=dt, device="cuda")
        _prefill(gdn, dev, out, gate=gate, state_slots=slots)
        outs.append(out.cpu())
    assert gdn.gdn_get_device_error() == 0
    o32, o = outs
    assert torch.all(o[1].float() == 7.0)
    _assert_norm_of(o[0::2], o32[0::2], z[0::2], w, True, "gated out")
    ref = oracle_full(inp)
    _assert_end_to_end(o[0::2], o32[0::2], ref.out[0::2], z[0::2], w, True,
                       "gated prefill 27B-shape T512 (rows 0, 2) vs oracle")


def test_prefill_fp32_mode(gdn):
    """All-fp32 mode (FMA-pipe prefill, then the norm as a pass of its own)."""
    sh = gi.GDNShape(2, 130, 4, 8, conv_width=0)
    inp = gi.make_inputs(sh, seed=6300, dtype="f32", state="normal")
    z, w = _gate_inputs((2, 130, 8, 128), 3, "f32")
    ref = oracle_full(inp)
    want = oracle.gated_rmsnorm(ref.out, z, w, EPS)
    dev = to_device(inp)
    out = torch.empty(2, 130, 8, 128, device="cuda")
    _prefill(gdn, dev, out, gate=(z.cuda(), w.cuda()))
    assert gdn.gdn_get_device_error() == 0
    assert_f32_parity(out.cpu(), want, what="gated out")


def _decode_run(gdn, dev, x_or_qkv, a, b, steps, gate_zs=None, w=None, out_dtype=torch.bfloat16):
    """`steps` decode steps from dev's state; returns the outputs [B, steps, Hv, 128]."""
    sh = dev.shape
    B, Hv = sh.batch, sh.num_v_heads
    outs = torch.empty(B, steps, Hv, 128, dtype=out_dtype, device="cuda")
    for t in range(steps):
        o = torch.empty(B, 1, Hv, 128, dtype=out_dtype, device="cuda")
        sl = lambda u: u[:, t:t + 1].contiguous()
        if sh.conv_width > 0:
            args = (sl(x_or_qkv), None, None)
            kw = dict(num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight,
                      conv_state=dev.conv_state)
        else:
            args = tuple(sl(u) for u in x_or_qkv)
            kw = {}
        args = args + (sl(a), sl(b), dev.A_log, dev.dt_bias, dev.state, o)
        if gate_zs is None:
            gdn.gdn_decode_step(*args, **kw)
        else:
            gdn.gdn_decode_step_gated(*args, gate_z=sl(gate_zs), gate_weight=w, gate_eps=EPS,
                                      **kw)
        outs[:, t:t + 1] = o
    return outs


@pytest.mark.parametrize("B", [1, 8, 32])
def test_decode_27b_shape(gdn, B):
    """27B shape decode, 4 steps from a random state: B = 1 and 8 run the per-item cluster
    kernel (the norm's partial sums cross CTAs), B = 32 the streaming kernel."""
    steps = 4
    sh = gi.GDNShape(B, steps, 16, 48, conv_width=4)
    inp = gi.make_inputs(sh, seed=6400 + B, dtype="bf16", state="normal", state_std=0.3)
    inp.conv_state = gi.to_bf16(np.random.default_rng(B).standard_normal(
        inp.conv_state.shape).astype(np.float32))
    z, w = _gate_inputs((B, steps, 48, 128), 4 + B, "bf16")
    ref = oracle_full(inp)
    plain, gated = to_device(inp), to_device(inp)
    out_p = _decode_run(gdn, plain, plain.x, plain.a, plain.b, steps, out_dtype=torch.float32)
    out = _decode_run(gdn, gated, gated.x, gated.a, gated.b, steps, z.cuda(), w.cuda())
    assert gdn.gdn_get_device_error() == 0
    _assert_end_to_end(out, out_p, ref.out, z, w, True, f"gated decode 27B-shape B{B} vs oracle")
    assert torch.equal(gated.state, plain.state)
    assert torch.equal(gated.conv_state, plain.conv_state)


@pytest.mark.parametrize("B", [2, 40])
def test_decode_fp32_mode(gdn, B):
    """All-fp32 decode, no conv, 16 key / 16 value heads: B = 2 on the cluster kernel,
    B = 40 (640 items) on the streaming kernel."""
    steps = 3
    sh = gi.GDNShape(B, steps, 16, 16, conv_width=0)
    inp = gi.make_inputs(sh, seed=6500 + B, dtype="f32", state="normal", state_std=0.3)
    z, w = _gate_inputs((B, steps, 16, 128), 5 + B, "f32")
    ref = oracle_full(inp)
    want = oracle.gated_rmsnorm(ref.out, z, w, EPS)
    dev = to_device(inp)
    out = _decode_run(gdn, dev, (dev.q, dev.k, dev.v), dev.a, dev.b, steps, z.cuda(), w.cuda(),
                      out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    assert_f32_parity(out.cpu(), want, what="gated decode out")
