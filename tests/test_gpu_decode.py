"""Parity of gdn_decode_step (one fused kernel per step, through the C ABI) with the oracle.

The 27B-shape batched decode (16/48 heads, GQA 1:3, width-4 conv): every batch row's state
comes from a 512-token prefill (4B-workload-style inputs: conv, half the heads strongly
decayed), then 256 decode steps run on the HBM-resident state.  Sampled (row, head) units
are checked against the fp64 oracle at every step's output and at steps 1, 16, 64, 256 for
the state, so drift would show.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import (assert_bf16_parity, assert_f32_parity, assert_state_parity,
                          head_slice, oracle_full, run_prefill, to_device)

pytestmark = pytest.mark.gpu

CHECK_STEPS = (1, 16, 64, 256)


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_13_gb300 as m
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def _decode_step(gdn, dev, dec, t, out):
    sh = dev.shape
    B, Hv = sh.batch, sh.num_v_heads
    a = dec["a"][t].view(B, 1, Hv)
    b = dec["b"][t].view(B, 1, Hv)
    if sh.conv_width > 0:
        x = dec["x"][t].view(B, 1, -1)
        gdn.gdn_decode_step(x, None, None, a, b, dev.A_log, dev.dt_bias, dev.state, out,
                            num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight,
                            conv_state=dev.conv_state)
    else:
        gdn.gdn_decode_step(dec["q"][t].view(B, 1, sh.num_k_heads, 128),
                            dec["k"][t].view(B, 1, sh.num_k_heads, 128),
                            dec["v"][t].view(B, 1, Hv, 128), a, b, dev.A_log, dev.dt_bias,
                            dev.state, out)


def _oracle_decode_segment(kw_state, dec, b, h, t0, t1, sh):
    """Oracle over decode steps [t0, t1) of unit (b, h), starting from kw_state."""
    d, Hk, Hv = 128, sh.num_k_heads, sh.num_v_heads
    kh = h // (Hv // Hk)
    cpu = lambda t: t.detach().float().cpu()
    idx = torch.cat([torch.arange(kh * d, (kh + 1) * d),
                     torch.arange(Hk * d + kh * d, Hk * d + (kh + 1) * d),
                     torch.arange(2 * Hk * d + h * d, 2 * Hk * d + (h + 1) * d)]).to(dec["x"].device)
    x = cpu(dec["x"][t0:t1, b].index_select(1, idx)).unsqueeze(0)
    a = cpu(dec["a"][t0:t1, b, h]).view(1, -1, 1)
    bb = cpu(dec["b"][t0:t1, b, h]).view(1, -1, 1)
    kw = dict(kw_state)
    kw.update(x=x, a=a, b=bb)
    return oracle.layer(**kw)


@pytest.mark.parametrize("B", gi.DECODE_BATCHES_27B)
def test_27b_decode_256_steps(gdn, B):
    sh = gi.GDNShape(B, 512, 16, 48, conv_width=4)
    pre = gi.make_inputs_device(sh, seed=3000 + B, device="cuda", strong_decay_half=True)
    units = sorted({(0, 0), (B - 1, 47), (B // 2, 23), (min(1, B - 1), 30)})
    # the oracle's inputs are taken before the prefill updates the states in place
    sliced = {u: head_slice(pre, *u) for u in units}
    out_pre = run_prefill(gdn, pre)
    steps = 256
    dec = gi.make_decode_inputs_device(gi.GDNShape(B, 1, 16, 48, conv_width=4), steps,
                                       seed=3500 + B, device="cuda")
    # oracle: the 512-token prefill of each sampled unit
    ostate = {}
    for (b, h) in units:
        kw = sliced[(b, h)]
        r = oracle.layer(**kw)
        assert_bf16_parity(out_pre[b, :, h].cpu(), r.out[0, :, 0], what=f"prefill {b},{h}")
        ostate[(b, h)] = dict(num_k_heads=1, num_v_heads=1, head_dim=128, A_log=kw["A_log"],
                              dt_bias=kw["dt_bias"], conv_weight=kw["conv_weight"],
                              state=r.state, conv_state=r.conv_state)
    dsh = gi.GDNShape(B, 1, 16, 48, conv_width=4)
    pre.shape = dsh
    outs = torch.empty(steps, B, 48, 128, dtype=torch.bfloat16, device="cuda")
    snaps = {}
    for t in range(steps):
        _decode_step(gdn, pre, dec, t, outs[t].view(B, 1, 48, 128))
        if t + 1 in CHECK_STEPS:
            snaps[t + 1] = {u: pre.state[u[0], u[1]].cpu() for u in units}
    assert gdn.gdn_get_device_error() == 0
    outs_h = outs.cpu()
    for (b, h) in units:
        st = ostate[(b, h)]
        t0 = 0
        for t1 in CHECK_STEPS:
            r = _oracle_decode_segment(st, dec, b, h, t0, t1, dsh)
            assert_bf16_parity(outs_h[t0:t1, b, h], r.out[0, :, 0], what=f"out {b},{h} steps<{t1}")
            assert_state_parity(snaps[t1][(b, h)], r.state[0, 0], what=f"state {b},{h} @ {t1}")
            st = dict(st, state=r.state, conv_state=r.conv_state)
            t0 = t1


def test_decode_fp32_mode(gdn):
    """All-fp32 decode (GQA 1:2, conv), 8 steps from a random state: rel error <= 1e-4."""
    sh = gi.GDNShape(2, 1, 2, 4, conv_width=4)
    inp = gi.make_inputs(sh, seed=3700, dtype="f32", state="normal", state_std=0.3)
    inp.conv_state = torch.randn(inp.conv_state.shape, generator=torch.Generator().manual_seed(3))
    ref_state, ref_cs = inp.state.clone(), inp.conv_state.clone()
    dev = to_device(inp)
    dec = gi.make_decode_inputs_device(sh, 8, seed=3701, device="cuda", dtype="f32")
    out = torch.empty(8, 2, 4, 128, device="cuda")
    for t in range(8):
        _decode_step(gdn, dev, dec, t, out[t].view(2, 1, 4, 128))
    kw = dict(num_k_heads=2, num_v_heads=4, x=dec["x"].transpose(0, 1).cpu(),
              a=dec["a"].transpose(0, 1).cpu(), b=dec["b"].transpose(0, 1).cpu(),
              A_log=inp.A_log, dt_bias=inp.dt_bias, conv_weight=inp.conv_weight,
              state=ref_state, conv_state=ref_cs)
    r = oracle.layer(**kw)
    assert_f32_parity(out.transpose(0, 1).cpu(), r.out)
    assert_state_parity(dev.state.cpu(), r.state, fp32=True)
    np.testing.assert_array_equal(dev.conv_state.cpu().numpy(), r.conv_state)


@pytest.mark.parametrize("Hk,Hv", [(4, 4), (2, 4), (1, 8)])
def test_decode_without_conv(gdn, Hk, Hv):
    """q, k, v given post-conv, GQA 1:1 / 1:2 / 1:8 (cluster sizes 8, 8, 8)."""
    B = 3
    sh = gi.GDNShape(B, 1, Hk, Hv)
    inp = gi.make_inputs(sh, seed=3800 + Hv, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = torch.empty(B, 1, Hv, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                        out)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


def test_decode_slots(gdn):
    """Decode rows addressed through state_slots, one padded row (-1) left untouched, and an
    out-of-range row reported."""
    sh = gi.GDNShape(3, 1, 2, 6, conv_width=4)
    inp = gi.make_inputs(sh, seed=3900, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    dev = to_device(inp)
    bank = torch.zeros(4, 6, 128, 128, device="cuda")
    cbank = torch.zeros(4, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    bank[2], bank[0] = dev.state[0], dev.state[2]
    cbank[2], cbank[0] = dev.conv_state[0], dev.conv_state[2]
    slots = torch.tensor([2, -1, 0], dtype=torch.int32, device="cuda")
    out = torch.zeros(3, 1, 6, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                        num_k_heads=2, conv_weight=dev.conv_weight, conv_state=cbank,
                        state_slots=slots)
    assert gdn.gdn_get_device_error() == 0
    o = out.cpu()
    assert_bf16_parity(o[0], ref.out[0])
    assert_bf16_parity(o[2], ref.out[2])
    assert torch.count_nonzero(o[1]) == 0
    assert_state_parity(bank[2].cpu(), ref.state[0])
    assert_state_parity(bank[0].cpu(), ref.state[2])
    assert torch.count_nonzero(bank[1]) == 0 and torch.count_nonzero(bank[3]) == 0
    np.testing.assert_array_equal(cbank[2].float().cpu().numpy(), ref.conv_state[0])
    np.testing.assert_array_equal(cbank[0].float().cpu().numpy(), ref.conv_state[2])
    bad = torch.tensor([9, -1, -1], dtype=torch.int32, device="cuda")
    gdn.gdn_decode_step(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                        num_k_heads=2, conv_weight=dev.conv_weight, conv_state=cbank,
                        state_slots=bad)
    assert gdn.gdn_get_device_error() == 6


def test_prefill_of_one_token_equals_decode(gdn):
    """prefill(T=1) and one decode step compute the same thing (both against the oracle and
    against each other)."""
    sh = gi.GDNShape(2, 1, 16, 48, conv_width=4)
    inp = gi.make_inputs(sh, seed=3950, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    d1, d2 = to_device(inp), to_device(inp)
    o1 = run_prefill(gdn, d1)
    o2 = torch.empty_like(o1)
    gdn.gdn_decode_step(d2.x, None, None, d2.a, d2.b, d2.A_log, d2.dt_bias, d2.state, o2,
                        num_k_heads=16, conv_weight=d2.conv_weight, conv_state=d2.conv_state)
    for o in (o1, o2):
        assert_bf16_parity(o.cpu(), ref.out)
    assert_bf16_parity(o1.cpu(), o2.cpu())
    assert_state_parity(d1.state.cpu(), d2.state.cpu())
    assert torch.equal(d1.conv_state, d2.conv_state)


def _streaming_batch(Hk):
    """A batch with at least two (sequence, key head) items per SM, so that gdn_decode_step
    takes its streaming kernel rather than the per-item cluster kernel."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (2 * sms + Hk - 1) // Hk + 1


@pytest.mark.parametrize("dtype,conv,Hk,Hv", [("bf16", True, 4, 12), ("f32", True, 4, 8),
                                                ("bf16", False, 2, 16), ("bf16", False, 8, 8)])
def test_decode_streaming_kernel(gdn, dtype, conv, Hk, Hv):
    """Batches large enough for the streaming decode kernel: bf16 / fp32, with and without the
    conv, GQA 1:3 / 1:2 / 1:8 / 1:1; two steps, every unit against the oracle."""
    B = _streaming_batch(Hk)
    sh = gi.GDNShape(B, 1, Hk, Hv, conv_width=4 if conv else 0)
    inp = gi.make_inputs(sh, seed=4100 + Hv + (7 if conv else 0), dtype=dtype, state="normal",
                         state_std=0.2)
    if conv:
        inp.conv_state = torch.randn(inp.conv_state.shape,
                                     generator=torch.Generator().manual_seed(41))
        if dtype == "bf16":
            inp.conv_state = inp.conv_state.to(torch.bfloat16)
    ref1 = oracle_full(inp)
    dev = to_device(inp)
    odt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.empty(B, 1, Hv, 128, dtype=odt, device="cuda")
    if conv:
        gdn.gdn_decode_step(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                            out, num_k_heads=Hk, conv_weight=dev.conv_weight,
                            conv_state=dev.conv_state)
    else:
        gdn.gdn_decode_step(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias,
                            dev.state, out)
    assert gdn.gdn_get_device_error() == 0
    if dtype == "bf16":
        assert_bf16_parity(out.cpu(), ref1.out)
        assert_state_parity(dev.state.cpu(), ref1.state)
    else:
        assert_f32_parity(out.cpu(), ref1.out)
        assert_state_parity(dev.state.cpu(), ref1.state, fp32=True)
    if conv:
        np.testing.assert_array_equal(dev.conv_state.float().cpu().numpy(), ref1.conv_state)


def test_decode_streaming_slots(gdn):
    """Streaming-size batch addressed through state_slots: padded rows (-1) untouched, the
    rest equal to the oracle, and an out-of-range slot reported."""
    Hk, Hv = 4, 12
    B = _streaming_batch(Hk)
    sh = gi.GDNShape(B, 1, Hk, Hv, conv_width=4)
    inp = gi.make_inputs(sh, seed=4200, dtype="bf16", state="normal", state_std=0.2)
    ref = oracle_full(inp)
    dev = to_device(inp)
    nbank = B + 3
    perm = torch.randperm(nbank, generator=torch.Generator().manual_seed(42))[:B]
    slots = perm.clone().to(torch.int32)
    slots[::7] = -1                                   # padded rows
    bank = torch.zeros(nbank, Hv, 128, 128, device="cuda")
    cbank = torch.zeros(nbank, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        if slots[b] >= 0:
            bank[slots[b]] = dev.state[b]
            cbank[slots[b]] = dev.conv_state[b]
    before = bank.clone()
    out = torch.zeros(B, 1, Hv, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                        num_k_heads=Hk, conv_weight=dev.conv_weight, conv_state=cbank,
                        state_slots=slots.cuda())
    assert gdn.gdn_get_device_error() == 0
    o = out.cpu()
    for b in range(B):
        s = int(slots[b])
        if s < 0:
            assert torch.count_nonzero(o[b]) == 0
            continue
        assert_bf16_parity(o[b], ref.out[b], what=f"out row {b}")
        assert_state_parity(bank[s].cpu(), ref.state[b], what=f"state row {b}")
        np.testing.assert_array_equal(cbank[s].float().cpu().numpy(), ref.conv_state[b])
    used = set(int(s) for s in slots if s >= 0)
    for s in range(nbank):
        if s not in used:
            assert torch.equal(bank[s], before[s])
    bad = slots.clone()
    bad[3] = nbank + 5
    gdn.gdn_decode_step(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                        num_k_heads=Hk, conv_weight=dev.conv_weight, conv_state=cbank,
                        state_slots=bad.cuda())
    assert gdn.gdn_get_device_error() == 6
