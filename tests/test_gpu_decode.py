"""Parity of gdn_decode_step (one fused kernel per step, through the C ABI) with the oracle.

The 27B-shape batched decode (16/48 heads, GQA 1:3, width-4 conv): every batch row's state
comes from a 512-token prefill (4B-workload-style inputs: conv, half the heads strongly
decayed), then 256 decode steps run on the HBM-resident state.  Every (row, head) unit is
checked against the fp64 oracle at every step's output (bf16 and fp32 outputs) and at steps
1, 16, 64, 256 for the state, so drift would show.
"""
import concurrent.futures as cf
import copy
import os

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import (BF16_MAXREL, BF16_OUT_ROUNDING, BF16_STATE_RELF, assert_bf16_parity,
                          assert_f32_parity, assert_state_parity, check_units, concat_units,
                          kh_slice, merge_units, oracle_full, run_prefill, to_device,
                          unit_metrics)

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


@pytest.mark.parametrize("B", gi.DECODE_BATCHES_27B)
def test_27b_decode_256_steps(gdn, B):
    """Every (row, value head) unit: the 512-token prefill that sets the state, then 256
    decode steps run twice from it, with bf16 and with fp32 outputs.  Against the oracle:
    every step's output (fp32: max|o - o_ref| / max|o_ref| <= 5e-3 per unit over the 256
    steps, bf16: that plus the output's own rounding; cosine >= 0.9999) and every unit's state
    after steps 1, 16, 64 and 256 (cosine >= 0.9999, rel-F <= 5e-3)."""
    Hk, Hv, d = 16, 48, 128
    r = Hv // Hk
    steps = 256
    sh = gi.GDNShape(B, 512, Hk, Hv, conv_width=4)
    pre = gi.make_inputs_device(sh, seed=3000 + B, device="cuda", strong_decay_half=True)
    # the oracle's inputs, taken before the prefill updates the states in place
    host = copy.copy(pre)
    for k, v in pre.__dict__.items():
        if isinstance(v, torch.Tensor):
            setattr(host, k, v.cpu())
    out_pre = run_prefill(gdn, pre)
    dsh = gi.GDNShape(B, 1, Hk, Hv, conv_width=4)
    dec = gi.make_decode_inputs_device(dsh, steps, seed=3500 + B, device="cuda")
    s0, c0 = pre.state.clone(), pre.conv_state.clone()
    pre.shape = dsh
    outs, snaps = {}, {}
    for odt in (torch.bfloat16, torch.float32):
        pre.state.copy_(s0)
        pre.conv_state.copy_(c0)
        o = torch.empty(steps, B, Hv, d, dtype=odt, device="cuda")
        sn = []
        for t in range(steps):
            _decode_step(gdn, pre, dec, t, o[t].view(B, 1, Hv, d))
            if t + 1 in CHECK_STEPS:
                sn.append(pre.state.clone())
        assert gdn.gdn_get_device_error() == 0
        outs[odt] = o.cpu()
        snaps[odt] = sn
    # the output dtype does not change the recurrence: the same states, bit for bit
    for a_, b_ in zip(snaps[torch.bfloat16], snaps[torch.float32]):
        assert torch.equal(a_, b_)
    snaps = {torch.bfloat16: [x.cpu() for x in snaps[torch.bfloat16]]}
    out_pre_h = out_pre.cpu()
    dec_h = {k: v.cpu() for k, v in dec.items()}
    C = dsh.conv_channels

    def rows(o):            # [t, r, d] -> [r, t*d]
        o = np.asarray(o, dtype=np.float64)
        return np.ascontiguousarray(o.transpose(1, 0, 2).reshape(o.shape[1], -1))

    def job(b, kh):
        kw = kh_slice(host, b, kh)
        res = oracle.layer(**kw)
        h0 = kh * r
        m = dict(pre=[unit_metrics(rows(out_pre_h[b, :, h0:h0 + r].double().numpy()),
                                   rows(res.out[0]))], o16=[], o32=[], state=[])
        idx = torch.cat([torch.arange(kh * d, (kh + 1) * d),
                         torch.arange(Hk * d + kh * d, Hk * d + (kh + 1) * d),
                         torch.arange(2 * Hk * d + h0 * d, 2 * Hk * d + (h0 + r) * d)])
        st, cst, t0 = res.state, res.conv_state, 0
        for ci, t1 in enumerate(CHECK_STEPS):
            kd = dict(kw, x=dec_h["x"][t0:t1, b].index_select(1, idx).unsqueeze(0),
                      a=dec_h["a"][t0:t1, b, h0:h0 + r].unsqueeze(0),
                      b=dec_h["b"][t0:t1, b, h0:h0 + r].unsqueeze(0), state=st, conv_state=cst)
            rd = oracle.layer(**kd)
            ref = rows(rd.out[0])
            m["o16"].append(unit_metrics(
                rows(outs[torch.bfloat16][t0:t1, b, h0:h0 + r].double().numpy()), ref))
            m["o32"].append(unit_metrics(
                rows(outs[torch.float32][t0:t1, b, h0:h0 + r].double().numpy()), ref))
            m["state"].append(unit_metrics(
                snaps[torch.bfloat16][ci][b, h0:h0 + r].double().numpy().reshape(r, -1),
                rd.state[0].reshape(r, -1)))
            st, cst, t0 = rd.state, rd.conv_state, t1
        return m

    with cf.ThreadPoolExecutor(max_workers=max(1, len(os.sched_getaffinity(0)) // r)) as ex:
        res = list(ex.map(lambda u: job(*u), [(b, kh) for b in range(B) for kh in range(Hk)]))
    parts = {k: [p for m in res for p in m[k]] for k in ("pre", "state")}
    case = f"qwen36_27b decode B{B}"
    check_units(parts["pre"], f"{case}: 512-token prefill out (bf16 out), per unit",
                maxrel=BF16_MAXREL + BF16_OUT_ROUNDING)
    # every unit over all 256 steps (its 4 segments merged); the per-segment figures (the first
    # segment is the single step 1) are recorded beside them
    for key, tag, bound in (("o32", "f32 out", BF16_MAXREL),
                            ("o16", "bf16 out", BF16_MAXREL + BF16_OUT_ROUNDING)):
        whole = concat_units([merge_units(m[key]) for m in res])
        check_units(whole, f"{case}: 256 steps out ({tag}), per unit", maxrel=bound)
        check_units([p for m in res for p in m[key]],
                    f"{case}: 256 steps out ({tag}), per unit and segment", maxrel=None, cos=None)
    check_units(parts["state"], f"{case}: state after steps 1/16/64/256", relf=BF16_STATE_RELF)


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
