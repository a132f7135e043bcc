"""Parity of gdn_chunk_prefill (CUDA, through the C ABI) with the fp64 oracle.

Workloads follow the Qwen3.5/3.6 gated-delta-net layer shapes (d = 128): the tiny fp32
layer, the 0.8B-shape sweep over T (ragged tails included), and the 4B-shape layer with conv
and strongly decayed heads (small, then at full size with every unit checked, fp32 and bf16
outputs).
"""
import math

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import (BF16_MAXREL, BF16_OUT_ROUNDING, BF16_STATE_RELF, assert_bf16_parity,
                          assert_f32_parity, assert_state_parity, assert_units, oracle_full,
                          run_prefill, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_13_gb300 as m
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def test_tiny_fp32_layer(gdn):
    """B=1, T=16, 16/16 heads, fp32 throughout, zero initial state: rel error <= 1e-4."""
    sh = gi.GDNShape(1, 16, 16, 16)
    inp = gi.make_inputs(sh, seed=0, dtype="f32", state="zero")
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = run_prefill(gdn, dev, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    assert_f32_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state, fp32=True)


@pytest.mark.parametrize("T", gi.SEQLEN_SWEEP_08B)
def test_08b_shape_sweep(gdn, T):
    """0.8B shape (16/16 heads), bf16 inputs, fp32 state ~ N(0, 0.02^2), T swept."""
    sh = gi.GDNShape(1, T, 16, 16)
    inp = gi.make_inputs(sh, seed=1000 + T, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = run_prefill(gdn, dev)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129])
def test_fp32_mode_ragged(gdn, T):
    """All-fp32 mode on ragged lengths around the chunk size, GQA 1:2, random state."""
    sh = gi.GDNShape(2, T, 2, 4)
    inp = gi.make_inputs(sh, seed=2000 + T, dtype="f32", state="normal", state_std=0.5)
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = run_prefill(gdn, dev, out_dtype=torch.float32)
    assert gdn.gdn_get_device_error() == 0
    assert_f32_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state, fp32=True)


def test_bf16_in_fp32_out(gdn):
    sh = gi.GDNShape(1, 100, 16, 16)
    inp = gi.make_inputs(sh, seed=3100, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = run_prefill(gdn, dev, out_dtype=torch.float32)
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


def test_4b_shape_conv_small(gdn):
    """4B shape (16/32 heads, GQA 1:2) with the width-4 conv, half the heads strongly
    decayed, B=2, T=300: every unit against the oracle, conv state bit-exact."""
    sh = gi.GDNShape(2, 300, 16, 32, conv_width=4)
    inp = gi.make_inputs(sh, seed=2001, dtype="bf16", strong_decay_half=True)
    inp.conv_state = gi.to_bf16(np.random.default_rng(5).standard_normal(
        inp.conv_state.shape).astype(np.float32))
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = run_prefill(gdn, dev)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)
    np.testing.assert_array_equal(dev.conv_state.float().cpu().numpy(), ref.conv_state)


@pytest.fixture(scope="module")
def full_4b():
    """The full 4B-shape workload (B=4, T=4096, 16/32 heads, conv, strong decay on value heads
    0..15) and the oracle over all of it (128 units x 4096 tokens)."""
    sh = gi.GDNShape(4, 4096, 16, 32, conv_width=4)
    inp = gi.make_inputs(sh, seed=2000, dtype="bf16", strong_decay_half=True)
    return inp, oracle_full(inp)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_4b_shape_full_size_every_unit(gdn, full_4b, out_dtype):
    """Every (batch, value head) unit of the full 4B-shape call against the oracle, over all
    4096 tokens: with fp32 outputs max|o - o_ref| / max|o_ref| <= 5e-3 per unit and cosine
    >= 0.9999 (the stated bar, no allowance); with bf16 outputs the same plus the output's own
    rounding.  The final state of every unit: cosine >= 0.9999, rel-F <= 5e-3."""
    inp, ref = full_4b
    sh = inp.shape
    B, T, Hv, d = sh.batch, sh.seqlen, sh.num_v_heads, sh.head_dim
    dev = to_device(inp)
    out = run_prefill(gdn, dev, out_dtype=out_dtype)
    assert gdn.gdn_get_device_error() == 0
    tag = "f32" if out_dtype == torch.float32 else "bf16"
    bound = BF16_MAXREL + (BF16_OUT_ROUNDING if out_dtype == torch.bfloat16 else 0.0)
    units = lambda o: np.ascontiguousarray(np.asarray(o, dtype=np.float64)
                                           .transpose(0, 2, 1, 3).reshape(B * Hv, T * d))
    assert_units(units(out.double().cpu().numpy()), units(ref.out),
                 f"qwen35_4b B4 T4096 out ({tag} out), per unit", maxrel=bound)
    assert_units(dev.state.double().cpu().numpy().reshape(B * Hv, -1),
                 ref.state.reshape(B * Hv, -1), f"qwen35_4b B4 T4096 final state ({tag} out)",
                 relf=BF16_STATE_RELF)
    # conv state: the last 3 pre-conv inputs of every channel, bit for bit
    np.testing.assert_array_equal(dev.conv_state.cpu().float().numpy(),
                                  inp.x[:, -3:].float().numpy())


def test_slots_skip_and_permutation(gdn):
    """state_slots maps batch entries to state rows; a negative entry skips the entry (its
    state row and outputs stay untouched)."""
    sh = gi.GDNShape(3, 70, 2, 4, conv_width=4)
    inp = gi.make_inputs(sh, seed=4000, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    dev = to_device(inp)
    # state bank of 5 rows; entry 0 -> row 3, entry 1 skipped, entry 2 -> row 0
    bank = torch.randn(5, 4, 128, 128, device="cuda") * 0.02
    cbank = torch.randn(5, 3, sh.conv_channels, device="cuda").to(torch.bfloat16)
    bank[3] = dev.state[0]
    bank[0] = dev.state[2]
    cbank[3] = dev.conv_state[0]
    cbank[0] = dev.conv_state[2]
    before = bank.clone()
    cbefore = cbank.clone()
    slots = torch.tensor([3, -1, 0], dtype=torch.int32, device="cuda")
    out = torch.full((3, 70, 4, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_chunk_prefill(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                          num_k_heads=2, conv_weight=dev.conv_weight, conv_state=cbank,
                          state_slots=slots)
    assert gdn.gdn_get_device_error() == 0
    o = out.cpu()
    assert_bf16_parity(o[0], ref.out[0])
    assert_bf16_parity(o[2], ref.out[2])
    assert torch.all(o[1].float() == 7.0)
    assert_state_parity(bank[3].cpu(), ref.state[0])
    assert_state_parity(bank[0].cpu(), ref.state[2])
    for row in (1, 2, 4):
        assert torch.equal(bank[row], before[row])
        assert torch.equal(cbank[row], cbefore[row])
    np.testing.assert_array_equal(cbank[3].float().cpu().numpy(), ref.conv_state[0])


def test_out_of_range_slot_is_reported(gdn):
    sh = gi.GDNShape(2, 20, 2, 2)
    dev = to_device(gi.make_inputs(sh, seed=4100, dtype="bf16", state="normal"))
    before = dev.state.clone()
    out = torch.zeros(2, 20, 2, 128, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([5, -1], dtype=torch.int32, device="cuda")
    gdn.gdn_chunk_prefill(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                          out, state_slots=slots)
    assert gdn.gdn_get_device_error() == 6
    assert gdn.gdn_get_device_error() == 0       # the word is cleared by reading it
    assert torch.equal(dev.state, before)
    assert torch.count_nonzero(out) == 0


def test_gates_precomputed(gdn):
    """a = g and b = beta given as fp32 arrays."""
    sh = gi.GDNShape(1, 77, 2, 2)
    inp = gi.make_inputs(sh, seed=4200, dtype="bf16", state="normal")
    g = torch.from_numpy(-np.random.default_rng(1).uniform(0, 4, (1, 77, 2)).astype(np.float32))
    beta = torch.from_numpy(np.random.default_rng(2).uniform(0, 1, (1, 77, 2)).astype(np.float32))
    kw = dict(num_k_heads=2, num_v_heads=2, q=inp.q, k=inp.k, v=inp.v, a=g, b=beta,
              state=inp.state, gates_precomputed=True)
    ref = oracle.layer(**kw)
    dev = to_device(inp)
    out = torch.empty(1, 77, 2, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_chunk_prefill(dev.q, dev.k, dev.v, g.cuda(), beta.cuda(), None, None, dev.state,
                          out, gates_precomputed=True)
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


def test_deterministic(gdn):
    sh = gi.GDNShape(1, 200, 16, 32, conv_width=4)
    inp = gi.make_inputs(sh, seed=4300, dtype="bf16")
    outs, states = [], []
    for _ in range(2):
        dev = to_device(inp)
        outs.append(run_prefill(gdn, dev))
        states.append(dev.state)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(states[0], states[1])


def test_split_call_matches_whole(gdn):
    """Two calls carrying (state, conv state) == one call: bit-exact when the split is a
    multiple of the chunk size, within tolerance otherwise."""
    sh = gi.GDNShape(1, 320, 2, 6, conv_width=4)
    inp = gi.make_inputs(sh, seed=4400, dtype="bf16")
    whole = to_device(inp)
    o_whole = run_prefill(gdn, whole)
    for split, exact in ((128, True), (100, False)):
        part = to_device(inp)
        x1, x2 = part.x[:, :split].contiguous(), part.x[:, split:].contiguous()
        a1, a2 = part.a[:, :split].contiguous(), part.a[:, split:].contiguous()
        b1, b2 = part.b[:, :split].contiguous(), part.b[:, split:].contiguous()
        outs = []
        for x, a, b in ((x1, a1, b1), (x2, a2, b2)):
            o = torch.empty(1, x.shape[1], 6, 128, dtype=torch.bfloat16, device="cuda")
            gdn.gdn_chunk_prefill(x, None, None, a, b, part.A_log, part.dt_bias, part.state, o,
                                  num_k_heads=2, conv_weight=part.conv_weight,
                                  conv_state=part.conv_state)
            outs.append(o)
        o_split = torch.cat(outs, 1)
        if exact:
            assert torch.equal(o_split, o_whole)
            assert torch.equal(part.state, whole.state)
        else:
            assert_bf16_parity(o_split.cpu(), o_whole.cpu())
            assert_state_parity(part.state.cpu(), whole.state.cpu())
        assert torch.equal(part.conv_state, whole.conv_state)


@pytest.mark.parametrize("Hk,Hv", [(2, 2), (2, 8), (1, 8)])
def test_conv_fused_group_sizes(gdn, Hk, Hv):
    """With conv width 4 the chunk-local kernel convolves the q / k channels itself, shared by
    the value heads of a key head as a cluster when there are 2 to 4 of them: one value head
    per key head (no sharing), four (a cluster of four) and eight (each CTA alone), against the
    oracle, over a ragged chunk and a non-zero conv state."""
    sh = gi.GDNShape(2, 150, Hk, Hv, conv_width=4)
    inp = gi.make_inputs(sh, seed=4300 + Hv, dtype="bf16", state="normal")
    g = torch.Generator().manual_seed(4301 + Hv)
    inp.conv_state = (torch.randn(inp.conv_state.shape, generator=g) * 0.5).to(torch.bfloat16)
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = torch.empty(2, 150, Hv, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_chunk_prefill(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state, out,
                          num_k_heads=Hk, conv_weight=dev.conv_weight, conv_state=dev.conv_state)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)
    np.testing.assert_array_equal(dev.conv_state.cpu().float().numpy(), ref.conv_state)
