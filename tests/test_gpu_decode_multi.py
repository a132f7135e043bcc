"""gdn_decode_multi (a decode step over T <= 16 tokens) against the fp64 oracle, through the
C ABI: outputs, final state and conv state for T = 1 .. 16 in bf16 and fp32, the 27B shape,
skipped rows, and the per-token snapshots (the state and conv state after every token, as a
speculative verifier restores them); small batches (the per-item kernel) and large ones (the
persistent kernel), up to the 27B-shape B = 128, T = 4 step with every unit checked.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import (assert_bf16_parity, assert_f32_parity, assert_state_parity,
                          head_slice, oracle_full, to_device)

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


def _inputs(B, T, Hk, Hv, W, dtype, seed):
    sh = gi.GDNShape(B, T, Hk, Hv, conv_width=W)
    inp = gi.make_inputs(sh, seed=seed, dtype=dtype, state="normal", state_std=0.3)
    if W > 0:
        cs = np.random.default_rng(seed).standard_normal(inp.conv_state.shape).astype(np.float32)
        inp.conv_state = gi.to_bf16(cs) if dtype == "bf16" else torch.from_numpy(cs)
    return sh, inp


def _run(gdn, dev, sh, out_dtype, state_slots=None, **snap):
    out = torch.full((sh.batch, sh.seqlen, sh.num_v_heads, 128), 7.0, dtype=out_dtype,
                     device="cuda")
    if sh.conv_width > 0:
        gdn.gdn_decode_multi(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                             out, num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight,
                             conv_state=dev.conv_state, state_slots=state_slots, **snap)
    else:
        gdn.gdn_decode_multi(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias,
                             dev.state, out, state_slots=state_slots, **snap)
    return out


@pytest.mark.parametrize("T", [1, 2, 5, 9, 16])
def test_bf16_conv_matches_oracle(gdn, T):
    sh, inp = _inputs(3, T, 2, 6, 4, "bf16", 8000 + T)
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = _run(gdn, dev, sh, torch.bfloat16)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)
    np.testing.assert_array_equal(dev.conv_state.float().cpu().numpy(), ref.conv_state)


def test_bf16_in_fp32_out(gdn):
    sh, inp = _inputs(2, 7, 2, 4, 4, "bf16", 8050)
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = _run(gdn, dev, sh, torch.float32)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


@pytest.mark.parametrize("T", [3, 16])
def test_fp32_mode(gdn, T):
    sh, inp = _inputs(2, T, 4, 4, 0, "f32", 8100 + T)
    ref = oracle_full(inp)
    dev = to_device(inp)
    out = _run(gdn, dev, sh, torch.float32)
    assert gdn.gdn_get_device_error() == 0
    assert_f32_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state, fp32=True)


def test_27b_shape_sampled(gdn):
    """16/48 heads (GQA 1:3), width-4 conv, B = 32, T = 4: sampled units against the oracle."""
    sh, inp = _inputs(32, 4, 16, 48, 4, "bf16", 8200)
    dev = to_device(inp)
    out = _run(gdn, dev, sh, torch.bfloat16)
    assert gdn.gdn_get_device_error() == 0
    for (b, h) in [(0, 0), (5, 47), (17, 23), (31, 30)]:
        r = oracle.layer(**head_slice(inp, b, h))
        assert_bf16_parity(out[b, :, h].cpu(), r.out[0, :, 0], what=f"out {b},{h}")
        assert_state_parity(dev.state[b, h].cpu(), r.state[0, 0], what=f"state {b},{h}")


def test_skipped_row(gdn):
    sh, inp = _inputs(3, 4, 2, 4, 4, "bf16", 8300)
    dev = to_device(inp)
    before = dev.state.clone()
    slots = torch.tensor([2, -1, 0], dtype=torch.int32, device="cuda")
    st = dev.state.clone()
    dev.state[2], dev.state[0] = st[0], st[2]
    cs = dev.conv_state.clone()
    dev.conv_state[2], dev.conv_state[0] = cs[0], cs[2]
    ref = oracle_full(inp)
    out = _run(gdn, dev, sh, torch.bfloat16, state_slots=slots)
    assert gdn.gdn_get_device_error() == 0
    assert torch.all(out[1].float() == 7.0)
    assert torch.equal(dev.state[1], before[1])
    assert_bf16_parity(out[0].cpu(), ref.out[0])
    assert_bf16_parity(out[2].cpu(), ref.out[2])
    assert_state_parity(dev.state[2].cpu(), ref.state[0])


@pytest.mark.parametrize("T", [5, 12])
def test_per_token_snapshots(gdn, T):
    """The state and conv state after every token of every row, into permuted bank rows with
    one pair masked: each equals the oracle after that many tokens (T = 12: two chunks of
    tokens, the second ragged)."""
    B = 2
    sh, inp = _inputs(B, T, 2, 6, 4, "bf16", 8400 + T)
    nb = B * T + 2
    perm = np.random.default_rng(1).permutation(nb)[:B * T].reshape(B, T)
    perm[1, 2] = -1
    slots = torch.tensor(perm, dtype=torch.int32, device="cuda")
    bank = torch.full((nb, 6, 128, 128), 12345.0, device="cuda")
    cbank = torch.zeros(nb, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    dev = to_device(inp)
    _run(gdn, dev, sh, torch.bfloat16, snap_state=bank, snap_conv_state=cbank, snap_slots=slots)
    assert gdn.gdn_get_device_error() == 0
    for b in range(B):
        for t in range(T):
            row = int(perm[b, t])
            if row < 0:
                continue
            sub = gi.GDNShape(1, t + 1, 2, 6, conv_width=4)
            part = gi.GDNInputs(sub, "bf16", None, None, None, inp.x[b:b + 1, :t + 1],
                                inp.a[b:b + 1, :t + 1], inp.b[b:b + 1, :t + 1], inp.A_log,
                                inp.dt_bias, inp.conv_weight, inp.state[b:b + 1],
                                inp.conv_state[b:b + 1])
            r = oracle_full(part)
            assert_state_parity(bank[row].cpu(), r.state[0], what=f"snapshot {b},{t}")
            np.testing.assert_array_equal(cbank[row].float().cpu().numpy(), r.conv_state[0])
    # the masked pair's row and the unused rows were not written
    used = set(int(v) for v in perm.ravel() if v >= 0)
    for row in range(nb):
        if row not in used:
            assert bool((bank[row] == 12345.0).all())


# ---------------------------------------------------------------- large batches
# Batches with more (sequence, key head) items than SMs take, for up to four tokens, the
# persistent warp-specialised kernel (a CTA per SM working through items in turn: row warps
# stream state rows while prologue warps prepare the next item from inputs staged by bulk
# copies); with more tokens, the per-item kernel.  The batches below give each persistent CTA
# two or more items.

def _persistent_batch(Hk, items_per_cta=2.5):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return int(items_per_cta * 2 * sms) // Hk + 1


def _run_ref(gdn, inp, sh, out_dtype, conv_bias=None, **kw):
    ref = oracle_full(inp, conv_bias=conv_bias)
    dev = to_device(inp)
    cb = None if conv_bias is None else conv_bias.to("cuda")
    out = torch.full((sh.batch, sh.seqlen, sh.num_v_heads, 128), 7.0, dtype=out_dtype,
                     device="cuda")
    if sh.conv_width > 0:
        gdn.gdn_decode_multi(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                             out, num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight,
                             conv_bias=cb, conv_state=dev.conv_state, **kw)
    else:
        gdn.gdn_decode_multi(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias,
                             dev.state, out, **kw)
    return ref, dev, out


@pytest.mark.parametrize("dtype,W,Hk,Hv,T,bias", [
    ("bf16", 4, 2, 6, 4, False),     # persistent: GQA 1:3, four tokens
    ("bf16", 4, 4, 8, 3, True),      # persistent: a conv bias
    ("bf16", 2, 2, 6, 4, False),     # persistent: conv width 2
    ("f32", 4, 2, 4, 3, True),       # persistent: fp32 inputs and outputs
    ("bf16", 0, 2, 4, 2, False),     # persistent: no conv
    ("bf16", 1, 2, 6, 4, False),     # persistent: conv width 1 (no conv state)
    ("bf16", 3, 4, 4, 2, True),      # persistent: conv width 3, GQA 1:1
    ("f32", 0, 2, 4, 4, False),      # persistent: fp32 without a conv
    ("bf16", 4, 4, 8, 7, True),      # per-item: seven tokens in the eight-token unroll
    ("bf16", 0, 2, 4, 16, False),    # per-item: no conv, sixteen tokens
])
def test_persistent_kernel_every_unit(gdn, dtype, W, Hk, Hv, T, bias):
    B = _persistent_batch(Hk)
    sh, inp = _inputs(B, T, Hk, Hv, W, dtype, 8500 + 10 * T + W)
    inp.dt_bias = torch.from_numpy(
        np.random.default_rng(T).standard_normal(Hv).astype(np.float32) * 0.5)
    cb = None
    if bias:
        cb = torch.from_numpy(np.random.default_rng(W).standard_normal(
            sh.conv_channels).astype(np.float32) * 0.1)
        cb = cb.to(torch.bfloat16) if dtype == "bf16" else cb
    odt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ref, dev, out = _run_ref(gdn, inp, sh, odt, conv_bias=cb)
    assert gdn.gdn_get_device_error() == 0
    if dtype == "bf16":
        assert_bf16_parity(out.cpu(), ref.out)
        assert_state_parity(dev.state.cpu(), ref.state)
    else:
        assert_f32_parity(out.cpu(), ref.out)
        assert_state_parity(dev.state.cpu(), ref.state, fp32=True)
    # every (sequence, value head) unit on its own, so that no unit hides in the aggregate
    o, s = out.cpu(), dev.state.cpu()
    for b in range(B):
        for h in range(Hv):
            if dtype == "bf16":
                assert_bf16_parity(o[b, :, h], ref.out[b, :, h], what=f"out {b},{h}")
            else:
                assert_f32_parity(o[b, :, h], ref.out[b, :, h], what=f"out {b},{h}")
            assert_state_parity(s[b, h], ref.state[b, h], fp32=dtype == "f32",
                                what=f"state {b},{h}")
    if W > 0:
        np.testing.assert_array_equal(dev.conv_state.float().cpu().numpy(), ref.conv_state)


def test_persistent_kernel_slots_and_snapshots(gdn):
    """Persistent-size batch through state_slots (permuted, padded rows -1) with per-token
    snapshots into permuted bank rows: the padded rows untouched, every other row's outputs,
    state, conv state and per-token snapshots equal to the oracle; then an out-of-range slot
    is reported."""
    Hk, Hv, T = 2, 6, 3
    B = _persistent_batch(Hk)
    sh, inp = _inputs(B, T, Hk, Hv, 4, "bf16", 8600)
    ref = oracle_full(inp)
    # the state after each token, for the snapshots (the oracle over the first t + 1 tokens)
    refs_t = []
    for t in range(T):
        part = gi.GDNInputs(gi.GDNShape(B, t + 1, Hk, Hv, conv_width=4), "bf16", None, None,
                            None, inp.x[:, :t + 1], inp.a[:, :t + 1], inp.b[:, :t + 1],
                            inp.A_log, inp.dt_bias, inp.conv_weight, inp.state, inp.conv_state)
        refs_t.append(oracle_full(part))
    dev = to_device(inp)
    nbank = B + 5
    g = torch.Generator().manual_seed(86)
    slots = torch.randperm(nbank, generator=g)[:B].to(torch.int32)
    slots[::9] = -1
    bank = torch.zeros(nbank, Hv, 128, 128, device="cuda")
    cbank = torch.zeros(nbank, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        if slots[b] >= 0:
            bank[slots[b]] = dev.state[b]
            cbank[slots[b]] = dev.conv_state[b]
    before, cbefore = bank.clone(), cbank.clone()
    nsnap = B * T + 4
    sperm = torch.randperm(nsnap, generator=g)[:B * T].view(B, T).to(torch.int32)
    sperm[5, 1] = -1
    sbank = torch.full((nsnap, Hv, 128, 128), 12345.0, device="cuda")
    scbank = torch.zeros(nsnap, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(B, T, Hv, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_multi(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                         num_k_heads=Hk, conv_weight=dev.conv_weight, conv_state=cbank,
                         state_slots=slots.cuda(), snap_state=sbank, snap_conv_state=scbank,
                         snap_slots=sperm.cuda())
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
        for t in range(T):
            row = int(sperm[b, t])
            if row < 0:
                continue
            assert_state_parity(sbank[row].cpu(), refs_t[t].state[b], what=f"snapshot {b},{t}")
            np.testing.assert_array_equal(scbank[row].float().cpu().numpy(),
                                          refs_t[t].conv_state[b])
    used = set(int(s) for s in slots if s >= 0)
    for s in range(nbank):
        if s not in used:
            assert torch.equal(bank[s], before[s]) and torch.equal(cbank[s], cbefore[s])
    # snapshot rows of padded sequences, the masked pair and the unused rows: not written
    written = set(int(sperm[b, t]) for b in range(B) for t in range(T)
                  if slots[b] >= 0 and sperm[b, t] >= 0)
    for row in range(nsnap):
        if row not in written:
            assert bool((sbank[row] == 12345.0).all())
    bad = slots.clone()
    bad[3] = nbank + 2
    gdn.gdn_decode_multi(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, bank, out,
                         num_k_heads=Hk, conv_weight=dev.conv_weight, conv_state=cbank,
                         state_slots=bad.cuda())
    assert gdn.gdn_get_device_error() == 6           # GDN_ERR_DEVICE_INDEX


def test_27b_shape_full_size_every_unit(gdn):
    """The bench's multi-token workload, 16/48 heads, width-4 conv, B = 128, T = 4, in the
    launch configuration it is timed in (the persistent kernel): every (sequence, value head)
    unit's outputs and state against the oracle, and the conv state exactly."""
    B, T = 128, 4
    sh, inp = _inputs(B, T, 16, 48, 4, "bf16", 8700)
    ref, dev, out = _run_ref(gdn, inp, sh, torch.bfloat16)
    assert gdn.gdn_get_device_error() == 0
    o, s = out.cpu(), dev.state.cpu()
    for b in range(B):
        for h in range(48):
            assert_bf16_parity(o[b, :, h], ref.out[b, :, h], what=f"out {b},{h}")
            assert_state_parity(s[b, h], ref.state[b, h], what=f"state {b},{h}")
    np.testing.assert_array_equal(dev.conv_state.float().cpu().numpy(), ref.conv_state)


@pytest.mark.parametrize("large", [False, True])
def test_options_both_kernels(gdn, large):
    """Precomputed gates (fp32 g and beta), a q scale, no q/k L2 norm and no SiLU, through the
    per-item kernel (B = 3) and the persistent kernel (a batch of more items than SMs), T = 3.
    x is scaled by 0.1 so that the unnormalised keys keep the delta rule stable."""
    Hk, Hv, T = 2, 6, 3
    B = _persistent_batch(Hk) if large else 3
    sh, inp = _inputs(B, T, Hk, Hv, 4, "bf16", 8800 + int(large))
    inp.x = (inp.x.float() * 0.1).to(torch.bfloat16)
    rng = np.random.default_rng(88)
    inp.a = torch.from_numpy(-rng.uniform(0, 4, (B, T, Hv)).astype(np.float32))
    inp.b = torch.from_numpy(rng.uniform(0, 1, (B, T, Hv)).astype(np.float32))
    opts = dict(scale=0.5, qk_l2norm=False, conv_silu=False, gates_precomputed=True)
    ref = oracle_full(inp, **opts)
    dev = to_device(inp)
    out = torch.full((B, T, Hv, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_multi(dev.x, None, None, dev.a, dev.b, None, None, dev.state, out,
                         num_k_heads=Hk, conv_weight=dev.conv_weight, conv_state=dev.conv_state,
                         **opts)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out, f"options B={B}")
    assert_state_parity(dev.state.cpu(), ref.state, what=f"options state B={B}")
    np.testing.assert_array_equal(dev.conv_state.float().cpu().numpy(), ref.conv_state)
