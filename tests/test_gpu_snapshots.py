"""gdn_chunk_prefill_snapshots on the GPU, through the C ABI.

One prefill call over a whole prompt that records the recurrent and conv state every
`snap_every` tokens must equal, bit for bit, the same prompt fed as buckets of `snap_every`
tokens with gdn_state_checkpoint(SAVE) after each (the chunk grid starts at the call start,
so both compute the same chunks): outputs, final live state and conv state, and every bank
row.  Cases put the boundaries inside the kernel's slices of chunks, on slice ends and at
the call end, with a ragged tail, masked and permuted bank rows, skipped batch rows, the fp32
path, and the full 27B-shape long-context workload (T = 131072, a snapshot per 512 tokens).
Sampled snapshots are also checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import assert_state_parity, head_slice, to_device

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0   # bank rows that must not be written keep this


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_13_gb300 as m
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def _banks(nb, sh, dtype):
    bank = torch.full((nb, sh.num_v_heads, 128, 128), SENTINEL, device="cuda")
    cbank = None
    if sh.conv_width > 1:
        cbank = torch.full((nb, sh.conv_width - 1, sh.conv_channels), SENTINEL, dtype=dtype,
                           device="cuda")
    return bank, cbank


def _layer_call(gdn, sh, dev, t0, t1, state, conv_state, out, state_slots, fn, **kw):
    """One prefill call over tokens [t0, t1) of `dev` (contiguous slices), writing out[:, t0:t1]."""
    seg = lambda t: t[:, t0:t1].contiguous()
    # (zeros: rows that state_slots skips are left as they are)
    o = torch.zeros(sh.batch, t1 - t0, sh.num_v_heads, 128, dtype=out.dtype, device="cuda")
    if sh.conv_width > 0:
        fn(seg(dev.x), None, None, seg(dev.a), seg(dev.b), dev.A_log, dev.dt_bias, state, o,
           num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight, conv_state=conv_state,
           state_slots=state_slots, **kw)
    else:
        fn(seg(dev.q), seg(dev.k), seg(dev.v), seg(dev.a), seg(dev.b), dev.A_log, dev.dt_bias,
           state, o, state_slots=state_slots, **kw)
    out[:, t0:t1] = o


def _bucketed(gdn, sh, dev, every, snap_slots, bank, cbank, out_dtype, state_slots=None):
    """The reference: buckets of `every` tokens, a SAVE of every recorded row after each."""
    state, conv = dev.state.clone(), dev.conv_state.clone() if sh.conv_width > 0 else None
    out = torch.zeros(sh.batch, sh.seqlen, sh.num_v_heads, 128, dtype=out_dtype, device="cuda")
    T = sh.seqlen
    live_rows = (state_slots if state_slots is not None
                 else torch.arange(sh.batch, dtype=torch.int32, device="cuda"))
    for j, t0 in enumerate(range(0, T, every)):
        t1 = min(T, t0 + every)
        _layer_call(gdn, sh, dev, t0, t1, state, conv, out, state_slots, gdn.gdn_chunk_prefill)
        if t1 - t0 == every:
            gdn.gdn_state_checkpoint("save", state, conv, bank, cbank, live_rows,
                                     snap_slots[:, j].contiguous(), num_k_heads=sh.num_k_heads)
    return out, state, conv


def _single(gdn, sh, dev, every, snap_slots, bank, cbank, out_dtype, state_slots=None):
    state, conv = dev.state.clone(), dev.conv_state.clone() if sh.conv_width > 0 else None
    out = torch.zeros(sh.batch, sh.seqlen, sh.num_v_heads, 128, dtype=out_dtype, device="cuda")
    _layer_call(gdn, sh, dev, 0, sh.seqlen, state, conv, out, state_slots,
                gdn.gdn_chunk_prefill_snapshots, snap_every=every, snap_state=bank,
                snap_conv_state=cbank, snap_slots=snap_slots)
    return out, state, conv


def _slot_table(B, n_snap, nb, seed, masked=()):
    """A permutation of bank rows, with the (b, j) pairs in `masked` set to -1."""
    perm = np.random.default_rng(seed).permutation(nb)[:B * n_snap].reshape(B, n_snap)
    for (b, j) in masked:
        perm[b, j] = -1
    return torch.tensor(perm, dtype=torch.int32, device="cuda")


def _compare(gdn, sh, dev, every, out_dtype, nb, seed, masked=(), state_slots=None):
    n_snap = sh.seqlen // every
    slots = _slot_table(sh.batch, n_snap, nb, seed, masked)
    dt = dev.x.dtype if sh.conv_width > 0 else dev.q.dtype
    bank_r, cbank_r = _banks(nb, sh, dt)
    bank_s, cbank_s = _banks(nb, sh, dt)
    ref = _bucketed(gdn, sh, dev, every, slots, bank_r, cbank_r, out_dtype, state_slots)
    got = _single(gdn, sh, dev, every, slots, bank_s, cbank_s, out_dtype, state_slots)
    assert gdn.gdn_get_device_error() == 0
    assert torch.equal(got[0], ref[0]), "out"
    assert torch.equal(got[1], ref[1]), "final state"
    if sh.conv_width > 0:
        assert torch.equal(got[2], ref[2]), "final conv state"
    assert torch.equal(bank_s, bank_r), "state bank"
    if cbank_s is not None:
        assert torch.equal(cbank_s, cbank_r), "conv-state bank"
    # masked pairs and unused bank rows were not written
    used = set(slots[slots >= 0].tolist())
    for r in range(nb):
        if r not in used:
            assert bool((bank_s[r] == SENTINEL).all()), f"bank row {r} written"
    return slots, bank_s


@pytest.mark.parametrize("T,every", [(640, 128), (640, 192), (700, 128), (640, 64)])
def test_27b_shape_multi_slice(gdn, T, every):
    """B = 8 at the 27B shape (16/48 heads, conv) makes a slice of the tensor-core path 3
    chunks long: boundaries fall inside slices, on slice ends and at the call end."""
    sh = gi.GDNShape(8, T, 16, 48, conv_width=4)
    inp = gi.make_inputs(sh, seed=5100 + T + every, dtype="bf16")
    inp.conv_state = gi.to_bf16(np.random.default_rng(7).standard_normal(
        inp.conv_state.shape).astype(np.float32))
    dev = to_device(inp)
    n_snap = T // every
    slots, bank = _compare(gdn, sh, dev, every, torch.bfloat16, nb=8 * n_snap + 3,
                           seed=T + every, masked=[(1, 0), (5, n_snap - 1)])
    # two recorded snapshots against the fp64 oracle
    for (b, h, j) in [(0, 7, 0), (6, 45, n_snap - 1)]:
        t1 = (j + 1) * every
        r = oracle.layer(**head_slice(inp, b, h, 0, t1))
        row = int(slots[b, j])
        assert_state_parity(bank[row, h].cpu(), r.state[0, 0], what=f"snapshot b{b} h{h} j{j}")


def test_state_slots_and_skipped_rows(gdn):
    """Batch rows mapped to live state rows by state_slots; a skipped row records nothing."""
    sh = gi.GDNShape(3, 256, 2, 6, conv_width=4)
    inp = gi.make_inputs(sh, seed=5200, dtype="bf16", state="normal")
    dev = to_device(inp)
    # live state with 5 rows, batch rows -> rows 4, skip, 0
    st = torch.randn(5, 6, 128, 128, device="cuda") * 0.02
    cs = torch.zeros(5, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    dev.state, dev.conv_state = st, cs
    state_slots = torch.tensor([4, -1, 0], dtype=torch.int32, device="cuda")
    slots, bank = _compare(gdn, sh, dev, 64, torch.bfloat16, nb=16, seed=3,
                           state_slots=state_slots)
    for j in range(4):
        assert bool((bank[int(slots[1, j])] == SENTINEL).all())


@pytest.mark.parametrize("T,every", [(266, 64), (256, 128)])
def test_fp32_path(gdn, T, every):
    """All-fp32 mode (the FMA-pipe kernel), without a conv."""
    sh = gi.GDNShape(2, T, 16, 16, conv_width=0)
    inp = gi.make_inputs(sh, seed=5300 + T, dtype="f32", state="normal")
    dev = to_device(inp)
    n_snap = T // every
    slots, bank = _compare(gdn, sh, dev, every, torch.float32, nb=2 * n_snap + 1, seed=T)
    r = oracle.layer(**head_slice(inp, 1, 3, 0, every))
    assert_state_parity(bank[int(slots[1, 0]), 3].cpu(), r.state[0, 0], fp32=True)


def test_out_of_range_bank_row_is_reported(gdn):
    sh = gi.GDNShape(1, 256, 2, 6, conv_width=4)
    dev = to_device(gi.make_inputs(sh, seed=5400, dtype="bf16"))
    bank, cbank = _banks(4, sh, torch.bfloat16)
    slots = torch.tensor([[0, 9]], dtype=torch.int32, device="cuda")
    _single(gdn, sh, dev, 128, slots, bank, cbank, torch.bfloat16)
    assert gdn.gdn_get_device_error() == 6
    # the valid one was still recorded
    assert not bool((bank[0] == SENTINEL).all())


def test_27b_long_context_single_call(gdn):
    """The 27B-shape long-context workload (B = 1, T = 131072) as one call with a snapshot
    per 512 tokens == 256 bucket calls with a SAVE after each, bit for bit."""
    T, every = 131072, 512
    sh = gi.GDNShape(1, T, 16, 48, conv_width=4)
    dev = gi.make_inputs_device(sh, seed=4000, device="cuda")
    nb = T // every
    slots = torch.arange(nb, dtype=torch.int32, device="cuda").view(1, nb)
    bank_r, cbank_r = _banks(nb, sh, torch.bfloat16)
    ref = _bucketed(gdn, sh, dev, every, slots, bank_r, cbank_r, torch.bfloat16)
    bank_s, cbank_s = _banks(nb, sh, torch.bfloat16)
    got = _single(gdn, sh, dev, every, slots, bank_s, cbank_s, torch.bfloat16)
    assert gdn.gdn_get_device_error() == 0
    assert torch.equal(got[0], ref[0])
    assert torch.equal(got[1], ref[1])
    assert torch.equal(got[2], ref[2])
    assert torch.equal(bank_s, bank_r)
    assert torch.equal(cbank_s, cbank_r)
