"""causal_conv1d_update and gdn_state_checkpoint on the GPU, through the C ABI.

The conv is checked against the oracle's conv (numpy.convolve-pinned) within one bf16
rounding of the output; its state, and every checkpoint copy, bit for bit.  The resume
test runs the 27B-shape layer over 131072 tokens in 512-token buckets with a checkpoint
after every bucket, restores a middle checkpoint, continues, and requires the continuation
to equal the uninterrupted run bit for bit (hybrid prefix-reuse semantics); sampled units
of that long run are checked against the oracle.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import assert_bf16_parity, assert_state_parity, head_slice, to_device

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


@pytest.mark.parametrize("dtype,W,T", [(torch.bfloat16, 4, 37), (torch.bfloat16, 2, 5),
                                       (torch.float32, 3, 70), (torch.bfloat16, 4, 1)])
def test_conv_matches_oracle(gdn, dtype, W, T):
    B, C = 3, 384
    g = torch.Generator().manual_seed(W * 100 + T)
    x = torch.randn(B, T, C, generator=g).to(dtype)
    w = (torch.randn(C, W, generator=g) / 2).to(dtype)
    bias = torch.randn(C, generator=g).to(dtype)
    cs = torch.randn(B, W - 1, C, generator=g).to(dtype)
    y_ref, cs_ref = oracle.conv1d(x, w, bias=bias, state=cs, silu=True)
    xd, wd, bd, csd = x.cuda(), w.cuda(), bias.cuda(), cs.cuda()
    y = torch.empty_like(xd)
    gdn.causal_conv1d_update(xd, wd, csd, y, bias=bd, silu=True)
    assert gdn.gdn_get_device_error() == 0
    err = np.abs(y.float().cpu().numpy() - y_ref)
    # fp32 accumulation of W + 1 terms of size ~1 (absolute part), plus one rounding of the
    # output to the storage type (relative part)
    rel = 2.0 ** -8 if dtype == torch.bfloat16 else 1e-6
    tol = rel * np.abs(y_ref) + 1e-5
    assert (err <= tol).all(), err.max()
    np.testing.assert_array_equal(csd.float().cpu().numpy(), cs_ref)


def test_conv_split_equals_whole_bitwise(gdn):
    B, T, C, W = 2, 100, 512, 4
    g = torch.Generator().manual_seed(5)
    x = torch.randn(B, T, C, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(C, W, generator=g).to(torch.bfloat16).cuda()
    cs0 = torch.randn(B, W - 1, C, generator=g).to(torch.bfloat16).cuda()
    y = torch.empty_like(x)
    cs = cs0.clone()
    gdn.causal_conv1d_update(x, w, cs, y)
    for split in (1, 2, 33):
        cs2 = cs0.clone()
        y1 = torch.empty(B, split, C, dtype=torch.bfloat16, device="cuda")
        y2 = torch.empty(B, T - split, C, dtype=torch.bfloat16, device="cuda")
        gdn.causal_conv1d_update(x[:, :split].contiguous(), w, cs2, y1)
        gdn.causal_conv1d_update(x[:, split:].contiguous(), w, cs2, y2)
        assert torch.equal(torch.cat([y1, y2], 1), y)
        assert torch.equal(cs2, cs)


def test_checkpoint_save_restore_masks(gdn):
    ns, nb, Hv, Hk, W = 3, 5, 6, 2, 4
    C = (2 * Hk + Hv) * 128
    state = torch.randn(ns, Hv, 128, 128, device="cuda")
    conv = torch.randn(ns, W - 1, C, device="cuda").to(torch.bfloat16)
    bank = torch.zeros(nb, Hv, 128, 128, device="cuda")
    cbank = torch.zeros(nb, W - 1, C, dtype=torch.bfloat16, device="cuda")
    rows = torch.tensor([0, 2, 1, -1], dtype=torch.int32, device="cuda")
    slots = torch.tensor([4, 1, -1, 0], dtype=torch.int32, device="cuda")
    gdn.gdn_state_checkpoint("save", state, conv, bank, cbank, rows, slots, num_k_heads=Hk)
    assert gdn.gdn_get_device_error() == 0
    assert torch.equal(bank[4], state[0]) and torch.equal(bank[1], state[2])
    assert torch.equal(cbank[4], conv[0]) and torch.equal(cbank[1], conv[2])
    for s in (0, 2, 3):
        assert torch.count_nonzero(bank[s]) == 0 and torch.count_nonzero(cbank[s]) == 0
    # restore into fresh live rows
    state2 = torch.zeros_like(state)
    conv2 = torch.zeros_like(conv)
    gdn.gdn_state_checkpoint("restore", state2, conv2, bank, cbank,
                             torch.tensor([1, 0], dtype=torch.int32, device="cuda"),
                             torch.tensor([4, 1], dtype=torch.int32, device="cuda"),
                             num_k_heads=Hk)
    assert torch.equal(state2[1], state[0]) and torch.equal(state2[0], state[2])
    assert torch.equal(conv2[1], conv[0]) and torch.equal(conv2[0], conv[2])
    assert torch.count_nonzero(state2[2]) == 0
    # an index past the bank is skipped and reported
    gdn.gdn_state_checkpoint("save", state, conv, bank, cbank,
                             torch.tensor([0], dtype=torch.int32, device="cuda"),
                             torch.tensor([nb], dtype=torch.int32, device="cuda"),
                             num_k_heads=Hk)
    assert gdn.gdn_get_device_error() == 6


def _bucket_run(gdn, dev, T_total, bucket, first_bucket, bank, cbank, out):
    """512-token bucket calls over [first_bucket*bucket, T_total) with a SAVE after each."""
    Hk = dev.shape.num_k_heads
    rows = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(first_bucket, T_total // bucket):
        t0 = i * bucket
        gdn.gdn_chunk_prefill(dev.x[:, t0:t0 + bucket], None, None, dev.a[:, t0:t0 + bucket],
                              dev.b[:, t0:t0 + bucket], dev.A_log, dev.dt_bias, dev.state,
                              out[:, t0:t0 + bucket], num_k_heads=Hk,
                              conv_weight=dev.conv_weight, conv_state=dev.conv_state)
        gdn.gdn_state_checkpoint("save", dev.state, dev.conv_state, bank, cbank, rows,
                                 torch.full((1,), i, dtype=torch.int32, device="cuda"),
                                 num_k_heads=Hk)


def test_27b_long_context_bucketed_with_resume(gdn):
    """27B shape (16/48 heads, conv), B=1, T=131072 = 256 buckets of 512 with a checkpoint
    after each; restore checkpoint 127 and continue: bit-identical to the uninterrupted run.
    Two sampled heads over all 131072 tokens against the oracle (state at 4 checkpoints)."""
    T, bucket = 131072, 512
    nbk = T // bucket
    sh = gi.GDNShape(1, T, 16, 48, conv_width=4)
    dev = gi.make_inputs_device(sh, seed=4000, device="cuda")
    # x slices along T must be contiguous per bucket for the C ABI: keep [B=1, T, C] layout
    bank = torch.empty(nbk, 48, 128, 128, device="cuda")
    cbank = torch.empty(nbk, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, T, 48, 128, dtype=torch.bfloat16, device="cuda")
    x0 = dev.x
    _bucket_run(gdn, dev, T, bucket, 0, bank, cbank, out)
    assert gdn.gdn_get_device_error() == 0
    final_state = dev.state.clone()
    final_conv = dev.conv_state.clone()
    # resume from checkpoint 127 (tokens [0, 65536) done) into fresh live state
    mid = 127
    dev.state = torch.full_like(final_state, float("nan"))
    dev.conv_state = torch.zeros_like(final_conv)
    gdn.gdn_state_checkpoint("restore", dev.state, dev.conv_state, bank, cbank,
                             torch.zeros(1, dtype=torch.int32, device="cuda"),
                             torch.full((1,), mid, dtype=torch.int32, device="cuda"),
                             num_k_heads=16)
    out2 = torch.full_like(out, float("nan"))
    bank2 = torch.empty_like(bank)
    cbank2 = torch.empty_like(cbank)
    _bucket_run(gdn, dev, T, bucket, mid + 1, bank2, cbank2, out2)
    assert gdn.gdn_get_device_error() == 0
    t_mid = (mid + 1) * bucket
    assert torch.equal(out2[:, t_mid:], out[:, t_mid:])
    assert torch.equal(dev.state, final_state)
    assert torch.equal(dev.conv_state, final_conv)
    # oracle on two sampled heads, in segments ending at checkpoints 0, 15, 127, 255
    out_h = out
    for (b, h) in [(0, 5), (0, 40)]:
        st, cst = None, None
        t0 = 0
        for ck in (0, 15, 127, 255):
            t1 = (ck + 1) * bucket
            kw = head_slice(dev, b, h, t0, t1)
            kw["x"] = kw["x"]  # pre-conv slice of [t0, t1)
            if st is not None:
                kw["state"], kw["conv_state"] = st, cst
            else:
                kw["state"] = torch.zeros(1, 1, 128, 128)
                kw["conv_state"] = torch.zeros(1, 3, 384)
            r = oracle.layer(**kw)
            assert_bf16_parity(out_h[0, t0:t1, h].cpu(), r.out[0, :, 0], what=f"out h{h} <{t1}")
            assert_state_parity(bank[ck, h].cpu(), r.state[0, 0], what=f"state h{h} @ ckpt {ck}")
            st, cst = r.state, r.conv_state
            t0 = t1
    del x0
