"""causal_conv1d_update and gdn_state_checkpoint on the GPU, through the C ABI.

The conv is checked against the oracle's conv (numpy.convolve-pinned) within one bf16
rounding of the output; its state, and every checkpoint copy, bit for bit.  The resume
test runs the 27B-shape layer over 131072 tokens in 512-token buckets with a checkpoint
after every bucket, restores a middle checkpoint, continues, and requires the continuation
to equal the uninterrupted run bit for bit (hybrid prefix-reuse semantics); every unit of
that long run is checked against the oracle, with bf16 and with fp32 outputs.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import (BF16_MAXREL, BF16_OUT_ROUNDING, BF16_STATE_RELF, assert_bf16_parity,
                          assert_state_parity, check_units, concat_units, kh_slice, merge_units,
                          to_device, unit_metrics)

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


CKPTS = (0, 15, 127, 255)


def test_27b_long_context_bucketed_with_resume(gdn):
    """27B shape (16/48 heads, conv), B=1, T=131072 = 256 buckets of 512 with a checkpoint
    after each; restore checkpoint 127 and continue: bit-identical to the uninterrupted run.
    The same bucketed run with fp32 outputs too; then every one of the 48 heads against the
    oracle over all 131072 tokens (outputs per segment, state at checkpoints 0, 15, 127, 255):
    fp32 outputs within max|o - o_ref| / max|o_ref| <= 5e-3 per unit and segment, bf16
    outputs within that plus their own rounding, cosine >= 0.9999; states cosine >= 0.9999
    and rel-F <= 5e-3."""
    T, bucket = 131072, 512
    nbk = T // bucket
    Hk, Hv, d = 16, 48, 128
    r = Hv // Hk
    sh = gi.GDNShape(1, T, Hk, Hv, conv_width=4)
    dev = gi.make_inputs_device(sh, seed=4000, device="cuda")
    bank = torch.empty(nbk, Hv, d, d, device="cuda")
    cbank = torch.empty(nbk, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, T, Hv, d, dtype=torch.bfloat16, device="cuda")
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
    del out2, bank2, cbank2
    # the same bucketed run with fp32 outputs, from the zero state
    dev.state = torch.zeros_like(final_state)
    dev.conv_state = torch.zeros_like(final_conv)
    out32 = torch.empty(1, T, Hv, d, dtype=torch.float32, device="cuda")
    bank32 = torch.empty_like(bank)
    cbank32 = torch.empty_like(cbank)
    _bucket_run(gdn, dev, T, bucket, 0, bank32, cbank32, out32)
    assert gdn.gdn_get_device_error() == 0
    # fp32 outputs do not change the recurrence: the same states, bit for bit
    assert torch.equal(dev.state, final_state)
    assert torch.equal(bank32[list(CKPTS)], bank[list(CKPTS)])
    del bank32, cbank32
    dev.state = torch.zeros_like(final_state)
    dev.conv_state = torch.zeros_like(final_conv)

    # the oracle: every key head (with its 3 value heads) in segments ending at the checkpoints
    bank_h = bank[list(CKPTS)].double().cpu().numpy()          # [4, Hv, d, d]
    parts = {k: [] for k in ("o32", "o16", "state")}    # [segment][key head] -> r units

    def unit_rows(o):       # [t, r, d] -> [r, t*d]
        return np.ascontiguousarray(np.asarray(o, dtype=np.float64).transpose(1, 0, 2)
                                    .reshape(o.shape[1], -1))

    def job(kh, t0, t1, st, cst, ci):
        kw = kh_slice(dev, 0, kh, t0, t1,
                      state=torch.zeros(1, r, d, d) if st is None else st,
                      conv_state=torch.zeros(1, 3, (2 + r) * d) if cst is None else cst)
        res = oracle.layer(**kw)
        ref = unit_rows(res.out[0])
        got32 = unit_rows(out32[0, t0:t1, kh * r:(kh + 1) * r].double().cpu().numpy())
        got16 = unit_rows(out[0, t0:t1, kh * r:(kh + 1) * r].double().cpu().numpy())
        m = (unit_metrics(got32, ref), unit_metrics(got16, ref),
             unit_metrics(bank_h[ci, kh * r:(kh + 1) * r].reshape(r, -1),
                          res.state[0].reshape(r, -1)))
        return m, res.state, res.conv_state

    carry = [(None, None)] * Hk
    t0 = 0
    with cf.ThreadPoolExecutor(max_workers=max(1, len(os.sched_getaffinity(0)) // r)) as ex:
        for ci, ck in enumerate(CKPTS):
            t1 = (ck + 1) * bucket
            res = list(ex.map(lambda kh: job(kh, t0, t1, carry[kh][0], carry[kh][1], ci),
                              range(Hk)))
            for kh, (m, st, cst) in enumerate(res):
                parts["o32"].append(m[0])
                parts["o16"].append(m[1])
                parts["state"].append(m[2])
                carry[kh] = (torch.from_numpy(st), torch.from_numpy(cst))
            t0 = t1
    # per unit over the whole call (the segments of a unit merged), then per segment
    for key, tag, bound in (("o32", "f32 out", BF16_MAXREL),
                            ("o16", "bf16 out", BF16_MAXREL + BF16_OUT_ROUNDING)):
        segs = parts[key]
        per_seg = [concat_units(segs[ci * Hk:(ci + 1) * Hk]) for ci in range(len(CKPTS))]
        check_units(merge_units(per_seg), f"qwen36_27b T131072 bucket512 out ({tag}), per unit",
                    maxrel=bound)
        check_units(per_seg, f"qwen36_27b T131072 bucket512 out ({tag}), per unit and segment",
                    maxrel=None, cos=None)
    check_units(parts["state"], "qwen36_27b T131072 bucket512 state at checkpoints 0/15/127/255",
                relf=BF16_STATE_RELF)
