"""gdn_chunk_prefill_varlen (packed variable-length batches) on the GPU, through the C ABI.

A packed call must equal one gdn_chunk_prefill call per sequence, bit for bit (every
sequence is its own recurrence with its own chunk grid): outputs, states and conv states.
Lengths cover empty sequences, sequences shorter than the conv window, chunk boundaries and
ragged tails; state rows are permuted and one sequence is skipped; a batch larger than one
slice of the tensor-core path has sequences crossing the slice boundary; the fp32 path and
the gated output norm are covered; sampled sequences are checked against the fp64 oracle;
bad offsets are reported and compute nothing.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from gdn_testutil import assert_bf16_parity, assert_state_parity, head_slice, to_device

pytestmark = pytest.mark.gpu

SENT = 7.0


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_13_gb300 as m
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def _packed_inputs(lengths, Hk, Hv, W, dtype, seed):
    """One packed input set (B = 1, T = sum of lengths) with a state row per sequence (random
    state and, with a conv, random conv state)."""
    T = int(sum(lengths))
    N = len(lengths)
    sh = gi.GDNShape(1, T, Hk, Hv, conv_width=W)
    inp = gi.make_inputs(sh, seed=seed, dtype=dtype, state="normal")
    rng = np.random.default_rng(seed + 1)
    inp.state = torch.from_numpy((rng.standard_normal((N, Hv, 128, 128)) * 0.05).astype(np.float32))
    if W > 0:
        cs = rng.standard_normal((N, W - 1, sh.conv_channels)).astype(np.float32)
        inp.conv_state = gi.to_bf16(cs) if dtype == "bf16" else torch.from_numpy(cs)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return sh, inp, torch.from_numpy(cu)


def _seq_call(gdn, dev, sh, t0, t1, rows, out, gate=None):
    """gdn_chunk_prefill of tokens [t0, t1) as a sequence of its own on state row(s) `rows`."""
    if t1 == t0:
        return
    seg = lambda u: u[:, t0:t1].contiguous()
    o = torch.empty(1, t1 - t0, sh.num_v_heads, 128, dtype=out.dtype, device="cuda")
    slots = torch.tensor([rows], dtype=torch.int32, device="cuda")
    kw = dict(state_slots=slots)
    if sh.conv_width > 0:
        args = (seg(dev.x), None, None)
        kw.update(num_k_heads=sh.num_k_heads, conv_weight=dev.conv_weight,
                  conv_state=dev.conv_state)
    else:
        args = (seg(dev.q), seg(dev.k), seg(dev.v))
    args = args + (seg(dev.a), seg(dev.b), dev.A_log, dev.dt_bias, dev.state, o)
    if gate is None:
        gdn.gdn_chunk_prefill(*args, **kw)
    else:
        gdn.gdn_chunk_prefill_gated(*args, gate_z=seg(gate[0]), gate_weight=gate[1], **kw)
    out[:, t0:t1] = o


def _packed_call(gdn, dev, sh, cu, slots, out, gate=None):
    kw = dict(cu_seqlens=cu, state_slots=slots)
    if gate is not None:
        kw.update(gate_z=gate[0], gate_weight=gate[1])
    if sh.conv_width > 0:
        gdn.gdn_chunk_prefill_varlen(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias,
                                     dev.state, out, num_k_heads=sh.num_k_heads,
                                     conv_weight=dev.conv_weight, conv_state=dev.conv_state,
                                     **kw)
    else:
        gdn.gdn_chunk_prefill_varlen(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias,
                                     dev.state, out, **kw)


def _compare(gdn, sh, inp, cu, slot_list, out_dtype, gate=None):
    """Packed call vs one call per sequence on the same slots; returns the packed run."""
    N = len(slot_list)
    cu_d = cu.cuda()
    slots = torch.tensor(slot_list, dtype=torch.int32, device="cuda")
    ref = to_device(inp)
    out_r = torch.full((1, sh.seqlen, sh.num_v_heads, 128), SENT, dtype=out_dtype, device="cuda")
    for n in range(N):
        if slot_list[n] >= 0:
            _seq_call(gdn, ref, sh, int(cu[n]), int(cu[n + 1]), slot_list[n], out_r, gate)
    got = to_device(inp)
    out_g = torch.full_like(out_r, SENT)
    _packed_call(gdn, got, sh, cu_d, slots, out_g, gate)
    assert gdn.gdn_get_device_error() == 0
    assert torch.equal(out_g, out_r), "outputs"
    assert torch.equal(got.state, ref.state), "states"
    if sh.conv_width > 0:
        assert torch.equal(got.conv_state, ref.conv_state), "conv states"
    return got, out_g


LENGTHS = [130, 0, 1, 2, 63, 64, 65, 200, 3, 70]


def test_packed_equals_per_sequence_bf16_conv(gdn):
    """bf16, GQA 1:3, width-4 conv; state rows permuted, sequence 4 skipped."""
    sh, inp, cu = _packed_inputs(LENGTHS, 2, 6, 4, "bf16", 7100)
    N = len(LENGTHS)
    slot_list = [int(v) for v in np.random.default_rng(3).permutation(N)]
    slot_list[4] = -1
    got, out = _compare(gdn, sh, inp, cu, slot_list, torch.bfloat16)
    # the skipped sequence's outputs are untouched
    t0, t1 = int(cu[4]), int(cu[5])
    assert torch.all(out[:, t0:t1].float() == SENT)
    # two sequences against the oracle (each with its own state and conv state)
    for n in (0, 7):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in (0, 5):
            kw = head_slice(inp, 0, h, t0, t1)
            sl = slot_list[n]                      # the row sequence n reads and updates
            kw["state"] = inp.state[sl:sl + 1, h:h + 1]
            kh, Hk = h // 3, 2                     # GQA 1:3 with 2 key heads
            idx = torch.cat([torch.arange(kh * 128, (kh + 1) * 128),
                             torch.arange((Hk + kh) * 128, (Hk + kh + 1) * 128),
                             torch.arange((2 * Hk + h) * 128, (2 * Hk + h + 1) * 128)])
            kw["conv_state"] = inp.conv_state[sl:sl + 1].index_select(2, idx)
            r = oracle.layer(**kw)
            assert_bf16_parity(out[0, t0:t1, h].cpu(), r.out[0, :, 0], what=f"seq {n} h{h}")
            assert_state_parity(got.state[sl, h].cpu(), r.state[0, 0],
                                what=f"state seq {n} h{h}")


def test_packed_fp32_path(gdn):
    sh, inp, cu = _packed_inputs([5, 64, 0, 77, 129], 4, 4, 0, "f32", 7200)
    _compare(gdn, sh, inp, cu, [4, 3, 2, 1, 0], torch.float32)


def test_packed_gated_norm(gdn):
    sh, inp, cu = _packed_inputs([100, 1, 64, 33], 2, 6, 4, "bf16", 7300)
    g = torch.Generator().manual_seed(9)
    z = torch.randn(1, sh.seqlen, 6, 128, generator=g).to(torch.bfloat16).cuda()
    w = (torch.rand(128, generator=g) + 0.5).cuda()
    _compare(gdn, sh, inp, cu, [0, 1, 2, 3], torch.bfloat16, gate=(z, w))


def test_packed_across_slices(gdn):
    """27B shape (16/48 heads): a slice of the tensor-core path holds 25 chunks of one packed
    axis, so these 4 sequences of 700 tokens (44 chunks) span two slices."""
    sh, inp, cu = _packed_inputs([700, 700, 650, 750], 16, 48, 4, "bf16", 7400)
    _compare(gdn, sh, inp, cu, [3, 0, 2, 1], torch.bfloat16)


def test_bad_offsets_compute_nothing(gdn):
    sh, inp, cu = _packed_inputs([40, 40, 40], 2, 2, 4, "bf16", 7500)
    dev = to_device(inp)
    before = dev.state.clone()
    cbefore = dev.conv_state.clone()
    out = torch.full((1, 120, 2, 128), SENT, dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([0, 50, 30, 120], dtype=torch.int32, device="cuda")   # not monotonic
    _packed_call(gdn, dev, sh, bad, None, out)
    assert gdn.gdn_get_device_error() == 6
    assert torch.equal(dev.state, before)
    assert torch.equal(dev.conv_state, cbefore)
    assert torch.all(out.float() == SENT)


def test_packed_fp32_gated_norm(gdn):
    """fp32 mode with the gated norm: the norm runs as a pass of its own that finds each
    token's sequence (and skips the skipped one) by bisection on the offsets."""
    sh, inp, cu = _packed_inputs([40, 0, 77, 64, 5], 4, 8, 0, "f32", 7600)
    g = torch.Generator().manual_seed(11)
    z = torch.randn(1, sh.seqlen, 8, 128, generator=g).cuda()
    w = (torch.rand(128, generator=g) + 0.5).cuda()
    _, out = _compare(gdn, sh, inp, cu, [3, 4, -1, 0, 1], torch.float32, gate=(z, w))
    t0, t1 = int(cu[2]), int(cu[3])
    assert torch.all(out[:, t0:t1] == SENT)
