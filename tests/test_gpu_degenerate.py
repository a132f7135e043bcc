"""Degenerate gates and the widest head grouping, every path against the fp64 oracle.

Gates are given precomputed (fp32 g and beta) so that the extremes are exact: g = 0 (no
decay), g = -1e-3, g = -5 and g = -50 (the state all but wiped; e^g underflows nothing in
fp32 but leaves nothing of the past), beta = 0 (the token writes nothing), beta = 1 (the
write replaces the value at k exactly) and beta = 0.5.  The paths: the tensor-core prefill
(bf16), the fp32 prefill, the decode step on both of its kernels, the multi-token step; and
GQA 1:8 (one key head for eight value heads) on the prefill and the multi-token step.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
from gdn_testutil import (assert_bf16_parity, assert_f32_parity, assert_state_parity,
                          oracle_full, to_device)

pytestmark = pytest.mark.gpu

G_VALUES = np.array([0.0, -1e-3, -5.0, -50.0], dtype=np.float32)
B_VALUES = np.array([0.0, 1.0, 0.5], dtype=np.float32)


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_13_gb300 as m
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def _extreme(B, T, Hk, Hv, dtype, seed):
    sh = gi.GDNShape(B, T, Hk, Hv, conv_width=0)
    inp = gi.make_inputs(sh, seed=seed, dtype=dtype, state="normal", state_std=0.3)
    rng = np.random.default_rng(seed)
    inp.a = torch.from_numpy(G_VALUES[rng.integers(0, len(G_VALUES), (B, T, Hv))])
    inp.b = torch.from_numpy(B_VALUES[rng.integers(0, len(B_VALUES), (B, T, Hv))])
    return sh, inp


def _oracle(inp):
    return oracle_full(inp, gates_precomputed=True)


def _prefill(gdn, dev, out):
    gdn.gdn_chunk_prefill(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                          out, gates_precomputed=True)


@pytest.mark.parametrize("Hk,Hv", [(2, 4), (1, 8)])
def test_prefill_tensor_core(gdn, Hk, Hv):
    sh, inp = _extreme(2, 150, Hk, Hv, "bf16", 9000 + Hv)
    ref = _oracle(inp)
    dev = to_device(inp)
    out = torch.empty(2, 150, Hv, 128, dtype=torch.bfloat16, device="cuda")
    _prefill(gdn, dev, out)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


def test_prefill_fp32(gdn):
    sh, inp = _extreme(2, 150, 2, 4, "f32", 9100)
    ref = _oracle(inp)
    dev = to_device(inp)
    out = torch.empty(2, 150, 4, 128, device="cuda")
    _prefill(gdn, dev, out)
    assert gdn.gdn_get_device_error() == 0
    assert_f32_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state, fp32=True)


@pytest.mark.parametrize("B,Hk", [(2, 2), (40, 16)])
def test_decode_steps(gdn, B, Hk):
    """8 single-token steps: B = 2 runs the cluster kernel, B = 40 x 16 key heads the
    streaming one."""
    steps = 8
    sh, inp = _extreme(B, steps, Hk, Hk * 2, "bf16", 9200 + B)
    ref = _oracle(inp)
    dev = to_device(inp)
    outs = []
    for t in range(steps):
        o = torch.empty(B, 1, Hk * 2, 128, dtype=torch.bfloat16, device="cuda")
        sl = lambda u: u[:, t:t + 1].contiguous()
        gdn.gdn_decode_step(sl(dev.q), sl(dev.k), sl(dev.v), sl(dev.a), sl(dev.b), dev.A_log,
                            dev.dt_bias, dev.state, o, gates_precomputed=True)
        outs.append(o)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(torch.cat(outs, 1).cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)


@pytest.mark.parametrize("Hk,Hv,T", [(2, 4, 8), (1, 8, 16)])
def test_multi_token_step(gdn, Hk, Hv, T):
    sh, inp = _extreme(3, T, Hk, Hv, "bf16", 9300 + T)
    ref = _oracle(inp)
    dev = to_device(inp)
    out = torch.empty(3, T, Hv, 128, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_multi(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                         out, gates_precomputed=True)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), ref.out)
    assert_state_parity(dev.state.cpu(), ref.state)
