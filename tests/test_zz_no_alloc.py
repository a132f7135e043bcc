"""gdn_chunk_prefill_noalloc: the prefill variant for callers that cannot allocate device memory
(e.g. code recorded into a CUDA graph, or a plug-in that is handed only input and output
pointers).  It keeps its scratch (post-conv activations, the tensor-core path's chunk tiles) in
the library's fixed device array instead of a caller workspace.  Both entry points run the
same deterministic kernels on the same inputs, so the outputs, the state and the conv state
must be bit-identical: checked through the C ABI against gdn_chunk_prefill on two calls in a
row, which also exercises the reuse of the shared array and the per-device set-up done by the
first call; then on the fp32 path (scratch holds only the post-conv activations) and on an
fp32 call without the conv (no scratch at all: nothing is looked up).

This file is collected last on purpose, so that a run stopping at the first failure has run
every other test first; it passes on its own in a fresh process too.
"""
import pytest
import torch

import gdn_inputs as gi
from gdn_testutil import to_device

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


def _call(fn, dev, out, **kw):
    if dev.shape.conv_width > 0:
        fn(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state, out,
           num_k_heads=dev.shape.num_k_heads, conv_weight=dev.conv_weight,
           conv_state=dev.conv_state, **kw)
    else:
        fn(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state, out, **kw)


def _same(gdn, sh, seed, dtype, what):
    inp = gi.make_inputs(sh, seed=seed, dtype=dtype, state="normal")
    ref_dev, dev = to_device(inp), to_device(inp)
    odt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o_ref = torch.empty(sh.batch, sh.seqlen, sh.num_v_heads, 128, dtype=odt, device="cuda")
    o = torch.full_like(o_ref, float("nan"))
    _call(gdn.gdn_chunk_prefill, ref_dev, o_ref)
    _call(gdn.gdn_chunk_prefill_noalloc, dev, o)
    assert gdn.gdn_get_device_error() == 0, what
    assert torch.equal(o, o_ref), what
    assert torch.equal(dev.state, ref_dev.state), what
    if sh.conv_width > 0:
        assert torch.equal(dev.conv_state, ref_dev.conv_state), what


def test_noalloc_matches_workspace_prefill_twice(gdn):
    # 27B head geometry with the conv; two different calls back to back through the same array
    for call, (B, T, seed) in enumerate([(2, 300, 9100), (1, 517, 9101)]):
        _same(gdn, gi.GDNShape(B, T, 16, 48, conv_width=4), seed, "bf16", f"bf16 call {call}")


def test_noalloc_fp32_paths(gdn):
    # fp32 with the conv: the array holds the post-conv activations only
    _same(gdn, gi.GDNShape(2, 150, 2, 6, conv_width=4), 9103, "f32", "fp32 with conv")
    # fp32 without the conv: the call needs no scratch and looks nothing up
    _same(gdn, gi.GDNShape(1, 70, 2, 4), 9104, "f32", "fp32 without conv")


def test_noalloc_rejects_oversized_call(gdn):
    # B*T*C_conv*2 bytes beyond the fixed array: refused before any launch, outputs untouched
    C = (2 * 16 + 48) * 128
    T = gdn.NOALLOC_SCRATCH_BYTES // (C * 2) + 1
    sh = gi.GDNShape(1, T, 16, 48, conv_width=4)
    dev = gi.make_inputs_device(sh, seed=9102, device="cuda")
    out = torch.zeros(1, T, 48, 128, dtype=torch.bfloat16, device="cuda")
    before = dev.state.clone()
    with pytest.raises(gdn.GDNError) as e:
        _call(gdn.gdn_chunk_prefill_noalloc, dev, out)
    assert e.value.status == 3
    assert torch.equal(dev.state, before)
    assert torch.count_nonzero(out) == 0
