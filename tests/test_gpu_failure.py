"""Failure detection on the GPU without a fault: a bounded wait that nothing ends.

Every wait of the library's copy / tensor-core pipelines is bounded.  When a copy or an MMA
never completes, the CTA gives up, records GDN_ERR_DEVICE_TIMEOUT in the device error word and
returns, leaving the context usable.  gdn_selftest_device_timeout drives that path on purpose
with a wait on an mbarrier that nothing arrives at (no copy, MMA or TMEM in flight, so nothing
can fault): the status must be reported once, cleared by reading it, and a prefill right
after must run normally.  The out-of-range state slot (GDN_ERR_DEVICE_INDEX) is covered in
test_gpu_prefill.py.
"""
import pytest
import torch

import gdn_inputs as gi
from gdn_testutil import assert_bf16_parity, oracle_full, run_prefill, to_device

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


@pytest.mark.parametrize("polls", [1, 1024])
def test_bounded_wait_timeout_is_reported_then_cleared(gdn, polls):
    assert gdn.gdn_get_device_error() == 0
    gdn.gdn_selftest_device_timeout(polls)
    assert gdn.gdn_get_device_error() == 5  # GDN_ERR_DEVICE_TIMEOUT
    assert gdn.gdn_get_device_error() == 0
    # the context survives: a prefill right after matches the oracle
    sh = gi.GDNShape(1, 100, 2, 6, conv_width=4)
    inp = gi.make_inputs(sh, seed=9300 + polls, dtype="bf16", state="normal")
    dev = to_device(inp)
    out = run_prefill(gdn, dev)
    assert gdn.gdn_get_device_error() == 0
    assert_bf16_parity(out.cpu(), oracle_full(inp).out, "prefill after the timeout")
