"""Pins against values the pages print (tests/golden/, each file with its citation).

The pages print no worked example of the recurrence itself (no test vector or reference
output); what they do print and what this build's layout depends on is the size of the 27B
model's 64-slot checkpoint bank.  A slot holds, per GDN layer, the recurrent state and the
conv state; with the layouts this library uses (state [Hv, d, d] fp32, conv state
[W - 1, C_conv] in the bf16 input type, W = 4, C_conv = (2 Hk + Hv) d) the bank comes to the
printed ~9.85 GB.  The neighbouring readings (W conv rows instead of W - 1, an fp32 conv
state, no conv state, a bf16 recurrent state) all miss it, so the figure pins the reading.
"""
import os

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _read(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split()
            vals[k] = float(v)
    return vals


def _slot_bytes(Hk, Hv, d, W, state_dtype, conv_dtype, conv_rows):
    """Bytes of one checkpoint slot of one layer, from tensors shaped as the library's
    state and conv-state rows (meta tensors: nothing is allocated)."""
    C = (2 * Hk + Hv) * d
    st = torch.empty(Hv, d, d, dtype=state_dtype, device="meta")
    cs = torch.empty(conv_rows, C, dtype=conv_dtype, device="meta")
    return st.numel() * st.element_size() + cs.numel() * cs.element_size()


def _bank_gb(g, **kw):
    per = _slot_bytes(int(g["key_heads"]), int(g["value_heads"]), int(g["head_dim"]), 4, **kw)
    return g["slots"] * g["gdn_layers"] * per / 1e9


def test_checkpoint_bank_matches_the_printed_size():
    g = _read("apc_checkpoint_bank.txt")
    gb = _bank_gb(g, state_dtype=torch.float32, conv_dtype=torch.bfloat16, conv_rows=3)
    assert abs(gb - g["bank_gb_decimal"]) <= g["half_unit_gb"], gb


@pytest.mark.parametrize("state_dtype,conv_dtype,conv_rows", [
    (torch.float32, torch.bfloat16, 4),      # W rows of conv state
    (torch.float32, torch.float32, 3),       # an fp32 conv state
    (torch.float32, torch.bfloat16, 0),      # no conv state
    (torch.bfloat16, torch.bfloat16, 3),     # a bf16 recurrent state
])
def test_other_layouts_miss_it(state_dtype, conv_dtype, conv_rows):
    g = _read("apc_checkpoint_bank.txt")
    gb = _bank_gb(g, state_dtype=state_dtype, conv_dtype=conv_dtype, conv_rows=conv_rows)
    assert abs(gb - g["bank_gb_decimal"]) > g["half_unit_gb"], gb


def test_the_bench_allocates_that_layout():
    """The bench's bank rows have the pinned shapes: fp32 [Hv, d, d] and bf16 [W-1, C_conv]."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    g = _read("apc_checkpoint_bank.txt")
    assert (bench.HK, bench.HV, bench.D, bench.W) == (int(g["key_heads"]),
                                                      int(g["value_heads"]),
                                                      int(g["head_dim"]), 4)
    assert bench.C_CONV == (2 * bench.HK + bench.HV) * bench.D
