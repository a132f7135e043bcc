"""The -DGDN_BOUNDS_CHECK build (libgdn_checked.so) on the GPU.

Its kernels check their computed global indices (workspace units, token rows, state and
conv-state rows, halo and tail rows) and record GDN_ERR_DEVICE_INDEX instead of faulting.
Small cases of every prefill form, the decode step, the multi-token step (both of its
kernels) and a checkpoint round trip run through it in a process of their own: each must match the oracle, report no index error, and give the
same bits on a second run (determinism).
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import os, sys
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))
import torch
import gdn_inputs as gi
import gated_deltanet_linear_13_gb300 as gdn
from gated_deltanet_linear_13_gb300 import build_lib
from gdn_testutil import assert_bf16_parity, assert_state_parity, oracle_full, to_device

gdn.load_library(build_lib.build(checked=True))


def clean(what):
    st = gdn.gdn_get_device_error()
    assert st == 0, f"{what}: {gdn.gdn_status_string(st)}"


def prefill(sh, seed, **kw):
    inp = gi.make_inputs(sh, seed=seed, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    outs = []
    for rep in range(2):
        dev = to_device(inp)
        out = torch.empty(sh.batch, sh.seqlen, sh.num_v_heads, 128, dtype=torch.bfloat16,
                          device="cuda")
        if sh.conv_width:
            gdn.gdn_chunk_prefill(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias,
                                  dev.state, out, num_k_heads=sh.num_k_heads,
                                  conv_weight=dev.conv_weight, conv_state=dev.conv_state, **kw)
        else:
            gdn.gdn_chunk_prefill(dev.q, dev.k, dev.v, dev.a, dev.b, dev.A_log, dev.dt_bias,
                                  dev.state, out, **kw)
        clean(f"prefill {sh}")
        outs.append((out, dev.state.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert_bf16_parity(outs[0][0].cpu(), ref.out, f"checked prefill {sh}")
    assert_state_parity(outs[0][1].cpu(), ref.state, what=f"checked prefill state {sh}")


# the tensor-core path with the conv fused: one slice; two slices (B = 8); ragged tails
prefill(gi.GDNShape(2, 97, 16, 48, conv_width=4), 11)
prefill(gi.GDNShape(8, 200, 16, 48, conv_width=4), 12)
# without a conv, and another conv width (separate conv kernels)
prefill(gi.GDNShape(2, 130, 2, 4), 13)
prefill(gi.GDNShape(2, 70, 2, 4, conv_width=2), 14)

# continued calls against plain calls
sh = gi.GDNShape(1, 3 * 128, 16, 48, conv_width=4)
dev = gi.make_inputs_device(sh, seed=15, device="cuda")
ws = [torch.empty(gdn.gdn_prefill_workspace_size(1, 128, 16, 48, 4), dtype=torch.uint8,
                  device="cuda") for _ in range(2)]
res = []
for chained in (False, True):
    st, cs = dev.state.clone(), dev.conv_state.clone()
    out = torch.empty(1, 3 * 128, 48, 128, dtype=torch.bfloat16, device="cuda")
    for i in range(3):
        sl = slice(128 * i, 128 * (i + 1))
        gdn.gdn_chunk_prefill_ex(dev.x[:, sl], None, None, dev.a[:, sl], dev.b[:, sl],
                                 dev.A_log, dev.dt_bias, st, out[:, sl], num_k_heads=16,
                                 conv_weight=dev.conv_weight, conv_state=cs, workspace=ws[i & 1],
                                 prev_workspace=ws[(i - 1) & 1] if (chained and i) else None)
    clean("continued calls")
    res.append((out, st, cs))
assert all(torch.equal(a, b) for a, b in zip(res[0], res[1])), "continued != plain"

# packed batch
sh = gi.GDNShape(1, 150, 2, 6, conv_width=4)
inp = gi.make_inputs(sh, seed=16, dtype="bf16", state="normal")
dev = to_device(inp)
dev.state = torch.cat([dev.state, dev.state, dev.state])
dev.conv_state = torch.cat([dev.conv_state, dev.conv_state, dev.conv_state])
cu = torch.tensor([0, 40, 41, 150], dtype=torch.int32, device="cuda")
out = torch.empty(1, 150, 6, 128, dtype=torch.bfloat16, device="cuda")
gdn.gdn_chunk_prefill_varlen(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                             out, num_k_heads=2, conv_weight=dev.conv_weight,
                             conv_state=dev.conv_state, cu_seqlens=cu)
clean("packed batch")

# multi-token steps: a small batch (per-item kernel, clusters), a batch of more items than
# SMs at T = 4 (the persistent kernel: staged inputs, bulk stores) and at T = 12 (chunks of 8)
sms = torch.cuda.get_device_properties(0).multi_processor_count
for (B, T, seed) in ((3, 4, 18), (sms // 2 + 7, 4, 19), (sms // 2 + 7, 12, 20)):
    sh = gi.GDNShape(B, T, 2, 6, conv_width=4)
    inp = gi.make_inputs(sh, seed=seed, dtype="bf16", state="normal")
    ref = oracle_full(inp)
    outs = []
    for rep in range(2):
        dev = to_device(inp)
        out = torch.empty(B, T, 6, 128, dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_multi(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state,
                             out, num_k_heads=2, conv_weight=dev.conv_weight,
                             conv_state=dev.conv_state)
        clean(f"multi-token B={B} T={T}")
        outs.append((out, dev.state.clone(), dev.conv_state.clone()))
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
    assert_bf16_parity(outs[0][0].cpu(), ref.out, f"checked multi-token B={B} T={T}")
    assert_state_parity(outs[0][1].cpu(), ref.state, what=f"checked multi-token state B={B}")

# a decode step, then a checkpoint round trip
sh = gi.GDNShape(3, 1, 16, 48, conv_width=4)
inp = gi.make_inputs(sh, seed=17, dtype="bf16", state="normal")
ref = oracle_full(inp)
dev = to_device(inp)
out = torch.empty(3, 1, 48, 128, dtype=torch.bfloat16, device="cuda")
gdn.gdn_decode_step(dev.x, None, None, dev.a, dev.b, dev.A_log, dev.dt_bias, dev.state, out,
                    num_k_heads=16, conv_weight=dev.conv_weight, conv_state=dev.conv_state)
clean("decode")
assert_bf16_parity(out.cpu(), ref.out, "checked decode")
bank = torch.zeros(4, 48, 128, 128, device="cuda")
cbank = torch.zeros(4, 3, sh.conv_channels, dtype=torch.bfloat16, device="cuda")
rows = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
slots = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
gdn.gdn_state_checkpoint("save", dev.state, dev.conv_state, bank, cbank, rows, slots,
                         num_k_heads=16)
clean("checkpoint")
assert torch.equal(bank[3], dev.state[0]) and torch.equal(bank[1], dev.state[2])
print("bounds-checked build: clean")
'''


def test_bounds_checked_build_runs_clean():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + SCRIPT],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "bounds-checked build: clean" in r.stdout
