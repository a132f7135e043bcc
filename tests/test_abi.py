"""The C ABI without a GPU: the library loads, exports every symbol that include/gdn.h
declares, and rejects bad arguments on the host before any CUDA call.

Every call below is built to FAIL validation (or to be a documented no-op): none of them
ever reaches a kernel launch, so they are safe on any machine, with or without a GPU.
"""
import ctypes
import os
import re

import pytest

import gated_deltanet_linear_13_gb300 as gdn
from gated_deltanet_linear_13_gb300 import GdnDims, GdnOpts, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return gdn.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", src)) - {"sizeof"})


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert set(declared) == set(gdn.EXPORTED), declared
    for name in declared:
        assert hasattr(L, name), f"libgdn.so does not export {name}"


def test_status_strings_and_version(L):
    for code, name in gdn.STATUS_NAMES.items():
        assert gdn.gdn_status_string(code) == name
    assert gdn.gdn_status_string(99) == "GDN_UNKNOWN_STATUS"
    assert L.gdn_version() == 104


def _dims(**kw):
    base = dict(batch=1, seqlen=16, num_k_heads=16, num_v_heads=16, head_dim=128,
                chunk_size=64, conv_width=0, num_slots=0)
    base.update(kw)
    return GdnDims(*[base[f] for f, _ in GdnDims._fields_])


def _opts(**kw):
    base = dict(in_dtype=gdn.GDN_BF16, out_dtype=gdn.GDN_BF16, qk_l2norm=1, l2_eps=1e-6,
                scale=1.0, conv_silu=1, gates_precomputed=0)
    base.update(kw)
    return GdnOpts(*[base[f] for f, _ in GdnOpts._fields_])


A = 0x10000   # fake, 16-byte aligned addresses: only ever used in calls that fail validation


def _prefill(L, dims, opts, q=A, k=A, v=A, a=A, b=A, A_log=A, state=A, out=A, ws=None, wsb=0,
             conv_w=None, conv_state=None):
    return L.gdn_chunk_prefill(ctypes.byref(dims), ctypes.byref(opts), q, k, v, a, b, A_log,
                               None, conv_w, None, state, conv_state, None, out, ws, wsb, None)


def _snap(L, dims, opts, every, snap_state=A, snap_conv=None, nbank=4, snap_slots=A,
          conv_w=None, conv_state=None, q=A, k=A, v=A):
    return L.gdn_chunk_prefill_snapshots(ctypes.byref(dims), ctypes.byref(opts), q, k, v, A, A,
                                         A, None, conv_w, None, A, conv_state, None, A, every,
                                         snap_state, snap_conv, nbank, snap_slots, None, 0, None)


def test_snapshot_prefill_rejects_bad_arguments(L):
    d = _dims(seqlen=256)
    # the boundary spacing: positive and a whole number of 64-token chunks
    for every in (0, -64, 100, 32):
        assert _snap(L, d, _opts(), every) == 1
    # with at least one boundary inside T: bank, slot table and bank size are required
    assert _snap(L, d, _opts(), 128, snap_state=None) == 1
    assert _snap(L, d, _opts(), 128, snap_state=A + 4) == 1          # misaligned
    assert _snap(L, d, _opts(), 128, snap_slots=None) == 1
    assert _snap(L, d, _opts(), 128, nbank=0) == 1
    # with a conv: the conv-state bank too (x arrives in q, k = v = NULL)
    dc = _dims(seqlen=256, conv_width=4)
    assert _snap(L, dc, _opts(), 128, conv_w=A, conv_state=A, k=None, v=None,
                 snap_conv=None) == 1
    # bad dims are still caught first
    assert _snap(L, _dims(seqlen=256, head_dim=64), _opts(), 128) == 2
    # an empty batch is a no-op
    assert _snap(L, _dims(batch=0, seqlen=256), _opts(), 128) == 0


def test_gated_entries_reject_bad_gate(L):
    d = _dims()
    g = gdn.GdnOutGate(A, A, 1e-6)
    args = [ctypes.byref(d), ctypes.byref(_opts()), A, A, A, A, A, A, None, None, None, A, None,
            None, A]
    # a gate is required, with z and weight present and aligned and eps >= 0
    for bad in (None, gdn.GdnOutGate(None, A, 1e-6), gdn.GdnOutGate(A + 4, A, 1e-6),
                gdn.GdnOutGate(A, None, 1e-6), gdn.GdnOutGate(A, A + 2, 1e-6),
                gdn.GdnOutGate(A, A, -1.0), gdn.GdnOutGate(A, A, float("nan"))):
        ref = None if bad is None else ctypes.byref(bad)
        assert L.gdn_chunk_prefill_gated(*args, ref, None, 0, None) == 1
        dd = _dims(seqlen=1)
        dargs = [ctypes.byref(dd)] + args[1:]
        assert L.gdn_decode_step_gated(*dargs, ref, None) == 1
    # the layer's own checks still come first
    bad_dims = [ctypes.byref(_dims(head_dim=64))] + args[1:]
    assert L.gdn_chunk_prefill_gated(*bad_dims, ctypes.byref(g), None, 0, None) == 2


def test_prefill_ex_rejects_bad_arguments(L):
    """gdn_chunk_prefill_ex: NULL ext is the plain call; each part is checked as in its own
    entry point; a continued call's previous workspace must be aligned and must not overlap
    this call's; with conv width 4 (bf16) the conv taps and biases must be 16-byte aligned."""
    dc = _dims(conv_width=4)
    o = _opts()
    need = L.gdn_prefill_workspace_size(ctypes.byref(dc), ctypes.byref(o))
    ws = 0x100000

    def call(ext, conv_w=A, ws_=ws, d=dc):
        return L.gdn_chunk_prefill_ex(ctypes.byref(d), ctypes.byref(o), A, None, None, A, A, A,
                                      None, conv_w, None, A, A, None, A,
                                      None if ext is None else ctypes.byref(ext), ws_, need, None)

    ext = gdn.GdnPrefillExt()
    ext.prev_workspace = ws + 64                      # inside this call's workspace
    assert call(ext) == 1
    ext.prev_workspace = ws - 16                      # its conv tail runs into this workspace
    assert call(ext) == 1
    ext.prev_workspace = ws + need + 8                # misaligned
    assert call(ext) == 1
    assert call(None, conv_w=A + 4) == 1              # taps not 16-byte aligned (fused conv)
    bad = gdn.GdnPrefillExt()
    bad.snap_every = 100                              # not a whole number of chunks
    assert call(bad) == 1
    g = gdn.GdnOutGate(A + 4, A, 1e-6)                # misaligned gate
    bg = gdn.GdnPrefillExt()
    bg.gate = ctypes.cast(ctypes.pointer(g), ctypes.c_void_p)
    assert call(bg) == 1
    assert call(None, d=_dims(conv_width=4, head_dim=64)) == 2
    assert call(None, d=_dims(batch=0, conv_width=4)) == 0


def test_decode_multi_rejects_bad_arguments(L):
    def call(d, snap_state=None, snap_conv=None, nb=0, snap_slots=None):
        return L.gdn_decode_multi(ctypes.byref(d), ctypes.byref(_opts()), A, A, A, A, A, A, None,
                                  None, None, A, None, None, A, snap_state, snap_conv, nb,
                                  snap_slots, None)
    assert call(_dims(seqlen=17)) == 2                      # more than 16 tokens: the prefill
    assert call(_dims(seqlen=4, head_dim=64)) == 2
    assert call(_dims(seqlen=4), snap_slots=A) == 1          # slots without a bank
    assert call(_dims(seqlen=4), snap_state=A, nb=0, snap_slots=A) == 1
    assert call(_dims(seqlen=4), snap_state=A + 4, nb=3, snap_slots=A) == 1
    assert call(_dims(seqlen=0)) == 0 and call(_dims(batch=0, seqlen=4)) == 0


def test_varlen_rejects_bad_arguments(L):
    d = _dims(batch=3, seqlen=200)
    args = [ctypes.byref(d), ctypes.byref(_opts()), A, A, A, A, A, A, None, None, None, A, None,
            None]
    # offsets are required and 4-byte aligned
    assert L.gdn_chunk_prefill_varlen(*args, None, A, None, A, 1 << 30, None) == 1
    assert L.gdn_chunk_prefill_varlen(*args, A + 2, A, None, A, 1 << 30, None) == 1
    # the workspace must hold the offsets' tables and the tiles
    need = L.gdn_prefill_varlen_workspace_size(ctypes.byref(d), ctypes.byref(_opts()))
    assert need > 0
    assert L.gdn_chunk_prefill_varlen(*args, A, A, None, A, need - 1, None) == 3
    assert L.gdn_chunk_prefill_varlen(*args, A, A, None, None, need, None) == 3
    # a bad gate is rejected; bad dims first
    bad = gdn.GdnOutGate(None, A, 1e-6)
    assert L.gdn_chunk_prefill_varlen(*args, A, A, ctypes.byref(bad), A, need, None) == 1
    bd = [ctypes.byref(_dims(batch=3, seqlen=200, head_dim=64))] + args[1:]
    assert L.gdn_chunk_prefill_varlen(*bd, A, A, None, A, need, None) == 2
    # no sequences or no tokens: nothing to do
    for dd in (_dims(batch=0, seqlen=200), _dims(batch=3, seqlen=0)):
        a0 = [ctypes.byref(dd)] + args[1:]
        assert L.gdn_chunk_prefill_varlen(*a0, A, A, None, None, 0, None) == 0


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, 2), ("chunk_size", 32, 2), ("conv_width", 5, 2),
    ("num_v_heads", 24 + 1, 1), ("batch", -1, 1), ("seqlen", -3, 1), ("num_k_heads", 0, 1),
    ("batch", 70000, 2),
])
def test_prefill_rejects_bad_dims(L, field, value, status):
    assert _prefill(L, _dims(**{field: value}), _opts()) == status


def test_prefill_rejects_bad_opts(L):
    assert _prefill(L, _dims(), _opts(in_dtype=7)) == 1
    assert _prefill(L, _dims(), _opts(in_dtype=gdn.GDN_F32, out_dtype=gdn.GDN_BF16)) == 2
    assert _prefill(L, _dims(), _opts(l2_eps=-1.0)) == 1
    assert _prefill(L, _dims(), _opts(scale=float("nan"))) == 1


def test_prefill_rejects_bad_pointers(L):
    d, o = _dims(), _opts()
    assert _prefill(L, d, o, q=None) == 1
    assert _prefill(L, d, o, state=None) == 1
    assert _prefill(L, d, o, out=None) == 1
    assert _prefill(L, d, o, q=A + 8) == 1          # misaligned tensor
    assert _prefill(L, d, o, a=A + 2) == 1          # misaligned gate input
    assert _prefill(L, d, o, A_log=None) == 1        # needed unless gates are precomputed
    assert _prefill(L, d, o, k=None) == 1            # no conv: k and v are required
    # with a conv, x arrives in q and k / v must be NULL; weight and conv state required
    dc = _dims(conv_width=4)
    assert _prefill(L, dc, o, conv_w=A, conv_state=A) == 1                  # k, v given
    assert _prefill(L, dc, o, k=None, v=None, conv_w=None, conv_state=A) == 1
    assert _prefill(L, dc, o, k=None, v=None, conv_w=A, conv_state=None) == 1
    # state with fewer rows than the batch and no slot map
    assert _prefill(L, _dims(batch=4, num_slots=2), o) == 1


def test_prefill_workspace_two_halves_past_one_slice(L):
    """The 27B shape (48 value heads) holds floor(96 MiB / (48 x 80 KiB)) = 25 chunks of tiles
    per slice. A call of 25 chunks needs one slice's tiles; one more chunk makes two slices,
    and the workspace then holds two slices' worth (one written while the other is read)."""
    o = _opts()
    half = 25 * 48 * 80 * 1024 + ((25 * 48 * 4 + 255) // 256) * 256
    one = _dims(seqlen=25 * 64, num_v_heads=48)
    two = _dims(seqlen=26 * 64, num_v_heads=48)
    assert L.gdn_prefill_workspace_size(ctypes.byref(one), ctypes.byref(o)) == half
    assert L.gdn_prefill_workspace_size(ctypes.byref(two), ctypes.byref(o)) == 2 * half
    # a longer call keeps the same two halves
    long_ = _dims(seqlen=2048 * 64, num_v_heads=48)
    assert L.gdn_prefill_workspace_size(ctypes.byref(long_), ctypes.byref(o)) == 2 * half


def test_prefill_workspace_fused_conv(L):
    """With conv width 4 (bf16) the chunk-local kernel convolves the q and k channels itself:
    the workspace holds the call's conv tail [B][3][C_conv] (bf16, 1 KiB rounded) at offset 0,
    then the post-conv v channels [B][T][Hv d], then the tiles (25 chunks per slice at 48
    value heads, as without the conv)."""
    o = _opts()
    cc = (2 * 16 + 48) * 128
    tail = ((3 * cc * 2 + 1023) // 1024) * 1024
    half = 25 * 48 * 80 * 1024 + ((25 * 48 * 4 + 255) // 256) * 256
    for T, halves in ((25 * 64, 1), (26 * 64, 2), (2048 * 64, 2)):
        d = _dims(seqlen=T, num_k_heads=16, num_v_heads=48, conv_width=4)
        v = ((T * 48 * 128 * 2 + 1023) // 1024) * 1024
        assert L.gdn_prefill_workspace_size(ctypes.byref(d), ctypes.byref(o)) == (
            tail + v + halves * half), T


def test_prefill_workspace_checked(L):
    dc, o = _dims(conv_width=4), _opts()
    need = L.gdn_prefill_workspace_size(ctypes.byref(dc), ctypes.byref(o))
    # bf16, conv width 4: the conv tail (3 rows of the 6144 channels) + the post-conv v
    # channels (16 tokens x 16 heads x 128) + one chunk x 16 value heads of 80 KB tiles + their
    # e^{G_C} (256-byte rounded)
    assert need == 3 * (2 * 16 + 16) * 128 * 2 + 16 * 16 * 128 * 2 + 1 * 16 * 80 * 1024 + 256
    # bf16, another conv width: the post-conv activations + 80 KB tiles
    tiles = 1 * 16 * 80 * 1024 + 256
    d2 = _dims(conv_width=2)
    assert (L.gdn_prefill_workspace_size(ctypes.byref(d2), ctypes.byref(o)) ==
            1 * 16 * (2 * 16 + 16) * 128 * 2 + tiles)
    assert L.gdn_prefill_workspace_size(ctypes.byref(_dims()), ctypes.byref(o)) == tiles
    # the all-fp32 path needs only the conv activations
    of = _opts(in_dtype=gdn.GDN_F32, out_dtype=gdn.GDN_F32)
    assert L.gdn_prefill_workspace_size(ctypes.byref(_dims()), ctypes.byref(of)) == 0
    assert L.gdn_prefill_workspace_size(ctypes.byref(dc), ctypes.byref(of)) == 1 * 16 * 6144 * 4
    assert L.gdn_prefill_workspace_size(ctypes.byref(_dims(head_dim=7)), ctypes.byref(o)) == 0
    assert _prefill(L, dc, o, k=None, v=None, conv_w=A, conv_state=A, ws=None) == 3
    assert _prefill(L, dc, o, k=None, v=None, conv_w=A, conv_state=A, ws=A, wsb=need - 1) == 3
    assert _prefill(L, dc, o, k=None, v=None, conv_w=A, conv_state=A, ws=A + 4, wsb=need) == 3


def test_empty_calls_are_noops(L):
    # B == 0 or T == 0: GDN_OK without touching any pointer or CUDA
    assert _prefill(L, _dims(batch=0), _opts(), q=None, state=None, out=None) == 0
    assert _prefill(L, _dims(seqlen=0), _opts(), q=None, state=None, out=None) == 0


def test_decode_rejects_bad_arguments(L):
    def dec(dims, opts, **kw):
        p = dict(q=A, k=A, v=A, a=A, b=A, A_log=A, state=A, out=A)
        p.update(kw)
        return L.gdn_decode_step(ctypes.byref(dims), ctypes.byref(opts), p["q"], p["k"], p["v"],
                                 p["a"], p["b"], p["A_log"], None, None, None, p["state"], None,
                                 None, p["out"], None)
    assert dec(_dims(seqlen=2), _opts()) == 1                     # one token per sequence
    assert dec(_dims(seqlen=1, num_k_heads=1, num_v_heads=16), _opts()) == 2   # Hv/Hk > 8
    assert dec(_dims(seqlen=1, head_dim=256), _opts()) == 2
    assert dec(_dims(seqlen=1), _opts(), state=A + 4) == 1
    assert dec(_dims(seqlen=1, batch=0), _opts(), q=None) == 0


def test_conv_rejects_bad_arguments(L):
    def conv(B=1, T=4, C=64, W=4, dt=gdn.GDN_BF16, x=A, w=A, cs=A, ns=0, y=A + 4096):
        return L.causal_conv1d_update(B, T, C, W, dt, x, w, None, cs, ns, None, 1, y, None)
    assert conv(W=5) == 2
    assert conv(W=1) == 2
    assert conv(C=12) == 2
    assert conv(dt=3) == 1
    assert conv(x=None) == 1
    assert conv(x=A + 8) == 1
    assert conv(y=A) == 1                      # y aliases x
    assert conv(B=2, ns=1) == 1                # fewer state rows than sequences, no slot map
    assert conv(T=0, x=None) == 0              # empty


def test_checkpoint_rejects_bad_arguments(L):
    d = _dims(conv_width=4, num_slots=2)
    def ck(op=0, dims=d, dt=gdn.GDN_BF16, st=A, cs=A, ss=A, scs=A, nb=4, rows=A, slots=A, n=1):
        return L.gdn_state_checkpoint(op, ctypes.byref(dims), dt, st, cs, ss, scs, nb, rows,
                                      slots, n, None)
    assert ck(op=2) == 1
    assert ck(n=-1) == 1
    assert ck(dims=_dims(head_dim=64)) == 2
    assert ck(st=None) == 1
    assert ck(rows=None) == 1
    assert ck(cs=None) == 1
    assert ck(ss=A + 8) == 1
    assert ck(n=70000) == 2
    assert ck(n=0, st=None) == 0


def test_selftest_rejects_bad_limits(L):
    # out-of-range poll limits are refused before any launch
    for n in (0, (1 << 20) + 1, 0xFFFFFFFF):
        assert L.gdn_selftest_device_timeout(n, None) == 1
