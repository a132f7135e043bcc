"""Continued prefill calls (gdn_chunk_prefill_ex with prev_workspace) on the GPU.

A long prompt prefilled in fixed-size calls, each continuing the previous one, must give
exactly what the same calls give one after the other without overlap: the outputs, the
state, the conv state and the per-call checkpoints, bit for bit.  (Each plain call is
checked against the oracle by the prefill tests; here the continued calls only have to
reproduce it.)  Cases: the 27B-shape 512-token buckets with in-call snapshots standing in
for the checkpoint saves, also replayed from a CUDA graph; ragged buckets of a batch on
permuted state slots; calls shorter than the conv window; calls spanning several slices;
no conv; the gated output norm.
"""
import ctypes

import pytest
import torch

import gdn_inputs as gi

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


def _split(t, n, T):
    return [t[:, i * T:(i + 1) * T].contiguous() for i in range(n)]


class _Case:
    def __init__(self, gdn, B, T, n, Hk=16, Hv=48, W=4, num_slots=None, slots=None, seed=5,
                 gate=False):
        self.gdn, self.B, self.T, self.n, self.Hk, self.Hv, self.W = gdn, B, T, n, Hk, Hv, W
        sh = gi.GDNShape(B, T * n, Hk, Hv, conv_width=W)
        self.dev = gi.make_inputs_device(sh, seed=seed, device="cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 1)
        self.num_slots = num_slots or B
        self.state0 = torch.randn(self.num_slots, Hv, 128, 128, generator=g, device="cuda") * 0.02
        self.conv0 = None
        if W > 0:
            self.conv0 = torch.randn(self.num_slots, W - 1, sh.conv_channels, generator=g,
                                     device="cuda").to(torch.bfloat16)
            self.conv_bias = (torch.randn(sh.conv_channels, generator=g, device="cuda") * 0.1
                              ).to(torch.bfloat16)
            self.xs = _split(self.dev.x, n, T)
        else:
            self.qs, self.ks, self.vs = (_split(t, n, T) for t in (self.dev.q, self.dev.k,
                                                                  self.dev.v))
        self.as_, self.bs = _split(self.dev.a, n, T), _split(self.dev.b, n, T)
        self.slots = None if slots is None else torch.tensor(slots, dtype=torch.int32,
                                                             device="cuda")
        self.rows = self.slots if self.slots is not None else torch.arange(
            B, dtype=torch.int32, device="cuda")
        self.gate = None
        if gate:
            self.zs = [torch.randn(B, T, Hv, 128, generator=g, device="cuda").to(torch.bfloat16)
                       for _ in range(n)]
            self.gw = torch.rand(128, generator=g, device="cuda") + 0.5
        self.gated = gate
        dims = gdn.GdnDims(B, T, Hk, Hv, 128, 64, W, self.num_slots)
        opts = gdn._opts(gi_dt(gdn), gi_dt(gdn), True, 1e-6, 1.0, True, False)
        need = int(gdn.load_library().gdn_prefill_workspace_size(ctypes.byref(dims),
                                                                  ctypes.byref(opts)))
        self.ws = [torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
                   for _ in range(2)]

    def fresh(self):
        st = self.state0.clone()
        cs = None if self.conv0 is None else self.conv0.clone()
        outs = [torch.full((self.B, self.T, self.Hv, 128), 7.0, dtype=torch.bfloat16,
                           device="cuda") for _ in range(self.n)]
        return st, cs, outs

    def call(self, i, st, cs, out, prev=None, snap=None):
        gdn = self.gdn
        if self.W > 0:
            args = (self.xs[i], None, None)
            kw = dict(num_k_heads=self.Hk, conv_weight=self.dev.conv_weight,
                      conv_bias=self.conv_bias, conv_state=cs)
        else:
            args = (self.qs[i], self.ks[i], self.vs[i])
            kw = {}
        kw.update(state_slots=self.slots, workspace=self.ws[i & 1], prev_workspace=prev)
        if self.gated:
            kw.update(gate_z=self.zs[i], gate_weight=self.gw)
        if snap is not None:
            kw.update(snap_every=self.T, snap_state=snap[0], snap_conv_state=snap[1],
                      snap_slots=snap[2])
        gdn.gdn_chunk_prefill_ex(*args, self.as_[i], self.bs[i], self.dev.A_log,
                                 self.dev.dt_bias, st, out, **kw)

    def banks(self):
        nb = self.n * self.B
        bank = torch.zeros(nb, self.Hv, 128, 128, device="cuda")
        cbank = None
        if self.W > 0:
            cbank = torch.zeros(nb, self.W - 1, (2 * self.Hk + self.Hv) * 128,
                                dtype=torch.bfloat16, device="cuda")
        return bank, cbank

    def plain(self, save=False):
        """One call after the other (each starts after the previous one has finished); with
        save, a gdn_state_checkpoint SAVE of every sequence after every call."""
        st, cs, outs = self.fresh()
        bank, cbank = self.banks()
        for i in range(self.n):
            self.call(i, st, cs, outs[i])
            if save:
                bslots = torch.arange(i * self.B, (i + 1) * self.B, dtype=torch.int32,
                                      device="cuda")
                self.gdn.gdn_state_checkpoint("save", st, cs, bank, cbank, self.rows, bslots,
                                              num_k_heads=self.Hk)
        torch.cuda.synchronize()
        assert self.gdn.gdn_get_device_error() == 0
        return st, cs, outs, bank, cbank

    def chained(self, snap=False, st=None, cs=None, outs=None, bank=None, cbank=None):
        """Each call continues the previous one; with snap, in-call snapshots at the call end
        into the same bank rows as plain(save=True)."""
        if st is None:
            st, cs, outs = self.fresh()
            bank, cbank = self.banks()
        for i in range(self.n):
            sn = None
            if snap:
                sl = torch.arange(i * self.B, (i + 1) * self.B, dtype=torch.int32,
                                  device="cuda").view(self.B, 1)
                sn = (bank, cbank, sl)
            self.call(i, st, cs, outs[i], prev=self.ws[(i - 1) & 1] if i > 0 else None, snap=sn)
        return st, cs, outs, bank, cbank


def gi_dt(gdn):
    return gdn.GDN_BF16


def _same(a, b, what):
    assert len(a) == len(b)
    for x, y, name in zip(a, b, ("state", "conv state", "outputs", "bank", "conv bank")):
        if x is None:
            assert y is None
            continue
        if isinstance(x, list):
            for j, (xx, yy) in enumerate(zip(x, y)):
                assert torch.equal(xx, yy), f"{what}: {name} of call {j}"
        else:
            assert torch.equal(x, y), f"{what}: {name}"


def test_27b_buckets_with_snapshots_equal_plain_calls_and_saves(gdn):
    c = _Case(gdn, 1, 512, 6)
    ref = c.plain(save=True)
    got = c.chained(snap=True)
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    _same(got, ref, "continued 512-token calls")


def test_27b_buckets_continued_inside_a_cuda_graph(gdn):
    c = _Case(gdn, 1, 512, 4, seed=9)
    ref = c.plain(save=True)
    st, cs, outs = c.fresh()
    bank, cbank = c.banks()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        c.chained(snap=True, st=st, cs=cs, outs=outs, bank=bank, cbank=cbank)   # warm-up
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st.copy_(c.state0)
            cs.copy_(c.conv0)
            c.chained(snap=True, st=st, cs=cs, outs=outs, bank=bank, cbank=cbank)
    torch.cuda.synchronize()
    for o in outs:
        o.fill_(3.0)
    bank.zero_()
    cbank.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    _same((st, cs, outs, bank, cbank), ref, "graph replay of continued calls")


@pytest.mark.parametrize("B,T,n,slots,num_slots", [
    (3, 200, 4, [2, 0, 3], 5),      # ragged chunks, permuted slots
    (1, 2, 6, None, None),          # calls shorter than the conv window
    (1, 67, 3, None, None),
    (8, 256, 3, None, None),        # B = 8: two slices per call
])
def test_continued_calls_equal_plain_calls(gdn, B, T, n, slots, num_slots):
    c = _Case(gdn, B, T, n, slots=slots, num_slots=num_slots, seed=B * 100 + T)
    ref = c.plain()
    got = c.chained()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    _same(got[:3], ref[:3], f"B={B} T={T}")


def test_continued_calls_without_conv(gdn):
    c = _Case(gdn, 2, 128, 3, Hk=16, Hv=32, W=0, seed=77)
    ref = c.plain()
    got = c.chained()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    _same(got[:3], ref[:3], "no conv")


def test_continued_calls_with_gated_norm(gdn):
    c = _Case(gdn, 1, 256, 3, seed=31, gate=True)
    ref = c.plain()
    got = c.chained()
    torch.cuda.synchronize()
    assert gdn.gdn_get_device_error() == 0
    _same(got[:3], ref[:3], "gated")
