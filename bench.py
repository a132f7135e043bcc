"""Throughput of the gated delta rule on GB300: one JSON line.

Step = one pass of the whole hot path over the 27B-shape long-context workload: a
Qwen3.6-27B-shape gated-delta-net layer (16 key / 48 value heads, d = 128, width-4 conv,
bf16 inputs, fp32 state), B = 1, T = 131072 tokens processed as 256 prefill calls of 512
tokens, each followed by a checkpoint SAVE of the recurrent + conv state into a slot bank.
`value` = prefill tokens/s.  In the same run the batched decode step of the same layer
shape (B = 128 sequences, 256 consecutive steps on HBM-resident state) is timed and
reported as HBM GB/s under "decode".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (independent
sequences: no data-path collective); the control plane (barrier, max of the times) uses
gloo.  `cpu_baseline`: the fp64 CPU oracle over each GPU workload in full, on the same
inputs, on this host's cores (rank 0, after the GPU timings).  `--impl reference` times the
fp64 CPU oracle on a bounded sample of the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import gdn_inputs as gi  # noqa: E402

METRIC = "GDN prefill tokens/s (27B layer shape) and decode state-update HBM GB/s"
HK, HV, D, W = 16, 48, 128, 4
T_TOTAL, BUCKET = 131072, 512
DECODE_B, DECODE_STEPS = 128, 256   # --prefill-tokens / --decode-batch shrink these for ncu
C_CONV = (2 * HK + HV) * D
# algorithmic work (chunked WY/UT form, d = 128, C = 64): 6 d^2 + 10 C d FLOP per token per
# value head on the tensor cores
FLOP_PER_TOKEN = HV * (6 * D * D + 10 * 64 * D)
# decode bytes per sequence per step (bf16 out): state r+w, conv state r+w, x, out, gates
DECODE_BYTES_PER_SEQ = (2 * HV * D * D * 4 + 2 * (W - 1) * C_CONV * 2 + C_CONV * 2
                        + HV * D * 2 + 2 * HV * 2)
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def measured_traffic(key: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json), or None
    when the kernel sources changed since that capture or it was of another workload."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[key]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("workload") != workload:
        return None
    for src, digest in rec.get("sources", {}).items():
        try:
            if hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest() != digest:
                return None
        except OSError:
            return None
    return rec["bytes"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ ranks

class ControlPlane:
    """The ranks of one node (torchrun sets RANK / WORLD_SIZE / LOCAL_RANK / MASTER_*): each
    runs the whole workload on its own GPU (independent sequences, no collective on the data
    path); gloo carries only the host-side barrier and the max of the timings."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max_over_ranks(self, x: float) -> float:
        if self.dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.barrier()
            self.dist.destroy_process_group()


def whole_job_rate(world: int, units_per_rank: float, max_ms: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (max_ms / 1e3)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while the timed region runs, written
    as CSV to $GDN_CLOCK_LOG_DIR (default: the system temp directory)."""

    def __init__(self, gpu_index: int):
        self.proc = None
        log_dir = os.environ.get("GDN_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_rank{gpu_index}.csv")
        self.gpu = gpu_index

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows), "samples": len(rows),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ workload

def make_prefill_workload(device):
    sh = gi.GDNShape(1, T_TOTAL, HK, HV, conv_width=W)
    inp = gi.make_inputs_device(sh, seed=4000, device=device)
    nbk = T_TOTAL // BUCKET
    bank = torch.empty(nbk, HV, D, D, device=device)
    cbank = torch.empty(nbk, W - 1, C_CONV, dtype=torch.bfloat16, device=device)
    out = torch.empty(1, T_TOTAL, HV, D, dtype=torch.bfloat16, device=device)
    import gated_deltanet_linear_13_gb300 as gdn
    # two workspaces, used by alternate buckets: each call continues the one before it
    ws = [torch.empty(gdn.gdn_prefill_workspace_size(1, BUCKET, HK, HV, W), dtype=torch.uint8,
                      device=device) for _ in range(2)]
    rows = torch.zeros(1, dtype=torch.int32, device=device)
    slot_ids = torch.arange(nbk, dtype=torch.int32, device=device)
    return dict(inp=inp, bank=bank, cbank=cbank, out=out, ws=ws, rows=rows, slots=slot_ids)


def bucket_call(gdn, wl, i, checkpoint=True, gate=None):
    """Bucket i of the sequence through the public API: a call that continues bucket i - 1
    (its kernels start while that call's state chain finishes); with `checkpoint`, the state
    and conv state after the bucket go to checkpoint-bank slot i (an in-call snapshot at the
    call's end: the same bank rows as a gdn_state_checkpoint SAVE after the call)."""
    inp = wl["inp"]
    sl = slice(i * BUCKET, (i + 1) * BUCKET)
    kw = dict(num_k_heads=HK, conv_weight=inp.conv_weight, conv_state=inp.conv_state,
              workspace=wl["ws"][i & 1], prev_workspace=wl["ws"][(i - 1) & 1] if i else None)
    if checkpoint:
        kw.update(snap_every=BUCKET, snap_state=wl["bank"], snap_conv_state=wl["cbank"],
                  snap_slots=wl["slots"][i:i + 1].view(1, 1))
    if gate is not None:
        kw.update(gate_z=gate[0][:, sl], gate_weight=gate[1])
    gdn.gdn_chunk_prefill_ex(inp.x[:, sl], None, None, inp.a[:, sl], inp.b[:, sl], inp.A_log,
                             inp.dt_bias, inp.state, wl["out"][:, sl], **kw)


def prefill_step(gdn, wl):
    """A fresh sequence: 256 bucket calls of 512 tokens, a checkpoint of the state and conv
    state after each."""
    inp = wl["inp"]
    inp.state.zero_()
    inp.conv_state.zero_()
    for i in range(T_TOTAL // BUCKET):
        bucket_call(gdn, wl, i)


def prefill_step_separate_saves(gdn, wl):
    """The step with a gdn_state_checkpoint SAVE after each bucket call instead of the
    in-call snapshot (each save ends the overlap of consecutive calls)."""
    inp = wl["inp"]
    inp.state.zero_()
    inp.conv_state.zero_()
    for i in range(T_TOTAL // BUCKET):
        bucket_call(gdn, wl, i, checkpoint=False)
        gdn.gdn_state_checkpoint("save", inp.state, inp.conv_state, wl["bank"], wl["cbank"],
                                 wl["rows"], wl["slots"][i:i + 1], num_k_heads=HK)


def prefill_calls_only(gdn, wl, gate=None):
    """The 256 bucket prefill calls of a step without the checkpoints (kernel timing); with
    `gate` = (z [1, T, Hv, d], weight [d]) the gated output norm too."""
    for i in range(T_TOTAL // BUCKET):
        bucket_call(gdn, wl, i, checkpoint=False, gate=gate)


def make_decode_workload(device):
    sh = gi.GDNShape(DECODE_B, 1, HK, HV, conv_width=W)
    dec = gi.make_decode_inputs_device(sh, DECODE_STEPS, seed=3628, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(3629)
    state = torch.randn(DECODE_B, HV, D, D, generator=g, device=device) * 0.02
    conv_state = torch.randn(DECODE_B, W - 1, C_CONV, generator=g, device=device).to(torch.bfloat16)
    cw = (torch.randn(C_CONV, W, generator=g, device=device) / 2).to(torch.bfloat16)
    A_log = torch.rand(HV, generator=g, device=device) * math.log(16.0)
    dt_bias = torch.zeros(HV, device=device)
    out = torch.empty(DECODE_STEPS, DECODE_B, HV, D, dtype=torch.bfloat16, device=device)
    return dict(dec=dec, state=state, conv_state=conv_state, cw=cw, A_log=A_log,
                dt_bias=dt_bias, out=out)


def decode_steps(gdn, wl, events=None, gate=None):
    """DECODE_STEPS decode steps; with `gate` = (z [steps, B, Hv, d], weight [d]) the
    gated-norm entry point instead."""
    dec = wl["dec"]
    for t in range(DECODE_STEPS):
        if events is not None:
            events[t][0].record()
        args = (dec["x"][t].view(DECODE_B, 1, C_CONV), None, None,
                dec["a"][t].view(DECODE_B, 1, HV), dec["b"][t].view(DECODE_B, 1, HV),
                wl["A_log"], wl["dt_bias"], wl["state"], wl["out"][t].view(DECODE_B, 1, HV, D))
        kw = dict(num_k_heads=HK, conv_weight=wl["cw"], conv_state=wl["conv_state"])
        if gate is None:
            gdn.gdn_decode_step(*args, **kw)
        else:
            gdn.gdn_decode_step_gated(*args, gate_z=gate[0][t].view(DECODE_B, 1, HV, D),
                                      gate_weight=gate[1], **kw)
        if events is not None:
            events[t][1].record()


# ------------------------------------------------------------------ CPU oracle baseline

def oracle_sample(tokens: int, heads: int = HV, seed: int = 4000, reps: int = 1):
    """fp64 oracle over the first `tokens` tokens of `heads` value heads of the 27B-shape
    workload (host-generated inputs, same distributions), run `reps` times back to back with
    the recurrent and conv state carried from one pass to the next, as consecutive buckets
    of one sequence.  Returns (seconds, threads)."""
    import oracle
    sh = gi.GDNShape(1, tokens, HK, HV, conv_width=W)
    inp = gi.make_inputs(sh, seed=seed, dtype="bf16")
    nthreads = len(os.sched_getaffinity(0))
    state, conv_state = None, inp.conv_state
    t = time.perf_counter()
    for _ in range(reps):
        res = oracle.layer(num_k_heads=HK, num_v_heads=HV, x=inp.x, a=inp.a, b=inp.b,
                           A_log=inp.A_log, dt_bias=inp.dt_bias, conv_weight=inp.conv_weight,
                           conv_state=conv_state, state=state, nthreads=nthreads)
        state, conv_state = res.state, res.conv_state
    return time.perf_counter() - t, nthreads


# Arm CPU part numbers (/proc/cpuinfo "CPU part") of the cores these hosts use
_ARM_PARTS = {"0xd4f": "Neoverse-V2", "0xd40": "Neoverse-V1", "0xd0c": "Neoverse-N1",
              "0xd49": "Neoverse-N2", "0xd8e": "Neoverse-N3", "0xd84": "Neoverse-V3"}


def cpu_model():
    """The host CPU's model name and the number of cores this process may run on."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not name or name == "-":
        try:
            for line in open("/proc/cpuinfo"):
                key = line.split(":", 1)[0].strip().lower()
                if key == "model name":
                    name = line.split(":", 1)[1].strip()
                    break
                if key == "cpu part":
                    part = line.split(":", 1)[1].strip().lower()
                    name = _ARM_PARTS.get(part, "Arm part " + part)
                    break
        except OSError:
            pass
    return f"{name or 'unknown'}, {len(os.sched_getaffinity(0))} cores"


def _kh_layer(inp, kh, x=None, a=None, b=None, state=None, conv_state=None):
    """Keyword arguments of oracle.layer for key head kh with its r value heads, as a layer of
    one key head (exact: the conv is depthwise and value head h reads key head h / r); the
    device tensors (or the given ones) are sliced and copied to the host."""
    sh = inp.shape
    r = sh.num_v_heads // sh.num_k_heads
    h0 = kh * r
    idx = torch.cat([torch.arange(kh * D, (kh + 1) * D),
                     torch.arange(sh.num_k_heads * D + kh * D, sh.num_k_heads * D + (kh + 1) * D),
                     torch.arange(2 * sh.num_k_heads * D + h0 * D,
                                  2 * sh.num_k_heads * D + (h0 + r) * D)]).to(inp.x.device)
    x = inp.x if x is None else x
    a = inp.a if a is None else a
    b = inp.b if b is None else b
    B = x.shape[0]
    return dict(num_k_heads=1, num_v_heads=r, head_dim=D, nthreads=r,
                x=x.index_select(2, idx).cpu(), a=a[:, :, h0:h0 + r].cpu(),
                b=b[:, :, h0:h0 + r].cpu(), A_log=inp.A_log[h0:h0 + r].cpu(),
                dt_bias=inp.dt_bias[h0:h0 + r].cpu(),
                conv_weight=inp.conv_weight.index_select(0, idx).cpu(),
                state=(torch.zeros(B, r, D, D) if state is None else state[:, h0:h0 + r].cpu()),
                conv_state=(torch.zeros(B, W - 1, (2 + r) * D) if conv_state is None
                            else conv_state.index_select(2, idx).cpu()))


def _oracle_jobs(jobs, cores):
    """oracle.layer over a list of keyword sets, as many at a time as the cores allow (the C
    oracle runs outside the interpreter lock); returns the wall seconds."""
    import concurrent.futures as cf
    import oracle
    workers = max(1, cores // max(1, jobs[0]["nthreads"]))
    t = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda kw: oracle.layer(**kw), jobs))
    return time.perf_counter() - t


def cpu_full_baselines(device, prefill_inp, dwl):
    """The fp64 oracle on the host cores over each GPU workload IN FULL, on the same inputs:
    the 27B-shape prefill (131072 tokens x 48 value heads), the 27B-shape decode (256 steps at
    B = 128), the 4B-shape prefill (B = 4, T = 4096).  Copying the inputs to the host is not
    timed; the oracle calls are."""
    cores = len(os.sched_getaffinity(0))
    out = {}
    jobs = [_kh_layer(prefill_inp, kh) for kh in range(HK)]
    secs = _oracle_jobs(jobs, cores)
    out["prefill"] = {"value": T_TOTAL / secs, "unit": "tokens/s", "seconds": secs,
                      "sample": f"the whole workload: {T_TOTAL} tokens x {HV} value heads in one "
                                f"pass (conv + norm + gates + recurrence, fp64)"}
    del jobs
    # decode: 256 consecutive tokens per row are 256 decode steps (the same recurrence)
    dec = dwl["dec"]
    xs = dec["x"].transpose(0, 1)                         # [B, steps, C]
    a_, b_ = dec["a"].transpose(0, 1), dec["b"].transpose(0, 1)
    dinp = gi.GDNInputs(gi.GDNShape(DECODE_B, DECODE_STEPS, HK, HV, conv_width=W), "bf16",
                        None, None, None, xs, a_, b_, dwl["A_log"], dwl["dt_bias"], dwl["cw"],
                        dwl["state"], dwl["conv_state"])
    jobs = [_kh_layer(dinp, kh, state=dwl["state"], conv_state=dwl["conv_state"])
            for kh in range(HK)]
    for kw in jobs:
        kw["nthreads"] = cores
    secs = _oracle_jobs(jobs, cores)
    out["decode"] = {"value": DECODE_STEPS / secs, "unit": "steps/s", "seconds": secs,
                     "sample": f"{DECODE_STEPS} decode steps at B = {DECODE_B} ({DECODE_B * HV} "
                               f"units), the whole decode workload"}
    del jobs
    sh4 = gi.GDNShape(4, 4096, 16, 32, conv_width=W)
    in4 = gi.make_inputs_device(sh4, seed=4400, device=device, strong_decay_half=True)
    jobs = [_kh_layer(in4, kh) for kh in range(16)]
    for kw in jobs:
        kw["nthreads"] = max(1, cores // 4)
    secs = _oracle_jobs(jobs, cores)
    out["prefill_4b"] = {"value": 4 * 4096 / secs, "unit": "tokens/s", "seconds": secs,
                         "sample": "the whole workload: B = 4 x 4096 tokens x 32 value heads"}
    return out


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    tokens = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample(min(tokens, 64))
    times = []
    nthreads = 1
    for _ in range(args.steps):
        s, nthreads = oracle_sample(tokens)
        times.append(s)
    tok_s = tokens * args.steps / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "qwen36_27b_gdn_prefill_T131072_bucket512",
                   "sample_tokens_per_step": tokens, "heads": HV},
        "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": nthreads,
                         "kind": "oracle", "cpu": cpu_model(),
                         "sample": f"first {tokens} tokens x {HV} value heads of the 27B-shape "
                                   f"workload (conv + norm + gates + recurrence, fp64)"},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ profiler cases

def varlen16_inputs(device):
    """The packed 27B-shape batch of the bench: 16 sequences of seeded lengths in [64, 2048]."""
    lens = torch.randint(64, 2049, (16,), generator=torch.Generator().manual_seed(77))
    cu = torch.zeros(17, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    Tv = int(cu[-1])
    inv = gi.make_inputs_device(gi.GDNShape(1, Tv, HK, HV, conv_width=W), seed=4600,
                                device=device)
    return lens, cu, Tv, inv


def run_case(args):
    """One workload, three calls, nothing printed but a status line (for ncu captures)."""
    import gated_deltanet_linear_13_gb300 as gdn
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    gdn.load_library()
    device = torch.device("cuda", 0)
    if args.case == "decode_multi_T4":
        B, Tm = DECODE_B, 4
        inm = gi.make_inputs_device(gi.GDNShape(B, Tm, HK, HV, conv_width=W), seed=4704,
                                    device=device)
        st = torch.randn(B, HV, D, D, device=device) * 0.02
        cs = torch.zeros(B, W - 1, C_CONV, dtype=torch.bfloat16, device=device)
        out = torch.empty(B, Tm, HV, D, dtype=torch.bfloat16, device=device)
        for _ in range(3):
            gdn.gdn_decode_multi(inm.x, None, None, inm.a, inm.b, inm.A_log, inm.dt_bias, st,
                                 out, num_k_heads=HK, conv_weight=inm.conv_weight,
                                 conv_state=cs)
    else:
        lens, cu, Tv, inv = varlen16_inputs(device)
        st = torch.zeros(16, HV, D, D, device=device)
        cs = torch.zeros(16, W - 1, C_CONV, dtype=torch.bfloat16, device=device)
        out = torch.empty(1, Tv, HV, D, dtype=torch.bfloat16, device=device)
        for _ in range(3):
            gdn.gdn_chunk_prefill_varlen(inv.x, None, None, inv.a, inv.b, inv.A_log,
                                         inv.dt_bias, st, out, cu_seqlens=cu.to(device),
                                         num_k_heads=HK, conv_weight=inv.conv_weight,
                                         conv_state=cs)
    torch.cuda.synchronize()
    st = gdn.gdn_get_device_error()
    if st != 0:
        raise RuntimeError(f"device error in case {args.case}: {gdn.gdn_status_string(st)}")
    print(f"case {args.case}: ok")
    return 0


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=2048)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode-sweep", action="store_true")
    ap.add_argument("--no-prefill-4b", action="store_true")
    ap.add_argument("--no-latency", action="store_true",
                    help="skip the small-call latency sweep")
    ap.add_argument("--no-multi", action="store_true",
                    help="skip the multi-token decode steps")
    ap.add_argument("--no-varlen", action="store_true",
                    help="skip the packed variable-length prefill")
    ap.add_argument("--no-gated", action="store_true",
                    help="skip the gated-norm prefill / decode variants")
    ap.add_argument("--no-single-call", action="store_true",
                    help="skip the one-call 27B prefill with in-kernel snapshots")
    ap.add_argument("--e2e-streams", type=int, default=1, help="upload streams of the e2e pipeline")
    ap.add_argument("--e2e-group", type=int, default=4,
                    help="buckets per host copy in the e2e pipeline")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--prefill-tokens", type=int, default=T_TOTAL,
                    help="tokens of the prefill workload (a multiple of 512; smaller only for "
                         "profiling captures, the reported workload is 131072)")
    ap.add_argument("--decode-batch", type=int, default=DECODE_B)
    ap.add_argument("--case", default=None, choices=["decode_multi_T4", "varlen16"],
                    help="run one workload three times and exit (for profiler captures)")
    args = ap.parse_args()
    globals()["T_TOTAL"] = args.prefill_tokens
    globals()["DECODE_B"] = args.decode_batch
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)

    cp = ControlPlane()
    world, rank, local = cp.world, cp.rank, cp.local
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    def barrier():
        torch.cuda.synchronize()
        cp.barrier()
        torch.cuda.synchronize()

    max_over_ranks = cp.max_over_ranks

    import gated_deltanet_linear_13_gb300 as gdn
    from gated_deltanet_linear_13_gb300 import build_lib
    build_lib.build()
    gdn.load_library()
    peaks = load_peaks()

    # ---------------- prefill (the step), replayed as one CUDA graph of public-API calls
    wl = make_prefill_workload(device)
    prefill_step(gdn, wl)                      # eager once: attribute set-up, errors surface
    st = gdn.gdn_get_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the eager step: {gdn.gdn_status_string(st)}")
    nbk = T_TOTAL // BUCKET
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        prefill_step(gdn, wl)
    g_calls = torch.cuda.CUDAGraph()          # the prefill calls alone, for the kernel timing
    with torch.cuda.graph(g_calls):
        prefill_calls_only(gdn, wl)
    g_saves = torch.cuda.CUDAGraph()          # the step with separate checkpoint saves
    with torch.cuda.graph(g_saves):
        prefill_step_separate_saves(gdn, wl)
    for _ in range(args.warmup):
        g_step.replay()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clk:
        t_start.record()
        for _ in range(args.steps):
            g_step.replay()
        t_end.record()
        barrier()
        # per-launch duration of the prefill call, inside the same sampled window
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        reps = max(1, args.steps)
        g_calls.replay()
        c0.record()
        for _ in range(reps):
            g_calls.replay()
        c1.record()
        barrier()
    prefill_ms = t_start.elapsed_time(t_end)
    call_ms = c0.elapsed_time(c1) / (reps * nbk)
    g_saves.replay()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record()
    g_saves.replay()
    s1.record()
    torch.cuda.synchronize()
    separate_saves_ms = s0.elapsed_time(s1)
    del g_saves
    clocks = clk.summary()
    st = gdn.gdn_get_device_error()
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {gdn.gdn_status_string(st)}")
    prefill_ms = max_over_ranks(prefill_ms)
    ms_per_step = prefill_ms / args.steps
    value = whole_job_rate(world, T_TOTAL * args.steps, prefill_ms)
    achieved_tflops = FLOP_PER_TOKEN * BUCKET / (call_ms / 1e3) / 1e12

    # ---------------- the 4B-shape prefill (16 / 32 heads, B = 4, T = 4096, conv, half the heads
    #                  strongly decayed) as one call: the same kernels with four sequences
    other_prefill = []
    if not args.no_prefill_4b:
        sh4 = gi.GDNShape(4, 4096, 16, 32, conv_width=W)
        in4 = gi.make_inputs_device(sh4, seed=4400, device=device, strong_decay_half=True)
        out4 = torch.empty(4, 4096, 32, D, dtype=torch.bfloat16, device=device)

        def call4():
            gdn.gdn_chunk_prefill(in4.x, None, None, in4.a, in4.b, in4.A_log, in4.dt_bias,
                                  in4.state, out4, num_k_heads=16, conv_weight=in4.conv_weight,
                                  conv_state=in4.conv_state)
        call4()
        g4 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g4):
            call4()
        for _ in range(3):
            g4.replay()
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        q0.record()
        for _ in range(5):
            g4.replay()
        q1.record()
        torch.cuda.synchronize()
        ms4 = q0.elapsed_time(q1) / 5
        st = gdn.gdn_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in the 4B prefill: {gdn.gdn_status_string(st)}")
        tok4 = 4 * 4096 / (ms4 / 1e3)
        tf4 = tok4 * 32 * (6 * D * D + 10 * 64 * D) / 1e12
        other_prefill.append({"workload": "qwen35_4b_gdn_prefill_B4_T4096", "tokens_per_s": tok4,
                              "ms_per_call": ms4, "tflops": tf4,
                              "frac_of_bf16_burst": tf4 / peaks["bf16"]})
        del g4, in4, out4

    # ---------------- the same 27B-shape long-context workload as ONE call that records the
    #                  state every 512 tokens in-kernel (into the same 256-slot bank)
    if not args.no_single_call:
        inp = wl["inp"]
        ws1 = torch.empty(gdn.gdn_prefill_workspace_size(1, T_TOTAL, HK, HV, W),
                          dtype=torch.uint8, device=device)
        snap_rows = wl["slots"].view(1, nbk)

        def call1():
            inp.state.zero_()
            inp.conv_state.zero_()
            gdn.gdn_chunk_prefill_snapshots(
                inp.x, None, None, inp.a, inp.b, inp.A_log, inp.dt_bias, inp.state, wl["out"],
                snap_every=BUCKET, snap_state=wl["bank"], snap_conv_state=wl["cbank"],
                snap_slots=snap_rows, num_k_heads=HK, conv_weight=inp.conv_weight,
                conv_state=inp.conv_state, workspace=ws1)
        call1()
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1):
            call1()
        for _ in range(2):
            g1.replay()
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        q0.record()
        for _ in range(3):
            g1.replay()
        q1.record()
        torch.cuda.synchronize()
        ms1 = q0.elapsed_time(q1) / 3
        st = gdn.gdn_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in the single-call prefill: {gdn.gdn_status_string(st)}")
        tok1 = T_TOTAL / (ms1 / 1e3)
        tf1 = tok1 * FLOP_PER_TOKEN / 1e12
        other_prefill.append({"workload": "qwen36_27b_prefill_T131072_one_call_snapshot_every512",
                              "tokens_per_s": tok1, "ms_per_call": ms1, "tflops": tf1,
                              "frac_of_bf16_burst": tf1 / peaks["bf16"]})
        del g1, ws1

    # ---------------- a packed variable-length batch of the 27B shape: 16 sequences of seeded
    #                  lengths in [64, 2048] (about 17k tokens) in one call
    if not args.no_varlen:
        lens, cu, Tv, inv = varlen16_inputs(device)
        stv = torch.zeros(16, HV, D, D, device=device)
        csv = torch.zeros(16, W - 1, C_CONV, dtype=torch.bfloat16, device=device)
        outv = torch.empty(1, Tv, HV, D, dtype=torch.bfloat16, device=device)
        cud = cu.to(device)
        wsv = torch.empty(gdn.gdn_prefill_varlen_workspace_size(16, Tv, HK, HV, W),
                          dtype=torch.uint8, device=device)

        def callv():
            gdn.gdn_chunk_prefill_varlen(inv.x, None, None, inv.a, inv.b, inv.A_log,
                                         inv.dt_bias, stv, outv, cu_seqlens=cud, num_k_heads=HK,
                                         conv_weight=inv.conv_weight, conv_state=csv,
                                         workspace=wsv)
        callv()
        gv = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gv):
            callv()
        for _ in range(3):
            gv.replay()
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        q0.record()
        for _ in range(5):
            gv.replay()
        q1.record()
        torch.cuda.synchronize()
        msv = q0.elapsed_time(q1) / 5
        st = gdn.gdn_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in the packed prefill: {gdn.gdn_status_string(st)}")
        tokv = Tv / (msv / 1e3)
        tfv = tokv * FLOP_PER_TOKEN / 1e12
        other_prefill.append({"workload": f"qwen36_27b_prefill_varlen_16seq_T{Tv}",
                              "tokens_per_s": tokv, "ms_per_call": msv, "tflops": tfv,
                              "frac_of_bf16_burst": tfv / peaks["bf16"],
                              "lengths": [int(x) for x in lens]})
        del gv, inv, stv, csv, outv, wsv

    # ---------------- small calls: the 0.8B-shape prefill (16 / 16 heads, no conv, bf16, B = 1)
    #                  per T of its sweep, and the tiny fp32 layer (B = 1, T = 16): device time
    #                  per call, from a CUDA graph of 10 calls (so that host launch overhead is
    #                  not timed), median of 50 replays after 5 warm-ups; for T <= 16 also the
    #                  multi-token step on the same inputs
    latency = []
    if not args.no_latency:
        def lat_ms(fn):
            fn()
            gl = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gl):
                for _ in range(10):
                    fn()
            for _ in range(5):
                gl.replay()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(50)]
            for a0, a1 in evs:
                a0.record()
                gl.replay()
                a1.record()
            torch.cuda.synchronize()
            return statistics.median(a0.elapsed_time(a1) for a0, a1 in evs) / 10
        for Tl, f32 in [(t, False) for t in gi.SEQLEN_SWEEP_08B] + [(16, True)]:
            shl = gi.GDNShape(1, Tl, 16, 16, conv_width=0)
            inl = gi.make_inputs_device(shl, seed=4900 + Tl, device=device,
                                        dtype="f32" if f32 else "bf16")
            stl = torch.randn(1, 16, D, D, device=device) * 0.02
            outl = torch.empty(1, Tl, 16, D, dtype=torch.float32 if f32 else torch.bfloat16,
                               device=device)
            wsl = torch.empty(max(16, gdn.gdn_prefill_workspace_size(
                1, Tl, 16, 16, 0, torch.float32 if f32 else torch.bfloat16)),
                dtype=torch.uint8, device=device)

            def callp():
                gdn.gdn_chunk_prefill(inl.q, inl.k, inl.v, inl.a, inl.b, inl.A_log, inl.dt_bias,
                                      stl, outl, workspace=wsl)

            row = {"workload": ("tiny_fp32_B1_T16_16h" if f32 else f"qwen35_08b_prefill_T{Tl}"),
                   "T": Tl, "prefill_call_us": 1e3 * lat_ms(callp)}
            if Tl <= 16:
                def callm():
                    gdn.gdn_decode_multi(inl.q, inl.k, inl.v, inl.a, inl.b, inl.A_log,
                                         inl.dt_bias, stl, outl)
                row["decode_multi_us"] = 1e3 * lat_ms(callm)
            latency.append(row)
            del inl, stl, outl, wsl
        st = gdn.gdn_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in the latency sweep: {gdn.gdn_status_string(st)}")

    # ---------------- decode (same run, HBM-resident state), 256 steps as one CUDA graph
    dwl = make_decode_workload(device)
    decode_steps(gdn, dwl)
    st = gdn.gdn_get_device_error()
    if st != 0:
        raise RuntimeError(f"device error in decode: {gdn.gdn_status_string(st)}")
    g_dec = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_dec):
        decode_steps(gdn, dwl)
    for _ in range(3):
        g_dec.replay()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    dreps = 3
    barrier()
    d0.record()
    for _ in range(dreps):
        g_dec.replay()
    d1.record()
    barrier()
    mean_ms = d0.elapsed_time(d1) / (dreps * DECODE_STEPS)
    # eager per-step timing (launch overhead included) for reference
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(DECODE_STEPS)]
    decode_steps(gdn, dwl, dev_ev)
    barrier()
    eager_ms = statistics.median(a.elapsed_time(b) for a, b in dev_ev)
    dec_bytes = DECODE_BYTES_PER_SEQ * DECODE_B
    dec_gbs = dec_bytes / (mean_ms / 1e3) / 1e9
    st = gdn.gdn_get_device_error()
    if st != 0:
        raise RuntimeError(f"device error in decode: {gdn.gdn_status_string(st)}")
    # the same decode with the gated RMS norm fused into the output (z adds B Hv d bf16 bytes)
    gated = None
    if not args.no_gated:
        gz = (torch.randn(DECODE_STEPS, DECODE_B, HV, D, device=device).to(torch.bfloat16),
              torch.rand(D, device=device) + 0.5)
        decode_steps(gdn, dwl, gate=gz)
        g_gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_gd):
            decode_steps(gdn, dwl, gate=gz)
        for _ in range(3):
            g_gd.replay()
        d0.record()
        for _ in range(dreps):
            g_gd.replay()
        d1.record()
        torch.cuda.synchronize()
        gd_ms = d0.elapsed_time(d1) / (dreps * DECODE_STEPS)
        gd_bytes = dec_bytes + DECODE_B * HV * D * 2
        # and the 27B bucket prefill calls with the norm (z [1, T, Hv, d] bf16)
        gzp = (torch.randn(1, T_TOTAL, HV, D, device=device).to(torch.bfloat16), gz[1])
        prefill_calls_only(gdn, wl, gate=gzp)
        g_gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_gp):
            prefill_calls_only(gdn, wl, gate=gzp)
        for _ in range(2):
            g_gp.replay()
        d0.record()
        for _ in range(3):
            g_gp.replay()
        d1.record()
        torch.cuda.synchronize()
        gp_ms = d0.elapsed_time(d1) / 3
        st = gdn.gdn_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in the gated runs: {gdn.gdn_status_string(st)}")
        gated = {"what": "gated RMS norm fused into the output (w o / rms(o) silu(z))",
                 "prefill_tokens_per_s": T_TOTAL / (gp_ms / 1e3),
                 "prefill_call_ms": gp_ms / nbk,
                 "decode_step_ms": gd_ms,
                 "decode_gbs": gd_bytes / (gd_ms / 1e3) / 1e9,
                 "decode_frac_of_hbm": gd_bytes / (gd_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        del g_gd, g_gp, gz, gzp
    del g_dec              # (the decode inputs stay for the CPU baseline)
    # multi-token steps (gdn_decode_multi) at B = 128: T = 4 and 16 new tokens per sequence in
    # one step, against T single-token steps; bytes are those of one step plus the extra
    # tokens' inputs and outputs
    multi = []
    if not args.no_multi:
        for Tm in (4, 16):
            shm = gi.GDNShape(DECODE_B, Tm, HK, HV, conv_width=W)
            inm = gi.make_inputs_device(shm, seed=4700 + Tm, device=device)
            stm = torch.randn(DECODE_B, HV, D, D, device=device) * 0.02
            csm = torch.zeros(DECODE_B, W - 1, C_CONV, dtype=torch.bfloat16, device=device)
            outm = torch.empty(DECODE_B, Tm, HV, D, dtype=torch.bfloat16, device=device)

            def callm():
                gdn.gdn_decode_multi(inm.x, None, None, inm.a, inm.b, inm.A_log, inm.dt_bias, stm,
                                     outm, num_k_heads=HK, conv_weight=inm.conv_weight,
                                     conv_state=csm)
            callm()
            gm = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gm):
                for _ in range(8):
                    callm()
            gm.replay()
            d0.record()
            for _ in range(3):
                gm.replay()
            d1.record()
            torch.cuda.synchronize()
            ms_m = d0.elapsed_time(d1) / 24
            st = gdn.gdn_get_device_error()
            if st != 0:
                raise RuntimeError(f"device error in the multi-token step: {gdn.gdn_status_string(st)}")
            mbytes = dec_bytes + (Tm - 1) * DECODE_B * (C_CONV * 2 + HV * D * 2 + 2 * HV * 2)
            multi.append({"tokens": Tm, "step_us": 1e3 * ms_m,
                          "us_per_token": 1e3 * ms_m / Tm,
                          "vs_single_token_steps": Tm * mean_ms / ms_m,
                          "gbs": mbytes / (ms_m / 1e3) / 1e9})
            del gm, inm, stm, csm, outm
    # the other batch sizes of the 27B decode workload (64-step graphs), for latency
    dec_batches = []
    if not args.no_decode_sweep:
        main_b, main_steps = DECODE_B, DECODE_STEPS
        for bsz in (1, 8, 32):
            globals()["DECODE_B"], globals()["DECODE_STEPS"] = bsz, 64
            swl = make_decode_workload(device)
            decode_steps(gdn, swl)
            g_sw = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_sw):
                decode_steps(gdn, swl)
            for _ in range(3):
                g_sw.replay()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record()
            for _ in range(3):
                g_sw.replay()
            s1.record()
            torch.cuda.synchronize()
            step_ms = s0.elapsed_time(s1) / (3 * 64)
            dec_batches.append({"batch": bsz, "step_us": 1e3 * step_ms,
                                "gbs": DECODE_BYTES_PER_SEQ * bsz / (step_ms / 1e3) / 1e9})
            del g_sw, swl
        globals()["DECODE_B"], globals()["DECODE_STEPS"] = main_b, main_steps
        st = gdn.gdn_get_device_error()
        if st != 0:
            raise RuntimeError(f"device error in decode: {gdn.gdn_status_string(st)}")

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        inp = wl["inp"]
        hx = torch.empty(inp.x.shape, dtype=inp.x.dtype, pin_memory=True)
        ha = torch.empty(inp.a.shape, dtype=inp.a.dtype, pin_memory=True)
        hb = torch.empty(inp.b.shape, dtype=inp.b.dtype, pin_memory=True)
        hout = torch.empty(wl["out"].shape, dtype=wl["out"].dtype, pin_memory=True)
        hx.copy_(inp.x)
        ha.copy_(inp.a)
        hb.copy_(inp.b)
        e2e_steps = max(1, min(args.steps, 3))
        # A serving-style pipeline through the public API: the gate inputs a, b of the step go
        # up first (two copies), then x in groups of `e2e_group` buckets on one stream while
        # earlier buckets compute, and each group's output comes down on another as soon as
        # its last bucket is done; every byte of every step's inputs and result crosses the
        # host link inside the timed region.  The whole step is captured once as a CUDA graph.
        n_up = args.e2e_streams
        grp = max(1, args.e2e_group)
        s_ups = [torch.cuda.Stream() for _ in range(n_up)]
        s_down = torch.cuda.Stream()
        nbk = T_TOTAL // BUCKET
        ngr = (nbk + grp - 1) // grp
        ev_ab = torch.cuda.Event()
        ev_in = [torch.cuda.Event() for _ in range(ngr)]
        ev_out = [torch.cuda.Event() for _ in range(ngr)]

        def e2e_body():
            comp = torch.cuda.current_stream()
            for su in s_ups:
                su.wait_stream(comp)
            s_down.wait_stream(comp)
            inp.state.zero_()
            inp.conv_state.zero_()
            with torch.cuda.stream(s_ups[0]):
                inp.a.copy_(ha, non_blocking=True)
                inp.b.copy_(hb, non_blocking=True)
                ev_ab.record(s_ups[0])
            comp.wait_event(ev_ab)
            for gi_ in range(ngr):
                gs = slice(gi_ * grp * BUCKET, min(nbk, (gi_ + 1) * grp) * BUCKET)
                s_up = s_ups[gi_ % n_up]
                with torch.cuda.stream(s_up):
                    inp.x[:, gs].copy_(hx[:, gs], non_blocking=True)
                    ev_in[gi_].record(s_up)
                comp.wait_event(ev_in[gi_])
                for i in range(gi_ * grp, min(nbk, (gi_ + 1) * grp)):
                    bucket_call(gdn, wl, i)
                ev_out[gi_].record(comp)
                with torch.cuda.stream(s_down):
                    s_down.wait_event(ev_out[gi_])
                    hout[:, gs].copy_(wl["out"][:, gs], non_blocking=True)
            for su in s_ups:
                comp.wait_stream(su)
            comp.wait_stream(s_down)

        e2e_body()                      # eager warm-up of the pipeline
        torch.cuda.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_body()

        def e2e_step():
            g_e2e.replay()

        e2e_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(e2e_steps):
            e2e_step()
        e1.record()
        barrier()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1))
        if not torch.equal(hout[0, -BUCKET:], wl["out"][0, -BUCKET:].cpu()):
            raise RuntimeError("end-to-end output differs from the device result")
        h2d = (hx.numel() * hx.element_size() + ha.numel() * ha.element_size() +
               hb.numel() * hb.element_size())
        d2h = hout.numel() * hout.element_size()
        e2e = {"value": whole_job_rate(world, T_TOTAL * e2e_steps, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / e2e_steps,
               "pipeline": f"a, b up once; x up and out down per {grp} buckets "
                           f"({args.e2e_streams} upload streams), compute per 512-token bucket"}

    # ---------------- CPU oracle baseline (rank 0): every GPU workload in full, same inputs
    cpu = None
    if rank == 0 and not args.no_cpu:
        full = cpu_full_baselines(device, wl["inp"], dwl)
        cpu = dict(full["prefill"], cores=len(os.sched_getaffinity(0)), kind="oracle",
                   cpu=cpu_model(),
                   other_workloads=[dict(full["decode"], workload=f"qwen36_27b_decode_B{DECODE_B}"),
                                    dict(full["prefill_4b"],
                                         workload="qwen35_4b_gdn_prefill_B4_T4096")])

    if rank == 0:
        # per bucket: the conv of the value channels, then (chunk-local kernel with the q / k
        # conv + state-chain kernel) per slice of chunks whose tiles fit the 96 MB slice budget
        # (80 KB per chunk and value head); the chains store the checkpoint rows themselves
        nch = BUCKET // 64
        per_slice = max(1, min(512, nch, (96 << 20) // (HV * 80 * 1024)))
        launches_per_step = nbk * (1 + 2 * (-(-nch // per_slice)))
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "qwen36_27b_gdn_prefill_T131072_bucket512",
                       "batch": 1, "seq_len": T_TOTAL, "bucket": BUCKET, "num_k_heads": HK,
                       "num_v_heads": HV, "head_dim": D, "conv_width": W, "chunk": 64,
                       "checkpoint_every": BUCKET,
                       "checkpoint": "state and conv state into bank slot i at the end of "
                                     "bucket call i (in-call snapshot); each call continues "
                                     "the previous one",
                       "step_ms_with_separate_checkpoint_saves": separate_saves_ms,
                       "l2": "inputs larger than L2 (2.7 GB x)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": achieved_tflops,
                         "peak": peaks["bf16"], "unit": "TFLOP/s",
                         "frac": achieved_tflops / peaks["bf16"],
                         "traffic": measured_traffic("prefill_call", f"qwen36_27b_prefill_bucket{BUCKET}"),
                         "kernel": "gdn_chunk_prefill (conv + chunked recurrence), 512 tokens",
                         "flop_per_launch": FLOP_PER_TOKEN * BUCKET,
                         "launch_ms": call_ms,
                         "peak_source": peaks["source"] + " burst (the call is timed in a "
                                        "sub-second region)"},
            "other_prefill": other_prefill,
            "latency": latency,
            "decode": {"metric": "decode state-update HBM GB/s", "value": dec_gbs,
                       "unit": "GB/s", "batch": DECODE_B, "steps": DECODE_STEPS,
                       "step_ms_graph_mean": mean_ms, "step_ms_eager_median": eager_ms,
                       "bytes_per_step": dec_bytes,
                       "roofline": {"bound": "hbm", "achieved": dec_gbs,
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": dec_gbs / peaks["hbm_gbs"],
                                    "traffic": measured_traffic("decode_step", f"qwen36_27b_decode_B{DECODE_B}"),
                                    "peak_source": peaks["source"]},
                       "l2": "state 805 MB > L2", "other_batches": dec_batches,
                       "multi_token": multi},
            "gated_rmsnorm": gated,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps,
        }
        print(json.dumps(line))
    cp.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
