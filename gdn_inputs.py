"""Seeded synthetic inputs for the gated delta rule (shared by the tests, the bench and smoke).

This module holds no arithmetic of the method: it only draws random numbers with the
distributions that the workloads prescribe and casts them to the storage dtype.  Both the
CUDA path and the fp64 oracle receive exactly the tensors produced here (the oracle after an
exact upcast to float64), so the two sides never share any step of the computation.

Distributions (Qwen3.5/3.6 gated-delta-net layer shapes, d_k = d_v = 128):
  * q, k, v ~ N(0, 1); with a causal conv the pre-conv activation x ~ N(0, 1) over the
    concatenated q|k|v channels (C_conv = (2*Hk + Hv) * d).
  * gate inputs a ~ N(0, 1) and b ~ N(0, 1) per token and value head (beta = sigmoid(b),
    g = -exp(A_log) * softplus(a + dt_bias) are formed by the consumer, not here).
  * A_log ~ U(0, ln 16) per value head; with ``strong_decay_half`` the first half of the value
    heads draw A_log ~ U(ln 8, ln 16).  dt_bias = 0.
  * conv weight ~ N(0, 1/W) per tap, no bias.
  * initial recurrent state: zeros, or N(0, 0.02^2) (0.02 read as the standard deviation).

Host generation uses numpy's PCG64 (``numpy.random.Generator(PCG64(seed))``) in float32,
then a round-to-nearest-even cast to bf16 through torch.  Device generation (for the
multi-GiB long-context workload) uses a seeded ``torch.Generator`` on the GPU with the same
distributions; those tensors are copied back to the host wherever the oracle checks them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

HEAD_DIM = 128


@dataclass
class GDNShape:
    """Geometry of one gated-delta-net layer call."""
    batch: int
    seqlen: int
    num_k_heads: int
    num_v_heads: int
    head_dim: int = HEAD_DIM
    conv_width: int = 0          # 0 = q/k/v given directly; 4 = causal depthwise conv first

    @property
    def conv_channels(self) -> int:
        return (2 * self.num_k_heads + self.num_v_heads) * self.head_dim


# Named workloads (sizes of the Qwen3.5/3.6 layer shapes these pages describe).
WORKLOADS = {
    # tiny fp32 layer, 16 tokens, 16/16 heads, zero initial state
    "tiny_fp32_T16": dict(B=1, T=16, Hk=16, Hv=16, W=0, dtype="f32", state="zero"),
    # 0.8B-shape prefill, 16/16 heads, T swept, state ~ N(0, 0.02^2)
    "qwen35_08b_prefill": dict(B=1, T=None, Hk=16, Hv=16, W=0, dtype="bf16", state="normal"),
    # 4B-shape prefill with conv, 16/32 heads, B=4, T=4096, half the heads strongly decayed
    "qwen35_4b_prefill_B4_T4096": dict(B=4, T=4096, Hk=16, Hv=32, W=4, dtype="bf16",
                                      state="zero", strong=True),
    # 27B-shape decode, 16/48 heads, conv
    "qwen36_27b_decode": dict(B=None, T=1, Hk=16, Hv=48, W=4, dtype="bf16", state="zero"),
    # 27B-shape long-context prefill, 16/48 heads, conv, T = 131072 in 512-token buckets
    "qwen36_27b_prefill_T131072": dict(B=1, T=131072, Hk=16, Hv=48, W=4, dtype="bf16",
                                      state="zero"),
}

SEQLEN_SWEEP_08B = (2, 10, 15, 16, 51, 100, 127, 129, 200)
DECODE_BATCHES_27B = (1, 8, 32, 128)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bf16 torch (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


@dataclass
class GDNInputs:
    shape: GDNShape
    dtype: str                      # "bf16" or "f32": storage dtype of q/k/v/x/a/b/conv
    q: Optional[torch.Tensor]       # [B,T,Hk,d]   (None when conv_width > 0)
    k: Optional[torch.Tensor]       # [B,T,Hk,d]
    v: Optional[torch.Tensor]       # [B,T,Hv,d]
    x: Optional[torch.Tensor]       # [B,T,C_conv] pre-conv (None when conv_width == 0)
    a: torch.Tensor                 # [B,T,Hv]
    b: torch.Tensor                 # [B,T,Hv]
    A_log: torch.Tensor             # [Hv] fp32
    dt_bias: torch.Tensor           # [Hv] fp32
    conv_weight: Optional[torch.Tensor]   # [C_conv, W]
    state: torch.Tensor             # [B,Hv,d,d] fp32, layout S[v][k]
    conv_state: Optional[torch.Tensor]    # [B,W-1,C_conv]
    extra: dict = field(default_factory=dict)

    def tensors(self):
        return {k: v for k, v in self.__dict__.items() if isinstance(v, torch.Tensor)}


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return to_bf16(a)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def make_inputs(shape: GDNShape, seed: int, dtype: str = "bf16", state: str = "zero",
                strong_decay_half: bool = False, state_std: float = 0.02) -> GDNInputs:
    """Host-side seeded inputs (numpy PCG64, float32, then cast)."""
    B, T, Hk, Hv, d, W = (shape.batch, shape.seqlen, shape.num_k_heads, shape.num_v_heads,
                          shape.head_dim, shape.conv_width)
    rng = np.random.Generator(np.random.PCG64(seed))
    f32 = np.float32
    q = k = v = x = cw = cs = None
    if W > 0:
        C = shape.conv_channels
        x = _cast(rng.standard_normal((B, T, C), dtype=f32), dtype)
        cw = _cast(rng.standard_normal((C, W), dtype=f32) * f32(1.0 / math.sqrt(W)), dtype)
        cs = _cast(np.zeros((B, W - 1, C), dtype=f32), dtype)
    else:
        q = _cast(rng.standard_normal((B, T, Hk, d), dtype=f32), dtype)
        k = _cast(rng.standard_normal((B, T, Hk, d), dtype=f32), dtype)
        v = _cast(rng.standard_normal((B, T, Hv, d), dtype=f32), dtype)
    a = _cast(rng.standard_normal((B, T, Hv), dtype=f32), dtype)
    b = _cast(rng.standard_normal((B, T, Hv), dtype=f32), dtype)
    A_log = rng.uniform(0.0, math.log(16.0), size=Hv).astype(f32)
    if strong_decay_half:
        A_log[: Hv // 2] = rng.uniform(math.log(8.0), math.log(16.0), size=Hv // 2).astype(f32)
    dt_bias = np.zeros(Hv, dtype=f32)
    if state == "zero":
        S = np.zeros((B, Hv, d, d), dtype=f32)
    elif state == "normal":
        S = rng.standard_normal((B, Hv, d, d), dtype=f32) * f32(state_std)
    else:
        raise ValueError(state)
    return GDNInputs(shape, dtype, q, k, v, x, a, b, torch.from_numpy(A_log),
                     torch.from_numpy(dt_bias), cw, torch.from_numpy(np.ascontiguousarray(S)), cs)


def make_inputs_device(shape: GDNShape, seed: int, device, dtype: str = "bf16",
                       strong_decay_half: bool = False) -> GDNInputs:
    """Device-side seeded inputs (torch.Generator on the GPU) for multi-GiB workloads.

    Same distributions as :func:`make_inputs`; zero initial recurrent and conv state.
    """
    B, T, Hk, Hv, d, W = (shape.batch, shape.seqlen, shape.num_k_heads, shape.num_v_heads,
                          shape.head_dim, shape.conv_width)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def randn(*s):
        return torch.randn(*s, generator=g, device=device, dtype=torch.float32).to(tdt)

    q = k = v = x = cw = cs = None
    if W > 0:
        C = shape.conv_channels
        x = randn(B, T, C)
        cw = (torch.randn(C, W, generator=g, device=device) / math.sqrt(W)).to(tdt)
        cs = torch.zeros(B, W - 1, C, device=device, dtype=tdt)
    else:
        q, k, v = randn(B, T, Hk, d), randn(B, T, Hk, d), randn(B, T, Hv, d)
    a, b = randn(B, T, Hv), randn(B, T, Hv)
    A_log = torch.rand(Hv, generator=g, device=device) * math.log(16.0)
    if strong_decay_half:
        A_log[: Hv // 2] = math.log(8.0) + torch.rand(Hv // 2, generator=g, device=device) * (
            math.log(16.0) - math.log(8.0))
    dt_bias = torch.zeros(Hv, device=device)
    S = torch.zeros(B, Hv, d, d, device=device)
    return GDNInputs(shape, dtype, q, k, v, x, a, b, A_log, dt_bias, cw, S, cs)


def make_decode_inputs_device(shape: GDNShape, steps: int, seed: int, device,
                              dtype: str = "bf16"):
    """Per-step decode inputs on the device: x [steps, B, C_conv] (or q/k/v [steps, B, H, d]
    without a conv), a, b [steps, B, Hv]; step t's slices are contiguous."""
    B, Hk, Hv, d = shape.batch, shape.num_k_heads, shape.num_v_heads, shape.head_dim
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def randn(*s):
        return torch.randn(*s, generator=g, device=device, dtype=torch.float32).to(tdt)

    out = {}
    if shape.conv_width > 0:
        out["x"] = randn(steps, B, shape.conv_channels)
    else:
        out["q"], out["k"], out["v"] = (randn(steps, B, Hk, d), randn(steps, B, Hk, d),
                                        randn(steps, B, Hv, d))
    out["a"], out["b"] = randn(steps, B, Hv), randn(steps, B, Hv)
    return out
