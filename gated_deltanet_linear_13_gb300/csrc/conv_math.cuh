// The per-token arithmetic of the causal depthwise conv (model card "Qwen3.5 Gated Delta Net
// NKI Kernel for AWS Neuron", "How It Works"), shared by the conv kernels and the chunk-local
// kernel's fused conv so that both give the same bits.
#pragma once

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

// One token of a thread's CPT channels: y = bias + sum_j w[j] win[j] (then SiLU), on channel
// pairs with the packed fp32x2 multiply-add (each lane the same fp32 FMA as fmaf, in the same
// order), and the SiLU x / (1 + 2^(-x log2 e)) with the hardware 2^x and reciprocal per lane.
template <int W, int CPT>
__device__ __forceinline__ void conv_token(const float (&wt)[W][CPT], const float (&bi)[CPT],
                                           const float (&win)[W][CPT], int silu,
                                           float (&out)[CPT]) {
#pragma unroll
  for (int e = 0; e < CPT; e += 2) {
    float2 acc = make_float2(bi[e], bi[e + 1]);
#pragma unroll
    for (int j = 0; j < W; ++j)
      acc = __ffma2_rn(make_float2(wt[j][e], wt[j][e + 1]), make_float2(win[j][e], win[j][e + 1]),
                       acc);
    if (silu) {
      const float2 m = __fmul2_rn(acc, make_float2(-1.4426950408889634f, -1.4426950408889634f));
      const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f),
                                  make_float2(ptx::ex2_approx(m.x), ptx::ex2_approx(m.y)));
      float r0, r1;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d.x));
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d.y));
      acc = __fmul2_rn(acc, make_float2(r0, r1));
    }
    out[e] = acc.x;
    out[e + 1] = acc.y;
  }
}

}  // namespace gdn
