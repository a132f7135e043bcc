// Causal depthwise conv1d with a carried conv state (the short conv in front of the gated
// delta rule; model card "Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron", "How It Works"
// and "Notice" on conv-state caching).
//
//   y[b,t,c] = bias[c] + sum_{j<W} w[c][j] * x[b, t-W+1+j, c]   (then SiLU if requested)
// positions before t = 0 read the conv state (the last W-1 pre-conv inputs, oldest first);
// afterwards the state holds the last W-1 inputs of this call.
//
// A thread owns 4 consecutive channels (8 bytes of bf16) of one sequence and a run of `TCH`
// tokens, sliding the window in registers, so each input element is read from HBM
// once (neighbouring token runs re-read W-1 halo tokens).  The thread holding the first
// token run is the only one that reads the old state of its channels, and it also writes
// the new state (taken from x, which nobody modifies), so no two threads race on it.
#include "common.cuh"

using namespace gdn;

static __device__ unsigned int g_err_conv;

unsigned gdn_take_error_conv() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_conv, sizeof(v));
  cudaMemcpyToSymbol(g_err_conv, &z, sizeof(z));
  return v;
}

constexpr int TCH = 4;    // tokens per thread (>= W - 1)
constexpr int CPT = 4;    // channels per thread (8 bytes of bf16, 16 bytes of fp32)

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 u;
  *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(v[0], v[1]);
  *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

template <typename T>
__global__ void __launch_bounds__(128) gdn_conv_kernel(int B, int T_, int C, int W, const T* x,
                                                       long long xs, const T* w, const T* bias,
                                                       T* cs, int num_slots,
                                                       const int32_t* slots, int silu, T* y,
                                                       long long ys) {
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * CPT;
  const int t0 = blockIdx.x * TCH;
  const int b = blockIdx.z;
  if (c0 >= C) return;
  const int slot = slots ? slots[b] : b;
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_err_conv, kErrIndex);
    return;
  }
  const T* xb = x + (size_t)b * T_ * xs + c0;
  T* yb = y + (size_t)b * T_ * ys + c0;
  T* csb = cs + (size_t)slot * (W - 1) * C + c0;
  const int t1 = min(T_, t0 + TCH);
  // this run's inputs first: independent loads, all in flight together
  float xr[TCH][CPT];
#pragma unroll
  for (int i = 0; i < TCH; ++i)
    if (t0 + i < t1) load4(xb + (size_t)(t0 + i) * xs, xr[i]);
  // window: win[0..W-2] = the W-1 inputs before token t0 (oldest first)
  float win[3][CPT];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) win[i][c] = 0.f;
    if (i < W - 1) {
      const int tau = t0 - (W - 1) + i;
      if (tau >= 0) load4(xb + (size_t)tau * xs, win[i]);
      else load4(csb + (size_t)(W - 1 + tau) * C, win[i]);
    }
  }
  // new conv state (first token run only): last W-1 inputs, read before anything is written
  float nst[3][CPT];
  const bool owner = (blockIdx.x == 0);
  if (owner) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      if (i < W - 1) {
        const int tau = T_ - (W - 1) + i;
        if (tau >= 0) load4(xb + (size_t)tau * xs, nst[i]);
        else load4(csb + (size_t)(W - 1 + tau) * C, nst[i]);
      }
    }
  }
  float wt[4][CPT];
  float bi[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) {
    bi[c] = bias ? ld_elem(bias + c0 + c) : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) wt[j][c] = (j < W) ? ld_elem(w + (size_t)(c0 + c) * W + j) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < TCH; ++i) {
    if (t0 + i >= t1) break;
    float out[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      float acc = bi[c];
#pragma unroll
      for (int j = 0; j < 3; ++j)
        if (j < W - 1) acc = fmaf(wt[j][c], win[j][c], acc);
      // the current token takes tap W-1
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j == W - 1) acc = fmaf(wt[j][c], xr[i][c], acc);
      out[c] = silu ? silu_f(acc) : acc;
      // shift the window
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (j < W - 2) win[j][c] = win[j + 1][c];
#pragma unroll
      for (int j = 0; j < 3; ++j)
        if (j == W - 2) win[j][c] = xr[i][c];
    }
    store4(yb + (size_t)(t0 + i) * ys, out);
  }
  if (owner) {
#pragma unroll
    for (int i = 0; i < 3; ++i)
      if (i < W - 1) store4(csb + (size_t)i * C, nst[i]);
  }
}

cudaError_t gdn_launch_conv(int B, int T, int C, int W, int bf16, const void* x,
                            long long x_tok_stride, const void* w, const void* bias,
                            void* conv_state, int num_slots, const int32_t* slots, int silu,
                            void* y, long long y_tok_stride, cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  const int threads = 128;
  dim3 grid((unsigned)((T + TCH - 1) / TCH), (unsigned)((C / CPT + threads - 1) / threads),
            (unsigned)B);
  if (bf16)
    gdn_conv_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(
        B, T, C, W, (const __nv_bfloat16*)x, x_tok_stride, (const __nv_bfloat16*)w,
        (const __nv_bfloat16*)bias, (__nv_bfloat16*)conv_state, num_slots, slots, silu,
        (__nv_bfloat16*)y, y_tok_stride);
  else
    gdn_conv_kernel<float><<<grid, threads, 0, stream>>>(
        B, T, C, W, (const float*)x, x_tok_stride, (const float*)w, (const float*)bias,
        (float*)conv_state, num_slots, slots, silu, (float*)y, y_tok_stride);
  return cudaGetLastError();
}
