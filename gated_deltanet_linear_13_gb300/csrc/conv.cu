// Causal depthwise conv1d with a carried conv state (the short conv in front of the gated
// delta rule; model card "Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron", "How It Works"
// and "Notice" on conv-state caching).
//
//   y[b,t,c] = bias[c] + sum_{j<W} w[c][j] * x[b, t-W+1+j, c]   (then SiLU if requested)
// positions before t = 0 read the conv state (the last W-1 pre-conv inputs, oldest first);
// afterwards the state holds the last W-1 inputs of this call.
//
// A CTA owns a tile of 64 tokens x 512 bytes of channels of one sequence: it loads the tile
// plus the W-1 rows before it (x, or the conv state before the sequence start) with
// independent 16-byte loads into shared memory, then each thread slides the window down 16
// tokens of one 4-byte column.  The thread holding a sequence's first tokens of a column is
// the only one that reads the old state of its channels, and it also writes the new state
// (taken from x, which nobody modifies), so no two threads race on it.
#include "common.cuh"

using namespace gdn;

static __device__ unsigned int g_err_conv;

unsigned gdn_take_error_conv() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_conv, sizeof(v));
  cudaMemcpyToSymbol(g_err_conv, &z, sizeof(z));
  return v;
}

constexpr int TT = 64;             // tokens per CTA tile
constexpr int TG = 16;             // tokens per thread (a CTA has TT / TG token groups)
constexpr int TILE_BYTES = 512;    // bytes of one token row of the tile (256 bf16 / 128 fp32)
constexpr int WORDS = TILE_BYTES / 4;                 // 4-byte words per row
constexpr int CONV_THREADS = WORDS * (TT / TG);       // a thread: one word x TG tokens

// one 4-byte word of a row: two bf16 channels or one fp32 channel
__device__ __forceinline__ void ld_word(const __nv_bfloat16* p, float (&v)[2]) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
  v[0] = f.x; v[1] = f.y;
}
__device__ __forceinline__ void ld_word(const float* p, float (&v)[1]) { v[0] = *p; }
__device__ __forceinline__ void st_word(__nv_bfloat16* p, const float (&v)[2]) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
}
__device__ __forceinline__ void st_word(float* p, const float (&v)[1]) { *p = v[0]; }

// x * sigmoid(x) = x / (1 + 2^(-x log2 e)): hardware 2^x and fast division (a few ulp; the
// limits x -> -inf and x -> +inf give 0 and x)
__device__ __forceinline__ float silu_fast(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * x));
  return __fdividef(x, 1.0f + e);
}

template <typename T, int W>
__global__ void __launch_bounds__(CONV_THREADS) gdn_conv_kernel(
    int B, int T_, int C, const T* x, long long xs, const T* w, const T* bias, T* cs,
    int num_slots, const int32_t* slots, int silu, T* y, long long ys) {
  constexpr int CC = TILE_BYTES / (int)sizeof(T);       // channels per tile
  constexpr int CPT = CC / WORDS;                       // channels per thread (2 or 1)
  constexpr int H = W - 1;                              // halo rows
  constexpr int ROWS = TT + H;
  __shared__ __align__(16) uint8_t tile[ROWS * TILE_BYTES];
  const int t0 = blockIdx.x * TT, cb = blockIdx.y * CC, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int slot = slots ? slots[b] : b;
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_err_conv, kErrIndex);
    return;
  }
  const T* xb = x + (size_t)b * T_ * xs;
  T* csb = cs + (size_t)slot * H * C;
  const int nt = min(TT, T_ - t0);
  // ---- tile rows r = 0 .. nt+H-1 hold the inputs of tokens t0 - H + r: x for tokens >= 0,
  //      the conv state for the (up to W-1) positions before the sequence start
  constexpr int CPR = TILE_BYTES / 16;                  // 16-byte pieces per row
  constexpr int NB = 2;                                 // loads in flight per thread per pass
  const int total = (nt + H) * CPR;
  for (int base = 0; base < total; base += NB * CONV_THREADS) {
    uint4 v[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int idx = base + u * CONV_THREADS + tid;
      const int r = idx / CPR, c = cb + (idx % CPR) * (16 / (int)sizeof(T));
      const int tau = t0 - H + r;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < total && c < C) {
        if (tau >= 0) v[u] = *reinterpret_cast<const uint4*>(xb + (size_t)tau * xs + c);
        else v[u] = *reinterpret_cast<const uint4*>(csb + (size_t)(H + tau) * C + c);
      }
    }
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int idx = base + u * CONV_THREADS + tid;
      if (idx < total) *reinterpret_cast<uint4*>(tile + idx * 16) = v[u];
    }
  }
  const int wi = tid % WORDS, tg = tid / WORDS;
  const int c0 = cb + wi * CPT;
  // ---- the new conv state (first token tile, first token group only): the last W-1
  //      inputs, read before any write; this thread is the only reader and writer of these
  //      channels' state
  const bool owner = (blockIdx.x == 0) && tg == 0 && c0 < C;
  float nst[H > 0 ? H : 1][CPT];
  if (owner) {
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const int tau = T_ - H + i;
      if (tau >= 0) ld_word(xb + (size_t)tau * xs + c0, nst[i]);
      else ld_word(csb + (size_t)(H + tau) * C + c0, nst[i]);
    }
  }
  float wt[W][CPT], bi[CPT];
#pragma unroll
  for (int e = 0; e < CPT; ++e) {
    const bool ok = c0 + e < C;
    bi[e] = (bias && ok) ? ld_elem(bias + c0 + e) : 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) wt[j][e] = ok ? ld_elem(w + (size_t)(c0 + e) * W + j) : 0.f;
  }
  __syncthreads();
  const int tb = tg * TG;                               // first token of this group in the tile
  if (c0 < C && tb < nt) {
    // sliding window down this thread's tile column
    const T* col = reinterpret_cast<const T*>(tile) + wi * CPT;
    float win[W][CPT];
#pragma unroll
    for (int i = 0; i < H; ++i) ld_word(col + (tb + i) * CC, win[i]);
    T* yb = y + ((size_t)b * T_ + t0 + tb) * ys + c0;
    const int n = min(TG, nt - tb);
#pragma unroll
    for (int t = 0; t < TG; ++t) {
      if (t < n) {
        ld_word(col + (tb + t + H) * CC, win[H]);
        float out[CPT];
#pragma unroll
        for (int e = 0; e < CPT; ++e) {
          float acc = bi[e];
#pragma unroll
          for (int j = 0; j < W; ++j) acc = fmaf(wt[j][e], win[j][e], acc);
          out[e] = silu ? silu_fast(acc) : acc;
        }
        st_word(yb + (size_t)t * ys, out);
#pragma unroll
        for (int j = 0; j < H; ++j)
#pragma unroll
          for (int e = 0; e < CPT; ++e) win[j][e] = win[j + 1][e];
      }
    }
  }
  if (owner) {
#pragma unroll
    for (int i = 0; i < H; ++i) st_word(csb + (size_t)i * C + c0, nst[i]);
  }
}

template <typename T>
void launch_conv_t(dim3 grid, cudaStream_t stream, int B, int Tn, int C, int W, const T* x,
                   long long xs, const T* w, const T* bias, T* cs, int ns, const int32_t* slots,
                   int silu, T* y, long long ys) {
  switch (W) {
    case 1: gdn_conv_kernel<T, 1><<<grid, CONV_THREADS, 0, stream>>>(B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys); break;
    case 2: gdn_conv_kernel<T, 2><<<grid, CONV_THREADS, 0, stream>>>(B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys); break;
    case 3: gdn_conv_kernel<T, 3><<<grid, CONV_THREADS, 0, stream>>>(B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys); break;
    default: gdn_conv_kernel<T, 4><<<grid, CONV_THREADS, 0, stream>>>(B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys); break;
  }
}

cudaError_t gdn_launch_conv(int B, int T, int C, int W, int bf16, const void* x,
                            long long x_tok_stride, const void* w, const void* bias,
                            void* conv_state, int num_slots, const int32_t* slots, int silu,
                            void* y, long long y_tok_stride, cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  if (W < 1 || W > 4) return cudaErrorInvalidValue;
  const int cc = bf16 ? TILE_BYTES / 2 : TILE_BYTES / 4;
  dim3 grid((unsigned)((T + TT - 1) / TT), (unsigned)((C + cc - 1) / cc), (unsigned)B);
  if (bf16)
    launch_conv_t<__nv_bfloat16>(grid, stream, B, T, C, W, (const __nv_bfloat16*)x, x_tok_stride,
                                 (const __nv_bfloat16*)w, (const __nv_bfloat16*)bias,
                                 (__nv_bfloat16*)conv_state, num_slots, slots, silu,
                                 (__nv_bfloat16*)y, y_tok_stride);
  else
    launch_conv_t<float>(grid, stream, B, T, C, W, (const float*)x, x_tok_stride,
                         (const float*)w, (const float*)bias, (float*)conv_state, num_slots,
                         slots, silu, (float*)y, y_tok_stride);
  return cudaGetLastError();
}
