// Causal depthwise conv1d with a carried conv state (the short conv in front of the gated
// delta rule; model card "Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron", "How It Works"
// and "Notice" on conv-state caching).
//
//   y[b,t,c] = bias[c] + sum_{j<W} w[c][j] * x[b, t-W+1+j, c]   (then SiLU if requested)
// positions before t = 0 read the conv state (the last W-1 pre-conv inputs, oldest first);
// afterwards the state holds the last W-1 inputs of this call.
//
// A CTA owns a tile of 64 tokens x 512 bytes of channels of one sequence: one TMA copy
// brings the tile plus the W-1 rows before it into shared memory (rows before the sequence
// start are then taken from the conv state), and each thread slides the window down 16
// tokens of one 8-byte column (256 threads, three CTAs per SM, so that a 512-token call's
// tiles run in one wave).  The thread holding a sequence's first tokens of a column is
// the only one that reads the old state of its channels, and it also writes the new state
// (taken from x, which nobody modifies), so no two threads race on it.
#include "common.cuh"
#include "conv_math.cuh"
#include "sm100_ptx.cuh"

using namespace gdn;
using namespace gdn::ptx;

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
constexpr int WORDS = TILE_BYTES / 8;                 // 8-byte words per row
constexpr int CONV_THREADS = WORDS * (TT / TG);       // a thread: one word x TG tokens
constexpr int MAX_HALO = 3;
constexpr int TILE_ROWS = TT + MAX_HALO;

// one 8-byte word of a row: four bf16 channels or two fp32 channels
__device__ __forceinline__ void ld_word(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = c.x; v[3] = c.y;
}
__device__ __forceinline__ void ld_word(const float* p, float (&v)[2]) {
  const float2 f = *reinterpret_cast<const float2*>(p);
  v[0] = f.x; v[1] = f.y;
}
__device__ __forceinline__ void st_word(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 u;
  *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(v[0], v[1]);
  *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void st_word(float* p, const float (&v)[2]) {
  *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}


// Where the inputs before the call's first token come from, and where the new conv state
// goes: halo == nullptr: the conv state rows of slot slots[b] (read, then overwritten);
// else rows [b or slot][W-1][C] of `halo` (halo_by_slot picks the index), and the new state
// goes to rows [b][W-1][C] of `tail` (the conv state is not touched).
template <typename T>
struct ConvEnds {
  const T* halo;
  int halo_by_slot;
  T* tail;
};

template <typename T, int W>
__device__ __forceinline__ void conv_tile(const CUtensorMap& tm_x, int B, int T_, int C,
                                          const T* x, long long xs, const T* w, const T* bias,
                                          T* cs, int num_slots, const int32_t* slots, int silu,
                                          T* y, long long ys, int c_base, int y_cbase,
                                          const ConvEnds<T>& ends);

template <typename T, int W>
__global__ void __launch_bounds__(CONV_THREADS, 3) gdn_conv_kernel(
    const __grid_constant__ CUtensorMap tm_x, int B, int T_, int C, const T* x, long long xs,
    const T* w, const T* bias, T* cs, int num_slots, const int32_t* slots, int silu, T* y,
    long long ys, int c_base, int late_wait, int y_cbase, const ConvEnds<T> ends) {
  conv_tile<T, W>(tm_x, B, T_, C, x, xs, w, bias, cs, num_slots, slots, silu, y, ys, c_base,
                  y_cbase, ends);
  // a launch that runs beside the kernel before it (which it does not depend on) completes
  // only after that kernel has: its last block waits for it, so that the kernel after this
  // one, which waits for this grid, may rely on both
  if (late_wait && blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 &&
      blockIdx.z == gridDim.z - 1)
    pdl_wait();
}

template <typename T, int W>
__device__ __forceinline__ void conv_tile(const CUtensorMap& tm_x, int B, int T_, int C,
                                          const T* x, long long xs, const T* w, const T* bias,
                                          T* cs, int num_slots, const int32_t* slots, int silu,
                                          T* y, long long ys, int c_base, int y_cbase,
                                          const ConvEnds<T>& ends) {
  constexpr int CC = TILE_BYTES / (int)sizeof(T);       // channels per tile
  constexpr int CPT = 8 / (int)sizeof(T);               // channels per thread (4 or 2)
  constexpr int H = W - 1;                              // halo rows
  __shared__ __align__(128) uint8_t tile[TILE_ROWS * TILE_BYTES];
  __shared__ uint64_t bar;
  const int t0 = blockIdx.x * TT, cb = c_base + blockIdx.y * CC, b = blockIdx.z;
  const int tid = threadIdx.x;
  pdl_trigger();              // the kernel that consumes y may start its set-up
  const int slot = slots ? slots[b] : b;
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_err_conv, kErrIndex);
    return;
  }
  const T* xb = x + (size_t)b * T_ * xs;
  T* csb = cs + (size_t)slot * H * C;
  if (!in_bounds(&g_err_conv, b < B && t0 < T_)) return;
  const T* oldb = ends.halo ? ends.halo + (size_t)(ends.halo_by_slot ? slot : b) * H * C : csb;
  T* newb = ends.tail ? ends.tail + (size_t)b * H * C : csb;
  const int nt = min(TT, T_ - t0);
  // ---- tile row r = the input of token t0 - H + r (the copy fills rows outside the
  //      sequence with zeros; rows before its start are replaced by the conv state below)
  const uint32_t bar_a = smem_addr(&bar);
  if (tid == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_a, (uint32_t)((TT + H) * TILE_BYTES));
    tma_load_3d(smem_addr(tile), &tm_x, cb, t0 - H, b, bar_a);
  }
  const int wi = tid % WORDS, tg = tid / WORDS;
  const int c0 = cb + wi * CPT;
  // ---- the new conv state (first token tile, first token group only): the last W-1
  //      inputs, read before any write; this thread is the only reader and writer of these
  //      channels' state
  const bool owner = (blockIdx.x == 0) && tg == 0 && c0 < C;
  float nst[H > 0 ? H : 1][CPT];
  float old[H > 0 ? H : 1][CPT];
  if (owner) {
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const int tau = T_ - H + i;
      ld_word(oldb + (size_t)i * C + c0, old[i]);
      if (tau >= 0) ld_word(xb + (size_t)tau * xs + c0, nst[i]);
    }
    // a sequence shorter than W-1 keeps part of the old state (position H + tau)
#pragma unroll
    for (int i = 0; i < H; ++i)
#pragma unroll
      for (int j = 0; j < H; ++j)
        if (j == T_ + i) {
#pragma unroll
          for (int e = 0; e < CPT; ++e) nst[i][e] = old[j][e];
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
  __syncthreads();                                      // barrier initialised
  const bool arrived = mbar_wait_bounded(bar_a, 0);
  if (owner && H > 0 && arrived) {
    // rows 0 .. H-1 of the first tile are the positions before the sequence start
    T* row0 = reinterpret_cast<T*>(tile) + wi * CPT;
#pragma unroll
    for (int i = 0; i < H; ++i) st_word(row0 + i * CC, old[i]);
  }
  if (!__syncthreads_and(arrived)) {
    if (tid == 0) atomicOr(&g_err_conv, kErrTimeout);
    return;
  }
  const int tb = tg * TG;                               // first token of this group in the tile
  if (c0 < C && tb < nt) {
    // sliding window down this thread's tile column
    const T* col = reinterpret_cast<const T*>(tile) + wi * CPT;
    float win[W][CPT];
#pragma unroll
    for (int i = 0; i < H; ++i) ld_word(col + (tb + i) * CC, win[i]);
    T* yp = y + ((size_t)b * T_ + t0 + tb) * ys + (c0 - y_cbase);
    if (!in_bounds(&g_err_conv, b < B && t0 + tb + min(TG, nt - tb) <= T_ && c0 >= y_cbase))
      return;
    const int n = min(TG, nt - tb);
#pragma unroll
    for (int t = 0; t < TG; ++t) {
      if (t < n) {
        ld_word(col + (tb + t + H) * CC, win[H]);
        float out[CPT];
        conv_token<W, CPT>(wt, bi, win, silu, out);
        st_word(yp, out);
        yp += ys;
#pragma unroll
        for (int j = 0; j < H; ++j)
#pragma unroll
          for (int e = 0; e < CPT; ++e) win[j][e] = win[j + 1][e];
      }
    }
  }
  if (owner) {
#pragma unroll
    for (int i = 0; i < H; ++i) st_word(newb + (size_t)i * C + c0, nst[i]);
  }
}

template <typename T, int W>
cudaError_t launch_conv_w(dim3 grid, cudaStream_t stream, const CUtensorMap& m, int B, int Tn,
                          int C, const T* x, long long xs, const T* w, const T* bias, T* cs,
                          int ns, const int32_t* slots, int silu, T* y, long long ys, int c_base,
                          bool pdl, bool late_wait, int y_cbase, const ConvEnds<T>& ends) {
  static unsigned done = 0u;       // room for several tiles per SM
  cudaError_t e = set_carveout_once(gdn_conv_kernel<T, W>, 100, &done);
  if (e != cudaSuccess) return e;
  return launch_pdl(pdl, gdn_conv_kernel<T, W>, grid, dim3(CONV_THREADS), 0, stream, m, B, Tn, C,
                    x, xs, w, bias, cs, ns, slots, silu, y, ys, c_base, late_wait ? 1 : 0,
                    y_cbase, ends);
}

template <typename T>
cudaError_t launch_conv_t(dim3 grid, cudaStream_t stream, const CUtensorMap& m, int B, int Tn,
                          int C, int W, const T* x, long long xs, const T* w, const T* bias,
                          T* cs, int ns, const int32_t* slots, int silu, T* y, long long ys,
                          int c_base, bool pdl, bool late_wait, int y_cbase,
                          const ConvEnds<T>& ends) {
  switch (W) {
    case 1: return launch_conv_w<T, 1>(grid, stream, m, B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys, c_base, pdl, late_wait, y_cbase, ends);
    case 2: return launch_conv_w<T, 2>(grid, stream, m, B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys, c_base, pdl, late_wait, y_cbase, ends);
    case 3: return launch_conv_w<T, 3>(grid, stream, m, B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys, c_base, pdl, late_wait, y_cbase, ends);
    default: return launch_conv_w<T, 4>(grid, stream, m, B, Tn, C, x, xs, w, bias, cs, ns, slots, silu, y, ys, c_base, pdl, late_wait, y_cbase, ends);
  }
}

cudaError_t gdn_launch_conv(int B, int T, int C, int W, int bf16, const void* x,
                            long long x_tok_stride, const void* w, const void* bias,
                            void* conv_state, int num_slots, const int32_t* slots, int silu,
                            void* y, long long y_tok_stride, cudaStream_t stream, int c_lo,
                            int c_hi, bool pdl, bool late_wait, const void* halo,
                            int halo_by_slot, void* tail, int y_cbase) {
  if (B == 0 || T == 0) return cudaSuccess;
  if (W < 1 || W > 4) return cudaErrorInvalidValue;
  const int eb = bf16 ? 2 : 4, cc = TILE_BYTES / eb;
  if (c_hi < 0) c_hi = C;
  if (c_lo < 0 || c_lo % cc != 0 || c_hi > C || c_lo >= c_hi) return cudaErrorInvalidValue;
  CUtensorMap m;
  if (!gdn_make_map(&m, x, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    eb, C, T, B, x_tok_stride, cc, TT + W - 1, false))
    return cudaErrorInvalidValue;
  dim3 grid((unsigned)((T + TT - 1) / TT), (unsigned)((c_hi - c_lo + cc - 1) / cc), (unsigned)B);
  if (bf16)
    return launch_conv_t<__nv_bfloat16>(
        grid, stream, m, B, T, C, W, (const __nv_bfloat16*)x, x_tok_stride,
        (const __nv_bfloat16*)w, (const __nv_bfloat16*)bias, (__nv_bfloat16*)conv_state,
        num_slots, slots, silu, (__nv_bfloat16*)y, y_tok_stride, c_lo, pdl, late_wait, y_cbase,
        ConvEnds<__nv_bfloat16>{(const __nv_bfloat16*)halo, halo_by_slot,
                                (__nv_bfloat16*)tail});
  return launch_conv_t<float>(grid, stream, m, B, T, C, W, (const float*)x, x_tok_stride,
                              (const float*)w, (const float*)bias, (float*)conv_state, num_slots,
                              slots, silu, (float*)y, y_tok_stride, c_lo, pdl, late_wait, y_cbase,
                              ConvEnds<float>{(const float*)halo, halo_by_slot, (float*)tail});
}

// ======================================================================= packed sequences
// Variable-length batches: N sequences packed back to back in x [T_total][C], sequence n on
// tokens [cu[n], cu[n+1]) (cu validated by the prep kernel), each with its own conv-state
// row.  The tile and the sliding window are those above; a thread finds the sequence of its
// first token by bisection and, when its window crosses into the next sequence, restarts the
// window from that sequence's old conv state.  The per-token arithmetic is the same as above,
// so each sequence's outputs equal those of a call of its own, bit for bit.  The new conv
// states are written by the kernel after this one (every old state is read here first).

template <typename T, int H>
__device__ __forceinline__ void conv_state_word(const T* cs, int C, int num_slots,
                                                const int32_t* slots, int n, int idx, int c0,
                                                float (&v)[8 / sizeof(T)]) {
  const int slot = slots ? slots[n] : n;
  if (slot < 0 || slot >= num_slots) {
#pragma unroll
    for (int e = 0; e < (int)(8 / sizeof(T)); ++e) v[e] = 0.f;
    return;
  }
  ld_word(cs + ((size_t)slot * H + idx) * C + c0, v);
}

template <typename T, int W>
__global__ void __launch_bounds__(CONV_THREADS, 3) gdn_conv_varlen_kernel(
    const __grid_constant__ CUtensorMap tm_x, int N, int T_, int C, const int32_t* cu,
    const T* w, const T* bias, const T* cs, int num_slots, const int32_t* slots, int silu,
    T* y, long long ys) {
  constexpr int CC = TILE_BYTES / (int)sizeof(T);
  constexpr int CPT = 8 / (int)sizeof(T);
  constexpr int H = W - 1;
  __shared__ __align__(128) uint8_t tile[TILE_ROWS * TILE_BYTES];
  __shared__ uint64_t bar;
  const int t0 = blockIdx.x * TT, cb = blockIdx.y * CC;
  const int tid = threadIdx.x;
  pdl_trigger();
  const int nt = min(TT, T_ - t0);
  const uint32_t bar_a = smem_addr(&bar);
  if (tid == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_a, (uint32_t)((TT + H) * TILE_BYTES));
    tma_load_3d(smem_addr(tile), &tm_x, cb, t0 - H, 0, bar_a);
  }
  const int wi = tid % WORDS, tg = tid / WORDS;
  const int c0 = cb + wi * CPT;
  float wt[W][CPT], bi[CPT];
#pragma unroll
  for (int e = 0; e < CPT; ++e) {
    const bool ok = c0 + e < C;
    bi[e] = (bias && ok) ? ld_elem(bias + c0 + e) : 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) wt[j][e] = ok ? ld_elem(w + (size_t)(c0 + e) * W + j) : 0.f;
  }
  __syncthreads();
  if (!__syncthreads_and(mbar_wait_bounded(bar_a, 0))) {
    if (tid == 0) atomicOr(&g_err_conv, kErrTimeout);
    return;
  }
  const int tb = tg * TG;
  const int tfirst = t0 + tb;
  if (c0 >= C || tb >= nt || tfirst >= cu[N]) return;
  // the sequence holding tfirst: cu[lo] <= tfirst < cu[lo + 1]
  int lo = 0, hi = N;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= tfirst) lo = mid; else hi = mid;
  }
  int n = lo, s0 = cu[n], s1 = cu[n + 1];
  const T* col = reinterpret_cast<const T*>(tile) + wi * CPT;
  float win[W][CPT];
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const int pos = tfirst - H + i;
    if (pos >= s0) ld_word(col + (tb + i) * CC, win[i]);
    else conv_state_word<T, H>(cs, C, num_slots, slots, n, pos - s0 + H, c0, win[i]);
  }
  T* yp = y + (size_t)tfirst * ys + c0;
  const int cnt = min(TG, nt - tb);
#pragma unroll
  for (int t = 0; t < TG; ++t) {
    if (t < cnt) {
      const int tt = tfirst + t;
      if (tt >= s1) {
        // the next non-empty sequence starts at tt: its window history is its conv state
        while (tt >= s1 && n < N - 1) {
          ++n;
          s0 = s1;
          s1 = cu[n + 1];
        }
#pragma unroll
        for (int i = 0; i < H; ++i) conv_state_word<T, H>(cs, C, num_slots, slots, n, i, c0, win[i]);
      }
      ld_word(col + (tb + t + H) * CC, win[H]);
      float out[CPT];
      conv_token<W, CPT>(wt, bi, win, silu, out);
      st_word(yp, out);
      yp += ys;
#pragma unroll
      for (int j = 0; j < H; ++j)
#pragma unroll
        for (int e = 0; e < CPT; ++e) win[j][e] = win[j + 1][e];
    }
  }
}

// New conv state of each packed sequence: its last W-1 inputs, the older ones from its old
// state when it is shorter than W-1.  CTA (sequence, block of words); a thread owns a word.
template <typename T, int W>
__global__ void __launch_bounds__(256) gdn_conv_state_varlen_kernel(
    int N, int C, const int32_t* cu, const T* x, long long xs, T* cs, int num_slots,
    const int32_t* slots) {
  constexpr int CPT = 8 / (int)sizeof(T);
  constexpr int H = W - 1;
  pdl_wait();
  const int n = blockIdx.x;
  const int slot = slots ? slots[n] : n;
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_err_conv, kErrIndex);
    return;
  }
  const int s0 = cu[n], s1 = cu[n + 1];
  T* csn = cs + (size_t)slot * H * C;
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * CPT;
  if (c0 < C) {
    float old[H > 0 ? H : 1][CPT], nst[H > 0 ? H : 1][CPT];
#pragma unroll
    for (int i = 0; i < H; ++i) ld_word(csn + (size_t)i * C + c0, old[i]);
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const int pos = s1 - H + i;
      if (pos >= s0) {
        ld_word(x + (size_t)pos * xs + c0, nst[i]);
      } else {
#pragma unroll
        for (int j = 0; j < H; ++j)
          if (j == pos - s0 + H) {
#pragma unroll
            for (int e = 0; e < CPT; ++e) nst[i][e] = old[j][e];
          }
      }
    }
#pragma unroll
    for (int i = 0; i < H; ++i) st_word(csn + (size_t)i * C + c0, nst[i]);
  }
}

template <typename T, int W>
static cudaError_t launch_conv_varlen_w(const CUtensorMap& m, int N, int Tn, int C,
                                        const int32_t* cu, const T* x, long long xs, const T* w,
                                        const T* bias, T* cs, int ns, const int32_t* slots,
                                        int silu, T* y, long long ys, cudaStream_t stream) {
  static unsigned done = 0;
  cudaError_t e = set_carveout_once(gdn_conv_varlen_kernel<T, W>, 100, &done);
  if (e != cudaSuccess) return e;
  constexpr int cc = TILE_BYTES / (int)sizeof(T);
  dim3 grid((unsigned)((Tn + TT - 1) / TT), (unsigned)((C + cc - 1) / cc), 1);
  gdn_conv_varlen_kernel<T, W><<<grid, CONV_THREADS, 0, stream>>>(m, N, Tn, C, cu, w, bias, cs,
                                                                   ns, slots, silu, y, ys);
  e = cudaGetLastError();
  if (e != cudaSuccess || W < 2) return e;
  constexpr int cpt = 8 / (int)sizeof(T);
  const unsigned wblocks = (unsigned)((C + 256 * cpt - 1) / (256 * cpt));
  return launch_pdl(true, gdn_conv_state_varlen_kernel<T, W>, dim3((unsigned)N, wblocks),
                    dim3(256), 0, stream, N, C, cu, x, xs, cs, ns, slots);
}

template <typename T>
static cudaError_t launch_conv_varlen_t(const CUtensorMap& m, int N, int Tn, int C, int W,
                                        const int32_t* cu, const T* x, long long xs, const T* w,
                                        const T* bias, T* cs, int ns, const int32_t* slots,
                                        int silu, T* y, long long ys, cudaStream_t stream) {
  switch (W) {
    case 1: return launch_conv_varlen_w<T, 1>(m, N, Tn, C, cu, x, xs, w, bias, cs, ns, slots, silu, y, ys, stream);
    case 2: return launch_conv_varlen_w<T, 2>(m, N, Tn, C, cu, x, xs, w, bias, cs, ns, slots, silu, y, ys, stream);
    case 3: return launch_conv_varlen_w<T, 3>(m, N, Tn, C, cu, x, xs, w, bias, cs, ns, slots, silu, y, ys, stream);
    default: return launch_conv_varlen_w<T, 4>(m, N, Tn, C, cu, x, xs, w, bias, cs, ns, slots, silu, y, ys, stream);
  }
}

cudaError_t gdn_launch_conv_varlen(int N, int T, int C, int W, int bf16, const int32_t* cu,
                                   const void* x, long long x_tok_stride, const void* w,
                                   const void* bias, void* conv_state, int num_slots,
                                   const int32_t* slots, int silu, void* y,
                                   long long y_tok_stride, cudaStream_t stream) {
  if (N == 0 || T == 0) return cudaSuccess;
  if (W < 1 || W > 4) return cudaErrorInvalidValue;
  const int eb = bf16 ? 2 : 4, cc = TILE_BYTES / eb;
  CUtensorMap m;
  if (!gdn_make_map(&m, x, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    eb, C, T, 1, x_tok_stride, cc, TT + W - 1, false))
    return cudaErrorInvalidValue;
  if (bf16)
    return launch_conv_varlen_t<__nv_bfloat16>(
        m, N, T, C, W, cu, (const __nv_bfloat16*)x, x_tok_stride, (const __nv_bfloat16*)w,
        (const __nv_bfloat16*)bias, (__nv_bfloat16*)conv_state, num_slots, slots, silu,
        (__nv_bfloat16*)y, y_tok_stride, stream);
  return launch_conv_varlen_t<float>(m, N, T, C, W, cu, (const float*)x, x_tok_stride,
                                     (const float*)w, (const float*)bias, (float*)conv_state,
                                     num_slots, slots, silu, (float*)y, y_tok_stride, stream);
}
