// Variable-length batches: N sequences packed back to back on one token axis, sequence n on
// tokens [cu[n], cu[n+1]).  Every sequence is its own recurrence with its own state row and
// its own chunk grid (chunks never cross a sequence boundary), so a packed call equals one
// call per sequence.
//
// The prep kernel checks the offsets on the device (cu[0] = 0, non-decreasing, cu[N] = the
// packed length) and lays out the per-chunk work for the prefill kernels:
//   cu_ok[N+1]   the offsets, or all zeros (no work at all) when they are not valid;
//   ccs[N+1]     chunk offsets: sequence n owns global chunks [ccs[n], ccs[n+1]);
//   ctab[U]      per global chunk u: {first token, tokens (1..64), sequence, 0};
//                entries past the last chunk have 0 tokens.
// U = ceil(T / 64) + N bounds the chunk count on the host, which never reads the offsets.
#include "common.cuh"

using namespace gdn;

static __device__ unsigned int g_err_varlen;

unsigned gdn_take_error_varlen() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_varlen, sizeof(v));
  cudaMemcpyToSymbol(g_err_varlen, &z, sizeof(z));
  return v;
}

constexpr int PREP_THREADS = 1024;

__global__ void __launch_bounds__(PREP_THREADS) gdn_varlen_prep_kernel(
    const int32_t* cu, int N, int T, int U, int32_t* cu_ok, int32_t* ccs, int4* ctab) {
  __shared__ int warp_tot[PREP_THREADS / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // ---- validity
  bool ok = true;
  for (int i = tid; i <= N; i += PREP_THREADS) {
    const int c = cu[i];
    if (i == 0 && c != 0) ok = false;
    if (i == N && c != T) ok = false;
    if (i > 0 && c < cu[i - 1]) ok = false;
  }
  ok = __syncthreads_and(ok);
  if (!ok && tid == 0) atomicOr(&g_err_varlen, kErrIndex);
  // ---- offsets and chunk offsets (a block-wide exclusive scan of ceil(len / 64), tile by tile)
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base <= N; base += PREP_THREADS) {
    const int i = base + tid;
    int nc = 0;
    if (ok && i < N) nc = (cu[i + 1] - cu[i] + kChunk - 1) / kChunk;
    int incl = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;                        // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - nc;
    if (i <= N) {
      ccs[i] = before;
      cu_ok[i] = ok ? cu[i] : 0;
    }
    __syncthreads();
    if (tid == PREP_THREADS - 1) carry = before + nc;
    __syncthreads();
  }
  // ---- the chunk table, one entry per thread: the sequence of chunk u by bisection on ccs
  const int used = ccs[N];
  for (int u = tid; u < U; u += PREP_THREADS) {
    int4 e = make_int4(0, 0, 0, 0);
    if (u < used) {
      int lo = 0, hi = N;                        // ccs[lo] <= u < ccs[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ccs[mid] <= u) lo = mid; else hi = mid;
      }
      const int c = u - ccs[lo], s0 = cu[lo] + c * kChunk;
      e = make_int4(s0, min(kChunk, cu[lo + 1] - s0), lo, 0);
    }
    ctab[u] = e;
  }
}

cudaError_t gdn_launch_varlen_prep(const int32_t* cu, int N, int T, int U, int32_t* cu_ok,
                                   int32_t* ccs, void* ctab, cudaStream_t stream) {
  gdn_varlen_prep_kernel<<<1, PREP_THREADS, 0, stream>>>(cu, N, T, U, cu_ok, ccs,
                                                         static_cast<int4*>(ctab));
  return cudaGetLastError();
}
