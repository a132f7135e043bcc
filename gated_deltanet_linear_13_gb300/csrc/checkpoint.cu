// Indexed save / restore of the recurrent state and conv state between live rows and a
// checkpoint-slot bank (PR #164 "Hybrid APC Runtime": checkpoint slots with restore and
// commit masks).  A plain bit copy with 128-bit loads and stores; a negative row or slot
// masks the pair out.
#include "common.cuh"

using namespace gdn;

static __device__ unsigned int g_err_ckpt;

unsigned gdn_take_error_checkpoint() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_ckpt, sizeof(v));
  cudaMemcpyToSymbol(g_err_ckpt, &z, sizeof(z));
  return v;
}

__global__ void __launch_bounds__(256) gdn_checkpoint_kernel(
    int op, long long state_v4, long long conv_v4, float4* state, uint4* conv_state,
    int num_rows, float4* slot_state, uint4* slot_conv, int num_bank, const int32_t* rows,
    const int32_t* slots, int n) {
  // launched with programmatic dependent launch: everything it reads may come from the
  // kernel before it, which has completed once this wait returns
  pdl_wait();
  const int i = blockIdx.y;
  const int row = rows[i], slot = slots[i];
  if (row < 0 || slot < 0) return;                       // masked pair
  if (row >= num_rows || slot >= num_bank) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_err_ckpt, kErrIndex);
    return;
  }
  float4* s_live = state + (size_t)row * state_v4;
  float4* s_bank = slot_state + (size_t)slot * state_v4;
  const float4* __restrict__ src = op == 0 ? s_live : s_bank;
  float4* __restrict__ dst = op == 0 ? s_bank : s_live;
  // one 16-byte element per thread and pass (the grid covers the state in one pass for the
  // usual sizes), every load of a thread issued before its stores
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long e0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long e = e0; e < state_v4; e += 2 * stride) {
    const float4 a = src[e];
    const bool two = e + stride < state_v4;
    const float4 b = two ? src[e + stride] : a;
    dst[e] = a;
    if (two) dst[e + stride] = b;
  }
  if (conv_v4 > 0) {
    uint4* c_live = conv_state + (size_t)row * conv_v4;
    uint4* c_bank = slot_conv + (size_t)slot * conv_v4;
    const uint4* __restrict__ csrc = op == 0 ? c_live : c_bank;
    uint4* __restrict__ cdst = op == 0 ? c_bank : c_live;
    for (long long e = e0; e < conv_v4; e += stride) cdst[e] = csrc[e];
  }
}

cudaError_t gdn_launch_checkpoint(int op, int Hv, int d, int conv_elems, int conv_elem_bytes,
                                  float* state, void* conv_state, int num_rows,
                                  float* slot_state, void* slot_conv_state, int num_bank,
                                  const int32_t* rows, const int32_t* slots, int n,
                                  cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const long long state_v4 = (long long)Hv * d * d / 4;
  const long long conv_v4 = (long long)conv_elems * conv_elem_bytes / 16;
  // one 16-byte element per thread: 4 KB per block (several pairs share the 65535-block limit
  // of grid.x only when a state is above 256 MB)
  long long bxl = (state_v4 + 255) / 256;
  if (bxl > 65535) bxl = 65535;
  int bx = (int)bxl;
  if (bx < 1) bx = 1;
  dim3 grid((unsigned)bx, (unsigned)n, 1);
  return launch_pdl(true, gdn_checkpoint_kernel, grid, dim3(256), 0, stream, op, state_v4,
                    conv_v4, (float4*)state, (uint4*)conv_state, num_rows,
                    (float4*)slot_state, (uint4*)slot_conv_state, num_bank, rows, slots, n);
}

// Conv-state snapshots of a prefill that records its state every `every` tokens: the conv
// state after token t is the W-1 pre-conv inputs t-W+2 .. t, which are rows of the call's own
// input x (every >= 64 > W-1), so each snapshot is a copy of `rows` rows of x.  One CTA per
// (sequence, snapshot); 16-byte elements.
constexpr int SN_ILP = 8;

__global__ void __launch_bounds__(256) gdn_conv_snapshot_kernel(
    const uint8_t* x, long long x_tok_bytes, long long x_seq_bytes, int row_v4, int rows,
    int every, int n_snap, uint4* bank, int num_bank, const int32_t* slots,
    const int32_t* row_slots) {
  // launched behind the prefill's kernels with programmatic dependent launch (x is an input
  // of the call and nothing else in the call touches the bank, so the wait only keeps the
  // copy in the call's order).  The kernel after it (a call continuing the sequence) reads
  // nothing this one writes: it may start at once
  pdl_trigger();
  pdl_wait();
  const long long i = blockIdx.x;                // b * n_snap + j
  const long long bb = i / n_snap, j = i % n_snap;
  const int slot = slots[i];
  if (slot < 0 || (row_slots && row_slots[bb] < 0)) return;   // masked pair, skipped row
  if (slot >= num_bank) {
    if (threadIdx.x == 0) atomicOr(&g_err_ckpt, kErrIndex);
    return;
  }
  const long long t0 = (j + 1) * every - rows;   // first copied token
  const uint8_t* src = x + bb * x_seq_bytes + t0 * x_tok_bytes;
  uint4* dst = bank + (size_t)slot * rows * row_v4;
  // SN_ILP elements per thread and pass, every load before the stores
  const int total = rows * row_v4;
  for (int e0 = threadIdx.x; e0 < total; e0 += SN_ILP * blockDim.x) {
    uint4 v[SN_ILP];
#pragma unroll
    for (int k = 0; k < SN_ILP; ++k) {
      const int e = e0 + k * blockDim.x;
      if (e < total) v[k] = reinterpret_cast<const uint4*>(src + (e / row_v4) * x_tok_bytes)[e % row_v4];
    }
#pragma unroll
    for (int k = 0; k < SN_ILP; ++k) {
      const int e = e0 + k * blockDim.x;
      if (e < total) dst[e] = v[k];
    }
  }
}

cudaError_t gdn_launch_conv_snapshots(int B, int T, int row_bytes, long long x_tok_bytes,
                                      int rows, const void* x, int every, int n_snap,
                                      void* bank, int num_bank, const int32_t* slots,
                                      const int32_t* row_slots, cudaStream_t stream) {
  if (B == 0 || n_snap == 0 || rows <= 0) return cudaSuccess;
  if (row_bytes % 16 != 0 || x_tok_bytes % 16 != 0) return cudaErrorInvalidValue;
  const int row_v4 = row_bytes / 16;
  const long long pairs = (long long)B * n_snap;
  if (pairs > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid((unsigned)pairs, 1, 1);
  return launch_pdl(true, gdn_conv_snapshot_kernel, grid, dim3(256), 0, stream,
                    static_cast<const uint8_t*>(x), x_tok_bytes, x_tok_bytes * T, row_v4, rows,
                    every, n_snap, static_cast<uint4*>(bank), num_bank, slots, row_slots);
}
