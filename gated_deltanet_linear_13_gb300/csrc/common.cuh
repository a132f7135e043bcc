// Internal helpers shared by the kernels of libgdn.so (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gdn.h"

namespace gdn {

constexpr int kHeadDim = 128;
constexpr int kChunk = 64;

// Bits of a translation unit's device error word.
enum : unsigned { kErrIndex = 1u, kErrTimeout = 2u };

// Index checks of the -DGDN_BOUNDS_CHECK build: in_bounds(word, ok) records kErrIndex in the
// translation unit's error word and returns false when a computed global index is out of its
// array (the caller then skips the access); in the normal build it is true and costs nothing.
#ifdef GDN_BOUNDS_CHECK
__device__ __forceinline__ bool in_bounds(unsigned int* word, bool ok) {
  if (!ok) atomicOr(word, kErrIndex);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(unsigned int*, bool) { return true; }
#endif

// ----------------------------------------------------------------- element access

__device__ __forceinline__ float ld_elem(const float* p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ----------------------------------------------------------------- gates

// softplus(x) = max(x, 0) + log(1 + exp(-|x|)), written with the library's log1pf / expf.
__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }
// SiLU for the output gate: z / (1 + e^-z) with the fast exponential and division (for
// z -> -inf the denominator overflows to inf and the quotient is 0).
__device__ __forceinline__ float silu_gate(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Gate of the model card's correctness contract: g = -exp(A_log) * softplus(a + dt_bias).
__device__ __forceinline__ float gate_g(float a, float A_log, float dt_bias) {
  return -expf(A_log) * softplus_f(a + dt_bias);
}

// Sets a kernel's dynamic shared-memory limit once per device (so that launches issued later,
// e.g. under CUDA-graph capture, make no attribute calls).
template <typename K>
inline cudaError_t set_smem_once(K kernel, int bytes, unsigned* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = 1u << (dev & 31);
  if (*done_mask & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) *done_mask |= bit;
  return e;
}

// Same, for the preferred shared-memory carveout (percent of the unified L1 / shared array).
template <typename K>
inline cudaError_t set_carveout_once(K kernel, int percent, unsigned* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = 1u << (dev & 31);
  if (*done_mask & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, percent);
  if (e == cudaSuccess) *done_mask |= bit;
  return e;
}

// ----------------------------------------------------------------- programmatic dependent launch
// A kernel launched with launch_pdl may start while the kernel before it in the stream is
// still running: it does its set-up, then pdl_wait() (every thread) blocks until that kernel
// has completed and its memory writes are visible; nothing it produced, and nothing it may
// still read, is touched before.  pdl_trigger() in the earlier kernel lets the later one be
// scheduled as soon as every CTA of the earlier one has issued it (else at its exit).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// `pdl` false launches normally: the kernel then starts only after all earlier work on the
// stream (e.g. the caller's kernels that produce its inputs) has completed, and its
// pdl_wait() returns at once.  A kernel whose pre-wait set-up reads caller inputs is
// launched that way when it is the first kernel of an API call.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                              size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- warp reductions

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace gdn

// ----------------------------------------------------------------- launchers (gdn_api.cu)

struct GdnLayerArgs {
  // geometry
  int B, T, Hk, Hv, W, C_conv, num_slots;
  // options
  int in_bf16, out_bf16, l2norm, silu, gates_pre;
  float eps, scale;
  // post-conv operands for the recurrence kernels: element pointers + token strides
  const void* q; const void* k; const void* v;
  long long q_tok_stride, k_tok_stride, v_tok_stride;   // elements between tokens
  // raw pre-conv activation (decode / conv)
  const void* x;
  const void* a; const void* b;
  const float* A_log; const float* dt_bias;
  const void* conv_w; const void* conv_b;
  float* state; void* conv_state;
  const int32_t* slots;
  void* out;
  // workspace of the tensor-core prefill (chunk tiles between its two kernels)
  void* scratch;
  size_t scratch_bytes;
  // in-call snapshots (prefill): the state after every snap_every tokens of the call goes to
  // bank row snap_slots[b * n_snap + j]; snap_every == 0 records none
  int snap_every, n_snap, num_snap_slots;
  float* snap_state;
  const int32_t* snap_slots;
  void* snap_conv_state;      // the conv-state bank (the tensor-core prefill with conv width 4
                              // writes it from its chains; other paths launch a copy kernel)
  // gated RMS norm of the output (gate != 0): out = w * o / sqrt(mean(o^2) + eps) * silu(z)
  int gate;
  const void* gate_z;         // [B, T, Hv, d] in the input type
  const float* gate_w;        // [d]
  float gate_eps;
  // packed variable-length batch (cu != nullptr): B sequences on one axis of T tokens,
  // sequence n on [cu[n], cu[n+1]) (validated offsets), global chunks [ccs[n], ccs[n+1]),
  // chunk table ctab[n_chunks] of int4 {first token, tokens, sequence, 0}
  const int32_t* cu;
  const int32_t* ccs;
  const void* ctab;
  int n_chunks;
  // the conv of the value channels [2 Hk d, C_conv) is still to be launched (tensor-core
  // prefill): the prefill launches it after its first chunk-local kernel, beside which it runs
  int vconv_pending;
  // the tensor-core prefill with conv width 4 (bf16, not a packed batch): the conv of the q
  // and k channels fused into the chunk-local kernel, that of the v channels (into `v`) the
  // call's first launch; the call's conv tail (its last W-1 inputs, [B][W-1][C_conv]) goes to
  // `tail` and from there, by the last state-chain kernel, into conv_state
  int fuse;
  void* tail;
  // the call continues the sequences of the call before it on the stream: the inputs before
  // its first token come from that call's conv tail `prev_tail` (not from conv_state), and its
  // first kernel may start while that call's last kernels still run
  int chained;
  const void* prev_tail;
};

// Workspace bytes the tensor-core prefill needs for B sequences of T tokens, Hv value heads.
size_t gdn_prefill_tc_scratch_bytes(int B, int T, int Hv);

cudaError_t gdn_launch_decode(const GdnLayerArgs& args, cudaStream_t stream);
// A decode step over args.T <= 16 tokens per sequence; with snap_slots ([B][T]) the state and
// conv state after every token go to those bank rows.
cudaError_t gdn_launch_decode_multi(const GdnLayerArgs& args, float* snap_state, int num_snap,
                                    const int32_t* snap_slots, void* snap_conv,
                                    cudaStream_t stream);
cudaError_t gdn_launch_prefill_simt(const GdnLayerArgs& args, cudaStream_t stream);
cudaError_t gdn_launch_prefill_tc(const GdnLayerArgs& args, cudaStream_t stream);
// The bounded-wait self-test (one CTA, an mbarrier nothing arrives at, max_iters polls).
cudaError_t gdn_launch_selftest_wait(uint32_t max_iters, cudaStream_t stream);
// 3-D tensor map over [B][T][width] elements starting at `base`, token stride `tok_stride`
// elements; box = {box0, box1 tokens, 1 sequence}; 128-byte swizzle or none.
bool gdn_make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
                  int width, int T, int B, long long tok_stride, int box0, int box1,
                  bool swizzle128);

// Channels [c_lo, c_hi) only (c_lo a multiple of the 512-byte channel tile; c_hi < 0: to C).
// pdl: launched with programmatic dependent launch; late_wait: the grid's last block waits at
// its end for the kernel before it, so that the grid completes only after that kernel (a
// launch that runs beside a kernel it does not depend on).  halo: the W-1 inputs before the
// first token come from rows [slot (halo_by_slot) or b][W-1][C] of halo instead of the conv
// state, and the new state goes to rows [b][W-1][C] of tail instead (the conv state is left
// alone).  Channel c is stored at column c - y_cbase of y.
cudaError_t gdn_launch_conv(int B, int T, int C, int W, int bf16, const void* x,
                            long long x_tok_stride, const void* w, const void* bias,
                            void* conv_state, int num_slots, const int32_t* slots, int silu,
                            void* y, long long y_tok_stride, cudaStream_t stream, int c_lo = 0,
                            int c_hi = -1, bool pdl = false, bool late_wait = false,
                            const void* halo = nullptr, int halo_by_slot = 1,
                            void* tail = nullptr, int y_cbase = 0);
// Conv-state snapshots of an in-call snapshot prefill: snapshot j of row b is the W-1
// pre-conv rows of x ending at token (j + 1) * every, copied to bank row slots[b * n_snap + j]
// (nothing for a row whose row_slots entry is negative; row_slots may be NULL).
cudaError_t gdn_launch_conv_snapshots(int B, int T, int row_bytes, long long x_tok_bytes,
                                      int rows, const void* x, int every, int n_snap,
                                      void* bank, int num_bank, const int32_t* slots,
                                      const int32_t* row_slots, cudaStream_t stream);
// Packed variable-length batches: validate the offsets and lay out the chunk table (above).
cudaError_t gdn_launch_varlen_prep(const int32_t* cu, int N, int T, int U, int32_t* cu_ok,
                                   int32_t* ccs, void* ctab, cudaStream_t stream);
// Conv of a packed batch (x, y: [T][C] with token strides), sequence n on [cu[n], cu[n+1]),
// then its new conv states.
cudaError_t gdn_launch_conv_varlen(int N, int T, int C, int W, int bf16, const int32_t* cu,
                                   const void* x, long long x_tok_stride, const void* w,
                                   const void* bias, void* conv_state, int num_slots,
                                   const int32_t* slots, int silu, void* y,
                                   long long y_tok_stride, cudaStream_t stream);
cudaError_t gdn_launch_checkpoint(int op, int Hv, int d, int conv_elems, int conv_elem_bytes,
                                  float* state, void* conv_state, int num_rows,
                                  float* slot_state, void* slot_conv_state, int num_bank,
                                  const int32_t* rows, const int32_t* slots, int n,
                                  cudaStream_t stream);

// The gated RMS norm as a pass of its own over out [B][T][Hv][d] (in place, fp32), for the
// FMA-pipe prefill; z [B][T][Hv][d] in fp32; rows of batch entries that `slots` skips are
// left alone.
cudaError_t gdn_launch_gated_norm_f32(float* out, const float* z, const float* w, float eps,
                                      int B, long long rows_per_seq, const int32_t* slots,
                                      int num_slots, cudaStream_t stream,
                                      const int32_t* cu = nullptr, int Hv = 0);

// Per-translation-unit device error words: read and clear (host side, synchronous copy).
unsigned gdn_take_error_decode();
unsigned gdn_take_error_conv();
unsigned gdn_take_error_checkpoint();
unsigned gdn_take_error_prefill_simt();
unsigned gdn_take_error_prefill_tc();
unsigned gdn_take_error_varlen();
unsigned gdn_take_error_decode_multi();
