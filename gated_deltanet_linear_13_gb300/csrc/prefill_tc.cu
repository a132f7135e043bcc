// Chunked gated-delta-rule prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Method: the chunked WY/UT form with a direct triangular solve (PR #164 "Fused DeltaNet
// Direct-Solve Follow-Up"), which unrolls the per-token recurrence of the model card
// "Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron" ("How It Works").  Per chunk of C = 64
// tokens with entering state S0 [v][k] (fp32) and in-chunk cumulative log-decay G_r:
//   A[r][s] = beta_r e^{G_r-G_s} (k^_r . k^_s), s < r        T = (I + A)^{-1}
//   W  = T diag(beta e^G) K^,     U' = T diag(beta) V,     U = U' - W S0^T
//   P[r][s] = e^{G_r-G_s} (q^_r . k^_s), s <= r
//   O  = diag(e^G) Q^ S0^T + P U,     S = e^{G_C} S0 + U^T diag(e^{G_C-G}) K^
// Normalisation and every diagonal factor are folded into small matrices or into row
// scalings of the raw tiles, so the tensor cores see raw bf16 q/k/v:
//   G = [K;Q][K;Q]^T (one M=N=128 MMA)  ->  A, P (with 1/||k||, scale/||q||, decays); the
//   squared norms are G's diagonal
//   T' = T diag(beta e^G / ||k||),  T'' = T diag(beta)      (the solve, fp32 FMA)
//   W^T = K^T T'^T,  U'^T = V^T T''^T                          (M = d = 128)
//   Q~ = diag(scale e^G / ||q||) Q,  K~ = diag(e^{G_C-G} / ||k||) K
//   U^T = U'^T - S0 W^T,  O^T = S0 Q~^T + U^T P^T,  S = e^{G_C} S0 + U^T K~
// T', T'', P and U^T enter the tensor cores as bf16 pairs hi + lo (hi = rn(x), lo = rn(x-hi)),
// which keeps ~16 mantissa bits in the small intra-chunk products; the state snapshot S0,
// W, Q~ and K~ are single bf16 (their rounding costs far less at the output).
// Everything is computed transposed so that the MMA M dimension (128 TMEM lanes) is the
// head dimension: state row i lives in TMEM lane i for the whole sequence.
//
// Two kernels per slice of chunks:
//   * gdn_chunk_local_kernel, one CTA per (chunk, value head, sequence), three CTAs per SM:
//     everything that does not depend on the state (gates, norms, G, A, P, the direct solve,
//     T', T'', W, Q~, K~).  Its results for the chain are five 16 KB tiles per chunk, already
//     in the swizzled layouts the chain's MMAs read, written with bulk copies to a workspace
//     slice small enough to stay in L2, plus e^{G_C}.
//   * gdn_chunk_chain_kernel, one CTA per (value head, sequence): the state chain only, with
//     eight epilogue warps, one MMA / copy issuer warp and four store warps.  Per chunk: U'^T
//     (MMA), S0 = bf16(S) into TMEM, S <- e^{G_C} S, U^T += S0 (-W)^T, O^T = S0 Q~^T, U^T ->
//     bf16 hi/lo in TMEM, S += U^T K~, O^T += U^T P^T; the next chunk's tiles stream in
//     meanwhile, the store warps send the previous chunk's output (optionally through the
//     gated RMS norm) by TMA, and the epilogue warps send the leaving state (and any in-call
//     snapshot).  A packed variable-length batch runs the same kernels on one token axis
//     with a per-chunk table (each sequence keeps its own chunk grid).
// Both kernels are launched with programmatic dependent launch (set-up overlaps the tail of
// the kernel before).  In a call of several slices the workspace is double-buffered and the
// local kernel of slice i+1 runs beside the chain of slice i: the chain releases its
// dependents right after its own grid wait, and the local kernel's last block waits for that
// chain before it exits, so that the grid (whose completion starts the next chain) cannot
// complete first.  No kernel spins on another's data.  The fp32 state stays in TMEM for a
// whole slice.  Every mbarrier wait is bounded: on timeout the CTA records
// GDN_ERR_DEVICE_TIMEOUT, waits (bounded) for its own copies and MMAs, frees TMEM and
// returns.
#include "common.cuh"
#include "conv_math.cuh"
#include "sm100_ptx.cuh"

using namespace gdn;
using namespace gdn::ptx;

static __device__ unsigned int g_err_tc;

unsigned gdn_take_error_prefill_tc() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(v));
  cudaMemcpyToSymbol(g_err_tc, &z, sizeof(z));
  return v;
}

namespace {

constexpr int C = kChunk, D = kHeadDim;
constexpr uint32_t KB = 1024;
// Row stride (floats) of the fp32 solve matrices: 64 + 4 pad, so that the rows a warp's lanes
// own start 16 bytes apart in the bank space (no conflicts when each lane writes its row).
constexpr int LA = 68;
constexpr uint32_t SOLVE_MAT = 64 * LA * 4;           // bytes of one solve matrix
constexpr int LGT = 256;                              // threads of the local kernel (barrier 1)

// ---- one chunk's tiles for the chain (bytes within a 80 KB unit of the workspace)
constexpr uint32_t U_NW = 0;          // -W^T   [128 rows d_k][128 B = 64 tokens], MN-major B
constexpr uint32_t U_QT = 16 * KB;    // Q~     [2 blocks of 64 d_k][64 rows r][128 B], K-major B
constexpr uint32_t U_P = 32 * KB;     // P hi | P lo  [64 rows r][128 B = 64 s], K-major B
constexpr uint32_t U_KT = 48 * KB;    // K~     [2 blocks of 64 d_k][64 rows s][128 B], MN-major B
constexpr uint32_t U_T2 = 64 * KB;    // T'' hi | T'' lo [64 rows r][128 B = 64 s], K-major B
constexpr uint32_t UNIT_BYTES = 80 * KB;
constexpr size_t SLICE_BUDGET = (size_t)96 << 20;   // workspace bytes for one slice of units

constexpr uint32_t ID_G = idesc_bf16(128, 128, false, false);  // [K;Q] [K;Q]^T
constexpr uint32_t ID_SW = idesc_bf16(128, 64, false, true);   // S0 (-W)^T
constexpr uint32_t ID_SQ = idesc_bf16(128, 64, false, false);  // S0 Q~^T, U^T P^T
constexpr uint32_t ID_UK = idesc_bf16(128, 128, false, true);  // U^T K~
// Products whose right factor is lower triangular in (output token r, summed token s) --
// X T'^T, X T''^T, X P^T with T', T'' zero for s > r and P zero for s > r: the 16-token K-block
// kb only reaches outputs r >= 16 kb, so it runs with N = 64 - 16 kb on columns 16 kb..63 (and
// B's rows from 16 kb on), 62.5% of the full work.
__host__ __device__ constexpr uint32_t id_tri_kt(int kb) { return idesc_bf16(128, 64 - 16 * kb, true, false); }
__host__ __device__ constexpr uint32_t id_tri_sq(int kb) { return idesc_bf16(128, 64 - 16 * kb, false, false); }

constexpr float LOG2E = 1.4426950408889634f;

struct TcParams {
  int T, Hk, Hv, num_slots, l2norm, gates_pre;
  int n0, ns;             // first chunk of this slice, chunks in this slice
  float eps, scale;
  const void* a;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  float* state;
  const int32_t* slots;
  uint8_t* units;         // workspace: ns * B * Hv units of UNIT_BYTES
  size_t n_units;         // units in one half of the workspace (bounds checks)
  int Bm;                 // batch extent of the token arrays (1 for a packed batch)
  float* egc;             // workspace: e^{G_C} per unit
  // in-call snapshots: the state entering chunk n (n > 0, n a multiple of se_c, n C <= T) goes
  // to bank row snap_slots[b * n_snap + n / se_c - 1]; se_c == 0: none
  int se_c, n_snap, n_snap_slots;
  const int32_t* snap_slots;
  // gated RMS norm of the output (the gate z arrives by TMA): out = w o / rms(o) silu(z)
  int gate;
  const float* gw;
  float geps;
  // packed variable-length batch (cu != nullptr): all tokens on one axis (batch index 0 of
  // the tensor maps); global chunk u of a slice is ctab[n0 + u] = {first token, tokens,
  // sequence}; sequence s owns global chunks [ccs[s], ccs[s+1]) and tokens [cu[s], cu[s+1])
  const int32_t* cu;
  const int32_t* ccs;
  const int4* ctab;
  void* out;              // for the ragged last chunk of a packed sequence (plain stores)
  // slices after the first of a call (and the first slice of a call that continues the one
  // before it): the local kernel waits for the kernel before it (the previous chain) only at
  // the end of its last block; the chain lets the kernel after it (the next slice's or call's
  // local kernel) start as soon as its own grid wait has returned
  int late_wait, early_trigger;
  // a late-waiting local kernel that releases its chain at its start (the first slice of an
  // ordinary call with the conv fused), or (trigger_end) once each block's unit is done, the
  // chain then reading the state only after its grid wait (state_late)
  int trigger_first, trigger_end, state_late;
  // the conv of the q and k channels fused into the local kernel (tm_q and tm_k then map the
  // pre-conv input x, [B][T][Cc]): the unit convolves its key head's q and k channels
  // (positions before the call's first token from `halo`: the conv state rows of slot
  // slots[b] when halo_by_slot, else rows [b][W-1][Cc] of the previous call's conv tail); the
  // units of the call's last chunk leave the q / k part of the call's conv tail in `tail`
  // [B][W-1][Cc] (the conv kernel before them leaves the v part); the last slice's chain
  // copies the tail into conv_state (cs_out, null before the last slice)
  int fuse, Cc, silu, halo_by_slot;
  const __nv_bfloat16* x;
  const __nv_bfloat16* cw;
  const __nv_bfloat16* cb;
  const __nv_bfloat16* halo;
  __nv_bfloat16* tail;
  __nv_bfloat16* cs_out;
  // with the conv fused and in-call snapshots: the conv-state bank [n_snap_slots][W-1][Cc]
  // (written by the chains), else null
  __nv_bfloat16* cbank;
  // with the conv fused: the post-conv v channels in the workspace [B][T][Hv d], else null
  const __nv_bfloat16* vbuf;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// hi = rn(x), lo = rn(x - hi) for a pair (x0, x1), packed
__device__ __forceinline__ void pack_hilo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 16-byte chunk `c` (0..7) of row `r` of a 128-byte-swizzled tile whose 8-row groups are
// 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128(uint32_t tile, int r, int c) {
  return tile + (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 32 fp32 values (times mul) -> bf16 -> 4 swizzled 16-byte chunks c0..c0+3 of row r.
__device__ __forceinline__ void store_row_bf16(uint32_t tile, int r, int c0, const float* v,
                                               float mul) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float* w = v + 8 * c;
    st_shared_v4(sw128(tile, r, c0 + c), pack_bf16(w[0] * mul, w[1] * mul),
                 pack_bf16(w[2] * mul, w[3] * mul), pack_bf16(w[4] * mul, w[5] * mul),
                 pack_bf16(w[6] * mul, w[7] * mul));
  }
}

// 32 fp32 values -> bf16 hi and lo rows (chunks c0..c0+3 of row r) of two tiles.
__device__ __forceinline__ void store_row_hilo(uint32_t tile_hi, uint32_t tile_lo, int r, int c0,
                                               const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pack_hilo(v[8 * c + 2 * e], v[8 * c + 2 * e + 1], h[e], l[e]);
    st_shared_v4(sw128(tile_hi, r, c0 + c), h[0], h[1], h[2], h[3]);
    st_shared_v4(sw128(tile_lo, r, c0 + c), l[0], l[1], l[2], l[3]);
  }
}

// ---- warp-level tensor-core products for the solve (mma.sync m16n8k16, bf16 in, fp32 out).
// A value x enters as the pair hi = rn(x), lo = rn(x - hi) and a product as hi*hi + hi*lo +
// lo*hi (the lo*lo term is below 2^-16 of it), which keeps about 16 bits of each operand.
// Fragment layouts (lane = 4 g + t): A (16 x 16, row-major) holds rows g and g + 8, columns
// 2t, 2t + 1 and 8 + 2t, 9 + 2t; B (16 x 8, k x n) holds k = 2t, 2t + 1 and 8 + 2t, 9 + 2t at
// n = g; the fp32 accumulator (16 x 8) holds rows g and g + 8 at columns 2t, 2t + 1.
struct FragA { uint32_t h[4], l[4]; };
struct FragB { uint32_t h[2], l[2]; };

__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d += a b with both operands as hi + lo pairs (small terms first)
__device__ __forceinline__ void mma_hilo(float (&d)[4], const FragA& a, const FragB& b) {
  mma_m16n8k16(d, a.l, b.h[0], b.h[1]);
  mma_m16n8k16(d, a.h, b.l[0], b.l[1]);
  mma_m16n8k16(d, a.h, b.h[0], b.h[1]);
}
// A fragment of the 16 x 16 block at (r0, c0) of a row-major fp32 matrix (row stride LA)
__device__ __forceinline__ void load_a_hilo(const float* M, int r0, int c0, int lane, FragA& f) {
  const int g = lane >> 2, t = lane & 3;
  const float* p0 = M + (r0 + g) * LA + c0 + 2 * t;
  const float* p1 = p0 + 8 * LA;
  const float2 x0 = *reinterpret_cast<const float2*>(p0);
  const float2 x1 = *reinterpret_cast<const float2*>(p1);
  const float2 x2 = *reinterpret_cast<const float2*>(p0 + 8);
  const float2 x3 = *reinterpret_cast<const float2*>(p1 + 8);
  pack_hilo(x0.x, x0.y, f.h[0], f.l[0]);
  pack_hilo(x1.x, x1.y, f.h[1], f.l[1]);
  pack_hilo(x2.x, x2.y, f.h[2], f.l[2]);
  pack_hilo(x3.x, x3.y, f.h[3], f.l[3]);
}
// B fragment of the 16 (k) x 8 (n) block at (k0, n0) of a row-major fp32 matrix [k][n]
__device__ __forceinline__ void load_b_hilo(const float* M, int k0, int n0, int lane, FragB& f) {
  const int g = lane >> 2, t = lane & 3;
  const float* p = M + (k0 + 2 * t) * LA + n0 + g;
  pack_hilo(p[0], p[LA], f.h[0], f.l[0]);
  pack_hilo(p[8 * LA], p[9 * LA], f.h[1], f.l[1]);
}
// The accumulators of two adjacent 16 x 8 tiles (columns 0-7, 8-15 of a 16 x 16 block) as the
// A fragment of that block: the accumulator and A layouts coincide.
__device__ __forceinline__ void acc_to_a_hilo(const float (&d0)[4], const float (&d1)[4],
                                              FragA& f) {
  pack_hilo(d0[0], d0[1], f.h[0], f.l[0]);
  pack_hilo(d0[2], d0[3], f.h[1], f.l[1]);
  pack_hilo(d1[0], d1[1], f.h[2], f.l[2]);
  pack_hilo(d1[2], d1[3], f.h[3], f.l[3]);
}
// -d into the 16 x 8 block at (r0, c0) of a row-major fp32 matrix
__device__ __forceinline__ void store_neg(float* M, int r0, int c0, int lane, const float (&d)[4]) {
  const int g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(M + (r0 + g) * LA + c0 + 2 * t) = make_float2(-d[0], -d[1]);
  *reinterpret_cast<float2*>(M + (r0 + g + 8) * LA + c0 + 2 * t) = make_float2(-d[2], -d[3]);
}

// T = (I + A)^{-1} for the strictly lower 64 x 64 matrix A (fp32, row stride LA), by the
// blocked form of forward substitution, on the 256 threads of a local group (named barrier
// bar_id).  For a unit lower triangular L = [[L11, 0], [L21, L22]],
//   L^{-1} = [[T11, 0], [-T22 L21 T11, T22]],   T11 = L11^{-1},  T22 = L22^{-1}.
// Level 0: warps 0-3 invert one diagonal 16 x 16 block each in fp32 (lane = column;
// right-looking: once t_s is final, every later row r subtracts A_rs t_s) while the other
// threads zero the strictly upper blocks.  Level 1 (16 -> 32) and level 2 (32 -> 64) form
// the off-diagonal blocks as (T22 A21) T11 on the tensor cores, four warps each.
__device__ __forceinline__ void solve_unit_lower(const float* As, float* Ts, int lt,
                                                 uint32_t bar_id) {
  const int w = lt >> 5, lane = lt & 31;
  if (w < 4 && lane < 16) {
    const int o = 16 * w, c = lane;
    float a[16][16];
#pragma unroll
    for (int r = 1; r < 16; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = *reinterpret_cast<const float4*>(As + (o + r) * LA + o + 4 * q);
        a[r][4 * q] = x.x; a[r][4 * q + 1] = x.y; a[r][4 * q + 2] = x.z; a[r][4 * q + 3] = x.w;
      }
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const float ts = acc[s];
#pragma unroll
      for (int r = s + 1; r < 16; ++r) acc[r] = fmaf(-a[r][s], ts, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Ts[(o + r) * LA + o + c] = acc[r];
  } else {
    // strictly upper blocks of T are zero: blocks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
    const int z = (w < 4) ? (w * 16 + lane - 16) : (64 + (lt - 128));   // 0..191
    for (int idx = z; idx < 6 * 256; idx += 192) {
      const int blk = idx >> 8, e = idx & 255;
      const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      Ts[(16 * bi + (e >> 4)) * LA + 16 * bj + (e & 15)] = 0.f;
    }
  }
  named_bar_sync(bar_id, LGT);
  // level 1: warp w forms columns 8 (w & 1) .. + 7 of block (i, j) = (1, 0) or (3, 2)
  if (w < 4) {
    const int i = 2 * (w >> 1) + 1, j = i - 1, nh = w & 1;
    FragA tii;
    load_a_hilo(Ts, 16 * i, 16 * i, lane, tii);
    float z[2][4] = {};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      FragB aij;
      load_b_hilo(As, 16 * i, 16 * j + 8 * nt, lane, aij);
      mma_hilo(z[nt], tii, aij);
    }
    FragA za;
    acc_to_a_hilo(z[0], z[1], za);
    FragB tjj;
    load_b_hilo(Ts, 16 * j, 16 * j + 8 * nh, lane, tjj);
    float r[4] = {};
    mma_hilo(r, za, tjj);
    store_neg(Ts, 16 * i, 16 * j + 8 * nh, lane, r);
  }
  named_bar_sync(bar_id, LGT);
  // level 2: the 32 x 32 block at rows 32.., columns 0..; warp w forms rows 32 + 16 (w >> 1)
  // .. + 15, columns 16 (w & 1) .. + 15
  if (w < 4) {
    const int r0 = 32 + 16 * (w >> 1), nh = w & 1;
    float z[4][4] = {};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      FragA tb;
      load_a_hilo(Ts, r0, 32 + 16 * kk, lane, tb);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        FragB ab;
        load_b_hilo(As, 32 + 16 * kk, 8 * nt, lane, ab);
        mma_hilo(z[nt], tb, ab);
      }
    }
    float r[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      FragA za;
      acc_to_a_hilo(z[2 * kk], z[2 * kk + 1], za);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        FragB ta;
        load_b_hilo(Ts, 16 * kk, 16 * nh + 8 * nt, lane, ta);
        mma_hilo(r[nt], za, ta);
      }
    }
    store_neg(Ts, r0, 16 * nh, lane, r[0]);
    store_neg(Ts, r0, 16 * nh + 8, lane, r[1]);
  }
  named_bar_sync(bar_id, LGT);
}

// Row scaling in place of the two 64-row blocks (kb = 0, 1; 16 KB apart) of a K or Q tile:
// row r of both blocks times f0[r] * f1[r].  Thread lt: block lt >> 7, row (lt >> 1) & 63,
// chunks 4 (lt & 1) .. + 3 visited in swizzled order (the lanes' rows hit different banks).
__device__ __forceinline__ void scale_rows_in_place(uint8_t* tile, const float* f0,
                                                    const float* f1, int lt) {
  const int kb = lt >> 7, r = (lt >> 1) & 63, c0 = 4 * (lt & 1);
  uint8_t* row = tile + kb * 16 * KB + r * 128;
  const float f = f0[r] * f1[r];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int pc = ((c0 + c) ^ r) & 7;
    uint4 w4 = reinterpret_cast<const uint4*>(row)[pc];
    __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&w4);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(hv[e]);
      hv[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
    }
    reinterpret_cast<uint4*>(row)[pc] = w4;
  }
}

// ======================================================================= chunk-local unit
// One unit = (chunk j of the slice, value head h, sequence b), processed by a group of 256
// threads with its own named barrier, TMEM columns and mbarriers (here a whole CTA of the
// chunk-local kernel).  Each tile for the chain is staged, in the swizzled layout the chain's MMAs read, in
// shared memory that is free at that point (P in the T region before the solve, Q~ in place,
// T'' beside T', K~ in place and -W^T over Q~ once K is read no more) and leaves with bulk
// copies of whole rows.
constexpr uint32_t L_KQ = 0;            // [kb][K 64 rows | Q 64 rows][128 B]
constexpr uint32_t L_SOLVE = 32 * KB;   // A | T fp32 [64][LA]; then T'h T'l
constexpr uint32_t L_MISC = L_SOLVE + 2 * SOLVE_MAT;   // factors, solve scratch, barriers
constexpr uint32_t L_SMEM = L_MISC + 6 * KB + KB;
constexpr uint32_t L_TMEM = 128;        // G (128 columns); later W^T in its first 64

// ======================================================================= fused conv
// The causal depthwise conv of width 4 (model card, "How It Works": the short conv in front of
// the recurrence) of the unit's q and k channels, computed inside the chunk-local unit in
// place on its K and Q tiles, which arrive by TMA as the pre-conv input x in the layout the
// MMAs read.  Thread lt owns one channel pair of one 64-channel tile block and 32 tokens, and
// slides up its column from the last token, so that each input is read before its row is
// overwritten; the three inputs below its first token are read before any thread writes (the
// rows of the thread below it, or, for the chunk's first rows, the tokens before the chunk:
// x, or at the call's start the halo rows).  The per-token arithmetic is the conv kernels'
// (conv_token), so the results are the same bits.  (The v channels are convolved by the conv
// kernel launched before the chunk-local kernel.)
constexpr int FC_W = 4, FC_H = FC_W - 1;

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}

// The pre-conv input pair at x channel ch of token t of the call (t >= -3; t < 0: halo row
// t + 3 -- the conv state rows of slot `slot`, or the previous call's conv tail of sequence b).
__device__ __forceinline__ uint32_t input_pair(const TcParams& p, int slot, int b, int t, int ch) {
  if (t < 0) {
    const size_t row = (size_t)(p.halo_by_slot ? slot : b) * FC_H + (t + FC_H);
    if (!in_bounds(&g_err_tc, row < (size_t)(p.halo_by_slot ? p.num_slots : p.Bm) * FC_H &&
                                  t >= -FC_H && ch < p.Cc))
      return 0u;
    return __ldcg(reinterpret_cast<const unsigned int*>(p.halo + row * p.Cc + ch));
  }
  if (!in_bounds(&g_err_tc, b < p.Bm && t < p.T && ch < p.Cc)) return 0u;
  return __ldg(reinterpret_cast<const unsigned int*>(p.x + ((size_t)b * p.T + t) * p.Cc + ch));
}

// One thread's share of the fused conv (see above).  Its first part (taps, biases and the three
// inputs below its rows) must complete in every thread before any thread runs its second part.
struct FusedConvQK {
  uint32_t tile, cofs;
  int q, th;
  float w[FC_W][2], bias[2];
  uint32_t below[FC_H];

  __device__ __forceinline__ uint32_t addr(int r) const {
    return tile + (uint32_t)r * 128u + ((uint32_t)(((q >> 2) ^ (r & 7)) << 4)) + cofs;
  }

  __device__ __forceinline__ void prepare(const TcParams& p, uint32_t sb, int lt, int kh, int b,
                                          int slot, int tok0) {
    const int pp = lt & 127, blk = pp >> 5, kb = blk & 1, isk = blk >> 1;
    q = pp & 31;
    th = lt >> 7;
    const int ch = (isk ? p.Hk * D : 0) + kh * D + 64 * kb + 2 * q;
    tile = sb + L_KQ + kb * 16 * KB + (isk ? 0u : 8 * KB);
    cofs = (uint32_t)((q & 3) * 4);
    // taps: conv_weight rows ch, ch + 1 (4 bf16 each); biases ch, ch + 1
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(p.cw + (size_t)ch * FC_W));
    const float2 a01 = bf2_to_f2(wv.x), a23 = bf2_to_f2(wv.y);
    const float2 b01 = bf2_to_f2(wv.z), b23 = bf2_to_f2(wv.w);
    w[0][0] = a01.x; w[1][0] = a01.y; w[2][0] = a23.x; w[3][0] = a23.y;
    w[0][1] = b01.x; w[1][1] = b01.y; w[2][1] = b23.x; w[3][1] = b23.y;
    const float2 bb = p.cb ? bf2_to_f2(__ldg(reinterpret_cast<const unsigned int*>(p.cb + ch)))
                           : make_float2(0.f, 0.f);
    bias[0] = bb.x;
    bias[1] = bb.y;
#pragma unroll
    for (int j = 0; j < FC_H; ++j) {
      const int r = 32 * th - FC_H + j;
      below[j] = th ? lds32(addr(r)) : input_pair(p, slot, b, tok0 + r, ch);
    }
  }

  // rows 32 th + 31 .. 32 th, bottom up; rows at or past ntok are zero
  __device__ __forceinline__ void run(int ntok, int silu) {
    const int r0 = 32 * th;
    uint32_t win[FC_W];
#pragma unroll
    for (int j = 0; j < FC_W; ++j) win[j] = lds32(addr(r0 + 31 - FC_H + j));
#pragma unroll
    for (int t = 31; t >= 0; --t) {
      const int r = r0 + t;
      float x2[FC_W][2], y2[2];
#pragma unroll
      for (int j = 0; j < FC_W; ++j) {
        const float2 f = bf2_to_f2(win[j]);
        x2[j][0] = f.x;
        x2[j][1] = f.y;
      }
      conv_token<FC_W, 2>(w, bias, x2, silu, y2);
      sts32(addr(r), r < ntok ? pack_bf16(y2[0], y2[1]) : 0u);
      if (t > 0) {
#pragma unroll
        for (int j = FC_W - 1; j > 0; --j) win[j] = win[j - 1];
        win[0] = t >= FC_W ? lds32(addr(r0 + t - FC_W)) : below[(t >= 1 && t <= FC_H) ? t - 1 : 0];
      }
    }
  }
};

// The call's conv tail of the q and k channels of key head kh (its last 3 inputs, from x or,
// for a call of fewer than 3 tokens, partly from the halo) -> tail rows [b][0..2].  Threads
// 0..95, one 16-byte word each.
__device__ __forceinline__ void fused_conv_tail_qk(const TcParams& p, int tid, int kh, int b,
                                                   int slot) {
  if (tid >= 96) return;
  const int j = tid >> 5, cc = tid & 31;
  const int ch = ((cc >> 4) ? p.Hk * D : 0) + kh * D + 8 * (cc & 15);
  const int t = p.T - FC_H + j;
  if (!in_bounds(&g_err_tc, b < p.Bm && ch + 8 <= p.Cc &&
                                (t >= 0 || (p.halo_by_slot ? slot < p.num_slots : true))))
    return;
  uint4 v;
  if (t < 0) {
    const size_t row = (size_t)(p.halo_by_slot ? slot : b) * FC_H + (t + FC_H);
    v = __ldcg(reinterpret_cast<const uint4*>(p.halo + row * p.Cc + ch));
  } else {
    v = __ldg(reinterpret_cast<const uint4*>(p.x + ((size_t)b * p.T + t) * p.Cc + ch));
  }
  *reinterpret_cast<uint4*>(p.tail + ((size_t)b * FC_H + j) * p.Cc + ch) = v;
}

// A group's resources: its 1024-byte aligned L_SMEM bytes (barriers and flags inside them),
// its 128 TMEM columns, its named barrier, and the parities of its two mbarriers.
struct LocalGroup {
  uint8_t* sm;
  uint32_t sb;
  uint32_t tmem;
  int lt;                  // thread index within the group, 0..255
  uint32_t bar_id;         // named barrier of the group's 256 threads
  uint32_t in_phase;       // parity of the next wait on bar_in
  bool tmem_pending;       // the TMEM address is still to be read from tmem_slot() after the
                           // unit's first group barrier (which publishes the allocation)
  __device__ void sync() const { named_bar_sync(bar_id, LGT); }
  __device__ bool sync_or(bool x) const { return named_bar_sync_or(bar_id, LGT, x); }
  __device__ uint64_t* barmem() const { return reinterpret_cast<uint64_t*>(sm + L_MISC + 5120); }
  __device__ uint32_t* tmem_slot() const {
    return reinterpret_cast<uint32_t*>(sm + L_MISC + 5120 + 32);
  }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(sm + L_MISC + 5120 + 36);
  }
};

// Thread 0 of the group: its two mbarriers and its abort flag.
__device__ __forceinline__ void local_group_init(const LocalGroup& g) {
  if (g.lt == 0) {
    mbar_init(smem_addr(&g.barmem()[0]), 1);
    mbar_init(smem_addr(&g.barmem()[1]), 1);
    *g.abort_flag() = 0;
    fence_mbar_init();
  }
}

// Tokens of unit jc of a slice: first token, count and sequence; false when the unit holds no
// work (past the last chunk of a packed batch, or a skipped / out-of-range state slot, which
// the chain reports).
__device__ __forceinline__ bool local_unit_tokens(const TcParams& p, int jc, int b, int& tok0,
                                                  int& ntok, int& seq) {
  tok0 = (p.n0 + jc) * C;
  ntok = min(C, p.T - tok0);
  seq = b;
  if (p.cu) {
    const int4 e = p.ctab[p.n0 + jc];
    tok0 = e.x;
    ntok = e.y;
    seq = e.z;
    if (ntok <= 0) return false;
  }
  const int slot = p.slots ? p.slots[seq] : seq;
  return slot >= 0 && slot < p.num_slots;
}

// Everything of one unit that does not depend on the state.  PDL_MID: the standalone local
// kernel of a call's first slice waits for the kernel before it (and releases its
// dependents) between the gates and the tile loads.  Returns false when a bounded wait gave
// up (the group's abort flag is then set and the condition recorded).
template <typename Tin, bool PDL_MID>
__device__ __forceinline__ bool local_unit(LocalGroup& g, const CUtensorMap* tm_q,
                                           const CUtensorMap* tm_k, const TcParams& p, int jc,
                                           int h, int b, int tok0, int ntok) {
  uint8_t* sm = g.sm;
  const uint32_t sb = g.sb;
  const int tid = g.lt, warp = tid >> 5, lane = tid & 31;
  const int kh = h / (p.Hv / p.Hk);
  const size_t u = ((size_t)b * p.Hv + h) * p.ns + jc;
  uint8_t* unit = p.units + u * UNIT_BYTES;
  const int slot = p.slots ? p.slots[b] : b;

  float* gl2 = reinterpret_cast<float*>(sm + L_MISC);   // G_r * log2(e)
  float* beta = gl2 + 64;
  float* nk = gl2 + 128;                                 // 1 / ||k_r||
  float* nq = gl2 + 192;                                 // scale / ||q_r||
  float* eG = gl2 + 256;                                 // e^{G_r}
  float* dK = gl2 + 320;                                 // e^{G_C - G_r}
  float* fT1 = gl2 + 384;                                // beta_s e^{G_s} / ||k_s||
  volatile int* sAbort = g.abort_flag();
  const uint32_t bar_in = smem_addr(&g.barmem()[0]), bar_mma = smem_addr(&g.barmem()[1]);

  // gates: g, beta and G = inclusive prefix sum of g (warp 1, two tokens per lane)
  if (warp == 1) {
    const float A_log_h = p.gates_pre ? 0.f : p.A_log[h];
    const float dtb_h = (p.gates_pre || !p.dt_bias) ? 0.f : p.dt_bias[h];
    float g2[2] = {0.f, 0.f}, b2[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 2 * lane + e;
      if (r < ntok) {
        const size_t gi = ((size_t)b * p.T + tok0 + r) * p.Hv + h;
        if (!in_bounds(&g_err_tc, gi < (size_t)p.Bm * p.T * p.Hv)) continue;
        if (p.gates_pre) {
          g2[e] = reinterpret_cast<const float*>(p.a)[gi];
          b2[e] = reinterpret_cast<const float*>(p.b)[gi];
        } else {
          g2[e] = gate_g(ld_elem(reinterpret_cast<const Tin*>(p.a) + gi), A_log_h, dtb_h);
          b2[e] = sigmoid_f(ld_elem(reinterpret_cast<const Tin*>(p.b) + gi));
        }
      }
    }
    float s = g2[0] + g2[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    gl2[2 * lane] = (s - g2[1]) * LOG2E;
    gl2[2 * lane + 1] = s * LOG2E;
    beta[2 * lane] = b2[0];
    beta[2 * lane + 1] = b2[1];
  }
  // the conv output (K, Q) and this slice's workspace belong to the kernels before until
  // here.  Only then may the state-chain kernel start its set-up, which reads the state: the
  // chain that last wrote it is then complete and visible.  A later slice of the call (its
  // own half of a double-buffered workspace; the conv output complete since the first slice)
  // skips this and waits at its end instead, running beside the previous slice's chain.
  if (PDL_MID && !p.late_wait) {
    pdl_wait();
    pdl_trigger();
  }
  if (tid == 0) {
    // the K and Q tiles (with the conv fused: the pre-conv q and k channels of x, which the
    // conv below then replaces in place)
    const int k0 = p.fuse ? p.Hk * D : 0;
    mbar_arrive_expect_tx(bar_in, 32 * KB);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_3d(sb + L_KQ + kb * 16 * KB, tm_k, k0 + kh * D + 64 * kb, tok0, b, bar_in);
      tma_load_3d(sb + L_KQ + kb * 16 * KB + 8 * KB, tm_q, kh * D + 64 * kb, tok0, b, bar_in);
    }
  }
  // the call's last chunk: the conv tail of the q / k channels (the first value head of a key
  // head writes it)
  if (p.fuse && p.tail && tok0 + C >= p.T && h % (p.Hv / p.Hk) == 0)
    fused_conv_tail_qk(p, tid, kh, b, slot);
  tc_fence_before();
  g.sync();
  tc_fence_after();
  if (g.tmem_pending) {
    g.tmem = *g.tmem_slot();
    g.tmem_pending = false;
  }
  const uint32_t TM_G = g.tmem, TM_W = g.tmem;
  const int gw = warp & 3, half = warp >> 2;
  const uint32_t lane_off = static_cast<uint32_t>(gw * 32) << 16;
  const int row = 32 * gw + lane;
  bool pend_mma = false;
  uint32_t mma_phase = 0;

  do {
    if (!mbar_wait_or_abort(bar_in, g.in_phase, sAbort)) *sAbort = 1;
    g.in_phase ^= 1;
    g.sync();
    if (*sAbort) break;
    if (p.fuse) {
      FusedConvQK fc;
      fc.prepare(p, sb, tid, kh, b, slot, tok0);
      g.sync();
      fc.run(ntok, p.silu);
      fence_proxy_async_smem();        // (the tensor cores read the K and Q tiles next)
      g.sync();
    }
    // ---- MMA 1: G = [K; Q] [K; Q]^T  (M = N = 128: k_0..k_63, q_0..q_63; K = 128).  Its
    //      k.k and q.k blocks feed A and P, its diagonal gives the squared row norms.
    if (warp == 0 && elect_one()) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t dkq = sdesc_sw128(sb + L_KQ + (k >> 2) * 16 * KB + (k & 3) * 32, 16, 1024);
        mma_bf16(TM_G, dkq, dkq, ID_G, k > 0);
      }
      mma_commit(bar_mma);
    }
    pend_mma = true;
    if (tid < 64) {
      eG[tid] = ex2_approx(gl2[tid]);
      dK[tid] = ex2_approx(gl2[63] - gl2[tid]);
    }
    if (tid == 0) p.egc[u] = ex2_approx(gl2[63]);
    if (!mbar_wait_or_abort(bar_mma, mma_phase, sAbort)) *sAbort = 1;
    mma_phase ^= 1;
    pend_mma = false;
    tc_fence_after();
    if (g.sync_or(*sAbort)) break;

    // ---- E1: G -> A (fp32 [r][s], strictly lower) and P (bf16 hi/lo [r][s], K-major)
    {
      float* As = reinterpret_cast<float*>(sm + L_SOLVE);
      const bool isq = row >= 64;                        // (warp-uniform)
      const int r = row & 63;
      float v[32], dg[32];
      tmem_ld32(TM_G + lane_off + 32 * half, v);
      // the diagonal entry of this row: k row r in column r (warps 0 and 5 hold it), q row r in
      // column 64 + r (read by the q warps of column half 0)
      if (isq && half == 0) tmem_ld32(TM_G + lane_off + 64 + 32 * (gw - 2), dg);
      tmem_wait_ld();
      tc_fence_before();                                 // (W^T later reuses these columns)
      if (isq ? (half == 0) : (half == gw)) {
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == lane) d = isq ? dg[j] : v[j];
        const float inv = p.l2norm ? 1.0f / sqrtf(d + p.eps) : 1.0f;
        if (isq) nq[r] = inv * p.scale; else nk[r] = inv;
      }
      g.sync();
      if (tid < 64) fT1[tid] = beta[tid] * eG[tid] * nk[tid];
      const float Gr = gl2[r], sr = (isq ? 1.0f : beta[r]) * (isq ? nq[r] : nk[r]);
      float gs[32], ns[32];
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 g4 = *reinterpret_cast<const float4*>(gl2 + 32 * half + 4 * j4);
        const float4 n4 = *reinterpret_cast<const float4*>(nk + 32 * half + 4 * j4);
        gs[4 * j4] = g4.x; gs[4 * j4 + 1] = g4.y; gs[4 * j4 + 2] = g4.z; gs[4 * j4 + 3] = g4.w;
        ns[4 * j4] = n4.x; ns[4 * j4 + 1] = n4.y; ns[4 * j4 + 2] = n4.z; ns[4 * j4 + 3] = n4.w;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int s = 32 * half + j;
        const bool keep = isq ? (s <= r) : (s < r);
        v[j] = keep ? ex2_approx(Gr - gs[j]) * v[j] * (sr * ns[j]) : 0.f;
      }
      if (isq) {
        // P staged in the T region of the solve (not written before the solve starts)
        store_row_hilo(sb + L_SOLVE + SOLVE_MAT, sb + L_SOLVE + SOLVE_MAT + 8 * KB, r, 4 * half, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(As + r * LA + 32 * half + j) =
              make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    // ---- Q~ = diag(scale e^G / ||q||) Q in place (Q is not read again).  Thread: half a row
    //      of one 64-column block (4 chunks, visited in swizzled order so that the lanes' rows
    //      hit different banks).
    scale_rows_in_place(sm + L_KQ + 8 * KB, eG, nq, tid);
    fence_proxy_async_smem();
    g.sync();
    if (tid == 0) {                  // (bulk-copy groups are per thread: thread 0 waits on them)
      bulk_store(unit + U_P, sb + L_SOLVE + SOLVE_MAT, 16 * KB);
      tma_store_commit();
      bulk_store(unit + U_QT, sb + L_KQ + 8 * KB, 8 * KB);
      bulk_store(unit + U_QT + 8 * KB, sb + L_KQ + 24 * KB, 8 * KB);
      tma_store_commit();
      tma_store_wait_read_1();       // P has been read: the solve may write T over it
    }
    g.sync();

    // ---- the direct solve T = (I + A)^{-1}, then T' and T'' as bf16 hi/lo B operands
    {
      float* As = reinterpret_cast<float*>(sm + L_SOLVE);
      float* Ts = reinterpret_cast<float*>(sm + L_SOLVE + SOLVE_MAT);
      solve_unit_lower(As, Ts, tid, g.bar_id);
      // the T'/T'' tiles reuse the A/T region: read this thread's T entries first
      float tv[2][8];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int idx = tid + LGT * jj, r = idx >> 3, c = idx & 7;
        const float4 x0 = *reinterpret_cast<const float4*>(Ts + r * LA + 8 * c);
        const float4 x1 = *reinterpret_cast<const float4*>(Ts + r * LA + 8 * c + 4);
        tv[jj][0] = x0.x; tv[jj][1] = x0.y; tv[jj][2] = x0.z; tv[jj][3] = x0.w;
        tv[jj][4] = x1.x; tv[jj][5] = x1.y; tv[jj][6] = x1.z; tv[jj][7] = x1.w;
      }
      g.sync();
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int idx = tid + LGT * jj, r = idx >> 3, c = idx & 7;
        uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int s = 8 * c + 2 * e;
          const float2 f1 = *reinterpret_cast<const float2*>(fT1 + s);
          const float2 f2 = *reinterpret_cast<const float2*>(beta + s);
          pack_hilo(tv[jj][2 * e] * f1.x, tv[jj][2 * e + 1] * f1.y, h1[e], l1[e]);
          pack_hilo(tv[jj][2 * e] * f2.x, tv[jj][2 * e + 1] * f2.y, h2[e], l2[e]);
        }
        st_shared_v4(sw128(sb + L_SOLVE, r, c), h1[0], h1[1], h1[2], h1[3]);
        st_shared_v4(sw128(sb + L_SOLVE + 8 * KB, r, c), l1[0], l1[1], l1[2], l1[3]);
        st_shared_v4(sw128(sb + L_SOLVE + 16 * KB, r, c), h2[0], h2[1], h2[2], h2[3]);
        st_shared_v4(sw128(sb + L_SOLVE + 24 * KB, r, c), l2[0], l2[1], l2[2], l2[3]);
      }
    }
    fence_proxy_async_smem();
    g.sync();
    if (tid == 0) {
      bulk_store(unit + U_T2, sb + L_SOLVE + 16 * KB, 16 * KB);
      tma_store_commit();
    }
    // ---- MMA 3: W^T = K^T T'^T (M = d_k, N = 64 tokens, K = 64 tokens)
    if (warp == 0 && elect_one()) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int kb = k & 3;          // (T' is lower triangular: see id_tri_kt)
        mma_bf16(TM_W + 16 * kb, sdesc_sw128(sb + L_KQ + kb * 2048, 16 * KB, 1024),
                 sdesc_sw128(sb + L_SOLVE + (k < 4 ? 0 : 8 * KB) + kb * (2048 + 32), 16, 1024),
                 id_tri_kt(kb), k > 0);
      }
      mma_commit(bar_mma);
    }
    pend_mma = true;
    if (!mbar_wait_or_abort(bar_mma, mma_phase, sAbort)) *sAbort = 1;
    mma_phase ^= 1;
    pend_mma = false;
    tc_fence_after();
    if (tid == 0) tma_store_wait_read_1();   // Q~ has been read out of the Q half
    if (g.sync_or(*sAbort)) break;
    // ---- K is read no more: K~ = diag(e^{G_C-G} / ||k||) K in place; E3: W^T -> -W^T bf16
    //      (MN-major: row = d_k index, 64 token columns) into the Q half
    scale_rows_in_place(sm + L_KQ, dK, nk, tid);
    {
      float v[32];
      tmem_ld32(TM_W + lane_off + 32 * half, v);
      tmem_wait_ld();
      store_row_bf16(sb + L_KQ + (row < 64 ? 8 * KB : 24 * KB), row & 63, 4 * half, v, -1.0f);
    }
    tc_fence_before();               // (the next unit's MMAs write these TMEM columns)
    fence_proxy_async_smem();
    g.sync();
    if (tid == 0) {
      bulk_store(unit + U_KT, sb + L_KQ, 8 * KB);
      bulk_store(unit + U_KT + 8 * KB, sb + L_KQ + 16 * KB, 8 * KB);
      bulk_store(unit + U_NW, sb + L_KQ + 8 * KB, 8 * KB);
      bulk_store(unit + U_NW + 8 * KB, sb + L_KQ + 24 * KB, 8 * KB);
      tma_store_commit();
    }
  } while (0);

  // ---- the unit's end: the bulk copies out have read shared memory (the next unit's loads
  //      may overwrite it), (abort path only) pending MMAs are done
  const bool aborted = *sAbort != 0;
  if (tid == 0) {
    tma_store_wait_read();
    if (pend_mma) mbar_wait_bounded(bar_mma, mma_phase, 1u << 16);
    if (aborted) atomicOr(&g_err_tc, kErrTimeout);
  }
  return !aborted;
}

// Standalone chunk-local kernel: one CTA (one group) per (chunk j of the slice, value head h,
// sequence b), 256 threads, three CTAs per SM.
template <typename Tin>
__global__ void __launch_bounds__(LGT, 3)
    gdn_chunk_local_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed by offsetting the shared array itself so that every
  // pointer derived from it stays in the shared state space
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int jc = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  // a later slice of the call: the grid's last block alone waits for the previous slice's
  // chain, at its end; that keeps the grid from completing before the chain has, and lets
  // every other block finish and free its SM for the blocks behind it
  const bool wait_late = p.late_wait && jc == (int)gridDim.x - 1 &&
                         h == (int)gridDim.y - 1 && b == (int)gridDim.z - 1;
  if (p.trigger_first) pdl_trigger();
  int tok0, ntok, seq;
  // (the -DGDN_BOUNDS_CHECK build also drops a unit whose workspace unit or token rows would
  // fall outside their arrays)
  if (!local_unit_tokens(p, jc, b, tok0, ntok, seq) ||
      !in_bounds(&g_err_tc, ((size_t)b * p.Hv + h) * p.ns + jc < p.n_units && b < p.Bm &&
                                tok0 >= 0 && tok0 + ntok <= p.T)) {
    if (wait_late) pdl_wait();
    return;
  }
  LocalGroup g{sm, smem_addr(sm), 0u, tid, 1u, 0u, true};
  local_group_init(g);
  if (warp == 0) {
    tmem_alloc(smem_addr(g.tmem_slot()), L_TMEM);
    tmem_relinquish();
  }
  // (local_unit publishes the barrier initialisation and the TMEM address with its first
  // group barrier, after the gates, before either is used)
  local_unit<Tin, true>(g, &tm_q, &tm_k, p, jc, h, b, tok0, ntok);
  // ---- teardown: TMEM is freed once every thread's last TMEM access is done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(g.tmem, L_TMEM);
  }
  // the chain after this grid may be launched (and set up) once every block's unit is done
  if (p.trigger_end) pdl_trigger();
  // a later slice: this grid completes only after the previous slice's chain has, so that the
  // next chain (released by this grid's completion) reads the state that chain left
  if (wait_late) pdl_wait();
}

// One level of a transposing warp reduction: lanes with bit M set keep the upper half of
// s[0, L) and send the lower half to lane ^ M, the others the reverse; afterwards s[0, L/2)
// holds the sums of the kept half.
template <int M, int L>
__device__ __forceinline__ void butterfly_half(float (&s)[32], int lane) {
  const bool up = lane & M;
#pragma unroll
  for (int i = 0; i < L / 2; ++i) {
    const float send = up ? s[i] : s[i + L / 2];
    const float keep = up ? s[i + L / 2] : s[i];
    s[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
  }
}

// SiLU of the output gate: for a bf16 output z sigmoid(z) = z (1 + tanh(z / 2)) / 2 with the
// hardware tanh (one special-function op, relative error ~2^-11, below the output's rounding);
// for an fp32 output the exponential and division form.
template <typename Tout> __device__ __forceinline__ float silu_out(float z);
template <> __device__ __forceinline__ float silu_out<__nv_bfloat16>(float z) {
  float t;
  asm("tanh.approx.f32 %0, %1;\n" : "=f"(t) : "f"(0.5f * z));
  const float hz = 0.5f * z;
  return fmaf(hz, t, hz);
}
template <> __device__ __forceinline__ float silu_out<float>(float z) { return silu_gate(z); }

// A warp's 32 rows x 64 tokens of output (v[t] = row lane, token t) through its staging block
// [ROWS tokens][32 rows] to HBM, one TMA store of ROWS tokens per pass; lane 0 issues the
// stores and waits for the previous pass's read of the block.
template <typename Tout, int ROWS>
__device__ __forceinline__ void store_tile_passes(const CUtensorMap* tm, Tout* stg,
                                                  const float (&v)[64], int lane, int c0,
                                                  int tok0, int b) {
#pragma unroll
  for (int pass = 0; pass < 64 / ROWS; ++pass) {
    if (lane == 0) tma_store_wait_read();
    __syncwarp();
#pragma unroll
    for (int jj = 0; jj < ROWS; ++jj) stg[jj * 32 + lane] = from_float<Tout>(v[pass * ROWS + jj]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tm, smem_addr(stg), c0, tok0 + pass * ROWS, b);
      tma_store_commit();
    }
  }
}

// ======================================================================= chain kernel
// One CTA per (value head h, sequence b): eight epilogue warps (warp w: TMEM lane quarter
// w % 4, column half w / 4), one issuer warp, one elected lane of which issues every copy
// and MMA, so that no epilogue thread ever stalls behind the tensor-core queue, and four
// store warps for the output.  They meet only at mbarriers.  Per chunk: the five tiles of the
// local kernel plus V, double-buffered.
//
// The chain S -> S0 -> U -> S is the critical path; per chunk it runs
//   C0 (S0 = bf16(S); S *= e^{G_C} after signalling S0)  ->  U^T += S0 (-W)^T  ->  C2 (U^T ->
//   bf16 hi / lo)  ->  S += U^T K~
// with one commit barrier after each of its two MMA groups.  The output MMAs (O^T = S0 Q~^T,
// O^T += U^T P^T) and the state-independent U'^T = V^T T''^T of the next chunk are issued
// behind them and run while the epilogue warps work on the next step.  The finished output
// tile of a chunk (double-buffered in TMEM) is read by the store warps, which transpose it
// through shared memory (each warp its 32 d_v rows) and send it with TMA stores, off the
// epilogue's path.  A buffer's tiles other than P are free once S of its chunk is final; P
// once the output MMAs are done.
constexpr uint32_t CH_BUF = 96 * KB;            // unit tiles (80 KB) + V [2][64][128 B] (16 KB)
constexpr uint32_t CH_V = 80 * KB;
// output staging: 2 KB per store warp with the gated norm, else 4 KB (over the gate tiles)
constexpr uint32_t CH_OUT = 2 * CH_BUF;
constexpr uint32_t CH_Z = CH_OUT + 8 * KB;      // gate tiles z [64 tokens][32 d_v], 4 KB per store warp
constexpr uint32_t CH_SQ = CH_Z + 16 * KB;      // per-token sums of squares [2][4 warps][64]
constexpr uint32_t CH_RI = CH_SQ + 2 * KB;      // per-token 1 / rms, [4 warps][64]
constexpr uint32_t CH_MISC = CH_RI + KB;        // e^{G_C} of the slice (2 KB), barriers
constexpr uint32_t CH_SMEM = CH_MISC + 3 * KB + KB;
constexpr int CH_EPI = 256;                     // epilogue threads
constexpr int CH_ISSUER = CH_EPI / 32;          // the issuer warp
constexpr int CH_STORE = CH_ISSUER + 1;         // first of the four store warps
constexpr int CH_THREADS = CH_EPI + 32 + 128;
constexpr int MAX_SLICE = 512;
// TMEM columns: S fp32 | U^T fp32 | O^T fp32 x 2 | S0 bf16 packed | U^T bf16 hi | lo
constexpr uint32_t TM_S = 0, TM_U = 128, TM_O = 192, TM_S0 = 320, TM_UH = 384, TM_UL = 416;
constexpr uint32_t CH_TMEM = 512;

template <typename Tout>
__global__ void __launch_bounds__(CH_THREADS, 1)
    gdn_chunk_chain_kernel(const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_o,
                           const __grid_constant__ CUtensorMap tm_s,
                           const __grid_constant__ CUtensorMap tm_snap,
                           const __grid_constant__ CUtensorMap tm_z, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv;
  // this CTA's chunks: chunks n0 .. n0 + ns - 1 of sequence b; for a packed batch, the part
  // of sequence b's chunks [ccs[b], ccs[b+1]) inside this slice (tokens from tbase, batch
  // coordinate 0; the last one may hold fewer than C tokens of this sequence)
  int ns = p.ns, tbase = p.n0 * C, bt = b, last_tok = C;
  size_t u0 = ((size_t)b * p.Hv + h) * p.ns;      // first unit of this CTA's chunks
  if (p.cu) {
    const int cb0 = p.ccs[b], cb1 = p.ccs[b + 1];
    const int c0 = max(cb0, p.n0), c1 = min(cb1, p.n0 + p.ns);
    if (c0 >= c1) return;
    ns = c1 - c0;
    tbase = p.cu[b] + (c0 - cb0) * C;
    bt = 0;
    u0 = (size_t)h * p.ns + (c0 - p.n0);
    last_tok = min(C, p.cu[b + 1] - (tbase + (ns - 1) * C));
  }
  const int slot = p.slots ? p.slots[b] : b;
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (tid == 0 && (p.cu || p.n0 == 0)) atomicOr(&g_err_tc, kErrIndex);
    return;
  }
  // (the -DGDN_BOUNDS_CHECK build: this CTA's units, token rows and state rows)
  if (!in_bounds(&g_err_tc, u0 + ns <= p.n_units && bt < p.Bm && tbase >= 0 &&
                                (p.cu || tbase + (ns - 1) * C < p.T) && h < p.Hv))
    return;
  float* sEgc = reinterpret_cast<float*>(sm + CH_MISC);
  uint64_t* barmem = reinterpret_cast<uint64_t*>(sm + CH_MISC + 2048);
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + CH_MISC + 2048 + 256);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sm + CH_MISC + 2048 + 260);
  const uint32_t bar_ld0 = smem_addr(&barmem[0]), bar_ld1 = smem_addr(&barmem[1]);
  const uint32_t bar_u = smem_addr(&barmem[2]);     // MMA: U^T += S0 (-W)^T done (and all before)
  const uint32_t bar_s = smem_addr(&barmem[3]);     // MMA: S += U^T K~ done (and all before)
  // MMA: output MMAs of a chunk done (and all before), one barrier per TMEM output buffer
  const uint32_t bar_o0 = smem_addr(&barmem[4]), bar_o1 = smem_addr(&barmem[10]);
  const uint32_t bar_fin = smem_addr(&barmem[5]);   // MMA: teardown, everything issued done
  const uint32_t bar_c0 = smem_addr(&barmem[6]);    // epilogue: S0 packed, S rescaled
  const uint32_t bar_c2 = smem_addr(&barmem[7]);    // epilogue: U^T hi / lo packed
  const uint32_t bar_p0 = smem_addr(&barmem[8]), bar_p1 = smem_addr(&barmem[9]);   // P copies
  // store warps: the output tile of a TMEM output buffer has been read out
  const uint32_t bar_r0 = smem_addr(&barmem[11]), bar_r1 = smem_addr(&barmem[12]);
  // store warps, gated norm: barmem[13 + w] = gate tile of store warp w landed;
  // barmem[17 + (chunk & 1)] = the four warps' sums of squares written (every lane arrives)
  const bool issuer_warp = (warp == CH_ISSUER);

  // copies of chunk nl into buffer nl & 1: everything but P, and P (16 KB, needed only by the
  // last MMA group) on a barrier of its own
  auto load_main = [&](int nl) {
    const uint32_t buf = sb + (nl & 1) * CH_BUF;
    const uint32_t bar = (nl & 1) ? bar_ld1 : bar_ld0;
    const uint8_t* unit = p.units + (u0 + nl) * UNIT_BYTES;
    mbar_arrive_expect_tx(bar, 80 * KB);
    bulk_load(buf + U_NW, unit + U_NW, 32 * KB, bar);     // -W^T, Q~
    bulk_load(buf + U_KT, unit + U_KT, 32 * KB, bar);     // K~, T''
    tma_load_3d(buf + CH_V, &tm_v, h * D, tbase + nl * C, bt, bar);
    tma_load_3d(buf + CH_V + 8 * KB, &tm_v, h * D + 64, tbase + nl * C, bt, bar);
  };
  auto load_p = [&](int nl) {
    const uint32_t bar = (nl & 1) ? bar_p1 : bar_p0;
    mbar_arrive_expect_tx(bar, 16 * KB);
    bulk_load(sb + (nl & 1) * CH_BUF + U_P, p.units + (u0 + nl) * UNIT_BYTES + U_P, 16 * KB, bar);
  };
  // per buffer (issuer warp): chunk of the main / P copy issued and not yet waited for, or -1
  int ld_chunk[2] = {-1, -1}, lp_chunk[2] = {-1, -1};
  if (tid == CH_EPI) {
    for (int i = 0; i < 19; ++i)
      mbar_init(smem_addr(&barmem[i]), (i == 6 || i == 7) ? CH_EPI / 32
                                       : (i == 11 || i == 12) ? 4 : (i >= 17 ? 128 : 1));
    *sAbort = 0;
    fence_mbar_init();
  }
  if (issuer_warp)
    for (int i = 0; i < 2 && i < ns; ++i) ld_chunk[i] = lp_chunk[i] = i;
  if (warp == 0) {
    tmem_alloc(smem_addr(sTmem), CH_TMEM);
    tmem_relinquish();
  }
  const int gw = warp & 3, hc = (warp >> 2) & 1;
  const uint32_t lane_off = static_cast<uint32_t>(gw * 32) << 16;
  const int row = 32 * gw + lane;                       // state row / d_v index of this thread
  float* Sg = p.state + ((size_t)slot * p.Hv + h) * D * D + (size_t)row * D + 64 * hc;
  // the entering state (fp32, row i -> TMEM lane i; this thread: 64 columns).  It was last
  // written by the chain of the previous slice or call, which completed before the local
  // kernel before this one did; this kernel is launched either then (the state is read while
  // TMEM is being allocated) or earlier (state_late: it is read after the grid wait)
  float sv[64];
  auto load_state = [&]() {
    if (tid < CH_EPI) {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 f = reinterpret_cast<const float4*>(Sg)[q];
        sv[4 * q] = f.x; sv[4 * q + 1] = f.y; sv[4 * q + 2] = f.z; sv[4 * q + 3] = f.w;
      }
    }
  };
  if (!p.state_late) load_state();
  // the local kernel's tiles and e^{G_C} (and the conv output V) from here on
  pdl_wait();
  // another slice follows: its local kernel may run beside this chain now (it writes the
  // other half of the workspace and waits for this grid before it completes)
  if (p.early_trigger) pdl_trigger();
  if (tid == CH_EPI)
    for (int i = 0; i < 2 && i < ns; ++i) {
      load_main(i);
      load_p(i);
    }
  if (p.state_late) load_state();
  for (int i = tid; i < ns; i += CH_THREADS) sEgc[i] = p.egc[u0 + i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;

  if (issuer_warp) {
    // ======================= issuer warp: the whole warp runs the loop and waits, one
    // elected lane issues the copies and MMAs (in chain order)
    const bool leader = elect_one();
    for (int nl = 0; nl < ns; ++nl) {
      const uint32_t buf = sb + (nl & 1) * CH_BUF;
      const uint32_t tmO = tmem + TM_O + 64 * (nl & 1);
      // U'^T = V^T T''^T of this chunk (T'' as hi + lo; M = d_v, N = K = 64 tokens).  TM_U
      // was last read by C2 of the previous chunk, which the previous C3 waited for.
      // (a wait that gives up makes every other wait of the CTA give up too)
      if (!__all_sync(0xffffffffu,
                      mbar_wait_or_abort((nl & 1) ? bar_ld1 : bar_ld0, (nl >> 1) & 1, sAbort))) {
        *sAbort = 1;
        break;
      }
      ld_chunk[nl & 1] = -1;
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int kb = k & 3;        // (T'' is lower triangular: see id_tri_kt)
          mma_bf16(tmem + TM_U + 16 * kb, sdesc_sw128(buf + CH_V + kb * 2048, 8 * KB, 1024),
                   sdesc_sw128(buf + U_T2 + (k < 4 ? 0 : 8 * KB) + kb * (2048 + 32), 16, 1024),
                   id_tri_kt(kb), k > 0);
        }
      }
      __syncwarp();
      // C1 once C0 is done: U^T += S0 (-W)^T (critical), then O^T = S0 Q~^T
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(bar_c0, nl & 1, sAbort))) {
        *sAbort = 1;
        break;
      }
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ta(tmem + TM_U, tmem + TM_S0 + 8 * k,
                      sdesc_sw128(buf + U_NW + k * 2048, 8 * KB, 1024), ID_SW, true);
        mma_commit(bar_u);
        // C0 waited for S of the previous chunk: the other buffer's tiles but P are free
        if (nl >= 1 && nl + 1 < ns) load_main(nl + 1);
      }
      __syncwarp();
      if (nl >= 1 && nl + 1 < ns) ld_chunk[(nl + 1) & 1] = nl + 1;
      // then O^T = S0 Q~^T, once the store warps have read this O buffer's tile of chunk nl - 2
      if (nl >= 2 && !__all_sync(0xffffffffu, mbar_wait_or_abort((nl & 1) ? bar_r1 : bar_r0,
                                                                  ((nl - 2) >> 1) & 1, sAbort))) {
        *sAbort = 1;
        break;
      }
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ta(tmO, tmem + TM_S0 + 8 * k,
                      sdesc_sw128(buf + U_QT + (k >> 2) * 8 * KB + (k & 3) * 32, 16, 1024),
                      ID_SQ, k > 0);
      }
      __syncwarp();
      // C3 once C2 is done: S += U^T K~ (Uh K~ + Ul K~; critical), then
      // O^T += U^T P^T (Uh Ph + Ul Ph + Uh Pl)
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(bar_c2, nl & 1, sAbort))) {
        *sAbort = 1;
        break;
      }
      tc_fence_after();
      if (leader) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ta(tmem + TM_S, tmem + (k < 4 ? TM_UH : TM_UL) + 8 * (k & 3),
                      sdesc_sw128(buf + U_KT + (k & 3) * 2048, 8 * KB, 1024), ID_UK, true);
        mma_commit(bar_s);
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu,
                      mbar_wait_or_abort((nl & 1) ? bar_p1 : bar_p0, (nl >> 1) & 1, sAbort))) {
        *sAbort = 1;
        break;
      }
      lp_chunk[nl & 1] = -1;
      // C2 waited for U^T, i.e. for every MMA before it, the previous output MMAs included:
      // the other buffer's P is free
      const bool refill_p = nl >= 1 && nl + 1 < ns;
      if (leader) {
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          const uint32_t ua = (k < 4 || k >= 8) ? TM_UH : TM_UL;
          const uint32_t pb = (k < 8) ? 0u : 8 * KB;
          const int kb = k & 3;        // (P is lower triangular: see id_tri_sq)
          mma_bf16_ta(tmO + 16 * kb, tmem + ua + 8 * kb,
                      sdesc_sw128(buf + U_P + pb + kb * (2048 + 32), 16, 1024), id_tri_sq(kb),
                      true);
        }
        mma_commit((nl & 1) ? bar_o1 : bar_o0);
        if (refill_p) load_p(nl + 1);
      }
      __syncwarp();
      if (refill_p) lp_chunk[(nl + 1) & 1] = nl + 1;
      // chunk nl's tiles in the workspace (and, with the conv fused, its V rows there) have
      // been copied in and are read no more: their L2 lines are dropped, not written back
      {
        const uint8_t* unit = p.units + (u0 + nl) * UNIT_BYTES;
        for (uint32_t off = (uint32_t)lane * 128u; off < UNIT_BYTES; off += 32u * 128u)
          l2_discard_line(unit + off);
        if (p.vbuf) {
          const int rows = min(C, p.T - (tbase + nl * C));   // (vbuf: not a packed batch)
          for (int i = lane; i < 2 * rows; i += 32)
            l2_discard_line(p.vbuf + ((size_t)bt * p.T + tbase + nl * C + (i >> 1)) * p.Hv * D +
                            h * D + 64 * (i & 1));
        }
      }
    }
  } else if (tid < CH_EPI) {
    // ======================= epilogue warps
    tmem_st32(tmem + lane_off + TM_S + 64 * hc, *reinterpret_cast<float(*)[32]>(&sv[0]));
    tmem_st32(tmem + lane_off + TM_S + 64 * hc + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
    tmem_wait_st();
    // in-call snapshots: bank rows of the next boundary inside this slice (loaded a step or
    // more ahead of its use) and of the boundary at the slice end, -1 for none
    const int32_t* snap_row = p.se_c > 0 ? p.snap_slots + (size_t)b * p.n_snap - 1 : nullptr;
    int snap_nb = p.se_c > 0 ? (p.n0 / p.se_c + 1) * p.se_c : 0x7fffffff;   // chunk index
    int snap_next = snap_nb < p.n0 + ns ? snap_row[snap_nb / p.se_c] : -1;
    const int n_end = p.n0 + ns;
    const int snap_end =
        (p.se_c > 0 && n_end % p.se_c == 0 && n_end * C <= p.T) ? snap_row[n_end / p.se_c] : -1;
    if (tid == 0 && (snap_next >= p.n_snap_slots || snap_end >= p.n_snap_slots))
      atomicOr(&g_err_tc, kErrIndex);
    bool ok = true;
    for (int nl = 0; nl < ns && ok; ++nl) {
      // ---- C0: S -> S0 (bf16, packed into TMEM as the A operand);  S <- e^{G_C} S
      // (every wait is decided warp-uniformly: the warp syncs below must not split)
      if (nl > 0 && !__all_sync(0xffffffffu, mbar_wait_or_abort(bar_s, (nl - 1) & 1, sAbort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const float egc = sEgc[nl];
        const uint32_t ta = tmem + lane_off + TM_S + 64 * hc;
        float v[64];
        tmem_ld32(ta, *reinterpret_cast<float(*)[32]>(&v[0]));
        tmem_ld32(ta + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
        tmem_wait_ld();
        // a snapshot boundary: this warp's 32 rows x 64 columns of the entering state, staged
        // as two 128-byte-swizzled 32 x 32 blocks in the other tile buffer outside its P
        // (every other tile of it was read by MMAs that S's completion covers; the next copy
        // into it waits for C0) -> two TMA stores, whose reads end before C0 is signalled
        const bool snap_here = p.n0 + nl == snap_nb;
        if (snap_here) {
          if (snap_next >= 0 && snap_next < p.n_snap_slots) {
            const uint32_t stg = sb + (((nl & 1) ^ 1) * CH_BUF) +
                                 (warp < 4 ? warp * 8 * KB : U_KT + (warp - 4) * 8 * KB);
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                st_shared_v4(sw128(stg + g * 4 * KB, lane, c), __float_as_uint(v[32 * g + 4 * c]),
                             __float_as_uint(v[32 * g + 4 * c + 1]),
                             __float_as_uint(v[32 * g + 4 * c + 2]),
                             __float_as_uint(v[32 * g + 4 * c + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int srow = ((snap_next * p.Hv + h) * D) + 32 * gw;
#pragma unroll
              for (int g = 0; g < 2; ++g)
                tma_store_3d(&tm_snap, stg + g * 4 * KB, 64 * hc + 32 * g, srow, 0);
              tma_store_commit();
            }
          }
          snap_nb += p.se_c;
          snap_next = snap_nb < n_end ? snap_row[snap_nb / p.se_c] : -1;
          if (tid == 0 && snap_next >= p.n_snap_slots) atomicOr(&g_err_tc, kErrIndex);
        }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t pk[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            pk[jj] = pack_bf16(v[32 * g + 2 * jj], v[32 * g + 2 * jj + 1]);
          tmem_st16(tmem + lane_off + TM_S0 + 32 * hc + 16 * g, pk);
        }
        tmem_wait_st();
        if (snap_here && lane == 0) tma_store_wait_read();
        // S0 is what the next MMAs read: signal it now, and rescale S (which only the S
        // update, issued after C2, accumulates into) while U^T += S0 (-W)^T runs
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_c0);
#pragma unroll
        for (int jj = 0; jj < 64; ++jj) v[jj] *= egc;
        tmem_st32(ta, *reinterpret_cast<float(*)[32]>(&v[0]));
        tmem_st32(ta + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
        tmem_wait_st();
      }
      // ---- C2: U^T (fp32) -> bf16 hi / lo, packed into TMEM as A operands
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(bar_u, nl & 1, sAbort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        float v[32];
        uint32_t hu[16], lu[16];
        tmem_ld32(tmem + lane_off + TM_U + 32 * hc, v);
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) pack_hilo(v[2 * jj], v[2 * jj + 1], hu[jj], lu[jj]);
        tmem_st16(tmem + lane_off + TM_UH + 16 * hc, hu);
        tmem_st16(tmem + lane_off + TM_UL + 16 * hc, lu);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_c2);
    }
    if (ok && ns > 0) {
      // the leaving state, as soon as the last S update is done (the last output MMAs may
      // still run): TMEM -> this warp's 32 rows x 64 columns, staged as two 128-byte-swizzled
      // 32 x 32 blocks in the tile buffer the last chunk does not use (its readers are done)
      // -> two TMA tensor stores (whole rows per request)
      if (__all_sync(0xffffffffu, mbar_wait_or_abort(bar_s, (ns - 1) & 1, sAbort))) {
        tc_fence_after();
        const uint32_t stg = sb + ((((ns - 1) & 1) ^ 1) * CH_BUF) + warp * 8 * KB;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float v[32];
          tmem_ld32(tmem + lane_off + TM_S + 64 * hc + 32 * g, v);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(sw128(stg + g * 4 * KB, lane, c), __float_as_uint(v[4 * c]),
                         __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                         __float_as_uint(v[4 * c + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int srow = ((slot * p.Hv + h) * D) + 32 * gw;
#pragma unroll
          for (int g = 0; g < 2; ++g) tma_store_3d(&tm_s, stg + g * 4 * KB, 64 * hc + 32 * g, srow, 0);
          // the slice ends on a snapshot boundary: the same rows to the bank
          if (snap_end >= 0 && snap_end < p.n_snap_slots) {
            const int brow = ((snap_end * p.Hv + h) * D) + 32 * gw;
#pragma unroll
            for (int g = 0; g < 2; ++g)
              tma_store_3d(&tm_snap, stg + g * 4 * KB, 64 * hc + 32 * g, brow, 0);
          }
          tma_store_commit();
        }
      } else {
        ok = false;
      }
    }
    // the state stores must have read their staging before the CTA exits (their writes
    // complete with the grid)
    if (lane == 0) tma_store_wait_read();
    if (!ok) *sAbort = 1;
  } else {
    // ======================= store warps: the output tile of each chunk (O^T in TMEM: lane =
    // d_v index, column = token).  Warp w reads TMEM lane quarter w % 4, i.e. 32 d_v rows x 64
    // tokens, tells the issuer that the buffer is free, optionally applies the gated RMS norm,
    // then sends the rows through its staging block [token][32 d_v] (2 KB with the norm, whose
    // gate tiles take the rest of the area, else 4 KB) with one TMA store per pass (the store
    // clips the rows past the sequence end).  Lane 0 issues the copies and is the one that
    // waits for their reads.
    const int sw = warp - CH_STORE;
    const int q = warp & 3;
    const uint32_t lq = static_cast<uint32_t>(q * 32) << 16;
    Tout* stg = reinterpret_cast<Tout*>(sm + CH_OUT + sw * (p.gate ? 2 : 4) * KB);
    // gated norm: this warp's gate tile z [64 tokens][32 d_v] (bf16, one TMA copy per chunk,
    // a chunk ahead), the four warps' per-token partial sums of squares, this lane's weight
    const uint32_t zst = sb + CH_Z + sw * 4 * KB;
    const __nv_bfloat16* zs = reinterpret_cast<const __nv_bfloat16*>(sm + CH_Z + sw * 4 * KB);
    float* sqp = reinterpret_cast<float*>(sm + CH_SQ);
    float* rinv = reinterpret_cast<float*>(sm + CH_RI) + sw * 64;
    const uint32_t bar_zw = smem_addr(&barmem[13 + sw]);
    const float wgt = p.gate ? p.gw[32 * q + lane] : 0.f;
    int z_chunk = -1;                                  // gate copy in flight, or -1
    auto load_z = [&](int nl) {
      if (lane == 0) {
        fence_proxy_async_smem();                      // after this warp's reads of the tile
        mbar_arrive_expect_tx(bar_zw, 4 * KB);
        tma_load_3d(zst, &tm_z, h * D + 32 * q, tbase + nl * C, bt, bar_zw);
        // and the tile after it into L2, so that its own copy is an L2 hit
        if (nl + 1 < ns) tma_prefetch_l2_3d(&tm_z, h * D + 32 * q, tbase + (nl + 1) * C, bt);
      }
      z_chunk = nl;
    };
    if (p.gate && ns > 0) load_z(0);
    // Conv-state rows of this CTA's channels (the conv fused into the local kernels): its v
    // channels and, for the first value head of a key head, that key head's q and k channels;
    // word k of the 3 rows x those channels -> (row j, channel ch)
    const int n_words = (h % (p.Hv / p.Hk) == 0) ? 48 + 96 : 48;
    auto conv_word = [&](int k, int& j, int& ch) {
      if (k < 48) {
        j = k >> 4;
        ch = 2 * p.Hk * D + h * D + 8 * (k & 15);
      } else {
        const int cc = (k - 48) & 31;
        j = (k - 48) >> 5;
        ch = ((cc >> 4) ? p.Hk * D : 0) + (h / (p.Hv / p.Hk)) * D + 8 * (cc & 15);
      }
    };
    // the last slice: the call's conv tail (left by the conv and local kernels, complete since
    // the grid wait) into the conv state
    if (p.cs_out) {
      for (int k = tid - CH_STORE * 32; k < n_words; k += 128) {
        int j, ch;
        conv_word(k, j, ch);
        if (!in_bounds(&g_err_tc, b < p.Bm && ch + 8 <= p.Cc && j < FC_H)) continue;
        *reinterpret_cast<uint4*>(p.cs_out + ((size_t)slot * FC_H + j) * p.Cc + ch) =
            __ldcg(reinterpret_cast<const uint4*>(p.tail + ((size_t)b * FC_H + j) * p.Cc + ch));
      }
    }
    // in-call snapshots of the conv state at the boundaries this slice ends a chunk on: the
    // W-1 inputs before the boundary token (rows of x) into conv bank row snap_slots[b][j]
    // (an out-of-range bank row is skipped; the state snapshot reports it)
    if (p.cbank) {
      for (int nb = (p.n0 / p.se_c + 1) * p.se_c; nb <= p.n0 + ns && nb * C <= p.T;
           nb += p.se_c) {
        const int bs = p.snap_slots[(size_t)b * p.n_snap + nb / p.se_c - 1];
        if (bs < 0 || bs >= p.n_snap_slots) continue;
        for (int k = tid - CH_STORE * 32; k < n_words; k += 128) {
          int j, ch;
          conv_word(k, j, ch);
          const size_t t = (size_t)b * p.T + (size_t)nb * C - FC_H + j;
          if (!in_bounds(&g_err_tc, b < p.Bm && nb * C <= p.T && ch + 8 <= p.Cc)) continue;
          *reinterpret_cast<uint4*>(p.cbank + ((size_t)bs * FC_H + j) * p.Cc + ch) =
              __ldg(reinterpret_cast<const uint4*>(p.x + t * p.Cc + ch));
        }
      }
    }
    bool ok = true;
    for (int nl = 0; nl < ns; ++nl) {
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort((nl & 1) ? bar_o1 : bar_o0,
                                                      (nl >> 1) & 1, sAbort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[64];
      tmem_ld32(tmem + lq + TM_O + 64 * (nl & 1), *reinterpret_cast<float(*)[32]>(&v[0]));
      tmem_ld32(tmem + lq + TM_O + 64 * (nl & 1) + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive((nl & 1) ? bar_r1 : bar_r0);
      if (p.gate) {
        // per-token sums of squares over this warp's 32 rows: a transposing butterfly leaves
        // lane l with the sums of tokens 2l and 2l + 1; the four warps meet at a barrier
        float s2[32];
        {
          const bool up = lane & 16;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float lo = v[i] * v[i], hi = v[i + 32] * v[i + 32];
            s2[i] = (up ? hi : lo) + __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16);
          }
        }
        butterfly_half<8, 32>(s2, lane);
        butterfly_half<4, 16>(s2, lane);
        butterfly_half<2, 8>(s2, lane);
        butterfly_half<1, 4>(s2, lane);
        float* sqb = sqp + (nl & 1) * 256;
        *reinterpret_cast<float2*>(sqb + q * 64 + 2 * lane) = make_float2(s2[0], s2[1]);
        const uint32_t bsq = smem_addr(&barmem[17 + (nl & 1)]);
        mbar_arrive(bsq);
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(bsq, (nl >> 1) & 1, sAbort) &&
                                         mbar_wait_or_abort(bar_zw, nl & 1, sAbort))) {
          ok = false;
          break;
        }
        z_chunk = -1;
        float tot0 = 0.f, tot1 = 0.f;
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          const float2 pp = *reinterpret_cast<const float2*>(sqb + w4 * 64 + 2 * lane);
          tot0 += pp.x;
          tot1 += pp.y;
        }
        // this lane's two tokens' 1 / rms, then all 64 back as broadcast vector loads
        *reinterpret_cast<float2*>(rinv + 2 * lane) =
            make_float2(rsqrtf(tot0 * (1.0f / D) + p.geps), rsqrtf(tot1 * (1.0f / D) + p.geps));
        __syncwarp();
#pragma unroll
        for (int t4 = 0; t4 < 16; ++t4) {
          const float4 r4 = reinterpret_cast<const float4*>(rinv)[t4];
          const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int t = 4 * t4 + u;
            const float zt = __bfloat162float(zs[t * 32 + lane]);
            v[t] = wgt * (v[t] * rr[u]) * silu_out<Tout>(zt);
          }
        }
        __syncwarp();
        if (nl + 1 < ns) load_z(nl + 1);
      }
      const int tok0 = tbase + nl * C;
      if (p.cu && nl == ns - 1 && last_tok < C) {
        // the ragged last chunk of a packed sequence: the next sequence's tokens follow it,
        // so only this sequence's rows are written, with plain stores (a warp's 32 lanes are
        // 32 consecutive channels of a token row)
        Tout* o = reinterpret_cast<Tout*>(p.out) + (size_t)tok0 * p.Hv * D + h * D + 32 * q +
                  lane;
#pragma unroll
        for (int t = 0; t < 64; ++t)
          if (t < last_tok) o[(size_t)t * p.Hv * D] = from_float<Tout>(v[t]);
      } else if (p.gate)
        store_tile_passes<Tout, (int)(2 * KB / (32 * sizeof(Tout)))>(&tm_o, stg, v, lane,
                                                                     h * D + 32 * q, tok0, bt);
      else
        store_tile_passes<Tout, (int)(4 * KB / (32 * sizeof(Tout)))>(&tm_o, stg, v, lane,
                                                                     h * D + 32 * q, tok0, bt);
    }
    // everything this kernel writes has been issued: a kernel after it may start its set-up
    pdl_trigger();
    if (lane == 0) {
      tma_store_wait_read();
      // a gate copy issued ahead of a chunk that an abort left unprocessed must land first
      if (z_chunk >= 0) mbar_wait_bounded(bar_zw, z_chunk & 1, 1u << 16);
    }
    if (!ok) *sAbort = 1;
  }
  if (tid == CH_EPI) {
    // nothing may still write this CTA's shared memory or TMEM when it exits: first every
    // MMA issued (after which every tile is free), then every copy issued
    mma_commit(bar_fin);
    mbar_wait_bounded(bar_fin, 0, 1u << 16);
    for (int i = 0; i < 2; ++i) {
      if (ld_chunk[i] >= 0) mbar_wait_bounded(i ? bar_ld1 : bar_ld0, (ld_chunk[i] >> 1) & 1, 1u << 16);
      if (lp_chunk[i] >= 0) mbar_wait_bounded(i ? bar_p1 : bar_p0, (lp_chunk[i] >> 1) & 1, 1u << 16);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *sAbort) atomicOr(&g_err_tc, kErrTimeout);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, CH_TMEM);
  }
}

// ======================================================================= self-test
// One CTA waits on an mbarrier that nothing arrives at, with nothing in flight (no copy, no
// MMA, no TMEM), through the same bounded wait, abort flag and error word as the prefill
// kernels: each thread gives up after max_iters polls (or once another has raised the
// flag), and the CTA records kErrTimeout, which gdn_get_device_error then reports as
// GDN_ERR_DEVICE_TIMEOUT.
__global__ void __launch_bounds__(128, 1) gdn_selftest_wait_kernel(uint32_t max_iters) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (!mbar_wait_or_abort(b, 0, &abort_flag, max_iters)) abort_flag = 1;
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) atomicOr(&g_err_tc, kErrTimeout);
}

// ======================================================================= host side

// One slice's workspace: its units' tiles, then e^{G_C} per unit (256-byte aligned size).
size_t scratch_half_bytes(size_t units) {
  return units * UNIT_BYTES + ((units * sizeof(float) + 255) & ~(size_t)255);
}

// Chunks per slice: as many as keep one slice's tiles within SLICE_BUDGET bytes.
int slice_chunks(int B, int Hv, int nch) {
  const size_t per_chunk = (size_t)B * Hv * UNIT_BYTES;
  size_t ns = SLICE_BUDGET / per_chunk;
  if (ns < 1) ns = 1;
  if (ns > (size_t)MAX_SLICE) ns = MAX_SLICE;
  if (ns > (size_t)nch) ns = nch;
  return (int)ns;
}

template <typename Tout>
cudaError_t launch_tc_t(const GdnLayerArgs& L, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo, ms;
  // tokens per output store: a 2 KB staging block with the gated norm, else 4 KB
  const int out_rows = (int)((L.gate ? 2 : 4) * KB / (32 * sizeof(Tout)));
  // a packed batch has all its tokens on one axis: batch extent 1 in the tensor maps
  const int MB = L.cu ? 1 : L.B;
  // the q / k conv fused into the local kernel: the K and Q maps are one map over the pre-conv
  // input x (the k channels at offset Hk d), the V map one over the conv kernel's output
  const bool fuse = L.fuse != 0;
  const bool maps_in =
      (fuse ? gdn_make_map(&mq, L.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.C_conv, L.T, MB,
                           L.C_conv, 64, 64, true)
            : (gdn_make_map(&mq, L.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hk * D, L.T, MB,
                            L.q_tok_stride, 64, 64, true) &&
               gdn_make_map(&mk, L.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hk * D, L.T, MB,
                            L.k_tok_stride, 64, 64, true))) &&
      gdn_make_map(&mv, L.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hv * D, L.T, MB,
                   L.v_tok_stride, 64, 64, true);
  if (fuse) mk = mq;
  const bool ok =
      maps_in &&
      gdn_make_map(&mo, L.out,
               sizeof(Tout) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
               (int)sizeof(Tout), L.Hv * D, L.T, MB, (long long)L.Hv * D, 32, out_rows, false) &&
      // the state as rows of 128 fp32: box = 32 columns x 32 rows, 128-byte swizzle
      gdn_make_map(&ms, L.state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D,
                   L.num_slots * L.Hv * D, 1, D, 32, 32, true);
  if (!ok) return cudaErrorInvalidValue;
  // the output gate z [B][T][Hv d] bf16: box = 32 channels x 64 tokens (the V map stands in
  // when there is no gate)
  CUtensorMap mz = mv;
  if (L.gate && !gdn_make_map(&mz, L.gate_z, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hv * D, L.T,
                              MB, (long long)L.Hv * D, 32, 64, false))
    return cudaErrorInvalidValue;
  // the snapshot bank, the same way (the state map stands in when nothing is recorded)
  CUtensorMap msn = ms;
  const bool snaps = L.snap_every > 0 && L.n_snap > 0;
  if (snaps) {
    if ((long long)L.num_snap_slots * L.Hv * D > 0x7fffffffLL ||
        !gdn_make_map(&msn, L.snap_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D,
                      L.num_snap_slots * L.Hv * D, 1, D, 32, 32, true))
      return cudaErrorInvalidValue;
  }
  static unsigned done_l = 0, done_c = 0, done_lc = 0;
  cudaError_t e = set_smem_once(gdn_chunk_local_kernel<__nv_bfloat16>, (int)L_SMEM, &done_l);
  if (e != cudaSuccess) return e;
  e = set_carveout_once(gdn_chunk_local_kernel<__nv_bfloat16>, 100, &done_lc);   // 3 CTAs per SM
  if (e != cudaSuccess) return e;
  e = set_smem_once(gdn_chunk_chain_kernel<Tout>, (int)CH_SMEM, &done_c);
  if (e != cudaSuccess) return e;
  // chunks per sequence, or of a packed batch (its chunk table's length, an upper bound)
  const int nch = L.cu ? L.n_chunks : (L.T + C - 1) / C;
  const int ns_max = slice_chunks(MB, L.Hv, nch);
  const size_t units = (size_t)ns_max * MB * L.Hv;
  if (!L.scratch || L.scratch_bytes < gdn_prefill_tc_scratch_bytes(MB, nch * C, L.Hv))
    return cudaErrorInvalidValue;
  if (fuse && (!L.tail || (L.chained && !L.prev_tail) || (!L.chained && !L.conv_state)))
    return cudaErrorInvalidValue;
  const int nslices = (nch + ns_max - 1) / ns_max;
  const size_t half_bytes = scratch_half_bytes(units);
  TcParams p;
  p.T = L.T; p.Hk = L.Hk; p.Hv = L.Hv; p.num_slots = L.num_slots; p.l2norm = L.l2norm;
  p.gates_pre = L.gates_pre; p.eps = L.eps; p.scale = L.scale; p.a = L.a; p.b = L.b;
  p.A_log = L.A_log; p.dt_bias = L.dt_bias; p.state = L.state; p.slots = L.slots;
  p.se_c = snaps ? L.snap_every / C : 0;
  p.n_snap = snaps ? L.n_snap : 0;
  p.n_snap_slots = snaps ? L.num_snap_slots : 0;
  p.snap_slots = snaps ? L.snap_slots : nullptr;
  p.cbank = (snaps && L.fuse) ? static_cast<__nv_bfloat16*>(L.snap_conv_state) : nullptr;
  p.vbuf = L.fuse ? static_cast<const __nv_bfloat16*>(L.v) : nullptr;
  p.gate = L.gate;
  p.gw = L.gate_w;
  p.geps = L.gate_eps;
  p.cu = L.cu;
  p.ccs = L.ccs;
  p.ctab = static_cast<const int4*>(L.ctab);
  p.out = L.out;
  p.fuse = fuse;
  p.Bm = MB;
  p.Cc = L.C_conv;
  p.silu = L.silu;
  p.x = static_cast<const __nv_bfloat16*>(L.x);
  p.cw = static_cast<const __nv_bfloat16*>(L.conv_w);
  p.cb = static_cast<const __nv_bfloat16*>(L.conv_b);
  p.halo_by_slot = !L.chained;
  p.halo = static_cast<const __nv_bfloat16*>(L.chained ? L.prev_tail : L.conv_state);
  p.tail = static_cast<__nv_bfloat16*>(L.tail);
  // a call that continues the one before it on the stream: its first local kernel starts
  // beside that call's last chain (which released it right after its own grid wait), reads
  // only this call's inputs and the previous conv tail before its grid wait, and waits for
  // that chain at its end like a later slice's local kernel
  const bool chained = L.chained != 0 && (fuse || L.W == 0);
  if (fuse) {
    // the v channels' conv first: it reads only this call's input and the halo, writes V (into
    // the workspace) and the v part of the conv tail, and lets the local kernel start at once;
    // its last block waits for the kernel before it, so that the call's kernels complete in
    // stream order behind it
    e = gdn_launch_conv(L.B, L.T, L.C_conv, L.W, 1, L.x, L.C_conv, L.conv_w, L.conv_b,
                        L.conv_state, L.num_slots, L.slots, L.silu, const_cast<void*>(L.v),
                        (long long)L.Hv * D, stream, 2 * L.Hk * D, -1, chained, true, p.halo,
                        p.halo_by_slot, L.tail, 2 * L.Hk * D);
    if (e != cudaSuccess) return e;
  }
  for (int si = 0; si < nslices; ++si) {
    const int n0 = si * ns_max;
    p.n0 = n0;
    p.ns = nch - n0 < ns_max ? nch - n0 : ns_max;
    // workspace half (si & 1) when the call has several slices
    p.units = static_cast<uint8_t*>(L.scratch) +
              (nslices > 1 ? (size_t)(si & 1) * half_bytes : 0);
    p.egc = reinterpret_cast<float*>(p.units + units * UNIT_BYTES);
    p.n_units = units;
    // (with the conv fused, every local kernel runs behind a kernel it does not depend on --
    // the v conv or the previous chain -- and waits for it at its end only; the first one of
    // an ordinary call releases its chain at once, whose set-up then reads the state early:
    // everything before this call had completed when the v conv started)
    p.late_wait = si > 0 || chained || fuse;
    p.trigger_first = fuse && si == 0 && !chained;
    p.trigger_end = p.late_wait && !p.trigger_first;
    p.state_late = p.trigger_end;
    // (every chain releases the kernel after it early: the next slice's local kernel, or the
    // next call's first kernel, each of which waits for the chain before reading what it wrote)
    p.early_trigger = 1;
    p.cs_out = (fuse && si + 1 == nslices) ? static_cast<__nv_bfloat16*>(L.conv_state) : nullptr;
    // (the first slice's local kernel reads the caller's gate inputs, and a packed batch's
    // chunk table, before its grid wait: it may start early only behind this call's own conv
    // kernels, which began after everything earlier had completed, or as a continuing call)
    e = launch_pdl(n0 > 0 || chained || L.W > 0, gdn_chunk_local_kernel<__nv_bfloat16>,
                   dim3((unsigned)p.ns, (unsigned)L.Hv, (unsigned)MB), dim3(LGT), L_SMEM, stream,
                   mq, mk, p);
    if (e != cudaSuccess) return e;
    if (si == 0 && L.vconv_pending) {
      // the value channels' conv, beside the first chunk-local kernel (which releases it right
      // after its own grid wait and reads no value channel); its last block waits for that
      // kernel, so the chain after it may rely on both.  It writes V into the conv output
      // (whose base L.q is) and the value channels' conv state.
      e = gdn_launch_conv(L.B, L.T, L.C_conv, L.W, 1, L.x, L.C_conv, L.conv_w, L.conv_b,
                          L.conv_state, L.num_slots, L.slots, L.silu, const_cast<void*>(L.q),
                          L.C_conv, stream, 2 * L.Hk * D, -1, true, true);
      if (e != cudaSuccess) return e;
    }
    e = launch_pdl(true, gdn_chunk_chain_kernel<Tout>, dim3((unsigned)(L.B * L.Hv)), dim3(CH_THREADS),
                   CH_SMEM, stream, mv, mo, ms, msn, mz, p);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t gdn_prefill_tc_scratch_bytes(int B, int T, int Hv) {
  const int nch = (T + C - 1) / C;
  if (B <= 0 || nch <= 0 || Hv <= 0) return 0;
  const int ns = slice_chunks(B, Hv, nch);
  const size_t half = scratch_half_bytes((size_t)ns * B * Hv);
  return ns < nch ? 2 * half : half;        // two halves when the call has several slices
}

cudaError_t gdn_launch_selftest_wait(uint32_t max_iters, cudaStream_t stream) {
  gdn_selftest_wait_kernel<<<1, 128, 0, stream>>>(max_iters);
  return cudaGetLastError();
}

cudaError_t gdn_launch_prefill_tc(const GdnLayerArgs& L, cudaStream_t stream) {
  if (L.B == 0 || L.T == 0) return cudaSuccess;
  if (!L.in_bf16) return cudaErrorInvalidValue;
  return L.out_bf16 ? launch_tc_t<__nv_bfloat16>(L, stream) : launch_tc_t<float>(L, stream);
}
