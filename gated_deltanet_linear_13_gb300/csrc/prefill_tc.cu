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
//   G = [K;Q] K^T (one M=128 MMA)  ->  A, P (with 1/||k||, scale/||q||, decays)
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
// Pipeline: one CTA per (sequence, value head), two warp groups (384 threads).
//   local group (warps 0-7, 256 threads), chunk m: norms, gates, G = [K;Q]K^T, A and P, Q~ (in place),
//     the direct solve, T'/T'', W^T and U'^T (MMA), -W^T.  Nothing here depends on the state.
//   chain group (warps 8-11, 128 threads), chunk n = m - 1: S0 = bf16(S) into TMEM, S <- e^{G_C} S,
//     U^T += S0 (-W)^T and O^T = S0 Q~^T, K~, U^T -> bf16 hi/lo in TMEM,
//     O^T += U^T P^T and S += U^T K~, then the output tile of chunk n-1 to HBM (TMA store).
// The groups hand chunks over through mbarriers (ready / free, one per buffer parity), so the
// state-independent work of chunk n+1 overlaps the state chain of chunk n.  Each group's
// thread 0 issues its own MMAs; S0 and U^T are A operands read straight from TMEM.
// TMEM (512 columns): S 128 | U^T x2 | O^T x2 | G / W^T | S0 (packed bf16) / U^T hi,lo.
// Every mbarrier wait is bounded: on timeout the CTA records GDN_ERR_DEVICE_TIMEOUT, both
// groups leave their loops, pending MMAs and copies are waited for (bounded), TMEM is freed.
#include "common.cuh"
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

constexpr int C = kChunk, D = kHeadDim, THREADS = 384, LGT = 256, CGT = 128;
constexpr uint32_t KB = 1024;
// ---- shared memory (byte offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_KQ0 = 0, OFF_KQ1 = 32 * KB;  // per 64-column block kb: K rows, then Q rows
constexpr uint32_t KQ_KB = 16 * KB, KQ_Q = 8 * KB;
constexpr uint32_t OFF_V = 64 * KB;                  // V [2][64 rows][128 B] (single buffer)
constexpr uint32_t OFF_P0 = 80 * KB, OFF_P1 = 96 * KB;     // P hi at +0, lo at +8 KB
constexpr uint32_t OFF_NW0 = 112 * KB, OFF_NW1 = 128 * KB; // -W^T [128 rows d_k][128 B]
constexpr uint32_t OFF_KT = 144 * KB;                // K~ [2][64][128 B]
constexpr uint32_t OFF_SOLVE = 160 * KB;             // A | T fp32 [64][64]; then T' / T'' tiles
constexpr uint32_t OFF_T1H = OFF_SOLVE, OFF_T1L = OFF_SOLVE + 8 * KB;
constexpr uint32_t OFF_T2H = OFF_SOLVE + 16 * KB, OFF_T2L = OFF_SOLVE + 24 * KB;
constexpr uint32_t OFF_OUT = 192 * KB;               // output staging, 16 KB
constexpr uint32_t OFF_MISC = 208 * KB;              // per-chunk factors x2, solve scratch, bars
constexpr uint32_t MISC_F = 0, F_STRIDE = 2048;      // 8 arrays of 64 floats per parity
constexpr uint32_t MISC_X = 4096;                    // 3 x 256 floats
constexpr uint32_t MISC_BAR = 7168;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 8 * KB + KB;   // + alignment slack
constexpr int LA = 64;                               // row stride (floats) of the solve matrices

// ---- TMEM columns
constexpr uint32_t TM_S = 0, TM_U = 128, TM_O = 256, TM_GW = 384, TM_SU = 448, TM_COLS = 512;

constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);   // [K;Q] K^T
constexpr uint32_t ID_KT = idesc_bf16(128, 64, true, false);   // K^T T'^T, V^T T''^T
constexpr uint32_t ID_SW = idesc_bf16(128, 64, false, true);   // S0 (-W)^T
constexpr uint32_t ID_SQ = idesc_bf16(128, 64, false, false);  // S0 Q~^T, U^T P^T
constexpr uint32_t ID_UK = idesc_bf16(128, 128, false, true);  // U^T K~

constexpr float LOG2E = 1.4426950408889634f;

struct TcParams {
  int T, Hk, Hv, num_slots, l2norm, gates_pre;
  float eps, scale;
  const void* a;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  float* state;
  const int32_t* slots;
};

// Per-chunk factor arrays (one set per buffer parity).
struct Factors {
  float* gl2;   // G_r * log2(e)
  float* beta;
  float* nk;    // 1 / ||k_r||
  float* nq;    // scale / ||q_r||
  float* eG;    // e^{G_r}
  float* dK;    // e^{G_C - G_r}
  float* ra;    // raw gate inputs a, b of the chunk (parked one chunk ahead)
  float* rb;
};

__device__ __forceinline__ Factors factors_at(uint8_t* misc, int par) {
  float* f = reinterpret_cast<float*>(misc + MISC_F + par * F_STRIDE);
  return Factors{f, f + 64, f + 128, f + 192, f + 256, f + 320, f + 384, f + 448};
}

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

// T = (I + A)^{-1} for the strictly lower 64 x 64 matrix A (fp32, row stride LA), by blocked
// forward substitution over 16 x 16 blocks, on the 256 threads of the local group (named
// barrier 1).  Warps 0-3 invert one diagonal block each (lane = column; right-looking: once
// t_s is final, every later row r subtracts A_rs t_s) while the other threads zero the
// strictly upper blocks; then the off-diagonal blocks by distance from the diagonal,
//   X_ij = sum_{k=j}^{i-1} A_ik T_kj,   T_ij = -T_ii X_ij,
// one block entry per thread, with every operand loaded before the multiply-adds.
__device__ __forceinline__ void solve_unit_lower(const float* As, float* Ts, float* X, int lt) {
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
  named_bar_sync(1, LGT);
  const int rr = lt >> 4, cc = lt & 15;
#pragma unroll
  for (int dist = 1; dist <= 3; ++dist) {
#pragma unroll
    for (int q = 0; q < 4 - dist; ++q) {
      const int i = dist + q, j = q;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = j; k < i; ++k) {
        float av[16], tv[16];
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const float4 x = *reinterpret_cast<const float4*>(As + (16 * i + rr) * LA + 16 * k + 4 * m4);
          av[4 * m4] = x.x; av[4 * m4 + 1] = x.y; av[4 * m4 + 2] = x.z; av[4 * m4 + 3] = x.w;
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) tv[m] = Ts[(16 * k + m) * LA + 16 * j + cc];
#pragma unroll
        for (int m = 0; m < 16; ++m) acc[m & 3] = fmaf(av[m], tv[m], acc[m & 3]);
      }
      X[q * 256 + lt] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    named_bar_sync(1, LGT);
#pragma unroll
    for (int q = 0; q < 4 - dist; ++q) {
      const int i = dist + q, j = q;
      float tv[16], xv[16];
#pragma unroll
      for (int m4 = 0; m4 < 4; ++m4) {
        const float4 x = *reinterpret_cast<const float4*>(Ts + (16 * i + rr) * LA + 16 * i + 4 * m4);
        tv[4 * m4] = x.x; tv[4 * m4 + 1] = x.y; tv[4 * m4 + 2] = x.z; tv[4 * m4 + 3] = x.w;
      }
#pragma unroll
      for (int m = 0; m < 16; ++m) xv[m] = X[q * 256 + m * 16 + cc];
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 16; ++m) acc[m & 3] = fmaf(tv[m], xv[m], acc[m & 3]);
      Ts[(16 * i + rr) * LA + 16 * j + cc] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
    named_bar_sync(1, LGT);
  }
}

struct Bars {
  uint32_t kq[2], v, ready[2], fr[2], mma_l, mma_c;
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(THREADS, 1)
    gdn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_o, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed by offsetting the shared array itself so that every
  // pointer derived from it stays in the shared state space
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv;
  const int kh = h / (p.Hv / p.Hk);

  const int slot = p.slots ? p.slots[b] : b;
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (tid == 0) atomicOr(&g_err_tc, kErrIndex);
    return;
  }

  uint8_t* misc = sm + OFF_MISC;
  float* sX = reinterpret_cast<float*>(misc + MISC_X);
  uint64_t* barmem = reinterpret_cast<uint64_t*>(misc + MISC_BAR);
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(misc + MISC_BAR + 80);
  volatile int* sAbort = reinterpret_cast<volatile int*>(misc + MISC_BAR + 84);   // any thread
  volatile int* sAbortL = reinterpret_cast<volatile int*>(misc + MISC_BAR + 88);  // local group
  volatile int* sAbortC = reinterpret_cast<volatile int*>(misc + MISC_BAR + 92);  // chain group
  Bars bars;
  bars.kq[0] = smem_addr(&barmem[0]);
  bars.kq[1] = smem_addr(&barmem[1]);
  bars.v = smem_addr(&barmem[2]);
  bars.ready[0] = smem_addr(&barmem[3]);
  bars.ready[1] = smem_addr(&barmem[4]);
  bars.fr[0] = smem_addr(&barmem[5]);
  bars.fr[1] = smem_addr(&barmem[6]);
  bars.mma_l = smem_addr(&barmem[7]);
  bars.mma_c = smem_addr(&barmem[8]);

  if (tid == 0) {
    mbar_init(bars.kq[0], 1);
    mbar_init(bars.kq[1], 1);
    mbar_init(bars.v, 1);
    mbar_init(bars.ready[0], LGT);
    mbar_init(bars.ready[1], LGT);
    mbar_init(bars.fr[0], CGT);
    mbar_init(bars.fr[1], CGT);
    mbar_init(bars.mma_l, 1);
    mbar_init(bars.mma_c, 1);
    *sAbort = 0;
    *sAbortL = 0;
    *sAbortC = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(sTmem), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const int nchunks = (p.T + C - 1) / C;
  const int gw = warp & 3;                                 // TMEM lane quarter of this warp
  const uint32_t lane_off = static_cast<uint32_t>(gw * 32) << 16;
  const int row = 32 * gw + lane;                          // TMEM lane owned by this thread
  bool pend_mma = false;                                   // own group's MMA in flight
  uint32_t mma_phase = 0;

  if (tid < LGT) {
    // ======================================================== local group (warps 0-7)
    const int lt = tid;
    const int hcol = warp >> 2;                            // column half of this warp
    auto fail = [&]() { *sAbort = 1; *sAbortL = 1; };
    auto load_v = [&](int m) {
      mbar_arrive_expect_tx(bars.v, 16 * KB);
      tma_load_3d(sb + OFF_V, &tm_v, h * D, m * C, b, bars.v);
      tma_load_3d(sb + OFF_V + 8 * KB, &tm_v, h * D + 64, m * C, b, bars.v);
    };
    if (lt == 0 && nchunks > 0) load_v(0);
    const float A_log_h = p.gates_pre ? 0.f : p.A_log[h];
    const float dtb_h = (p.gates_pre || !p.dt_bias) ? 0.f : p.dt_bias[h];
    // raw gate inputs of a chunk: warp 0 loads them one chunk ahead into registers and parks
    // them in shared memory at the end of the chunk (by then the loads have long returned)
    float ra[2] = {0.f, 0.f}, rb[2] = {0.f, 0.f};
    auto load_gates = [&](int m) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = min(m * C + 2 * lane + e, p.T - 1);
        const size_t gi = ((size_t)b * p.T + t) * p.Hv + h;
        if (p.gates_pre) {
          ra[e] = reinterpret_cast<const float*>(p.a)[gi];
          rb[e] = reinterpret_cast<const float*>(p.b)[gi];
        } else {
          ra[e] = ld_elem(reinterpret_cast<const Tin*>(p.a) + gi);
          rb[e] = ld_elem(reinterpret_cast<const Tin*>(p.b) + gi);
        }
      }
    };
    auto park_gates = [&](int m) {
      const Factors Fm = factors_at(misc, m & 1);
      Fm.ra[2 * lane] = ra[0];
      Fm.ra[2 * lane + 1] = ra[1];
      Fm.rb[2 * lane] = rb[0];
      Fm.rb[2 * lane + 1] = rb[1];
    };
    if (warp == 0) {
      load_gates(0);
      park_gates(0);
    }

    for (int m = 0; m < nchunks; ++m) {
      const int par = m & 1;
      const Factors F = factors_at(misc, par);
      const uint32_t KQ = sb + (par ? OFF_KQ1 : OFF_KQ0);
      const uint8_t* KQp = sm + (par ? OFF_KQ1 : OFF_KQ0);
      const uint32_t Pt = sb + (par ? OFF_P1 : OFF_P0);
      const uint32_t NWt = sb + (par ? OFF_NW1 : OFF_NW0);
      const uint32_t tmU = tmem + TM_U + 64 * par;
      // this parity's buffers (P, -W^T, U^T, factors) are free once chunk m-2 left the chain
      if (m >= 2 && !mbar_wait_or_abort(bars.fr[par], ((m >> 1) - 1) & 1, sAbort)) fail();
      // gates: g, beta, G = inclusive prefix sum of g (two tokens per lane of warp 0)
      if (warp == 0) {
        float g2[2] = {0.f, 0.f}, b2[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (m * C + 2 * lane + e < p.T) {
            const float xa = F.ra[2 * lane + e], xb = F.rb[2 * lane + e];
            g2[e] = p.gates_pre ? xa : gate_g(xa, A_log_h, dtb_h);
            b2[e] = p.gates_pre ? xb : sigmoid_f(xb);
          }
        }
        if (m + 1 < nchunks) load_gates(m + 1);    // parked at the end of this iteration
        float s = g2[0] + g2[1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, s, o);
          if (lane >= o) s += y;
        }
        F.gl2[2 * lane] = (s - g2[1]) * LOG2E;
        F.gl2[2 * lane + 1] = s * LOG2E;
        F.beta[2 * lane] = b2[0];
        F.beta[2 * lane + 1] = b2[1];
      }
      if (!mbar_wait_or_abort(bars.kq[par], (m >> 1) & 1, sAbort)) fail();
      named_bar_sync(1, LGT);
      if (*sAbortL) break;

      // ---- MMA 1: G = [K; Q] K^T  (M = 128: k_0..k_63, q_0..q_63; N = 64; K = 128)
      if (lt == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * KQ_KB + (k & 3) * 32;
          mma_bf16(tmem + TM_GW, sdesc_sw128(KQ + off, 16, 1024), sdesc_sw128(KQ + off, 16, 1024),
                   ID_G, k > 0);
        }
        mma_commit(bars.mma_l);
      }
      pend_mma = true;
      // ---- row norms of k (rows 0..63) and q (rows 64..127) from the raw tiles
      {
        const int nr = lt >> 1, kb = lt & 1;
        const uint8_t* rp = KQp + kb * KQ_KB + (nr < 64 ? 0 : KQ_Q) + (nr & 63) * 128;
        uint4 u[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) u[c] = reinterpret_cast<const uint4*>(rp)[c];
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u[c]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(hv[e]);
            s4[e] = fmaf(f.x, f.x, fmaf(f.y, f.y, s4[e]));
          }
        }
        float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        if (kb == 0) {
          const float inv = p.l2norm ? 1.0f / sqrtf(ss + p.eps) : 1.0f;
          if (nr < 64) F.nk[nr] = inv; else F.nq[nr - 64] = inv * p.scale;
        }
      }
      named_bar_sync(1, LGT);
      if (lt < 64) {
        F.eG[lt] = ex2_approx(F.gl2[lt]);
        F.dK[lt] = ex2_approx(F.gl2[63] - F.gl2[lt]);
      }
      if (!mbar_wait_or_abort(bars.mma_l, mma_phase, sAbort)) fail();
      mma_phase ^= 1;
      pend_mma = false;
      tc_fence_after();
      named_bar_sync(1, LGT);
      if (*sAbortL) break;

      // ---- E1: G -> A (fp32 [r][s], strictly lower) and P (bf16 hi/lo [r][s], K-major)
      {
        float* As = reinterpret_cast<float*>(sm + OFF_SOLVE);
        const bool isq = row >= 64;
        const int r = row & 63;
        const float Gr = F.gl2[r], sr = (isq ? 1.0f : F.beta[r]) * (isq ? F.nq[r] : F.nk[r]);
        const int half = hcol;
        float v[32], gs[32], ns[32];
        tmem_ld32(tmem + lane_off + TM_GW + 32 * half, v);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 g4 = *reinterpret_cast<const float4*>(F.gl2 + 32 * half + 4 * j4);
          const float4 n4 = *reinterpret_cast<const float4*>(F.nk + 32 * half + 4 * j4);
          gs[4 * j4] = g4.x; gs[4 * j4 + 1] = g4.y; gs[4 * j4 + 2] = g4.z; gs[4 * j4 + 3] = g4.w;
          ns[4 * j4] = n4.x; ns[4 * j4 + 1] = n4.y; ns[4 * j4 + 2] = n4.z; ns[4 * j4 + 3] = n4.w;
        }
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int s = 32 * half + j;
          const bool keep = isq ? (s <= r) : (s < r);
          v[j] = keep ? ex2_approx(Gr - gs[j]) * v[j] * (sr * ns[j]) : 0.f;
        }
        if (isq) {
          store_row_hilo(Pt, Pt + 8 * KB, r, 4 * half, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(As + r * LA + 32 * half + j) =
                make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
      // ---- Q~ = diag(scale e^G / ||q||) Q, in place (the raw Q is no longer needed)
      for (int idx = lt; idx < 1024; idx += LGT) {
        const int kb = idx >> 9, off = (idx & 511) * 16, r = (idx & 511) >> 3;
        uint8_t* qp = const_cast<uint8_t*>(KQp) + kb * KQ_KB + KQ_Q + off;
        const float f = F.eG[r] * F.nq[r];
        uint4 u = *reinterpret_cast<const uint4*>(qp);
        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(hv[e]);
          hv[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
        }
        *reinterpret_cast<uint4*>(qp) = u;
      }
      named_bar_sync(1, LGT);

      // ---- the direct solve T = (I + A)^{-1}, then T' and T'' as bf16 hi/lo B operands
      {
        float* As = reinterpret_cast<float*>(sm + OFF_SOLVE);
        float* Ts = reinterpret_cast<float*>(sm + OFF_SOLVE + 16 * KB);
        solve_unit_lower(As, Ts, sX, lt);
        // the T'/T'' tiles reuse the A/T region: read this thread's T entries first
        float tv[2][8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int idx = lt + LGT * j, r = idx >> 3, c = idx & 7;
          const float4 x0 = *reinterpret_cast<const float4*>(Ts + r * LA + 8 * c);
          const float4 x1 = *reinterpret_cast<const float4*>(Ts + r * LA + 8 * c + 4);
          tv[j][0] = x0.x; tv[j][1] = x0.y; tv[j][2] = x0.z; tv[j][3] = x0.w;
          tv[j][4] = x1.x; tv[j][5] = x1.y; tv[j][6] = x1.z; tv[j][7] = x1.w;
        }
        named_bar_sync(1, LGT);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int idx = lt + LGT * j, r = idx >> 3, c = idx & 7;
          uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 8 * c + 2 * e;
            const float f10 = F.beta[s] * F.eG[s] * F.nk[s];
            const float f11 = F.beta[s + 1] * F.eG[s + 1] * F.nk[s + 1];
            pack_hilo(tv[j][2 * e] * f10, tv[j][2 * e + 1] * f11, h1[e], l1[e]);
            pack_hilo(tv[j][2 * e] * F.beta[s], tv[j][2 * e + 1] * F.beta[s + 1], h2[e], l2[e]);
          }
          st_shared_v4(sw128(sb + OFF_T1H, r, c), h1[0], h1[1], h1[2], h1[3]);
          st_shared_v4(sw128(sb + OFF_T1L, r, c), l1[0], l1[1], l1[2], l1[3]);
          st_shared_v4(sw128(sb + OFF_T2H, r, c), h2[0], h2[1], h2[2], h2[3]);
          st_shared_v4(sw128(sb + OFF_T2L, r, c), l2[0], l2[1], l2[2], l2[3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, LGT);

      // ---- MMA 3/4: W^T = K^T T'^T (M = d_k), U'^T = V^T T''^T (M = d_v), K = 64 tokens
      if (lt == 0) {
        if (!mbar_wait_or_abort(bars.v, m & 1, sAbort)) {
          fail();
        } else {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16(tmem + TM_GW, sdesc_sw128(KQ + (k & 3) * 2048, KQ_KB, 1024),
                     sdesc_sw128(sb + (k < 4 ? OFF_T1H : OFF_T1L) + (k & 3) * 32, 16, 1024),
                     ID_KT, k > 0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16(tmU, sdesc_sw128(sb + OFF_V + (k & 3) * 2048, 8 * KB, 1024),
                     sdesc_sw128(sb + (k < 4 ? OFF_T2H : OFF_T2L) + (k & 3) * 32, 16, 1024),
                     ID_KT, k > 0);
          mma_commit(bars.mma_l);
        }
      }
      pend_mma = true;
      if (!mbar_wait_or_abort(bars.mma_l, mma_phase, sAbort)) fail();
      mma_phase ^= 1;
      pend_mma = false;
      tc_fence_after();
      // the V buffer is free again
      if (lt == 0 && m + 1 < nchunks && !*sAbort) load_v(m + 1);
      // ---- E3: W^T -> -W^T bf16 (B operand, MN-major: row = d_k index, 64 token columns)
      {
        float v[32];
        tmem_ld32(tmem + lane_off + TM_GW + 32 * hcol, v);
        tmem_wait_ld();
        store_row_bf16(NWt, row, 4 * hcol, v, -1.0f);
      }
      // ---- park the next chunk's raw gates (loaded at the top of this iteration)
      if (warp == 0 && m + 1 < nchunks) park_gates(m + 1);
      // ---- hand the chunk to the chain group
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bars.ready[par]);
      named_bar_sync(1, LGT);
      if (*sAbortL) break;
    }
  } else {
    // ======================================================== chain group (warps 4-7)
    const int ct = tid - LGT;
    auto fail = [&]() { *sAbort = 1; *sAbortC = 1; };
    auto load_kq = [&](int n) {
      const uint32_t buf = sb + ((n & 1) ? OFF_KQ1 : OFF_KQ0);
      const uint32_t bar = bars.kq[n & 1];
      mbar_arrive_expect_tx(bar, 32 * KB);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d(buf + kb * KQ_KB, &tm_k, kh * D + 64 * kb, n * C, b, bar);
        tma_load_3d(buf + kb * KQ_KB + KQ_Q, &tm_q, kh * D + 64 * kb, n * C, b, bar);
      }
    };
    if (ct == 0) {
      if (nchunks > 0) load_kq(0);
      if (nchunks > 1) load_kq(1);
    }
    // the entering state -> TMEM (fp32, row i in lane i)
    float* Sg = p.state + ((size_t)slot * p.Hv + h) * D * D + (size_t)row * D;
    {
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 f = reinterpret_cast<const float4*>(Sg + 32 * q)[j];
          v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
        }
        tmem_st32(tmem + lane_off + TM_S + 32 * q, v);
      }
      tmem_wait_st();
    }
    constexpr int OUT_ROWS = (int)(16 * KB / (D * sizeof(Tout)));   // tokens per staging pass
    // output tile of chunk n (O^T in TMEM, lane = d_v index, column = token) -> HBM
    auto store_out = [&](int n) {
      const uint32_t tmO = tmem + lane_off + TM_O + 64 * (n & 1);
      Tout* stg = reinterpret_cast<Tout*>(sm + OFF_OUT);
#pragma unroll
      for (int pass = 0; pass < 64 / OUT_ROWS; ++pass) {
        if (ct == 0) tma_store_wait_read();      // the staging buffer is free again
        named_bar_sync(2, CGT);
        float v[32];
#pragma unroll
        for (int half = 0; half < OUT_ROWS / 32; ++half) {
          tmem_ld32(tmO + pass * OUT_ROWS + 32 * half, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) stg[(32 * half + j) * D + row] = from_float<Tout>(v[j]);
        }
        fence_proxy_async_smem();
        named_bar_sync(2, CGT);
        if (ct == 0) {
          tma_store_3d(&tm_o, sb + OFF_OUT, h * D, n * C + pass * OUT_ROWS, b);
          tma_store_commit();
        }
      }
    };

    bool aborted = false;
    for (int n = 0; n < nchunks; ++n) {
      const int par = n & 1;
      const Factors F = factors_at(misc, par);
      const uint32_t KQ = sb + (par ? OFF_KQ1 : OFF_KQ0);
      const uint8_t* KQp = sm + (par ? OFF_KQ1 : OFF_KQ0);
      const uint32_t Pt = sb + (par ? OFF_P1 : OFF_P0);
      const uint32_t NWt = sb + (par ? OFF_NW1 : OFF_NW0);
      const uint32_t tmU = tmem + TM_U + 64 * par;
      const uint32_t tmO = tmem + TM_O + 64 * par;
      if (!mbar_wait_or_abort(bars.ready[par], (n >> 1) & 1, sAbort)) fail();
      tc_fence_after();
      named_bar_sync(2, CGT);
      if (*sAbortC) { aborted = true; break; }

      // ---- C0: S -> S0 (bf16, packed into TMEM as the A operand);  S <- e^{G_C} S
      {
        const float eGC = F.eG[63];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t ta = tmem + lane_off + TM_S + 32 * g;
          float v[32];
          uint32_t pk[16];
          tmem_ld32(ta, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(v[2 * j], v[2 * j + 1]);
          tmem_st16(tmem + lane_off + TM_SU + 16 * g, pk);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= eGC;
          tmem_st32(ta, v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      named_bar_sync(2, CGT);
      // ---- C1: U^T += S0 (-W)^T ;  O^T = S0 Q~^T   (M = d_v, N = 64 tokens, K = d_k)
      if (ct == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ta(tmU, tmem + TM_SU + 8 * k, sdesc_sw128(NWt + k * 2048, 8 * KB, 1024), ID_SW,
                      true);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ta(tmO, tmem + TM_SU + 8 * k,
                      sdesc_sw128(KQ + (k >> 2) * KQ_KB + KQ_Q + (k & 3) * 32, 16, 1024), ID_SQ,
                      k > 0);
        mma_commit(bars.mma_c);
      }
      pend_mma = true;
      // while C1 runs: the output of chunk n-1, then K~ of chunk n
      if (n > 0) store_out(n - 1);
      for (int idx = ct; idx < 1024; idx += CGT) {
        const int kb = idx >> 9, off = (idx & 511) * 16, r = (idx & 511) >> 3;
        uint4 u = *reinterpret_cast<const uint4*>(KQp + kb * KQ_KB + off);
        const float f = F.dK[r] * F.nk[r];
        __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(hv[e]);
          hv[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
        }
        *reinterpret_cast<uint4*>(sm + OFF_KT + kb * 8 * KB + off) = u;
      }
      fence_proxy_async_smem();
      if (!mbar_wait_or_abort(bars.mma_c, mma_phase, sAbort)) fail();
      mma_phase ^= 1;
      pend_mma = false;
      tc_fence_after();
      named_bar_sync(2, CGT);
      if (*sAbortC) { aborted = true; break; }
      // the K|Q buffer of this parity has been fully read: load chunk n+2 into it
      if (ct == 0 && n + 2 < nchunks) load_kq(n + 2);

      // ---- C2: U^T (fp32) -> bf16 hi / lo, packed into TMEM as A operands
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float v[32];
        uint32_t hu[16], lu[16];
        tmem_ld32(tmU + lane_off + 32 * g, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) pack_hilo(v[2 * j], v[2 * j + 1], hu[j], lu[j]);
        tmem_st16(tmem + lane_off + TM_SU + 16 * g, hu);
        tmem_st16(tmem + lane_off + TM_SU + 32 + 16 * g, lu);
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(2, CGT);
      // ---- C3: O^T += U^T P^T (Uh Ph + Ul Ph + Uh Pl) ;  S += U^T K~ (Uh K~ + Ul K~)
      if (ct == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 12; ++k) {
          const uint32_t ua = (k < 4 || k >= 8) ? 0u : 32u;
          const uint32_t pb = (k < 8) ? 0u : 8 * KB;
          mma_bf16_ta(tmO, tmem + TM_SU + ua + 8 * (k & 3),
                      sdesc_sw128(Pt + pb + (k & 3) * 32, 16, 1024), ID_SQ, true);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ta(tmem + TM_S, tmem + TM_SU + (k < 4 ? 0u : 32u) + 8 * (k & 3),
                      sdesc_sw128(sb + OFF_KT + (k & 3) * 2048, 8 * KB, 1024), ID_UK, true);
        mma_commit(bars.mma_c);
      }
      pend_mma = true;
      if (!mbar_wait_or_abort(bars.mma_c, mma_phase, sAbort)) fail();
      mma_phase ^= 1;
      pend_mma = false;
      tc_fence_after();
      // chunk n has left the chain: its P, -W^T, U^T buffers and factors are free
      tc_fence_before();
      mbar_arrive(bars.fr[par]);
    }
    if (!aborted && !*sAbortC && nchunks > 0) {
      store_out(nchunks - 1);
      // the leaving state: TMEM -> HBM (fp32)
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        tmem_ld32(tmem + lane_off + TM_S + 32 * q, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          reinterpret_cast<float4*>(Sg + 32 * q)[j] =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
    }
    if (ct == 0) tma_store_wait_all();
  }

  // ---- teardown: pending MMAs (abort path only) are waited for, then TMEM is freed
  if (pend_mma && (tid == 0 || tid == LGT))
    mbar_wait_bounded(tid == 0 ? bars.mma_l : bars.mma_c, mma_phase, 1u << 16);
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *sAbort) atomicOr(&g_err_tc, kErrTimeout);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 3-D map over [B][T][width] elements starting at `base`, token stride `tok_stride`
// elements; box = {box0, box1 tokens, 1 sequence}.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
              int width, int T, int B, long long tok_stride, int box0, int box1,
              bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)(tok_stride * elem_bytes),
                           (cuuint64_t)(tok_stride * elem_bytes) * (cuuint64_t)T};
  cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename Tout>
cudaError_t launch_tc_t(const GdnLayerArgs& L, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  constexpr int out_rows = (int)(16 * KB / (D * sizeof(Tout)));
  const bool ok =
      make_map(&mq, L.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hk * D, L.T, L.B, L.q_tok_stride,
               64, 64, true) &&
      make_map(&mk, L.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hk * D, L.T, L.B, L.k_tok_stride,
               64, 64, true) &&
      make_map(&mv, L.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hv * D, L.T, L.B, L.v_tok_stride,
               64, 64, true) &&
      make_map(&mo, L.out,
               sizeof(Tout) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
               (int)sizeof(Tout), L.Hv * D, L.T, L.B, (long long)L.Hv * D, 128, out_rows, false);
  if (!ok) return cudaErrorInvalidValue;
  static unsigned done = 0;
  cudaError_t e = set_smem_once(gdn_prefill_tc_kernel<__nv_bfloat16, Tout>, (int)SMEM_BYTES, &done);
  if (e != cudaSuccess) return e;
  TcParams p;
  p.T = L.T; p.Hk = L.Hk; p.Hv = L.Hv; p.num_slots = L.num_slots; p.l2norm = L.l2norm;
  p.gates_pre = L.gates_pre; p.eps = L.eps; p.scale = L.scale; p.a = L.a; p.b = L.b;
  p.A_log = L.A_log; p.dt_bias = L.dt_bias; p.state = L.state; p.slots = L.slots;
  gdn_prefill_tc_kernel<__nv_bfloat16, Tout>
      <<<dim3((unsigned)(L.B * L.Hv)), THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gdn_launch_prefill_tc(const GdnLayerArgs& L, cudaStream_t stream) {
  if (L.B == 0 || L.T == 0) return cudaSuccess;
  if (!L.in_bf16) return cudaErrorInvalidValue;
  return L.out_bf16 ? launch_tc_t<__nv_bfloat16>(L, stream) : launch_tc_t<float>(L, stream);
}
