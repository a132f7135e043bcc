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
// scalings of the raw tiles, so the tensor cores always see raw bf16 q/k/v:
//   G = [K;Q] K^T (one M=128 MMA)  ->  A, P (with 1/||k||, scale/||q||, decays)
//   T' = T diag(beta e^G / ||k||),  T'' = T diag(beta)      (the solve, fp32 FMA)
// T', T'', P and U^T enter the tensor cores as bf16 pairs hi + lo (hi = rn(x), lo = rn(x-hi)),
// which keeps ~16 mantissa bits in the small intra-chunk products; the state snapshot S0,
// W, Q~ and K~ are single bf16 (their rounding costs far less at the output).
//   W^T = K^T T'^T,  U'^T = V^T T''^T                          (M = d = 128)
//   Q~ = diag(scale e^G / ||q||) Q,  K~ = diag(e^{G_C-G} / ||k||) K
//   U^T = U'^T - S0 W^T,  O^T = S0 Q~^T + U^T P^T,  S = e^{G_C} S0 + U^T K~
// Everything is computed transposed so that the MMA M dimension (128 TMEM lanes) is the
// head dimension: the state row i lives in TMEM lane i for the whole sequence and every
// epilogue thread owns one row.
//
// One CTA per (sequence, value head), 256 threads (8 warps: TMEM lane quarter = warp % 4,
// column half = warp / 4).  Thread 0 issues TMA loads and MMAs.  TMEM: S 128 columns, U^T 64,
// O^T 64, G 64, W^T 64 (512 allocated).  Q/K/V chunk tiles are double-buffered and loaded
// one chunk ahead with TMA (128-byte swizzle = the canonical UMMA K-major layout; the same
// bytes read as MN-major give K^T / V^T).  Outputs are staged in shared memory and written
// with a TMA store.  Every mbarrier wait is bounded: on timeout the CTA records
// GDN_ERR_DEVICE_TIMEOUT, waits (bounded) for its own copies, frees TMEM and returns.
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

constexpr int C = kChunk, D = kHeadDim, THREADS = 256;
constexpr uint32_t KB = 1024;
// shared-memory layout (byte offsets from a 1024-byte aligned base)
constexpr uint32_t IN_BYTES = 48 * KB;            // K|Q interleaved per 64-col block + V
constexpr uint32_t OFF_IN0 = 0, OFF_IN1 = IN_BYTES;
constexpr uint32_t IN_Q = 8 * KB;                 // Q rows after K rows inside a KQ block
constexpr uint32_t IN_KQ_KB = 16 * KB;            // stride of the two 64-column KQ blocks
constexpr uint32_t IN_V = 32 * KB;                // V tile: [2][64 rows][128 B]
constexpr uint32_t OFF_KT = 96 * KB;              // K~  [2][64][128 B]
constexpr uint32_t OFF_NW = 112 * KB;             // -W^T [128 rows d_k][128 B]
constexpr uint32_t OFF_S0 = 128 * KB;             // S0 bf16 [2][128][128 B] | solve A, T fp32
// T', T'' (hi, lo) [64][128 B] each; later U^T (hi, lo) [128][128 B]; later output staging
constexpr uint32_t OFF_TU = 160 * KB;
constexpr uint32_t OFF_T1H = OFF_TU, OFF_T1L = OFF_TU + 8 * KB;
constexpr uint32_t OFF_T2H = OFF_TU + 16 * KB, OFF_T2L = OFF_TU + 24 * KB;
constexpr uint32_t OFF_UTH = OFF_TU, OFF_UTL = OFF_TU + 16 * KB;
constexpr uint32_t OFF_OUT = OFF_TU;
constexpr uint32_t OFF_PH = 192 * KB, OFF_PL = 200 * KB;   // P (hi, lo) [64][128 B]
constexpr uint32_t OFF_MISC = 208 * KB;
constexpr uint32_t MISC_X = 2048;                 // solve scratch, 3 x 16 x 16 fp32
constexpr uint32_t MISC_BAR = 5120;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 6 * KB + KB;   // + alignment slack
constexpr int LA = 64;                            // row stride (floats) of the solve matrices

// TMEM column map
constexpr uint32_t TM_S = 0, TM_U = 128, TM_O = 192, TM_G = 256, TM_W = 320, TM_COLS = 512;

constexpr uint32_t ID_G = idesc_bf16(128, 64, false, false);   // [K;Q] K^T
constexpr uint32_t ID_KT = idesc_bf16(128, 64, true, false);   // K^T T'^T, V^T T''^T
constexpr uint32_t ID_SW = idesc_bf16(128, 64, false, true);   // S0 (-W)^T
constexpr uint32_t ID_SQ = idesc_bf16(128, 64, false, false);  // S0 Q~^T, U^T P^T
constexpr uint32_t ID_UK = idesc_bf16(128, 128, false, true);  // U^T K~

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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte chunk `c` (0..7) of row `r` of a 128-byte-swizzled tile whose 8-row groups are
// 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128(uint32_t row_base, int r, int c) {
  return row_base + (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 32 fp32 values -> 4 swizzled 16-byte chunks (chunk indices c0..c0+3) of row r.
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

// 32 fp32 values -> bf16 hi = rn(v) and lo = rn(v - hi) rows of two tiles (v = hi + lo to
// about 2^-16 relative): the small intra-chunk matrices keep ~16 mantissa bits this way.
__device__ __forceinline__ void store_row_hilo(uint32_t tile_hi, uint32_t tile_lo, int r, int c0,
                                               const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = v[8 * c + 2 * e], x1 = v[8 * c + 2 * e + 1];
      const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
      const float2 hf = __bfloat1622float2(h);
      const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
      hw[e] = *reinterpret_cast<const uint32_t*>(&h);
      lw[e] = *reinterpret_cast<const uint32_t*>(&l);
    }
    st_shared_v4(sw128(tile_hi, r, c0 + c), hw[0], hw[1], hw[2], hw[3]);
    st_shared_v4(sw128(tile_lo, r, c0 + c), lw[0], lw[1], lw[2], lw[3]);
  }
}

template <typename Tin>
__device__ __forceinline__ float ld_gate(const void* p, size_t i) {
  return ld_elem(reinterpret_cast<const Tin*>(p) + i);
}

// T = (I + A)^{-1} for the strictly lower 64 x 64 matrix A (fp32, row stride LA), by blocked
// forward substitution over 16 x 16 blocks: warps 0-3 invert one diagonal block each (lane =
// column, rows in order); then the off-diagonal blocks by distance from the diagonal,
//   T_ij = -T_ii * sum_{k=j}^{i-1} A_ik T_kj,
// one thread per block entry.  All 256 threads must call it.
__device__ void solve_unit_lower(const float* As, float* Ts, float* X, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 4) {
    if (lane < 16) {
      const int o = 16 * warp, c = lane;
      float t[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float val = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int s = 0; s < r; ++s) val = fmaf(-As[(o + r) * LA + o + s], t[s], val);
        t[r] = val;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) Ts[(o + r) * LA + o + c] = t[r];
    }
  } else {
    // strictly upper blocks of T are zero
    for (int idx = tid - 128; idx < 6 * 256; idx += 128) {
      const int blk = idx >> 8, e = idx & 255;
      const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
      Ts[(16 * bi + (e >> 4)) * LA + 16 * bj + (e & 15)] = 0.f;
    }
  }
  __syncthreads();
  const int rr = tid >> 4, cc = tid & 15;
  for (int dist = 1; dist <= 3; ++dist) {
    const int nblk = 4 - dist;
    // X_i = sum_{k=j}^{i-1} A_ik T_kj  for each block (i, j = i - dist)
    for (int q = 0; q < nblk; ++q) {
      const int i = dist + q, j = q;
      float acc = 0.f;
      for (int k = j; k < i; ++k) {
        const float* arow = As + (16 * i + rr) * LA + 16 * k;
        const float* tcol = Ts + (16 * k) * LA + 16 * j + cc;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(arow[m], tcol[m * LA], acc);
      }
      X[q * 256 + rr * 16 + cc] = acc;
    }
    __syncthreads();
    for (int q = 0; q < nblk; ++q) {
      const int i = dist + q, j = q;
      const float* trow = Ts + (16 * i + rr) * LA + 16 * i;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc = fmaf(trow[m], X[q * 256 + m * 16 + cc], acc);
      Ts[(16 * i + rr) * LA + 16 * j + cc] = -acc;
    }
    __syncthreads();
  }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(THREADS, 1)
    gdn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_o, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed by offsetting the shared array itself so that every
  // pointer derived from it stays in the shared state space (no generic accesses)
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hc = warp >> 2;
  const int b = blockIdx.x / p.Hv, h = blockIdx.x % p.Hv;
  const int kh = h / (p.Hv / p.Hk);

  const int slot = p.slots ? p.slots[b] : b;
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (tid == 0) atomicOr(&g_err_tc, kErrIndex);
    return;
  }

  float* sG = reinterpret_cast<float*>(sm + OFF_MISC);
  float* sBeta = sG + 64;
  float* sNk = sG + 128;   // 1 / ||k_r||
  float* sNq = sG + 192;   // scale / ||q_r||
  float* sEG = sG + 256;   // e^{G_r}
  float* sDK = sG + 320;   // e^{G_C - G_r}
  float* sX = reinterpret_cast<float*>(sm + OFF_MISC + MISC_X);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC + MISC_BAR);
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + OFF_MISC + MISC_BAR + 32);
  int* sAbort = reinterpret_cast<int*>(sm + OFF_MISC + MISC_BAR + 40);
  float* As = reinterpret_cast<float*>(sm + OFF_S0);
  float* Ts = reinterpret_cast<float*>(sm + OFF_S0 + 16 * KB);
  const uint32_t bar_in0 = smem_addr(&bars[0]), bar_in1 = smem_addr(&bars[1]);
  const uint32_t bar_mma = smem_addr(&bars[2]);

  if (tid == 0) {
    mbar_init(bar_in0, 1);
    mbar_init(bar_in1, 1);
    mbar_init(bar_mma, 1);
    *sAbort = 0;
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
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  const int row = 32 * q4 + lane;   // TMEM lane owned by this thread (a head-dim index)

  // ---- the entering state -> TMEM (fp32, row i in lane i)
  float* Sg = p.state + ((size_t)slot * p.Hv + h) * D * D + (size_t)row * D + 64 * hc;
  {
    float v[32];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 f = reinterpret_cast<const float4*>(Sg + 32 * half)[j];
        v[4 * j] = f.x; v[4 * j + 1] = f.y; v[4 * j + 2] = f.z; v[4 * j + 3] = f.w;
      }
      tmem_st32(tmem + lane_off + TM_S + 64 * hc + 32 * half, v);
    }
    tmem_wait_st();
  }

  const int nchunks = (p.T + C - 1) / C;
  auto issue_loads = [&](int n, uint32_t buf, uint32_t bar) {
    const int t0 = n * C;
    mbar_arrive_expect_tx(bar, 6 * 8 * KB);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_3d(buf + kb * IN_KQ_KB, &tm_k, kh * D + 64 * kb, t0, b, bar);
      tma_load_3d(buf + kb * IN_KQ_KB + IN_Q, &tm_q, kh * D + 64 * kb, t0, b, bar);
      tma_load_3d(buf + IN_V + kb * 8 * KB, &tm_v, h * D + 64 * kb, t0, b, bar);
    }
  };
  if (tid == 0 && nchunks > 0) issue_loads(0, sb + OFF_IN0, bar_in0);

  const float A_log_h = p.gates_pre ? 0.f : p.A_log[h];
  const float dtb_h = (p.gates_pre || !p.dt_bias) ? 0.f : p.dt_bias[h];
  uint32_t mma_phase = 0;
  bool aborted = false;

  // raw gate inputs of the next chunk, loaded one chunk ahead by warp 0 (2 tokens per lane)
  float ra[2] = {0.f, 0.f}, rb[2] = {0.f, 0.f};
  auto load_gates = [&](int n) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = n * C + 2 * lane + e;
      ra[e] = rb[e] = 0.f;
      if (t < p.T) {
        const size_t gi = ((size_t)b * p.T + t) * p.Hv + h;
        if (p.gates_pre) {
          ra[e] = reinterpret_cast<const float*>(p.a)[gi];
          rb[e] = reinterpret_cast<const float*>(p.b)[gi];
        } else {
          ra[e] = ld_gate<Tin>(p.a, gi);
          rb[e] = ld_gate<Tin>(p.b, gi);
        }
      }
    }
  };
  if (warp == 0) load_gates(0);

  for (int n = 0; n < nchunks; ++n) {
    const int t0 = n * C;
    const uint32_t buf = sb + ((n & 1) ? OFF_IN1 : OFF_IN0);
    const uint32_t bar_in = (n & 1) ? bar_in1 : bar_in0;
    const uint8_t* bufp = sm + ((n & 1) ? OFF_IN1 : OFF_IN0);

    // ---- gates of this chunk (warp 0): g, beta, inclusive prefix sum G
    if (warp == 0) {
      float g2[2] = {0.f, 0.f}, b2[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (t0 + 2 * lane + e < p.T) {
          g2[e] = p.gates_pre ? ra[e] : gate_g(ra[e], A_log_h, dtb_h);
          b2[e] = p.gates_pre ? rb[e] : sigmoid_f(rb[e]);
        }
      }
      if (n + 1 < nchunks) load_gates(n + 1);
      float s = g2[0] + g2[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      sG[2 * lane] = s - g2[1];
      sG[2 * lane + 1] = s;
      sBeta[2 * lane] = b2[0];
      sBeta[2 * lane + 1] = b2[1];
    }
    // the previous chunk's output store must have finished reading its staging (UT/P/T1)
    if (tid == 0) tma_store_wait_read();
    // ---- inputs of this chunk
    if (!mbar_wait_bounded(bar_in, (n >> 1) & 1)) atomicExch(sAbort, 1);
    __syncthreads();
    if (*sAbort) { aborted = true; break; }
    if (tid == 0 && n + 1 < nchunks)
      issue_loads(n + 1, sb + ((n & 1) ? OFF_IN0 : OFF_IN1), (n & 1) ? bar_in0 : bar_in1);

    // ---- MMA 1: G = [K; Q] K^T  (M = 128 rows: k_0..k_63, q_0..q_63; N = 64; K = 128)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t off = (k >> 2) * IN_KQ_KB + (k & 3) * 32;
        mma_bf16(tmem + TM_G, sdesc_sw128(buf + off, 16, 1024), sdesc_sw128(buf + off, 16, 1024),
                 ID_G, k > 0);
      }
      mma_commit(bar_mma);
    }
    // ---- row norms of k (rows 0..63) and q (rows 64..127) from the raw tiles
    {
      const int r = tid >> 1, kb = tid & 1;
      const uint8_t* rp = bufp + kb * IN_KQ_KB + (r < 64 ? 0 : IN_Q) + (r & 63) * 128;
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 u = reinterpret_cast<const uint4*>(rp)[c];
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(hv[e]);
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (kb == 0) {
        const float inv = p.l2norm ? 1.0f / sqrtf(ss + p.eps) : 1.0f;
        if (r < 64) sNk[r] = inv; else sNq[r - 64] = inv * p.scale;
      }
    }
    __syncthreads();
    if (tid < 64) {
      sEG[tid] = expf(sG[tid]);
      sDK[tid] = expf(sG[63] - sG[tid]);
    }
    if (!mbar_wait_bounded(bar_mma, mma_phase)) atomicExch(sAbort, 1);
    mma_phase ^= 1;
    tc_fence_after();
    __syncthreads();
    if (*sAbort) { aborted = true; break; }

    // ---- E1: G -> A (fp32, for the solve) and P (bf16 B operand [r][s], K-major)
    {
      float v[32];
      tmem_ld32(tmem + lane_off + TM_G + 32 * hc, v);
      tmem_wait_ld();
      if (q4 < 2) {
        const int r = row;
        const float br = sBeta[r], Gr = sG[r], nr = sNk[r];
        float* arow = As + r * LA + 32 * hc;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 o;
          float* of = reinterpret_cast<float*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 32 * hc + j + e;
            of[e] = (s < r) ? br * expf(Gr - sG[s]) * v[j + e] * nr * sNk[s] : 0.f;
          }
          *reinterpret_cast<float4*>(arow + j) = o;
        }
      } else {
        const int r = row - 64;
        const float Gr = sG[r], mr = sNq[r];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int s = 32 * hc + j;
          v[j] = (s <= r) ? expf(Gr - sG[s]) * v[j] * mr * sNk[s] : 0.f;
        }
        store_row_hilo(sb + OFF_PH, sb + OFF_PL, r, 4 * hc, v);
      }
    }
    // ---- Q~ = diag(scale e^G / ||q||) Q in place;  K~ = diag(e^{G_C-G} / ||k||) K -> KT
    for (int idx = tid; idx < 2048; idx += THREADS) {
      const int isk = idx >> 10, c = idx & 1023;
      const int kb = c >> 9, off = (c & 511) * 16, r = (c & 511) >> 3;
      const uint8_t* src = bufp + kb * IN_KQ_KB + (isk ? 0 : IN_Q) + off;
      uint8_t* dst = isk ? sm + OFF_KT + kb * 8 * KB + off : const_cast<uint8_t*>(src);
      const float f = isk ? sDK[r] * sNk[r] : sEG[r] * sNq[r];
      uint4 u = *reinterpret_cast<const uint4*>(src);
      __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(hv[e]);
        hv[e] = __floats2bfloat162_rn(x.x * f, x.y * f);
      }
      *reinterpret_cast<uint4*>(dst) = u;
    }
    __syncthreads();

    // ---- the direct solve T = (I + A)^{-1}, then T' and T'' as bf16 (hi, lo) B operands
    solve_unit_lower(As, Ts, sX, tid);
    for (int idx = tid; idx < 1024; idx += THREADS) {
      const int which = idx >> 9, r = (idx >> 3) & 63, c = idx & 7;
      const float* trow = Ts + r * LA + 8 * c;
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int s = 8 * c + 2 * e;
        const float f0 = which ? sBeta[s] : sBeta[s] * sEG[s] * sNk[s];
        const float f1 = which ? sBeta[s + 1] : sBeta[s + 1] * sEG[s + 1] * sNk[s + 1];
        const float x0 = trow[2 * e] * f0, x1 = trow[2 * e + 1] * f1;
        const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
        hw[e] = *reinterpret_cast<const uint32_t*>(&h);
        lw[e] = *reinterpret_cast<const uint32_t*>(&l);
      }
      st_shared_v4(sw128(sb + (which ? OFF_T2H : OFF_T1H), r, c), hw[0], hw[1], hw[2], hw[3]);
      st_shared_v4(sw128(sb + (which ? OFF_T2L : OFF_T1L), r, c), lw[0], lw[1], lw[2], lw[3]);
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA 3/4: W^T = K^T T'^T (M = d_k), U'^T = V^T T''^T (M = d_v)  (K = 64 tokens),
    //      T' and T'' each as hi + lo
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(tmem + TM_W, sdesc_sw128(buf + (k & 3) * 2048, IN_KQ_KB, 1024),
                 sdesc_sw128(sb + (k < 4 ? OFF_T1H : OFF_T1L) + (k & 3) * 32, 16, 1024), ID_KT,
                 k > 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(tmem + TM_U, sdesc_sw128(buf + IN_V + (k & 3) * 2048, 8 * KB, 1024),
                 sdesc_sw128(sb + (k < 4 ? OFF_T2H : OFF_T2L) + (k & 3) * 32, 16, 1024), ID_KT,
                 k > 0);
      mma_commit(bar_mma);
    }
    // ---- C0 (overlaps MMA 3/4): S -> S0 (bf16 A operand [i][j], K-major); S <- e^{G_C} S
    {
      const float eGC = sEG[63];
      float v[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t ta = tmem + lane_off + TM_S + 64 * hc + 32 * half;
        tmem_ld32(ta, v);
        tmem_wait_ld();
        store_row_bf16(sb + OFF_S0 + hc * 16 * KB, row, 4 * half, v, 1.0f);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= eGC;
        tmem_st32(ta, v);
      }
      tmem_wait_st();
    }
    if (!mbar_wait_bounded(bar_mma, mma_phase)) atomicExch(sAbort, 1);
    mma_phase ^= 1;
    tc_fence_after();
    // ---- E3: W^T -> -W^T bf16 (B operand, MN-major: row = d_k index, 64 token columns)
    {
      float v[32];
      tmem_ld32(tmem + lane_off + TM_W + 32 * hc, v);
      tmem_wait_ld();
      store_row_bf16(sb + OFF_NW, row, 4 * hc, v, -1.0f);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*sAbort) { aborted = true; break; }

    // ---- C1: U^T += S0 (-W)^T ;  O^T = S0 Q~^T   (M = d_v, N = 64 tokens, K = d_k)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(tmem + TM_U, sdesc_sw128(sb + OFF_S0 + (k >> 2) * 16 * KB + (k & 3) * 32, 16, 1024),
                 sdesc_sw128(sb + OFF_NW + k * 2048, 8 * KB, 1024), ID_SW, true);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(tmem + TM_O, sdesc_sw128(sb + OFF_S0 + (k >> 2) * 16 * KB + (k & 3) * 32, 16, 1024),
                 sdesc_sw128(buf + (k >> 2) * IN_KQ_KB + IN_Q + (k & 3) * 32, 16, 1024), ID_SQ,
                 k > 0);
      mma_commit(bar_mma);
    }
    if (!mbar_wait_bounded(bar_mma, mma_phase)) atomicExch(sAbort, 1);
    mma_phase ^= 1;
    tc_fence_after();
    // ---- C2: U^T -> bf16 (hi, lo) A operands [i][s], K-major
    {
      float v[32];
      tmem_ld32(tmem + lane_off + TM_U + 32 * hc, v);
      tmem_wait_ld();
      store_row_hilo(sb + OFF_UTH, sb + OFF_UTL, row, 4 * hc, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*sAbort) { aborted = true; break; }

    // ---- C3: O^T += U^T P^T (as Uh Ph + Ul Ph + Uh Pl) ;  S += U^T K~ (as Uh K~ + Ul K~)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 12; ++k) {
        const uint32_t ua = (k < 4 || k >= 8) ? OFF_UTH : OFF_UTL;
        const uint32_t pb = (k < 8) ? OFF_PH : OFF_PL;
        mma_bf16(tmem + TM_O, sdesc_sw128(sb + ua + (k & 3) * 32, 16, 1024),
                 sdesc_sw128(sb + pb + (k & 3) * 32, 16, 1024), ID_SQ, true);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(tmem + TM_S, sdesc_sw128(sb + (k < 4 ? OFF_UTH : OFF_UTL) + (k & 3) * 32, 16, 1024),
                 sdesc_sw128(sb + OFF_KT + (k & 3) * 2048, 8 * KB, 1024), ID_UK, true);
      mma_commit(bar_mma);
    }
    if (!mbar_wait_bounded(bar_mma, mma_phase)) atomicExch(sAbort, 1);
    mma_phase ^= 1;
    tc_fence_after();
    // ---- C4: O^T -> staging [64 tokens][128] (row-major, out dtype) -> TMA store
    {
      float v[32];
      tmem_ld32(tmem + lane_off + TM_O + 32 * hc, v);
      tmem_wait_ld();
      Tout* stg = reinterpret_cast<Tout*>(sm + OFF_OUT);
#pragma unroll
      for (int j = 0; j < 32; ++j) stg[(32 * hc + j) * D + row] = from_float<Tout>(v[j]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*sAbort) { aborted = true; break; }
    if (tid == 0) {
      tma_store_3d(&tm_o, sb + OFF_OUT, h * D, t0, b);
      tma_store_commit();
    }
  }

  if (aborted) {
    if (tid == 0) {
      atomicOr(&g_err_tc, kErrTimeout);
      // bounded waits for this CTA's own copies / MMAs still in flight
      mbar_wait_bounded(bar_mma, mma_phase, 1u << 16);
      mbar_wait_bounded(bar_in0, 0, 1u << 16);
      mbar_wait_bounded(bar_in1, 0, 1u << 16);
      tma_store_wait_all();
    }
  } else {
    // ---- the leaving state: TMEM -> HBM (fp32)
    float v[32];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      tmem_ld32(tmem + lane_off + TM_S + 64 * hc + 32 * half, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        reinterpret_cast<float4*>(Sg + 32 * half)[j] =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    if (tid == 0) tma_store_wait_all();
  }
  tc_fence_before();
  __syncthreads();
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
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D map over [B][T][width] elements starting at `base`, token stride `tok_stride`
// elements; box = {box0, 64 tokens, 1 sequence}.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem_bytes,
              int width, int T, int B, long long tok_stride, int box0, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)(tok_stride * elem_bytes),
                           (cuuint64_t)(tok_stride * elem_bytes) * (cuuint64_t)T};
  cuuint32_t box[3] = {(cuuint32_t)box0, 64u, 1u};
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
  const bool ok =
      make_map(&mq, L.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hk * D, L.T, L.B, L.q_tok_stride,
               64, true) &&
      make_map(&mk, L.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hk * D, L.T, L.B, L.k_tok_stride,
               64, true) &&
      make_map(&mv, L.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, L.Hv * D, L.T, L.B, L.v_tok_stride,
               64, true) &&
      make_map(&mo, L.out,
               sizeof(Tout) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
               (int)sizeof(Tout), L.Hv * D, L.T, L.B, (long long)L.Hv * D, 128, false);
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
