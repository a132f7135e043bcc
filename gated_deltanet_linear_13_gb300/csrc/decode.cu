// Batched single-token decode of the gated delta rule: one fused kernel.
//
// Per (sequence b, value head h) the step is the model card's "How It Works" loop for one
// token (decay, read, delta, write, output) on the fp32 state S[v][k] already in HBM, with
// the causal conv update (+SiLU), the L2 norm of q and k and the gates fused in front.
//
// Row independence: row i of S only needs v_i, and the output o_i only needs row i:
//     alpha = s_i . k,  gamma = s_i . q,  delta_i = beta (v_i - e^g alpha),
//     s_i <- e^g s_i + delta_i k,        o_i = e^g gamma + delta_i (k . q)
// (o = S_new q = e^g S q + delta (k . q)), so each row is streamed through once.
//
// Work split: a persistent grid of four CTAs per SM; a CTA takes whole (sequence, key head)
// items in turn.  Per item it runs the conv (+SiLU) of the key head's q/k channels and of its
// r = Hv/Hk value heads' v channels once, writes their new conv state itself (no other CTA
// touches those channels, so no ordering across CTAs is needed), forms the L2 norms and the
// gates, and then streams the item's r x 128 state rows through shared memory in 32-row
// blocks of 16 KB: a three-stage ring of TMA bulk copies (loads run two blocks ahead, across
// item boundaries, while the updated blocks leave with bulk stores).  In shared memory one
// warp handles a 512-byte row with 128-bit accesses and two warp-wide dot products.
//
// With the gated output norm (out = w o / sqrt(mean(o^2) + eps) silu(z) over the 128 outputs
// of a value head) the outputs of an item wait in shared memory, in the slots of the v values
// they replace, and the head's last block normalises and stores all 128 of them.
#include "common.cuh"
#include "sm100_ptx.cuh"

using namespace gdn;
using namespace gdn::ptx;

static __device__ unsigned int g_err_decode;

unsigned gdn_take_error_decode() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_decode, sizeof(v));
  cudaMemcpyToSymbol(g_err_decode, &z, sizeof(z));
  return v;
}

// Conv of one channel: window = [old state (W-1 values, oldest first), new input]; the new
// state (the last W-1 inputs) is written back by the caller through conv_store_state.
template <typename Tin>
__device__ __forceinline__ float conv_channel(const GdnLayerArgs& p, int slot, int b, int ch,
                                              float (&win)[4]) {
  const int W = p.W, C = p.C_conv;
  const Tin* cs = (const Tin*)p.conv_state + (size_t)slot * (W - 1) * C;
  const float xn = ld_elem((const Tin*)p.x + (size_t)b * C + ch);
#pragma unroll
  for (int i = 0; i < 4; ++i) win[i] = 0.f;
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (i < W - 1) win[i] = ld_elem(cs + (size_t)i * C + ch);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i == W - 1) win[i] = xn;
  float y = p.conv_b ? ld_elem((const Tin*)p.conv_b + ch) : 0.f;
  const Tin* w = (const Tin*)p.conv_w + (size_t)ch * W;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < W) y = fmaf(ld_elem(w + i), win[i], y);
  return p.silu ? silu_f(y) : y;
}

template <typename Tin>
__device__ __forceinline__ void conv_store_state(const GdnLayerArgs& p, int slot, int ch,
                                                 const float (&win)[4]) {
  const int W = p.W, C = p.C_conv;
  Tin* cs = (Tin*)p.conv_state + (size_t)slot * (W - 1) * C;
#pragma unroll
  for (int i = 0; i < 3; ++i)
    if (i < W - 1) st_elem(cs + (size_t)i * C + ch, win[i + 1]);
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

constexpr int DEC_THREADS = 256;
constexpr int DEC_RB = 32;                           // state rows per streamed block
constexpr int DEC_NS = 3;                            // ring stages
constexpr int DEC_CPS = 4;                           // CTAs per SM
constexpr int DEC_MAXR = 8;                          // value heads per key head (at most)
constexpr int DEC_BPH = kHeadDim / DEC_RB;          // blocks per value head
constexpr uint32_t DEC_BLOCK_BYTES = DEC_RB * kHeadDim * 4;
// shared memory: ring | q^ | k^ | v (r heads) | e^g, beta per head | outputs x 2 | reduce | bars
constexpr uint32_t DEC_OFF_Q = DEC_NS * DEC_BLOCK_BYTES;
constexpr uint32_t DEC_OFF_K = DEC_OFF_Q + kHeadDim * 4;
constexpr uint32_t DEC_OFF_V = DEC_OFF_K + kHeadDim * 4;
constexpr uint32_t DEC_OFF_G = DEC_OFF_V + DEC_MAXR * kHeadDim * 4;
constexpr uint32_t DEC_OFF_O = DEC_OFF_G + 2 * DEC_MAXR * 4;
constexpr uint32_t DEC_OFF_RED = DEC_OFF_O + 2 * DEC_RB * 4;
constexpr uint32_t DEC_OFF_BAR = DEC_OFF_RED + 32 * 4;
constexpr uint32_t DEC_SMEM = DEC_OFF_BAR + DEC_NS * 8 + 128;   // + alignment slack

// The sequence of (item, block) pairs a CTA processes: items blockIdx.x, +gridDim.x, ...
// whose sequence has a valid state slot, r * DEC_BPH blocks each.
struct DecCursor {
  int item, blk;
};

__device__ __forceinline__ bool dec_item_valid(const GdnLayerArgs& p, int item) {
  const int b = item / p.Hk;
  const int slot = p.slots ? p.slots[b] : b;
  if (slot >= p.num_slots) {
    if ((item % p.Hk) == 0 && threadIdx.x == 0) atomicOr(&g_err_decode, kErrIndex);
    return false;
  }
  return slot >= 0;
}

__device__ __forceinline__ void dec_first(const GdnLayerArgs& p, int nitems, DecCursor& c) {
  c.item = blockIdx.x;
  c.blk = 0;
  while (c.item < nitems && !dec_item_valid(p, c.item)) c.item += gridDim.x;
}

__device__ __forceinline__ void dec_advance(const GdnLayerArgs& p, int nitems, int nblk,
                                            DecCursor& c) {
  if (c.item >= nitems) return;
  if (++c.blk < nblk) return;
  c.blk = 0;
  do {
    c.item += gridDim.x;
  } while (c.item < nitems && !dec_item_valid(p, c.item));
}

// GATE: the gated output norm (a separate instantiation, so that the plain step keeps its
// own schedule).
template <typename Tin, typename Tout, bool GATE>
__global__ void __launch_bounds__(DEC_THREADS, DEC_CPS) gdn_decode_stream_kernel(GdnLayerArgs p) {
  constexpr int D = kHeadDim;
  constexpr int RPW = DEC_RB / (DEC_THREADS / 32);    // rows per warp in a block
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((128u - (smem_addr(dsm_raw) & 127u)) & 127u);
  float* ring = reinterpret_cast<float*>(dsm);
  float* sq = reinterpret_cast<float*>(dsm + DEC_OFF_Q);
  float* sk = reinterpret_cast<float*>(dsm + DEC_OFF_K);
  float* sv = reinterpret_cast<float*>(dsm + DEC_OFF_V);
  float* sg = reinterpret_cast<float*>(dsm + DEC_OFF_G);
  float* so = reinterpret_cast<float*>(dsm + DEC_OFF_O);
  float* red = reinterpret_cast<float*>(dsm + DEC_OFF_RED);
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + DEC_OFF_BAR);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = p.Hv / p.Hk, nblk = DEC_BPH * r, nitems = p.B * p.Hk;

  // state rows of block (item, blk): value head kh * r + blk / DEC_BPH, rows from
  // (blk % DEC_BPH) * DEC_RB
  auto block_src = [&](const DecCursor& c) -> float* {
    const int b = c.item / p.Hk, kh = c.item % p.Hk;
    const int slot = p.slots ? p.slots[b] : b;
    const int h = kh * r + c.blk / DEC_BPH;
    // (the -DGDN_BOUNDS_CHECK build: a row out of the state array is recorded and replaced by
    // row 0, so that the copy pipeline keeps its shape)
    if (!in_bounds(&g_err_decode, slot >= 0 && slot < p.num_slots && h < p.Hv && b < p.B))
      return p.state;
    return p.state + (((size_t)slot * p.Hv + h) * D + (size_t)(c.blk % DEC_BPH) * DEC_RB) * D;
  };
  // ---- producer state (thread 0): loads run DEC_NS - 1 blocks ahead of the consumers
  DecCursor pc;
  int pk = 0;                                          // ordinal of the next block to load
  bool ok = true;
  if (tid == 0) {
    for (int s = 0; s < DEC_NS; ++s) mbar_init(smem_addr(&full[s]), 1);
    fence_mbar_init();
    dec_first(p, nitems, pc);
    for (; pk < DEC_NS - 1 && pc.item < nitems; ++pk) {
      const uint32_t bar = smem_addr(&full[pk % DEC_NS]);
      mbar_arrive_expect_tx(bar, DEC_BLOCK_BYTES);
      bulk_load(smem_addr(ring) + (pk % DEC_NS) * DEC_BLOCK_BYTES, block_src(pc), DEC_BLOCK_BYTES,
                bar);
      dec_advance(p, nitems, nblk, pc);
    }
  }
  __syncthreads();

  DecCursor c;
  dec_first(p, nitems, c);
  float kq = 0.f;
  float zg = 0.f;                                      // gate of output channel tid (< 128)
  int k = 0;                                           // ordinal of the block being consumed
  for (; c.item < nitems; ++k) {
    const int b = c.item / p.Hk, kh = c.item % p.Hk;
    const int slot = p.slots ? p.slots[b] : b;
    if (c.blk == 0) {
      // (gated: the previous item's last head may still be reading its outputs out of sv)
      if (GATE) __syncthreads();
      // ---- item prologue: conv (+SiLU) of q, k (threads 0..127: q_j, 128..255: k_j) and of
      //      the r value heads' v channels, their new conv state, norms, k.q, gates
      const int j = tid & (D - 1);
      const bool isk = tid >= D;
      float val, win[4];
      if (p.W > 0) {
        const int ch = (isk ? p.Hk * D : 0) + kh * D + j;
        val = conv_channel<Tin>(p, slot, b, ch, win);
        if (p.W > 1) conv_store_state<Tin>(p, slot, ch, win);
      } else {
        const Tin* src = isk ? (const Tin*)p.k : (const Tin*)p.q;
        val = ld_elem(src + ((size_t)b * p.Hk + kh) * D + j);
      }
      for (int cv = tid; cv < r * D; cv += DEC_THREADS) {
        float vv;
        if (p.W > 0) {
          const int ch = 2 * p.Hk * D + kh * r * D + cv;
          float wv[4];
          vv = conv_channel<Tin>(p, slot, b, ch, wv);
          if (p.W > 1) conv_store_state<Tin>(p, slot, ch, wv);
        } else {
          vv = ld_elem((const Tin*)p.v + ((size_t)b * p.Hv + kh * r) * D + cv);
        }
        sv[cv] = vv;
      }
      if (tid < r) {
        const int h = kh * r + tid;
        const size_t gi = (size_t)b * p.Hv + h;
        float g, beta;
        if (p.gates_pre) {
          g = ((const float*)p.a)[gi];
          beta = ((const float*)p.b)[gi];
        } else {
          g = gate_g(ld_elem((const Tin*)p.a + gi), p.A_log[h], p.dt_bias ? p.dt_bias[h] : 0.f);
          beta = sigmoid_f(ld_elem((const Tin*)p.b + gi));
        }
        sg[2 * tid] = expf(g);
        sg[2 * tid + 1] = beta;
      }
      const float ss = warp_sum(val * val);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      {
        const float n2 = isk ? (red[4] + red[5] + red[6] + red[7])
                             : (red[0] + red[1] + red[2] + red[3]);
        const float inv = p.l2norm ? 1.0f / sqrtf(n2 + p.eps) : 1.0f;
        const float hat = val * inv * (isk ? 1.0f : p.scale);
        if (isk) sk[j] = hat; else sq[j] = hat;
      }
      __syncthreads();
      if (tid < D) {
        const float t = warp_sum(sq[tid] * sk[tid]);
        if (lane == 0) red[8 + warp] = t;
      }
      __syncthreads();
      kq = red[8] + red[9] + red[10] + red[11];
    }
    // ---- the block: rows r0 .. r0 + DEC_RB - 1 of value head hh
    const int hh = c.blk / DEC_BPH, r0 = (c.blk % DEC_BPH) * DEC_RB;
    const int h = kh * r + hh;
    if (GATE && c.blk % DEC_BPH == 0 && tid < D)        // used at the head's last block
      zg = ld_elem((const Tin*)p.gate_z + ((size_t)b * p.Hv + h) * D + tid);
    const float eg = sg[2 * hh], beta = sg[2 * hh + 1];
    const float4 k4 = reinterpret_cast<const float4*>(sk)[lane];
    const float4 q4 = reinterpret_cast<const float4*>(sq)[lane];
    const int st = k % DEC_NS;
    float* blkp = ring + st * (DEC_BLOCK_BYTES / 4);
    if (!mbar_wait_bounded(smem_addr(&full[st]), (k / DEC_NS) & 1)) ok = false;
    float* Sw = blkp + warp * RPW * D;
    float4 s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) s[i] = reinterpret_cast<const float4*>(Sw + i * D)[lane];
    float* sob = so + (k & 1) * DEC_RB;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int row = warp * RPW + i;
      float vi = 0.f;
      if (GATE) vi = sv[hh * D + r0 + row];
      const float al = warp_sum(dot4(s[i], k4));
      const float ga = warp_sum(dot4(s[i], q4));
      if (!GATE) vi = sv[hh * D + r0 + row];
      const float delta = beta * (vi - eg * al);
      float4 t;
      t.x = fmaf(eg, s[i].x, delta * k4.x);
      t.y = fmaf(eg, s[i].y, delta * k4.y);
      t.z = fmaf(eg, s[i].z, delta * k4.z);
      t.w = fmaf(eg, s[i].w, delta * k4.w);
      reinterpret_cast<float4*>(Sw + i * D)[lane] = t;
      const float o = fmaf(eg, ga, delta * kq);
      if (GATE) {
        __syncwarp();                                  // every lane has read v_i
        if (lane == 0) sv[hh * D + r0 + row] = o;
      } else if (lane == 0) {
        sob[row] = o;
      }
    }
    fence_proxy_async_smem();
    if (!__syncthreads_and(ok)) {
      if (tid == 0) atomicOr(&g_err_decode, kErrTimeout);
      break;
    }
    if (tid == 0) {
      bulk_store(block_src(c), smem_addr(blkp), DEC_BLOCK_BYTES);
      tma_store_commit();
      // refill the stage of the previous block once its store has read shared memory
      if (pc.item < nitems) {
        tma_store_wait_read_1();
        const int ps = pk % DEC_NS;
        const uint32_t bar = smem_addr(&full[ps]);
        mbar_arrive_expect_tx(bar, DEC_BLOCK_BYTES);
        bulk_load(smem_addr(ring) + ps * DEC_BLOCK_BYTES, block_src(pc), DEC_BLOCK_BYTES, bar);
        dec_advance(p, nitems, nblk, pc);
        ++pk;
      }
    }
    if (!GATE) {
      if (tid < DEC_RB) {
        Tout* o = (Tout*)p.out + ((size_t)b * p.Hv + h) * D + r0 + tid;
        *o = from_float<Tout>(sob[tid]);
      }
    } else if (c.blk % DEC_BPH == DEC_BPH - 1 && tid < D) {
      // the head's 128 outputs are complete: gated RMS norm over them (warps 0-3)
      const float ov = sv[hh * D + tid];
      const float ssum = warp_sum(ov * ov);
      if (lane == 0) red[16 + warp] = ssum;
      named_bar_sync(1, D);
      const float inv = rsqrtf((red[16] + red[17] + red[18] + red[19]) * (1.0f / D) + p.gate_eps);
      Tout* o = (Tout*)p.out + ((size_t)b * p.Hv + h) * D + tid;
      *o = from_float<Tout>(p.gate_w[tid] * (ov * inv) * silu_gate(zg));
    }
    dec_advance(p, nitems, nblk, c);
  }
  // Stores must have read shared memory before it is released; so must every load issued
  // ahead of a block that an abort left unconsumed (ordinals k .. pk - 1) have landed.
  if (tid == 0) {
    tma_store_wait_read();
    for (int o = k; o < pk; ++o)
      mbar_wait_bounded(smem_addr(&full[o % DEC_NS]), (o / DEC_NS) & 1, 1u << 16);
  }
}

// ======================================================================= small batches
// When there are fewer (sequence, key head) items than about two per SM, the stream above
// leaves SMs idle.  Then a thread-block cluster per item spreads it over r value heads times
// `nsplit` row blocks of R = 128/nsplit rows, one CTA each: every CTA recomputes the conv of
// the shared q/k channels, and the cluster barrier orders all CTAs' reads of the old q/k
// conv state before the one CTA that writes the new one (the v channels of rows
// [r0, r0+R) belong to one CTA only).  A CTA's R rows move with one bulk copy in, issued
// before the prologue, and one bulk store out.
// Relaxed arrive: the only ordering needed is "every CTA's loads of the old conv state have
// returned before the writer stores the new one", and those loaded values are consumed (a
// data dependence) before the arrive.  A release arrive would also wait for the state-row
// loads already in flight, which stalls the stream.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
// A float in the shared memory of cluster CTA `rank`, at the offset of `local` here.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
               : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <typename Tin, typename Tout, int R>
__global__ void __launch_bounds__(256) gdn_decode_cluster_kernel(GdnLayerArgs p, int nsplit) {
  constexpr int D = kHeadDim;
  constexpr int RPW = R / 8;  // rows per warp
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = p.Hv / p.Hk;
  const int csize = r * nsplit;
  const int crank = blockIdx.x % csize;
  const int group = blockIdx.x / csize;
  const int b = group / p.Hk, kh = group % p.Hk;
  const int hh = crank / nsplit, sp = crank % nsplit;
  const int h = kh * r + hh;
  const int r0 = sp * R;

  // Skip decisions depend on b only, so a whole cluster leaves together.
  const int slot = p.slots ? p.slots[b] : b;
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (tid == 0 && crank == 0) atomicOr(&g_err_decode, kErrIndex);
    return;
  }

  // The state rows do not depend on the conv / norm / gates: one bulk copy brings this CTA's
  // R rows into shared memory while the prologue runs.
  extern __shared__ __align__(128) float sS[];   // [R][D]
  __shared__ __align__(8) uint64_t sbar;
  float* Sg = p.state + (((size_t)slot * p.Hv + h) * D + r0) * D;
  const uint32_t bar = smem_addr(&sbar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, R * D * 4);
    bulk_load(smem_addr(sS), Sg, R * D * 4, bar);
  }

  __shared__ __align__(16) float sq[D];
  __shared__ __align__(16) float sk[D];
  __shared__ float sv[R];
  __shared__ float so[R];
  __shared__ float red[16];
  __shared__ float sgate[2];
  __shared__ float spart;                        // gated norm: sum of squares of this CTA's outputs
  // gated norm: the gate of this CTA's output channel r0 + tid
  const float zg = (p.gate && tid < R)
                       ? ld_elem((const Tin*)p.gate_z + ((size_t)b * p.Hv + h) * D + r0 + tid)
                       : 0.f;

  // ---- 1. conv (+SiLU) or plain load of q, k (threads 0..127: q_j, 128..255: k_j)
  const int j = tid & (D - 1);
  const bool isk = tid >= D;
  float win[4];
  float val;
  int ch = 0;
  if (p.W > 0) {
    ch = (isk ? p.Hk * D : 0) + kh * D + j;
    val = conv_channel<Tin>(p, slot, b, ch, win);
  } else {
    const Tin* src = isk ? (const Tin*)p.k : (const Tin*)p.q;
    val = ld_elem(src + ((size_t)b * p.Hk + kh) * D + j);
  }
  // v channels of this CTA's rows
  float winv[4];
  float vval = 0.f;
  int chv = 0;
  if (tid < R) {
    if (p.W > 0) {
      chv = 2 * p.Hk * D + h * D + r0 + tid;
      vval = conv_channel<Tin>(p, slot, b, chv, winv);
    } else {
      vval = ld_elem((const Tin*)p.v + ((size_t)b * p.Hv + h) * D + r0 + tid);
    }
    sv[tid] = vval;
  }
  // gates
  if (tid == 0) {
    const size_t gi = (size_t)b * p.Hv + h;
    float g, beta;
    if (p.gates_pre) {
      g = ((const float*)p.a)[gi];
      beta = ((const float*)p.b)[gi];
    } else {
      g = gate_g(ld_elem((const Tin*)p.a + gi), p.A_log[h], p.dt_bias ? p.dt_bias[h] : 0.f);
      beta = sigmoid_f(ld_elem((const Tin*)p.b + gi));
    }
    sgate[0] = g;
    sgate[1] = beta;
  }
  // ---- 2. L2 norms of q (warps 0-3) and k (warps 4-7)
  float ss = warp_sum(val * val);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  // every CTA of the cluster has now read the old conv state it needs
  cluster_arrive_relaxed();
  {
    const float n2 = isk ? (red[4] + red[5] + red[6] + red[7]) : (red[0] + red[1] + red[2] + red[3]);
    const float inv = p.l2norm ? 1.0f / sqrtf(n2 + p.eps) : 1.0f;
    const float hat = val * inv * (isk ? 1.0f : p.scale);
    if (isk) sk[j] = hat; else sq[j] = hat;
  }
  __syncthreads();
  if (tid < D) {
    float kq = warp_sum(sq[tid] * sk[tid]);
    if (lane == 0) red[8 + warp] = kq;
  }
  __syncthreads();
  const float kq = red[8] + red[9] + red[10] + red[11];
  const float g = sgate[0], beta = sgate[1];
  const float eg = expf(g);

  // ---- 3. update this CTA's R rows of S in shared memory: each warp owns RPW rows
  const float4 k4 = reinterpret_cast<const float4*>(sk)[lane];
  const float4 q4 = reinterpret_cast<const float4*>(sq)[lane];
  const bool landed = mbar_wait_bounded(bar, 0);
  if (!landed && tid == 0) atomicOr(&g_err_decode, kErrTimeout);
  float* Sw = sS + warp * RPW * D;
  float4 s[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) s[i] = reinterpret_cast<const float4*>(Sw + i * D)[lane];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const float al = warp_sum(dot4(s[i], k4));
    const float ga = warp_sum(dot4(s[i], q4));
    const int row = warp * RPW + i;
    const float delta = beta * (sv[row] - eg * al);
    float4 t;
    t.x = fmaf(eg, s[i].x, delta * k4.x);
    t.y = fmaf(eg, s[i].y, delta * k4.y);
    t.z = fmaf(eg, s[i].z, delta * k4.z);
    t.w = fmaf(eg, s[i].w, delta * k4.w);
    reinterpret_cast<float4*>(Sw + i * D)[lane] = t;
    if (lane == 0) so[row] = fmaf(eg, ga, delta * kq);
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0 && landed) {
    bulk_store(Sg, smem_addr(sS), R * D * 4);
    tma_store_commit();
  }
  // ---- 4. outputs and conv state
  if (!p.gate) {
    if (tid < R) {
      Tout* o = (Tout*)p.out + ((size_t)b * p.Hv + h) * D + r0 + tid;
      *o = from_float<Tout>(so[tid]);
      if (p.W > 1) conv_store_state<Tin>(p, slot, chv, winv);
    }
    cluster_wait_acquire();
    if (p.W > 1 && hh == 0 && sp == 0) conv_store_state<Tin>(p, slot, ch, win);
  } else {
    // gated RMS norm over the head's 128 outputs, spread over its nsplit CTAs: each CTA's
    // sum of squares goes to its shared memory, a cluster barrier publishes it, every CTA
    // adds the head's partial sums, and a last barrier keeps every CTA (and its partial sum)
    // alive until all reads are done
    if (warp == 0) {
      float acc = 0.f;
      for (int i = lane; i < R; i += 32) acc = fmaf(so[i], so[i], acc);
      acc = warp_sum(acc);
      if (lane == 0) spart = acc;
    }
    if (tid < R && p.W > 1) conv_store_state<Tin>(p, slot, chv, winv);
    cluster_wait_acquire();
    if (p.W > 1 && hh == 0 && sp == 0) conv_store_state<Tin>(p, slot, ch, win);
    cluster_arrive_release();
    cluster_wait_acquire();
    float tot = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) tot += ld_cluster_f32(&spart, (uint32_t)(hh * nsplit + s2));
    const float inv = rsqrtf(tot * (1.0f / D) + p.gate_eps);
    if (tid < R) {
      Tout* o = (Tout*)p.out + ((size_t)b * p.Hv + h) * D + r0 + tid;
      *o = from_float<Tout>(p.gate_w[r0 + tid] * (so[tid] * inv) * silu_gate(zg));
    }
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  if (tid == 0) tma_store_wait_read();    // the bulk store has read shared memory
}

template <typename Tin, typename Tout, int R>
static cudaError_t launch_decode_cluster_t(const GdnLayerArgs& p, int nsplit, cudaStream_t stream) {
  static unsigned done = 0;
  cudaError_t e = set_smem_once(gdn_decode_cluster_kernel<Tin, Tout, R>, R * kHeadDim * 4, &done);
  if (e != cudaSuccess) return e;
  const int r = p.Hv / p.Hk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.Hk * r * nsplit), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = (size_t)R * kHeadDim * 4;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)(r * nsplit);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gdn_decode_cluster_kernel<Tin, Tout, R>, p, nsplit);
}

static cudaError_t launch_decode_cluster(const GdnLayerArgs& p, cudaStream_t stream) {
  const int r = p.Hv / p.Hk;
  int nsplit = 8 / r;           // cluster of r * nsplit <= 8 CTAs
  if (nsplit >= 8) nsplit = 8;
  else if (nsplit >= 4) nsplit = 4;
  else if (nsplit >= 2) nsplit = 2;
  else nsplit = 1;
  const int R = kHeadDim / nsplit;
#define GDN_DEC(TI, TO)                                                         \
  switch (R) {                                                                  \
    case 16: return launch_decode_cluster_t<TI, TO, 16>(p, nsplit, stream);             \
    case 32: return launch_decode_cluster_t<TI, TO, 32>(p, nsplit, stream);             \
    case 64: return launch_decode_cluster_t<TI, TO, 64>(p, nsplit, stream);             \
    default: return launch_decode_cluster_t<TI, TO, 128>(p, nsplit, stream);            \
  }
  if (p.in_bf16) {
    if (p.out_bf16) { GDN_DEC(__nv_bfloat16, __nv_bfloat16) }
    GDN_DEC(__nv_bfloat16, float)
  }
  GDN_DEC(float, float)
#undef GDN_DEC
}

template <typename Tin, typename Tout, bool GATE>
static cudaError_t launch_stream(const GdnLayerArgs& p, int grid, unsigned (*done)[2],
                                 cudaStream_t stream) {
  cudaError_t e = set_smem_once(gdn_decode_stream_kernel<Tin, Tout, GATE>, (int)DEC_SMEM,
                                &(*done)[GATE ? 1 : 0]);
  if (e != cudaSuccess) return e;
  gdn_decode_stream_kernel<Tin, Tout, GATE><<<grid, DEC_THREADS, DEC_SMEM, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t gdn_launch_decode(const GdnLayerArgs& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  static unsigned done_bb[2] = {0, 0}, done_bf[2] = {0, 0}, done_ff[2] = {0, 0};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int nitems = p.B * p.Hk;
  if (nitems < 2 * sms) return launch_decode_cluster(p, stream);
  const int grid = nitems < sms * DEC_CPS ? nitems : sms * DEC_CPS;
  if (p.in_bf16 && p.out_bf16)
    return p.gate ? launch_stream<__nv_bfloat16, __nv_bfloat16, true>(p, grid, &done_bb, stream)
                  : launch_stream<__nv_bfloat16, __nv_bfloat16, false>(p, grid, &done_bb, stream);
  if (p.in_bf16)
    return p.gate ? launch_stream<__nv_bfloat16, float, true>(p, grid, &done_bf, stream)
                  : launch_stream<__nv_bfloat16, float, false>(p, grid, &done_bf, stream);
  return p.gate ? launch_stream<float, float, true>(p, grid, &done_ff, stream)
                : launch_stream<float, float, false>(p, grid, &done_ff, stream);
}
