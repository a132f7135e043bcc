// A decode step over T <= 16 new tokens per sequence (speculative multi-token verification,
// short prefill): the gated delta rule on the fp32 state already in HBM, as in the decode
// step, with the conv, the L2 norms and the gates fused in front, and optionally the state
// after every token written to checkpoint slots (so that a verifier can keep any accepted
// prefix).
//
// For the T tokens of one (sequence, value head) the chunked form of the recurrence holds
// with a T x T chunk (the same algebra as the prefill's 64-token chunks): with G_t the
// cumulative log-decay, A_ts = beta_t e^{G_t - G_s} (k_t . k_s) for s < t and
// P_ts = e^{G_t - G_s} (q_t . k_s) for s <= t,
//     u = (I + A)^{-1} (beta (v_i - e^{G} (k . s0_i)))          (per state row i)
//     o_t = e^{G_t} (q_t . s0_i) + sum_{s<=t} P_ts u_s
//     s_i <- e^{g_t} s_i + u_t k_t   after token t (t = 0 .. T-1).
// Row independence again: row i needs only its own T values of v, and its 2T dot products
// with the k_t and q_t are independent of each other, so a warp forms all 2T at once and one
// transposing warp reduction (31 shuffles) leaves lane l with dot product l.
//
// One CTA per (sequence, key head), or, at small batches, a thread-block cluster of nsplit
// CTAs that split the rows of each value head.  The prologue convolves the T tokens of the
// key head's q/k channels and of its own rows' v channels (and writes their new conv state),
// forms the norms, the gates and, per value head, (I + A)^{-1} and P in shared memory.  Then
// each warp streams state rows: one 512-byte row per warp access, coalesced.  All CTAs of a
// cluster read the old q/k conv state; a cluster barrier orders those reads before the one
// CTA (rank 0) that writes the new one.
#include "common.cuh"

using namespace gdn;

static __device__ unsigned int g_err_multi;

unsigned gdn_take_error_decode_multi() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_multi, sizeof(v));
  cudaMemcpyToSymbol(g_err_multi, &z, sizeof(z));
  return v;
}

namespace {

constexpr int D = kHeadDim;
constexpr int MT_THREADS = 256;
constexpr int MT_MAXT = 16;

__device__ __forceinline__ void cluster_arrive_relaxed_mt() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_mt() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

template <int V> struct Log2 { static constexpr int value = 1 + Log2<V / 2>::value; };
template <> struct Log2<1> { static constexpr int value = 0; };

// transposing warp reduction of V values per lane (V a power of two <= 32): log2 V halving
// levels, then plain butterfly levels; value v ends in lanes v * 32/V .. (v+1) * 32/V - 1
// (V - 1 + 5 - log2 V shuffles)
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&x)[V], int lane) {
  constexpr int LV = Log2<V>::value;
#pragma unroll
  for (int lvl = 0; lvl < LV; ++lvl) {
    const int m = 16 >> lvl, L = V >> lvl;
    const bool up = lane & m;
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      if (i < L / 2) {
        const float send = up ? x[i] : x[i + L / 2];
        const float keep = up ? x[i + L / 2] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
  }
  float r = x[0];
#pragma unroll
  for (int lvl = LV; lvl < 5; ++lvl) r += __shfl_xor_sync(0xffffffffu, r, 16 >> lvl);
  return r;
}

// shared-memory layout (floats) for T tokens and r value heads
struct MtLayout {
  int qh, kh, vv, kk, qk, mats, ostage, red, total;
  __host__ __device__ MtLayout(int T, int r) {
    qh = 0;
    kh = qh + T * D;
    vv = kh + T * D;
    kk = vv + T * r * D;
    qk = kk + T * T;
    mats = qk + T * T;                       // per value head: Tm [T][T], P [T][T], 4 x [T]
    ostage = mats + r * (2 * T * T + 4 * T);
    red = ostage + T * D;
    total = red + 64;
  }
};

// TM: the token capacity the loops are unrolled for (T <= TM)
template <typename Tin, typename Tout, int TM>
__global__ void __launch_bounds__(MT_THREADS) gdn_decode_multi_kernel(GdnLayerArgs p, int T,
                                                                      float* snap_state,
                                                                      int num_snap,
                                                                      const int32_t* snap_slots,
                                                                      Tin* snap_conv,
                                                                      int nsplit) {
  extern __shared__ __align__(16) float ms[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = p.Hv / p.Hk;
  const int item = blockIdx.x / nsplit, sp = blockIdx.x % nsplit;
  const int b = item / p.Hk, kh = item % p.Hk;
  const int R = D / nsplit, r_lo = sp * R;          // this CTA's rows of every value head
  const int slot = p.slots ? p.slots[b] : b;
  if (slot < 0) return;
  if (slot >= p.num_slots) {            // (decided per sequence: a whole cluster leaves)
    if (tid == 0 && kh == 0 && sp == 0) atomicOr(&g_err_multi, kErrIndex);
    return;
  }
  const MtLayout lay(T, r);
  float* qh = ms + lay.qh;
  float* khat = ms + lay.kh;
  float* vv = ms + lay.vv;
  float* KK = ms + lay.kk;
  float* QK = ms + lay.qk;
  float* red = ms + lay.red;
  const int W = p.W, H = W > 0 ? W - 1 : 0, C = p.C_conv;
  const int ch_qk = 2 * D, ch_all = ch_qk + r * R;
  // ---- 1. conv (+SiLU) of this CTA's channels over the T tokens, or plain loads; the new
  //      conv state, and the conv state after every token for the snapshots (for the q/k
  //      channels, which every CTA of a cluster reads, once the cluster's reads are done)
  float qkwin[3 + TM];                                  // this thread's q/k channel (tid < 256)
  int qkch = -1;
  for (int cl = tid; cl < ch_all; cl += MT_THREADS) {
    // local channel cl: q (0..127), k (128..255), then v of value head vh, row r_lo + vi
    const int vh = (cl - ch_qk) / R, vi = r_lo + (cl - ch_qk) % R;
    const int ch = cl < D ? kh * D + cl
                   : cl < ch_qk ? p.Hk * D + kh * D + (cl - D)
                                : 2 * p.Hk * D + (kh * r + vh) * D + vi;
    float win[3 + TM];
    if (W > 0) {
      const Tin* cs = (const Tin*)p.conv_state + (size_t)slot * H * C + ch;
      for (int i = 0; i < H; ++i) win[i] = ld_elem(cs + (size_t)i * C);
      for (int t = 0; t < T; ++t)
        win[H + t] = ld_elem((const Tin*)p.x + ((size_t)b * T + t) * C + ch);
      const float bias = p.conv_b ? ld_elem((const Tin*)p.conv_b + ch) : 0.f;
      const Tin* w = (const Tin*)p.conv_w + (size_t)ch * W;
      float wt[4];
      for (int j = 0; j < W; ++j) wt[j] = ld_elem(w + j);
      for (int t = 0; t < T; ++t) {
        float y = bias;
        for (int j = 0; j < W; ++j) y = fmaf(wt[j], win[t + j], y);
        y = p.silu ? silu_f(y) : y;
        if (cl < D) qh[t * D + cl] = y;
        else if (cl < ch_qk) khat[t * D + cl - D] = y;
        else vv[t * r * D + vh * D + vi] = y;
      }
      // new conv state: the last W-1 window entries; after token t: entries t+1 .. t+W-1
      if (cl < ch_qk) {
        qkch = ch;
        for (int i = 0; i < H + T; ++i) qkwin[i] = win[i];
      } else {
        Tin* csw = (Tin*)p.conv_state + (size_t)slot * H * C + ch;
        for (int i = 0; i < H; ++i) st_elem(csw + (size_t)i * C, win[T + i]);
        if (snap_conv && snap_slots)
          for (int t = 0; t < T; ++t) {
            const int sl = snap_slots[b * T + t];
            if (sl >= 0 && sl < num_snap)
              for (int i = 0; i < H; ++i)
                st_elem(snap_conv + ((size_t)sl * H + i) * C + ch, win[t + 1 + i]);
          }
      }
    } else {
      for (int t = 0; t < T; ++t) {
        float y;
        if (cl < D) {
          y = ld_elem((const Tin*)p.q + (((size_t)b * T + t) * p.Hk + kh) * D + cl);
          qh[t * D + cl] = y;
        } else if (cl < ch_qk) {
          y = ld_elem((const Tin*)p.k + (((size_t)b * T + t) * p.Hk + kh) * D + cl - D);
          khat[t * D + cl - D] = y;
        } else {
          y = ld_elem((const Tin*)p.v + (((size_t)b * T + t) * p.Hv + kh * r + vh) * D + vi);
          vv[t * r * D + vh * D + vi] = y;
        }
      }
    }
  }
  // every CTA of the cluster has read the old q/k conv state (the values are consumed)
  if (nsplit > 1) cluster_arrive_relaxed_mt();
  __syncthreads();
  // ---- 2. L2 norms of q_t and k_t (one warp per vector), q also times `scale`
  for (int vec = warp; vec < 2 * T; vec += MT_THREADS / 32) {
    float* x = (vec < T ? qh : khat) + (vec % T) * D;
    float4 v4 = reinterpret_cast<float4*>(x)[lane];
    const float ss = warp_sum(dot4(v4, v4));
    const float inv = (p.l2norm ? 1.0f / sqrtf(ss + p.eps) : 1.0f) * (vec < T ? p.scale : 1.0f);
    v4.x *= inv; v4.y *= inv; v4.z *= inv; v4.w *= inv;
    reinterpret_cast<float4*>(x)[lane] = v4;
  }
  __syncthreads();
  // ---- 3. KK_ts = k_t . k_s and QK_ts = q_t . k_s (a thread per pair, 2 T^2 <= 512; the
  //      thread walks its two vectors from rotated starting points so that a warp's lanes
  //      read different banks)
  for (int pr = tid; pr < 2 * T * T; pr += MT_THREADS) {
    const int which = pr / (T * T), t = (pr / T) % T, s2 = pr % T;
    const float4* a4 = reinterpret_cast<const float4*>((which ? qh : khat) + t * D);
    const float4* k4 = reinterpret_cast<const float4*>(khat + s2 * D);
    float d = 0.f;
#pragma unroll 8
    for (int j = 0; j < D / 4; ++j) {
      const int jj = (j + lane) & (D / 4 - 1);
      d += dot4(a4[jj], k4[jj]);
    }
    (which ? QK : KK)[t * T + s2] = d;
  }
  __syncthreads();
  // ---- 4. per value head: gates, G, (I + A)^{-1} and P (warp hh, lanes = tokens)
  for (int hh = warp; hh < r; hh += MT_THREADS / 32) {
    float* Tm = ms + lay.mats + hh * (2 * T * T + 4 * T);
    float* P = Tm + T * T;
    float* eG = P + T * T;          // e^{G_t}
    float* bt = eG + T;             // beta_t
    float* dk = bt + T;             // e^{G_{T-1} - G_t}
    float* eg = dk + T;             // e^{g_t}
    const int h = kh * r + hh;
    float g = 0.f, beta = 0.f;
    if (lane < T) {
      const size_t gi = ((size_t)b * T + lane) * p.Hv + h;
      if (p.gates_pre) {
        g = ((const float*)p.a)[gi];
        beta = ((const float*)p.b)[gi];
      } else {
        g = gate_g(ld_elem((const Tin*)p.a + gi), p.A_log[h], p.dt_bias ? p.dt_bias[h] : 0.f);
        beta = sigmoid_f(ld_elem((const Tin*)p.b + gi));
      }
    }
    float G = g;                    // inclusive prefix over tokens
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, G, o);
      if (lane >= o) G += y;
    }
    const float GT = __shfl_sync(0xffffffffu, G, T - 1);
    if (lane < T) {
      eG[lane] = expf(G);
      bt[lane] = beta;
      dk[lane] = expf(GT - G);
      eg[lane] = expf(g);
    }
    // A and P rows (lane t), then (I + A)^{-1} by forward substitution, column by column
    // (lane j owns column j; rows t > j in order)
    for (int s2 = 0; s2 < TM; ++s2) {
      const float Gs = __shfl_sync(0xffffffffu, G, s2 & 31);
      float a = 0.f, pp = 0.f;
      if (lane < T && s2 < T && s2 <= lane) {
        const float e = expf(G - Gs);
        if (s2 < lane) a = beta * e * KK[lane * T + s2];
        pp = e * QK[lane * T + s2];
      }
      if (lane < T && s2 < T) P[lane * T + s2] = pp;
      if (lane < T && s2 < T) Tm[lane * T + s2] = a;     // A for now
    }
    __syncwarp();
    if (lane < T) {
      const int j = lane;
      float col[TM];
      for (int t = 0; t < TM; ++t) col[t] = (t == j) ? 1.f : 0.f;
      for (int t = 0; t < TM; ++t) {
        if (t > j && t < T) {
          float acc = 0.f;
          for (int s2 = 0; s2 < TM; ++s2)
            if (s2 >= j && s2 < t) acc = fmaf(Tm[t * T + s2], col[s2], acc);
          col[t] = -acc;
        }
      }
      __syncwarp(__activemask());
      for (int t = 0; t < T; ++t) Tm[t * T + j] = col[t];
    }
  }
  __syncthreads();
  // ---- 5. the state rows: value head hh, rows warp, warp + 8, ... (the next row's load is
  //      issued before the current row's arithmetic)
  int* ssl = reinterpret_cast<int*>(red);              // this sequence's snapshot rows
  if (tid < TM) ssl[tid] = (snap_state && snap_slots && tid < T) ? snap_slots[b * T + tid] : -1;
  __syncthreads();
  constexpr int V = 2 * TM, SV = 32 / V;               // reduced values; lanes per value
  for (int hh = 0; hh < r; ++hh) {
    const int h = kh * r + hh;
    const float* Tm = ms + lay.mats + hh * (2 * T * T + 4 * T);
    const float* P = Tm + T * T;
    const float* eG = P + T * T;
    const float* bt = eG + T;
    const float* eg = bt + 2 * T;
    float* ost = ms + lay.ostage;
    float* Sh = p.state + ((size_t)slot * p.Hv + h) * D * D;
    // rows i, i + 8, ... two at a time for short token counts (independent chains that the
    // scheduler interleaves), one at a time for long ones (registers)
    constexpr int RPI = TM <= 8 ? 2 : 1;
    constexpr int STEP = RPI * (MT_THREADS / 32);
    float4 s_next[RPI];
#pragma unroll
    for (int q = 0; q < RPI; ++q)
      s_next[q] = reinterpret_cast<const float4*>(Sh + (size_t)(r_lo + warp + q * 8) * D)[lane];
    for (int i0 = r_lo + warp; i0 < r_lo + R; i0 += STEP) {
      float4 sr[RPI];
#pragma unroll
      for (int q = 0; q < RPI; ++q) {
        sr[q] = s_next[q];
        if (i0 + STEP < r_lo + R)
          s_next[q] = reinterpret_cast<const float4*>(Sh + (size_t)(i0 + STEP + q * 8) * D)[lane];
      }
      float red_v[RPI];
#pragma unroll
      for (int q = 0; q < RPI; ++q) {
        float x[V];
#pragma unroll
        for (int t = 0; t < TM; ++t) {
          const bool on = t < T;
          x[t] = on ? dot4(sr[q], reinterpret_cast<const float4*>(khat + t * D)[lane]) : 0.f;
          x[TM + t] = on ? dot4(sr[q], reinterpret_cast<const float4*>(qh + t * D)[lane]) : 0.f;
        }
        // value v (v < TM: k_v . s0_i; TM <= v: q_{v-TM} . s0_i) lands in lanes v * SV ..
        red_v[q] = transpose_reduce<V>(x, lane);
      }
      const int t = lane;
      float rhs[RPI], u[RPI], o[RPI];
#pragma unroll
      for (int q = 0; q < RPI; ++q) {
        const int i = i0 + q * 8;
        const float ai = __shfl_sync(0xffffffffu, red_v[q], (t * SV) & 31);
        const float ci = __shfl_sync(0xffffffffu, red_v[q], ((TM + t) * SV) & 31);
        rhs[q] = (t < T) ? bt[t] * (vv[t * r * D + hh * D + i] - eG[t] * ai) : 0.f;
        o[q] = (t < T) ? eG[t] * ci : 0.f;
        u[q] = 0.f;
      }
      // u = (I + A)^{-1} rhs, lane t
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2) {
        const float tm = (s2 < T && t < T && s2 <= t) ? Tm[t * T + s2] : 0.f;
#pragma unroll
        for (int q = 0; q < RPI; ++q) u[q] = fmaf(tm, __shfl_sync(0xffffffffu, rhs[q], s2), u[q]);
      }
      // outputs and the state after each token
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2) {
        if (s2 < T) {
          const float pv = (t < T && s2 <= t) ? P[t * T + s2] : 0.f;
          const float4 k4 = reinterpret_cast<const float4*>(khat + s2 * D)[lane];
          const float e = eg[s2];
          const int sl = ssl[s2];
#pragma unroll
          for (int q = 0; q < RPI; ++q) {
            const float us = __shfl_sync(0xffffffffu, u[q], s2);
            o[q] = fmaf(pv, us, o[q]);
            sr[q].x = fmaf(e, sr[q].x, us * k4.x);
            sr[q].y = fmaf(e, sr[q].y, us * k4.y);
            sr[q].z = fmaf(e, sr[q].z, us * k4.z);
            sr[q].w = fmaf(e, sr[q].w, us * k4.w);
            if (sl >= 0 && sl < num_snap)
              reinterpret_cast<float4*>(snap_state +
                                        (((size_t)sl * p.Hv + h) * D + i0 + q * 8) * D)[lane] = sr[q];
          }
        }
      }
#pragma unroll
      for (int q = 0; q < RPI; ++q) {
        const int i = i0 + q * 8;
        reinterpret_cast<float4*>(Sh + (size_t)i * D)[lane] = sr[q];
        if (t < T) ost[t * D + i] = o[q];
      }
    }
    __syncthreads();
    // this head's outputs, token rows of 128 channels
    for (int e = tid; e < T * R; e += MT_THREADS) {
      const int tt = e / R, c = r_lo + e % R;
      st_elem((Tout*)p.out + (((size_t)b * T + tt) * p.Hv + h) * D + c, ost[tt * D + c]);
    }
    __syncthreads();
  }
  // the q/k channels' new conv state (and per-token snapshots): rank 0, after the cluster's
  // reads of the old one
  if (nsplit > 1) cluster_wait_mt();
  if (sp == 0 && W > 0 && qkch >= 0) {
    Tin* csw = (Tin*)p.conv_state + (size_t)slot * H * C + qkch;
    for (int i = 0; i < H; ++i) st_elem(csw + (size_t)i * C, qkwin[T + i]);
    if (snap_conv && snap_slots)
      for (int t = 0; t < T; ++t) {
        const int sl = snap_slots[b * T + t];
        if (sl >= 0 && sl < num_snap)
          for (int i = 0; i < H; ++i)
            st_elem(snap_conv + ((size_t)sl * H + i) * C + qkch, qkwin[t + 1 + i]);
      }
  }
  if (tid == 0 && sp == 0 && snap_slots)
    for (int t = 0; t < T; ++t)
      if (snap_slots[b * T + t] >= num_snap && kh == 0) atomicOr(&g_err_multi, kErrIndex);
}

template <typename Tin, typename Tout, int TM>
cudaError_t launch_multi_tm(const GdnLayerArgs& p, int T, float* snap_state, int num_snap,
                            const int32_t* snap_slots, void* snap_conv, cudaStream_t stream) {
  const MtLayout lay(T, p.Hv / p.Hk);
  const size_t smem = sizeof(float) * lay.total;
  static unsigned done = 0;
  cudaError_t e = set_smem_once(gdn_decode_multi_kernel<Tin, Tout, TM>,
                                (int)(sizeof(float) * MtLayout(TM, 8).total), &done);
  if (e != cudaSuccess) return e;
  // rows of each value head split over a cluster of nsplit CTAs when the (sequence, key head)
  // items alone would leave most SMs idle
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int nitems = p.B * p.Hk;
  int nsplit = 1;
  while (nsplit < 8 && nitems * nsplit * 2 <= 2 * sms) nsplit *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nitems * nsplit), 1, 1);
  cfg.blockDim = dim3(MT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nsplit > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gdn_decode_multi_kernel<Tin, Tout, TM>, p, T, snap_state,
                            num_snap, snap_slots, static_cast<Tin*>(snap_conv), nsplit);
}

template <typename Tin, typename Tout>
cudaError_t launch_multi_t(const GdnLayerArgs& p, int T, float* snap_state, int num_snap,
                           const int32_t* snap_slots, void* snap_conv, cudaStream_t stream) {
  if (T <= 2) return launch_multi_tm<Tin, Tout, 2>(p, T, snap_state, num_snap, snap_slots, snap_conv, stream);
  if (T <= 4) return launch_multi_tm<Tin, Tout, 4>(p, T, snap_state, num_snap, snap_slots, snap_conv, stream);
  if (T <= 8) return launch_multi_tm<Tin, Tout, 8>(p, T, snap_state, num_snap, snap_slots, snap_conv, stream);
  return launch_multi_tm<Tin, Tout, 16>(p, T, snap_state, num_snap, snap_slots, snap_conv, stream);
}

}  // namespace

cudaError_t gdn_launch_decode_multi(const GdnLayerArgs& p, float* snap_state, int num_snap,
                                    const int32_t* snap_slots, void* snap_conv,
                                    cudaStream_t stream) {
  if (p.B == 0 || p.T == 0) return cudaSuccess;
  if (p.T > MT_MAXT) return cudaErrorInvalidValue;
  if (p.in_bf16 && p.out_bf16)
    return launch_multi_t<__nv_bfloat16, __nv_bfloat16>(p, p.T, snap_state, num_snap,
                                                         snap_slots, snap_conv, stream);
  if (p.in_bf16)
    return launch_multi_t<__nv_bfloat16, float>(p, p.T, snap_state, num_snap, snap_slots,
                                                snap_conv, stream);
  return launch_multi_t<float, float>(p, p.T, snap_state, num_snap, snap_slots, snap_conv,
                                      stream);
}
