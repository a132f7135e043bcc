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
// Row independence again: row i needs only its own T values of v and its 2T dot products
// with the k_t and q_t.  Eight lanes share a row (16 elements each), and a lane carries RL
// rows (two when T <= 8, else one), so that each k_t / q_t slice it reads from shared memory
// serves RL rows: a 128-bit shared load costs the same four wavefronts however many lanes
// share its addresses, so rows per lane is what sets the operand traffic.  A warp pass covers
// 4 RL rows.  The 2T partial sums of a row meet in a transposing reduction over its eight
// lanes (TM = T rounded up to 4, 8 or 16), after which each lane holds TM RL / 4 of one row's
// k_t . s0_i or q_t . s0_i.  With M = [(I + A)^{-1}; P (I + A)^{-1}], one pass of broadcasts
// of the right-hand side gives u in the lanes of the k-dots and the P u part of the outputs in
// those of the q-dots.  Without per-token snapshots the state update is taken relative to the
// last token, s_i <- e^{G_{T-1}} s_i + sum_t e^{G_{T-1} - G_t} u_t k_t (one FMA per element and
// token, no factor above 1); with them, token by token.
//
// One CTA per (sequence, key head), or, at small batches, a thread-block cluster of nsplit
// CTAs that split the rows of each value head.  The prologue convolves the T tokens of the
// key head's q/k channels and of its own rows' v channels (and writes their new conv state),
// forms the norms, the gates and, per value head, M in shared memory.  Then each warp
// streams state rows, 512 contiguous bytes per eight lanes, coalesced: asynchronous copies
// put the next pass's rows into one of two per-warp shared buffers a pass ahead (the first
// pass's at kernel entry, in flight during the prologue), and stores write the new rows.  All CTAs of a
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
// 16-byte asynchronous copy global -> shared (no registers held while it is in flight)
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// acc + a . b
__device__ __forceinline__ float fma4(float4 a, float4 b, float acc) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// transposing reduction of V values (a power of two >= 8) over the eight lanes of a row
// group: three halving levels (xor 4, 2, 1; 7 V / 8 shuffles); afterwards x[i], i < V / 8,
// holds value gl * V / 8 + i summed over the group (gl = lane & 7)
template <int V>
__device__ __forceinline__ void transpose_reduce8(float (&x)[V], int lane) {
#pragma unroll
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int m = 4 >> lvl, L = V >> lvl;
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
}

// shared-memory layout (floats) for T tokens, TM >= T the unrolled capacity, r value heads
struct MtLayout {
  int qh, kh, vv, kk, qk, mats, ostage, red, stage, total;
  // per value head: Mt [TM][2 TM] (column s of (I + A)^{-1}, then of P (I + A)^{-1}),
  // P [TM][TM], e^{G_t}, beta_t, e^{G_{T-1} - G_t}, e^{g_t}
  static __host__ __device__ int head_block(int TM) { return 3 * TM * TM + 4 * TM; }
  __host__ __device__ MtLayout(int T, int TM, int r) {
    qh = 0;
    kh = qh + T * D;
    vv = kh + T * D;
    kk = vv + T * r * D;
    qk = kk + T * T;
    mats = (qk + T * T + 3) & ~3;
    ostage = mats + r * head_block(TM);      // outputs [T][r][D]
    red = ostage + T * r * D;
    stage = red + 64;                        // per warp: two buffers of one pass's rows
    total = stage + (MT_THREADS / 32) * 2 * 4 * (TM <= 8 ? 2 : 1) * D;
  }
};

// TM: the token capacity the loops are unrolled for (T <= TM)
template <typename Tin, typename Tout, int TM>
__global__ void __launch_bounds__(MT_THREADS, 2) gdn_decode_multi_kernel(GdnLayerArgs p, int T,
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
  const MtLayout lay(T, TM, r);
  constexpr int HB = 3 * TM * TM + 4 * TM;
  // state-row geometry of step 5; the first pass's rows are copied now, so that they are in
  // flight while the prologue runs
  constexpr int RL = TM <= 8 ? 2 : 1;                  // state rows per lane
  constexpr int V = RL * 2 * TM, VPL = V / 8;          // reduced values; values per lane
  const int gl = lane & 7, grp = lane >> 3;
  const int QO = R / (4 * RL), NQ = r * QO;            // warp passes per head; in all
  auto pass_base = [&](int q, int& hh) {               // first row of pass q; its head
    hh = q / QO;
    return r_lo + (q - hh * QO) * 4 * RL + grp;
  };
  auto row_ptr = [&](int hh, int i) {
    return reinterpret_cast<float4*>(p.state + (((size_t)slot * p.Hv + kh * r + hh) * D + i) * D);
  };
  // a pass's rows go to one of this warp's two staging buffers by asynchronous copies, each
  // lane copying (and later reading) only its own 16-byte pieces: element
  // (rr, grp, 4 (gl + 8 m)); the k-th pass of this warp uses buffer k & 1
  constexpr int SBUF = 4 * RL * D / 4;                 // float4s per buffer
  float4* stg = reinterpret_cast<float4*>(ms + lay.stage) + warp * 2 * SBUF;
  auto prefetch_pass = [&](int q, int buf) {
    int hh;
    const int i0 = pass_base(q, hh);
    float4* dst = stg + buf * SBUF;
#pragma unroll
    for (int rr = 0; rr < RL; ++rr) {
      const float4* src = row_ptr(hh, i0 + 4 * rr);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        cp_async16(dst + (rr * 4 + grp) * (D / 4) + gl + 8 * m, src + gl + 8 * m);
    }
    cp_async_commit();
  };
  if (warp < NQ) prefetch_pass(warp, 0);
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
  // the window of a channel, right-aligned in 3 + TM registers: conv-state entries at
  // 3 - H .. 2, the new inputs at 3 .. 3 + T - 1 (zeros elsewhere), so that every register
  // index is a compile-time constant; window entries shift .. shift + H - 1 are a conv state
  auto store_window = [&](const float (&wv)[3 + TM], Tin* dst, int shift) {
#pragma unroll
    for (int pos = 0; pos < 3 + TM; ++pos) {
      const int i = pos - shift;
      if (i >= 0 && i < H) st_elem(dst + (size_t)i * C, wv[pos]);
    }
  };
  float qkwin[3 + TM];                                  // this thread's q/k channel (tid < 256)
  int qkch = -1;
  for (int cl = tid; cl < ch_all; cl += MT_THREADS) {
    // local channel cl: q (0..127), k (128..255), then v of value head vh, row r_lo + vi
    const int vh = (cl - ch_qk) / R, vi = r_lo + (cl - ch_qk) % R;
    const int ch = cl < D ? kh * D + cl
                   : cl < ch_qk ? p.Hk * D + kh * D + (cl - D)
                                : 2 * p.Hk * D + (kh * r + vh) * D + vi;
    if (W > 0) {
      const Tin* cs = (const Tin*)p.conv_state + (size_t)slot * H * C + ch;
      float win[3 + TM], w4[4];
#pragma unroll
      for (int j = 0; j < 3; ++j) win[j] = j >= 3 - H ? ld_elem(cs + (size_t)(j - 3 + H) * C) : 0.f;
#pragma unroll
      for (int t = 0; t < TM; ++t)
        win[3 + t] = t < T ? ld_elem((const Tin*)p.x + ((size_t)b * T + t) * C + ch) : 0.f;
      const float bias = p.conv_b ? ld_elem((const Tin*)p.conv_b + ch) : 0.f;
      const Tin* w = (const Tin*)p.conv_w + (size_t)ch * W;
#pragma unroll
      for (int j = 0; j < 4; ++j) w4[j] = j >= 4 - W ? ld_elem(w + j - 4 + W) : 0.f;
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < T) {
          float y = bias;
#pragma unroll
          for (int j = 0; j < 4; ++j) y = fmaf(w4[j], win[t + j], y);
          y = p.silu ? silu_f(y) : y;
          if (cl < D) qh[t * D + cl] = y;
          else if (cl < ch_qk) khat[t * D + cl - D] = y;
          else vv[t * r * D + vh * D + vi] = y;
        }
      }
      // new conv state: window entries T + 3 - H ..; after token t: t + 4 - H ..
      if (cl < ch_qk) {
        qkch = ch;
#pragma unroll
        for (int i = 0; i < 3 + TM; ++i) qkwin[i] = win[i];
      } else {
        store_window(win, (Tin*)p.conv_state + (size_t)slot * H * C + ch, T + 3 - H);
        if (snap_conv && snap_slots)
          for (int t = 0; t < T; ++t) {
            const int sl = snap_slots[b * T + t];
            if (sl >= 0 && sl < num_snap)
              store_window(win, snap_conv + (size_t)sl * H * C + ch, t + 4 - H);
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
  // ---- 4. per value head: gates, G, (I + A)^{-1}, P and P (I + A)^{-1} (warp hh, lanes =
  //      tokens); entries of tokens T .. TM-1 are zero
  for (int hh = warp; hh < r; hh += MT_THREADS / 32) {
    float* Mt = ms + lay.mats + hh * HB;
    float* P = Mt + 2 * TM * TM;
    float* eG = P + TM * TM;        // e^{G_t}
    float* bt = eG + TM;            // beta_t
    float* dk = bt + TM;            // e^{G_{T-1} - G_t}
    float* eg = dk + TM;            // e^{g_t}
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
    if (lane < TM) {
      const bool on = lane < T;
      eG[lane] = on ? expf(G) : 0.f;
      bt[lane] = on ? beta : 0.f;
      dk[lane] = on ? expf(GT - G) : 0.f;
      eg[lane] = on ? expf(g) : 1.f;
    }
    // A (strictly lower) into the Mt area for now, and P (lower with the diagonal): row t in
    // lane t
#pragma unroll
    for (int s2 = 0; s2 < TM; ++s2) {
      const float Gs = __shfl_sync(0xffffffffu, G, s2);
      float a = 0.f, pp = 0.f;
      if (lane < T && s2 < T && s2 <= lane) {
        const float e = expf(G - Gs);
        if (s2 < lane) a = beta * e * KK[lane * T + s2];
        pp = e * QK[lane * T + s2];
      }
      if (lane < TM) {
        Mt[lane * TM + s2] = a;
        P[lane * TM + s2] = pp;
      }
    }
    __syncwarp();
    // column j of (I + A)^{-1} by forward substitution (lane j), then column j of
    // P (I + A)^{-1}
    const int j = lane;
    float col[TM], pt[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) col[t] = (t == j && j < T) ? 1.f : 0.f;
    if (j < TM) {
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t > j && t < T) {
          float acc = 0.f;
#pragma unroll
          for (int s2 = 0; s2 < TM; ++s2)
            if (s2 >= j && s2 < t) acc = fmaf(Mt[t * TM + s2], col[s2], acc);
          col[t] = -acc;
        }
      }
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        float acc = 0.f;
#pragma unroll
        for (int s2 = 0; s2 <= t; ++s2) acc = fmaf(P[t * TM + s2], col[s2], acc);
        pt[t] = acc;
      }
    }
    __syncwarp();                   // every lane has read A
    if (j < TM) {
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        Mt[j * 2 * TM + t] = col[t];
        Mt[j * 2 * TM + TM + t] = pt[t];
      }
    }
  }
  __syncthreads();
  // ---- 5. the state rows: eight lanes a row (elements 4 (gl + 8 m) .. + 3, m < 4) and RL
  //      rows a lane (rows i0 + 4 rho + grp), so that each k / q slice read from shared memory
  //      serves RL rows; a warp pass covers 4 RL rows of one value head, warp w taking passes
  //      w, w + 8, ...; the next pass's rows are copied to shared memory (cp.async, no
  //      registers held) while this one's arithmetic runs
  int* ssl = reinterpret_cast<int*>(red);              // this sequence's snapshot rows
  if (tid < TM) ssl[tid] = (snap_state && snap_slots && tid < T) ? snap_slots[b * T + tid] : -1;
  __syncthreads();
  // after the reduction lane gl holds values gl VPL .. + VPL-1 of [row rho][k-dots, q-dots]
  const int rho = gl * VPL / (2 * TM), tr0 = gl * VPL - rho * 2 * TM;
  const bool role_a = tr0 < TM;                        // k-dots (-> u) or q-dots (-> o)
  const int tk0 = role_a ? tr0 : tr0 - TM;             // token of value slot 0
  const bool per_token = snap_state != nullptr && snap_slots != nullptr;
  const float4* q4 = reinterpret_cast<const float4*>(qh);
  const float4* k4 = reinterpret_cast<const float4*>(khat);
  float* ost = ms + lay.ostage;
  for (int q = warp, pk = 0; q < NQ; q += MT_THREADS / 32, pk ^= 1) {
    int hh;
    const int i0 = pass_base(q, hh);
    const int h = kh * r + hh, irow = i0 + 4 * rho;
    float4 st[RL][4];
    cp_async_wait_all();                               // this pass's rows (buffer pk)
#pragma unroll
    for (int rr = 0; rr < RL; ++rr)
#pragma unroll
      for (int m = 0; m < 4; ++m)
        st[rr][m] = stg[pk * SBUF + (rr * 4 + grp) * (D / 4) + gl + 8 * m];
    // the next pass's rows into the other buffer (read by this lane a pass ago)
    if (q + MT_THREADS / 32 < NQ) prefetch_pass(q + MT_THREADS / 32, pk ^ 1);
    const float* Mt = ms + lay.mats + hh * HB;
    const float* eG = Mt + 3 * TM * TM;
    const float* bt = eG + TM;
    const float* dk = bt + TM;
    const float* eg = dk + TM;
    // 2T partial dot products per row over this lane's 16 elements, reduced over the row's
    // eight lanes
    float x[V];
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      float a[RL], c[RL];
#pragma unroll
      for (int rr = 0; rr < RL; ++rr) a[rr] = c[rr] = 0.f;
      if (t < T) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 kv = k4[t * (D / 4) + gl + 8 * m];
          const float4 qv = q4[t * (D / 4) + gl + 8 * m];
#pragma unroll
          for (int rr = 0; rr < RL; ++rr) {
            a[rr] = fma4(st[rr][m], kv, a[rr]);
            c[rr] = fma4(st[rr][m], qv, c[rr]);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < RL; ++rr) {
        x[rr * 2 * TM + t] = a[rr];
        x[rr * 2 * TM + TM + t] = c[rr];
      }
    }
    transpose_reduce8<V>(x, lane);
    // x[k]: k_t . s0 (role_a) or q_t . s0 of row irow, t = tk0 + k
    float rhs[VPL], acc[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int t = tk0 + k;
      rhs[k] = (role_a && t < T) ? bt[t] * (vv[(t * r + hh) * D + irow] - eG[t] * x[k]) : 0.f;
      acc[k] = 0.f;
    }
    // role_a lanes: u = (I + A)^{-1} rhs; the others: P (I + A)^{-1} rhs
#pragma unroll
    for (int s2 = 0; s2 < TM; ++s2) {
      if (s2 < T) {
        const float rs =
            __shfl_sync(0xffffffffu, rhs[s2 % VPL], (rho * 2 * TM + s2) / VPL, 8);
        const float* mrow = Mt + s2 * 2 * TM + tr0;
#pragma unroll
        for (int k = 0; k < VPL; ++k) acc[k] = fmaf(mrow[k], rs, acc[k]);
      }
    }
    if (!role_a) {
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const int t = tk0 + k;
        if (t < T) ost[(t * r + hh) * D + irow] = fmaf(eG[t], x[k], acc[k]);
      }
    }
    // the state: token by token with snapshots, else relative to the last token; u_s of row
    // rr sits in lane (rr 2 TM + s) / VPL, slot s % VPL
    if (per_token) {
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2) {
        if (s2 < T) {
          float us[RL];
#pragma unroll
          for (int rr = 0; rr < RL; ++rr)
            us[rr] = __shfl_sync(0xffffffffu, acc[s2 % VPL], (rr * 2 * TM + s2) / VPL, 8);
          const float e = eg[s2];
          const int sl = ssl[s2];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 kv = k4[s2 * (D / 4) + gl + 8 * m];
#pragma unroll
            for (int rr = 0; rr < RL; ++rr) {
              st[rr][m].x = fmaf(e, st[rr][m].x, us[rr] * kv.x);
              st[rr][m].y = fmaf(e, st[rr][m].y, us[rr] * kv.y);
              st[rr][m].z = fmaf(e, st[rr][m].z, us[rr] * kv.z);
              st[rr][m].w = fmaf(e, st[rr][m].w, us[rr] * kv.w);
            }
          }
          if (sl >= 0 && sl < num_snap) {
#pragma unroll
            for (int rr = 0; rr < RL; ++rr) {
              float4* dst = reinterpret_cast<float4*>(
                  snap_state + (((size_t)sl * p.Hv + h) * D + i0 + 4 * rr) * D);
#pragma unroll
              for (int m = 0; m < 4; ++m) dst[gl + 8 * m] = st[rr][m];
            }
          }
        }
      }
    } else {
      const float eT = eG[T - 1];
#pragma unroll
      for (int rr = 0; rr < RL; ++rr)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          st[rr][m].x *= eT; st[rr][m].y *= eT; st[rr][m].z *= eT; st[rr][m].w *= eT;
        }
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2) {
        if (s2 < T) {
          float us[RL];
#pragma unroll
          for (int rr = 0; rr < RL; ++rr)
            us[rr] = __shfl_sync(0xffffffffu, acc[s2 % VPL], (rr * 2 * TM + s2) / VPL, 8) *
                     dk[s2];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 kv = k4[s2 * (D / 4) + gl + 8 * m];
#pragma unroll
            for (int rr = 0; rr < RL; ++rr) {
              st[rr][m].x = fmaf(us[rr], kv.x, st[rr][m].x);
              st[rr][m].y = fmaf(us[rr], kv.y, st[rr][m].y);
              st[rr][m].z = fmaf(us[rr], kv.z, st[rr][m].z);
              st[rr][m].w = fmaf(us[rr], kv.w, st[rr][m].w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < RL; ++rr) {
      float4* Sr = row_ptr(hh, i0 + 4 * rr);
#pragma unroll
      for (int m = 0; m < 4; ++m) Sr[gl + 8 * m] = st[rr][m];
    }
  }
  __syncthreads();
  // the outputs, token rows of Hv x 128 channels: this CTA's rows of its r value heads
  {
    const int lgR = __ffs(R) - 1;                      // R is a power of two
    for (int tt = 0; tt < T; ++tt) {
      Tout* orow = (Tout*)p.out + (((size_t)b * T + tt) * p.Hv + kh * r) * D;
      const float* srow = ost + tt * r * D;
      for (int j = tid; j < r * R; j += MT_THREADS) {
        const int e = (j >> lgR) * D + r_lo + (j & (R - 1));       // hh * D + c
        st_elem(orow + e, srow[e]);
      }
    }
  }
  // the q/k channels' new conv state (and per-token snapshots): rank 0, after the cluster's
  // reads of the old one
  if (nsplit > 1) cluster_wait_mt();
  if (sp == 0 && W > 0 && qkch >= 0) {
    store_window(qkwin, (Tin*)p.conv_state + (size_t)slot * H * C + qkch, T + 3 - H);
    if (snap_conv && snap_slots)
      for (int t = 0; t < T; ++t) {
        const int sl = snap_slots[b * T + t];
        if (sl >= 0 && sl < num_snap)
          store_window(qkwin, snap_conv + (size_t)sl * H * C + qkch, t + 4 - H);
      }
  }
  if (tid == 0 && sp == 0 && snap_slots)
    for (int t = 0; t < T; ++t)
      if (snap_slots[b * T + t] >= num_snap && kh == 0) atomicOr(&g_err_multi, kErrIndex);
}

template <typename Tin, typename Tout, int TM>
cudaError_t launch_multi_tm(const GdnLayerArgs& p, int T, float* snap_state, int num_snap,
                            const int32_t* snap_slots, void* snap_conv, cudaStream_t stream) {
  const MtLayout lay(T, TM, p.Hv / p.Hk);
  const size_t smem = sizeof(float) * lay.total;
  static unsigned done = 0;
  cudaError_t e = set_smem_once(gdn_decode_multi_kernel<Tin, Tout, TM>,
                                (int)(sizeof(float) * MtLayout(TM, TM, 8).total), &done);
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
  if (T <= 4)
    return launch_multi_tm<Tin, Tout, 4>(p, T, snap_state, num_snap, snap_slots, snap_conv,
                                         stream);
  if (T <= 8)
    return launch_multi_tm<Tin, Tout, 8>(p, T, snap_state, num_snap, snap_slots, snap_conv,
                                         stream);
  return launch_multi_tm<Tin, Tout, 16>(p, T, snap_state, num_snap, snap_slots, snap_conv,
                                        stream);
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
