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
// Work of one (sequence, key head) item: a prologue convolves the T tokens of the key head's
// q/k channels and of its value heads' v channels (and writes their new conv state), forms
// the norms, the gates and, per value head, M in shared memory.  Then warps stream the state
// rows, 512 contiguous bytes per eight lanes, coalesced: asynchronous copies put a warp's
// coming passes' rows into its shared buffers ahead of use, and stores write the new rows.
// More than eight tokens are taken in chunks of eight, the rows' state carried in registers
// from one chunk to the next.  Two kernels run it:
//  - large batches of up to four tokens: a persistent, warp-specialised CTA per SM.  Twelve
//    row warps stream state rows without a break (three buffers per warp, the copies running
//    two passes ahead across item boundaries), while four prologue warps prepare the next
//    item into the other half of a double-buffered prologue area: its inputs (x rows, conv
//    state, conv weights and bias, a few contiguous runs each) bulk-copied into a staging
//    area while the item before is prepared, its gates loaded into registers ahead of use;
//    the conv four channels a thread with the q/k norms as warp reductions, the dot products
//    four lanes a pair, M one thread per (value head, column).  The new conv state leaves by
//    bulk stores straight from the staged rows, the outputs by bulk stores from shared
//    memory, so that neither role issues per-thread global stores into the row stream.
//    mbarriers hand each prologue buffer to the row warps ("ready") and back ("free"); the
//    first item's prologue is computed by all warps together.
//  - small batches, and more than four tokens: one CTA per item, or a thread-block cluster
//    of nsplit CTAs that split the rows of each value head.  All CTAs of a cluster read the
//    old q/k conv state; a cluster barrier orders those reads before the one CTA (rank 0)
//    that writes the new one.
#include "common.cuh"
#include "sm100_ptx.cuh"

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
constexpr int MT_WARPS = MT_THREADS / 32;
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
// wait until at most n (0 .. 3) of this thread's newest copy groups are in flight
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  switch (n) {
    case 3: asm volatile("cp.async.wait_group 3;\n" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;\n" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;\n" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 0;\n" ::: "memory"); break;
  }
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

// state-row geometry: RL rows a lane, a warp pass of 4 RL rows of one value head
template <int TM>
struct RowGeo {
  static constexpr int RL = TM <= 8 ? 2 : 1;          // state rows per lane (TM <= 8: two)
  static constexpr int V = RL * 2 * TM, VPL = V / 8;  // reduced values; values per lane
  static constexpr int SBUF = 4 * RL * D / 4;         // float4s per pass buffer
};
__host__ __device__ constexpr int rows_per_lane(int TM) { return TM <= 8 ? 2 : 1; }

// The T tokens of a step are taken in chunks of TM (the unrolled capacity; one chunk when
// T <= TM), the state carried from chunk to chunk: the chunked form of the recurrence again,
// with chunks of TM tokens.
__host__ __device__ inline int token_chunks(int T, int TM) { return (T + TM - 1) / TM; }

// The per-item prologue results in shared memory (floats) for T tokens in NC chunks of TM,
// r value heads: q^_t, k^_t, v_t of the item's rows, KK, QK, per value head and chunk
// Mt [TM][2 TM] (column s of (I + A)^{-1}, then of P (I + A)^{-1}), P [TM][TM], e^{G_t},
// beta_t, e^{G_last - G_t}, e^{g_t} (G from the chunk's start); the gates g_t, beta_t per
// value head and token (NC TM of them); the snapshot rows of the tokens (ints).
struct ProOffsets {
  int qh, kh, vv, kk, qk, mats, gb, ssl, total;      // total: a multiple of 4
  static __host__ __device__ int head_block(int TM) { return 3 * TM * TM + 4 * TM; }
  __host__ __device__ ProOffsets(int T, int TM, int r, int R) {
    const int NC = token_chunks(T, TM), TS = NC * TM;
    qh = 0;
    kh = qh + T * D;
    vv = kh + T * D;
    kk = vv + T * r * R;
    qk = kk + T * T;
    mats = (qk + T * T + 3) & ~3;
    gb = mats + r * NC * head_block(TM);
    ssl = gb + 2 * TS * r;
    total = (ssl + TS + 3) & ~3;
  }
};

struct ProView {
  float *qh, *kh, *vv, *kk, *qk, *mats, *gb;
  int* ssl;
  __device__ ProView(float* base, const ProOffsets& o)
      : qh(base + o.qh), kh(base + o.kh), vv(base + o.vv), kk(base + o.kk), qk(base + o.qk),
        mats(base + o.mats), gb(base + o.gb), ssl(reinterpret_cast<int*>(base + o.ssl)) {}
};

// the new conv state (or the one after token t) from a channel's window, right-aligned in
// 3 + TM registers: window entries shift .. shift + H - 1 are that conv state
template <int TM, typename Tin>
__device__ __forceinline__ void store_window(const float (&wv)[3 + TM], Tin* dst, int shift,
                                             int H, int C) {
#pragma unroll
  for (int pos = 0; pos < 3 + TM; ++pos) {
    const int i = pos - shift;
    if (i >= 0 && i < H) st_elem(dst + (size_t)i * C, wv[pos]);
  }
}

// the conv (+SiLU) outputs of one channel over the T tokens from its window (conv-state
// entries at 3 - H .. 2, inputs at 3 .. 3 + T - 1); w4 right-aligned (zeros below 4 - W)
template <int TM>
__device__ __forceinline__ void conv_tokens(const float (&win)[3 + TM], const float (&w4)[4],
                                            float bias, bool silu, int T, float* dst,
                                            int dst_stride) {
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    if (t < T) {
      float y = bias;
#pragma unroll
      for (int j = 0; j < 4; ++j) y = fmaf(w4[j], win[t + j], y);
      dst[t * dst_stride] = silu ? silu_f(y) : y;
    }
  }
}

// The raw gate inputs of one (token, value head) of an item (index i < T r: token i / r,
// head i % r), loaded ahead of their use.
struct GateRaw {
  float a, b, A_log, dt_bias;
};

template <typename Tin>
__device__ __forceinline__ GateRaw load_gate_raw(const GdnLayerArgs& p, int b, int T, int kh,
                                                 int r, int i) {
  GateRaw g{0.f, 0.f, 0.f, 0.f};
  if (i < T * r) {
    const int t = i / r, h = kh * r + (i - t * r);
    const size_t gi = ((size_t)b * T + t) * p.Hv + h;
    if (p.gates_pre) {
      g.a = ((const float*)p.a)[gi];
      g.b = ((const float*)p.b)[gi];
    } else {
      g.a = ld_elem((const Tin*)p.a + gi);
      g.b = ld_elem((const Tin*)p.b + gi);
      g.A_log = p.A_log[h];
      g.dt_bias = p.dt_bias ? p.dt_bias[h] : 0.f;
    }
  }
  return g;
}

// g_t and beta_t into gb[(hh TS + t) 2 + {0, 1}], TS = the tokens rounded up to whole chunks
template <int TM>
__device__ __forceinline__ void store_gate(const GdnLayerArgs& p, const GateRaw& g, float* gb,
                                           int T, int r, int i) {
  if (i < T * r) {
    const int t = i / r, hh = i - t * r, ts = token_chunks(T, TM) * TM;
    gb[(hh * ts + t) * 2] = p.gates_pre ? g.a : gate_g(g.a, g.A_log, g.dt_bias);
    gb[(hh * ts + t) * 2 + 1] = p.gates_pre ? g.b : sigmoid_f(g.b);
  }
}

// ---- 2. L2 norms of q_t and k_t (one warp per vector, warps w0 + j nw), q also times `scale`
__device__ __forceinline__ void mt_norms(const GdnLayerArgs& p, const ProView& v, int T, int w0,
                                         int nw, int lane) {
  for (int vec = w0; vec < 2 * T; vec += nw) {
    float* x = (vec < T ? v.qh : v.kh) + (vec % T) * D;
    float4 v4 = reinterpret_cast<float4*>(x)[lane];
    const float ss = warp_sum(dot4(v4, v4));
    const float inv = (p.l2norm ? 1.0f / sqrtf(ss + p.eps) : 1.0f) * (vec < T ? p.scale : 1.0f);
    v4.x *= inv; v4.y *= inv; v4.z *= inv; v4.w *= inv;
    reinterpret_cast<float4*>(x)[lane] = v4;
  }
}

// ---- 3. KK_ts = k_t . k_s and QK_ts = q_t . k_s for t, s in the same chunk of TM tokens:
//      eight lanes a pair (16 elements each, a group's 128-bit loads covering all banks
//      once), reduced over the group
__device__ __forceinline__ void mt_dots(const ProView& v, int T, int TM, int w0, int nw,
                                        int lane) {
  const int gl = lane & 7, np = 2 * T * T;
  for (int base = w0 * 4; base < np; base += nw * 4) {
    const int pr = base + (lane >> 3);
    const int which = pr / (T * T), t = (pr / T) % T, s2 = pr % T;
    const bool on = pr < np && t / TM == s2 / TM;
    float d = 0.f;
    if (on) {
      const float4* a4 = reinterpret_cast<const float4*>((which ? v.qh : v.kh) + t * D);
      const float4* k4 = reinterpret_cast<const float4*>(v.kh + s2 * D);
#pragma unroll
      for (int m = 0; m < 4; ++m) d = fma4(a4[gl + 8 * m], k4[gl + 8 * m], d);
    }
    d += __shfl_xor_sync(0xffffffffu, d, 4);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    if (on && gl == 0) (which ? v.qk : v.kk)[t * T + s2] = d;
  }
}

// ---- 4. per value head and chunk: G, (I + A)^{-1}, P and P (I + A)^{-1} (warp w0 + j nw
//      takes job j = (chunk c, value head hh), lanes = the chunk's tokens); entries of tokens
//      past the chunk's end are zero
template <int TM>
__device__ __forceinline__ void mt_mats(const ProView& v, int T, int r, int w0, int nw,
                                        int lane) {
  constexpr int HB = 3 * TM * TM + 4 * TM;
  const int NC = token_chunks(T, TM), TS = NC * TM, Tall = T;
  for (int job = w0; job < r * NC; job += nw) {
    const int c = job / r, hh = job - c * r, t0 = c * TM;
    const int T = min(TM, Tall - t0);                  // tokens of this chunk
    float* Mt = v.mats + (c * r + hh) * HB;
    float* P = Mt + 2 * TM * TM;
    float* eG = P + TM * TM;        // e^{G_t}
    float* bt = eG + TM;            // beta_t
    float* dk = bt + TM;            // e^{G_{T-1} - G_t}
    float* eg = dk + TM;            // e^{g_t}
    float g = 0.f, beta = 0.f;
    if (lane < T) {
      g = v.gb[(hh * TS + t0 + lane) * 2];
      beta = v.gb[(hh * TS + t0 + lane) * 2 + 1];
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
        if (s2 < lane) a = beta * e * v.kk[(t0 + lane) * Tall + t0 + s2];
        pp = e * v.qk[(t0 + lane) * Tall + t0 + s2];
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
}

// The rows of one item's value heads that a CTA streams: value heads kh r .. kh r + r - 1 of
// state slot `slot`, rows r_lo .. r_lo + R - 1 of each (4 RL rows a pass, QO passes a head).
struct RowItem {
  int b, kh, slot, r_lo, R;
};

// A pass's rows go to one of a warp's shared buffers by asynchronous copies, each lane
// copying (and later reading) only its own 16-byte pieces: element (rr, grp, 4 (gl + 8 m)).
// The copies form one commit group (empty when `on` is false, so that every pass commits one).
template <int TM>
__device__ __forceinline__ void prefetch_pass(const GdnLayerArgs& p, const RowItem& it, int r,
                                              int q, float4* dst, int lane, bool on = true) {
  constexpr int RL = RowGeo<TM>::RL;
  if (on) {
    const int gl = lane & 7, grp = lane >> 3;
    const int QO = it.R / (4 * RL), hh = q / QO;
    const int i0 = it.r_lo + (q - hh * QO) * 4 * RL + grp;
    // (the -DGDN_BOUNDS_CHECK build: rows out of the state array are recorded and replaced by
    // row 0, so that the copy groups keep their shape)
    const bool ok = in_bounds(&g_err_multi, it.slot >= 0 && it.slot < p.num_slots &&
                                                it.kh * r + hh < p.Hv && i0 + 4 * (RL - 1) < D);
#pragma unroll
    for (int rr = 0; rr < RL; ++rr) {
      const float4* src = reinterpret_cast<const float4*>(
          ok ? p.state + (((size_t)it.slot * p.Hv + it.kh * r + hh) * D + i0 + 4 * rr) * D
             : p.state);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        cp_async16(dst + (rr * 4 + grp) * (D / 4) + gl + 8 * m, src + gl + 8 * m);
    }
  }
  cp_async_commit();
}

// this lane's pieces of a pass's rows, from its shared buffer
template <int TM>
__device__ __forceinline__ void read_pass(const float4* buf, float4 (&st)[RowGeo<TM>::RL][4],
                                          int lane) {
  const int gl = lane & 7, grp = lane >> 3;
#pragma unroll
  for (int rr = 0; rr < RowGeo<TM>::RL; ++rr)
#pragma unroll
    for (int m = 0; m < 4; ++m) st[rr][m] = buf[(rr * 4 + grp) * (D / 4) + gl + 8 * m];
}

// ---- 5. one warp pass of an item's state rows (pass q: value head q / QO), whose rows
//      (st) this lane has read: eight lanes a row (elements 4 (gl + 8 m) .. + 3, m < 4) and
//      RL rows a lane (rows i0 + 4 rho + grp), so that each k / q slice read from shared
//      memory serves RL rows; the tokens chunk by chunk.  Writes the outputs into
//      ost [T][r][R'] (R' = the rows of a value head the CTA holds; fp32, or the output type)
//      and the new rows (and per-token snapshots) to HBM.
template <int TM, int NCMAX, typename OT>
__device__ __forceinline__ void mt_pass(const GdnLayerArgs& p, const ProView& v, OT* ost,
                                        const RowItem& it, int T, int r, int q,
                                        float* snap_state, int num_snap,
                                        float4 (&st)[RowGeo<TM>::RL][4], int lane) {
  constexpr int RL = RowGeo<TM>::RL, V = RowGeo<TM>::V, VPL = RowGeo<TM>::VPL;
  constexpr int HB = 3 * TM * TM + 4 * TM;
  const int gl = lane & 7, grp = lane >> 3;
  const int QO = it.R / (4 * RL), hh = q / QO;
  const int i0 = it.r_lo + (q - hh * QO) * 4 * RL + grp;      // this lane's first row
  // after the reduction lane gl holds values gl VPL .. + VPL-1 of [row rho][k-dots, q-dots]
  const int rho = gl * VPL / (2 * TM), tr0 = gl * VPL - rho * 2 * TM;
  const bool role_a = tr0 < TM;                        // k-dots (-> u) or q-dots (-> o)
  const int tk0 = role_a ? tr0 : tr0 - TM;             // token of value slot 0
  const int h = it.kh * r + hh, irow = i0 + 4 * rho;   // the row of the reduced values
  const int lrow = irow - it.r_lo;                     // ... among the CTA's rows of the head
  const int Rv = it.R;                                 // v / output rows held per head
  // the chunks of TM tokens in turn (at most NCMAX), the rows' state carried in registers
  // from one to the next
#pragma unroll
  for (int c = 0; c < NCMAX; ++c) {
    const int t0 = c * TM, Tc = NCMAX == 1 ? T : min(TM, T - t0);
    if (NCMAX > 1 && Tc <= 0) break;
    const float4* q4 = reinterpret_cast<const float4*>(v.qh + t0 * D);
    const float4* k4 = reinterpret_cast<const float4*>(v.kh + t0 * D);
    const float* Mt = v.mats + (c * r + hh) * HB;
    const float* eG = Mt + 3 * TM * TM;
    const float* bt = eG + TM;
    const float* dk = bt + TM;
    const float* eg = dk + TM;
    // 2 Tc partial dot products per row over this lane's 16 elements, reduced over the row's
    // eight lanes
    float x[V];
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      float a[RL], cq[RL];
#pragma unroll
      for (int rr = 0; rr < RL; ++rr) a[rr] = cq[rr] = 0.f;
      if (t < Tc) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 kv = k4[t * (D / 4) + gl + 8 * m];
          const float4 qv = q4[t * (D / 4) + gl + 8 * m];
#pragma unroll
          for (int rr = 0; rr < RL; ++rr) {
            a[rr] = fma4(st[rr][m], kv, a[rr]);
            cq[rr] = fma4(st[rr][m], qv, cq[rr]);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < RL; ++rr) {
        x[rr * 2 * TM + t] = a[rr];
        x[rr * 2 * TM + TM + t] = cq[rr];
      }
    }
    transpose_reduce8<V>(x, lane);
    // x[k]: k_t . s (role_a) or q_t . s of row irow, t = t0 + tk0 + k, s the state at the
    // chunk's start
    float rhs[VPL], acc[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int t = tk0 + k;
      rhs[k] = (role_a && t < Tc)
                   ? bt[t] * (v.vv[((t0 + t) * r + hh) * Rv + lrow] - eG[t] * x[k]) : 0.f;
      acc[k] = 0.f;
    }
    // role_a lanes: u = (I + A)^{-1} rhs; the others: P (I + A)^{-1} rhs
#pragma unroll
    for (int s2 = 0; s2 < TM; ++s2) {
      if (s2 < Tc) {
        const float rs = __shfl_sync(0xffffffffu, rhs[s2 % VPL], (rho * 2 * TM + s2) / VPL, 8);
        const float* mrow = Mt + s2 * 2 * TM + tr0;
#pragma unroll
        for (int k = 0; k < VPL; ++k) acc[k] = fmaf(mrow[k], rs, acc[k]);
      }
    }
    if (!role_a) {
#pragma unroll
      for (int k = 0; k < VPL; ++k) {
        const int t = tk0 + k;
        if (t < Tc)
          ost[((t0 + t) * r + hh) * Rv + lrow] = from_float<OT>(fmaf(eG[t], x[k], acc[k]));
      }
    }
    // the state: token by token with snapshots, else relative to the chunk's last token;
    // u_s of row rr sits in lane (rr 2 TM + s) / VPL, slot s % VPL
    if (snap_state) {
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2) {
        if (s2 < Tc) {
          float us[RL];
#pragma unroll
          for (int rr = 0; rr < RL; ++rr)
            us[rr] = __shfl_sync(0xffffffffu, acc[s2 % VPL], (rr * 2 * TM + s2) / VPL, 8);
          const float e = eg[s2];
          const int sl = v.ssl[t0 + s2];
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
      const float eT = eG[Tc - 1];
#pragma unroll
      for (int rr = 0; rr < RL; ++rr)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          st[rr][m].x *= eT; st[rr][m].y *= eT; st[rr][m].z *= eT; st[rr][m].w *= eT;
        }
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2) {
        if (s2 < Tc) {
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
  }
  if (!in_bounds(&g_err_multi, it.slot >= 0 && it.slot < p.num_slots && h < p.Hv &&
                                  i0 + 4 * (RL - 1) < D))
    return;
#pragma unroll
  for (int rr = 0; rr < RL; ++rr) {
    float4* Sr = reinterpret_cast<float4*>(
        p.state + (((size_t)it.slot * p.Hv + h) * D + i0 + 4 * rr) * D);
#pragma unroll
    for (int m = 0; m < 4; ++m) Sr[gl + 8 * m] = st[rr][m];
  }
}

// the outputs, token rows of Hv x 128 channels: an item's rows r_lo .. r_lo + R - 1 of its
// r value heads, from ost [T][r][R] (threads t0 + j nt)
template <typename Tout>
__device__ __forceinline__ void mt_outputs(const GdnLayerArgs& p, const float* ost,
                                           const RowItem& it, int T, int r, int t0, int nt) {
  const int lgR = __ffs(it.R) - 1;                     // R is a power of two
  for (int tt = 0; tt < T; ++tt) {
    Tout* orow = (Tout*)p.out + (((size_t)it.b * T + tt) * p.Hv + it.kh * r) * D;
    const float* srow = ost + tt * r * it.R;
    for (int j = t0; j < r * it.R; j += nt)
      st_elem(orow + (j >> lgR) * D + it.r_lo + (j & (it.R - 1)), srow[j]);
  }
}

// a snapshot row at or past the bank's end (reported once per sequence)
__device__ __forceinline__ void check_snap_rows(const int32_t* snap_slots, int num_snap, int b,
                                                int T) {
  for (int t = 0; t < T; ++t)
    if (snap_slots[b * T + t] >= num_snap) atomicOr(&g_err_multi, kErrIndex);
}

// ======================================================================= small batches
// shared memory of the per-item kernel (floats): the prologue results, the outputs
// [T][r][R], per warp two buffers of one pass's rows
struct MtLayout {
  ProOffsets pro;
  int ost, stage, total;
  __host__ __device__ MtLayout(int T, int TM, int r, int R)
      : pro(T, TM, r, R) {
    ost = pro.total;
    stage = ost + ((T * r * R + 3) & ~3);
    total = stage + MT_WARPS * 2 * 4 * rows_per_lane(TM) * D;
  }
};

// TM: the chunk of tokens the row loops are unrolled for; TT >= T: the tokens the conv window
// is unrolled for
template <typename Tin, typename Tout, int TM, int TT>
__global__ void __launch_bounds__(MT_THREADS, 2) gdn_decode_multi_kernel(GdnLayerArgs p, int T,
                                                                      float* snap_state,
                                                                      int num_snap,
                                                                      const int32_t* snap_slots,
                                                                      Tin* snap_conv,
                                                                      int nsplit) {
  extern __shared__ __align__(16) float ms[];
  constexpr int SBUF = RowGeo<TM>::SBUF;
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
  const MtLayout lay(T, TM, r, R);
  const ProView v(ms, lay.pro);
  float* ost = ms + lay.ost;
  const RowItem it{b, kh, slot, r_lo, R};
  const int NQ = r * (R / (4 * RowGeo<TM>::RL));       // warp passes in all
  // the first pass's rows are copied now, so that they are in flight while the prologue runs
  float4* stg = reinterpret_cast<float4*>(ms + lay.stage) + warp * 2 * SBUF;
  if (warp < NQ) prefetch_pass<TM>(p, it, r, warp, stg, lane);
  // the gates, likewise in flight during the conv
  for (int i = tid; i < T * r; i += MT_THREADS)
    store_gate<TM>(p, load_gate_raw<Tin>(p, b, T, kh, r, i), v.gb, T, r, i);
  const int W = p.W, H = W > 0 ? W - 1 : 0, C = p.C_conv;
  const int ch_qk = 2 * D, ch_all = ch_qk + r * R;
  // ---- 1. conv (+SiLU) of this CTA's channels over the T tokens, or plain loads; the new
  //      conv state, and the conv state after every token for the snapshots (for the q/k
  //      channels, which every CTA of a cluster reads, once the cluster's reads are done)
  float qkwin[3 + TT];                                  // this thread's q/k channel (tid < 256)
  int qkch = -1;
  for (int cl = tid; cl < ch_all; cl += MT_THREADS) {
    // local channel cl: q (0..127), k (128..255), then v of value head vh, row r_lo + vi
    const int vh = (cl - ch_qk) / R, vi = (cl - ch_qk) % R;
    const int ch = cl < D ? kh * D + cl
                   : cl < ch_qk ? p.Hk * D + kh * D + (cl - D)
                                : 2 * p.Hk * D + (kh * r + vh) * D + r_lo + vi;
    float* dst = cl < D ? v.qh + cl : cl < ch_qk ? v.kh + cl - D : v.vv + vh * R + vi;
    const int dstride = cl < ch_qk ? D : r * R;
    if (W > 0) {
      const Tin* cs = (const Tin*)p.conv_state + (size_t)slot * H * C + ch;
      float win[3 + TT], w4[4];
#pragma unroll
      for (int j = 0; j < 3; ++j) win[j] = j >= 3 - H ? ld_elem(cs + (size_t)(j - 3 + H) * C) : 0.f;
#pragma unroll
      for (int t = 0; t < TT; ++t)
        win[3 + t] = t < T ? ld_elem((const Tin*)p.x + ((size_t)b * T + t) * C + ch) : 0.f;
      const float bias = p.conv_b ? ld_elem((const Tin*)p.conv_b + ch) : 0.f;
      const Tin* w = (const Tin*)p.conv_w + (size_t)ch * W;
#pragma unroll
      for (int j = 0; j < 4; ++j) w4[j] = j >= 4 - W ? ld_elem(w + j - 4 + W) : 0.f;
      conv_tokens<TT>(win, w4, bias, p.silu, T, dst, dstride);
      // new conv state: window entries T + 3 - H ..; after token t: t + 4 - H ..
      if (cl < ch_qk) {
        qkch = ch;
#pragma unroll
        for (int i = 0; i < 3 + TT; ++i) qkwin[i] = win[i];
      } else {
        store_window<TT>(win, (Tin*)p.conv_state + (size_t)slot * H * C + ch, T + 3 - H, H, C);
        if (snap_conv && snap_slots)
          for (int t = 0; t < T; ++t) {
            const int sl = snap_slots[b * T + t];
            if (sl >= 0 && sl < num_snap)
              store_window<TT>(win, snap_conv + (size_t)sl * H * C + ch, t + 4 - H, H, C);
          }
      }
    } else {
      for (int t = 0; t < T; ++t) {
        const Tin* src = cl < D ? (const Tin*)p.q + (((size_t)b * T + t) * p.Hk + kh) * D + cl
                         : cl < ch_qk
                             ? (const Tin*)p.k + (((size_t)b * T + t) * p.Hk + kh) * D + cl - D
                             : (const Tin*)p.v + (((size_t)b * T + t) * p.Hv + kh * r + vh) * D +
                                   r_lo + vi;
        dst[t * dstride] = ld_elem(src);
      }
    }
  }
  // every CTA of the cluster has read the old q/k conv state (the values are consumed)
  if (nsplit > 1) cluster_arrive_relaxed_mt();
  const bool per_token = snap_state && snap_slots;
  if (tid < token_chunks(T, TM) * TM)
    v.ssl[tid] = (per_token && tid < T) ? snap_slots[b * T + tid] : -1;
  __syncthreads();
  mt_norms(p, v, T, warp, MT_WARPS, lane);
  __syncthreads();
  mt_dots(v, T, TM, warp, MT_WARPS, lane);
  __syncthreads();
  mt_mats<TM>(v, T, r, warp, MT_WARPS, lane);
  __syncthreads();
  // ---- 5. the state rows: warp w takes passes w, w + 8, ...; the next pass's rows are
  //      copied into the warp's other buffer while this one's arithmetic runs
  for (int q = warp, pk = 0; q < NQ; q += MT_WARPS, pk ^= 1) {
    float4 st[RowGeo<TM>::RL][4];
    cp_async_wait_all();                               // this pass's rows (buffer pk)
    read_pass<TM>(stg + pk * SBUF, st, lane);
    if (q + MT_WARPS < NQ) prefetch_pass<TM>(p, it, r, q + MT_WARPS, stg + (pk ^ 1) * SBUF, lane);
    mt_pass<TM, TT / TM>(p, v, ost, it, T, r, q, per_token ? snap_state : nullptr, num_snap, st,
                         lane);
  }
  __syncthreads();
  mt_outputs<Tout>(p, ost, it, T, r, tid, MT_THREADS);
  // the q/k channels' new conv state (and per-token snapshots): rank 0, after the cluster's
  // reads of the old one
  if (nsplit > 1) cluster_wait_mt();
  if (sp == 0 && W > 0 && qkch >= 0) {
    store_window<TT>(qkwin, (Tin*)p.conv_state + (size_t)slot * H * C + qkch, T + 3 - H, H, C);
    if (snap_conv && snap_slots)
      for (int t = 0; t < T; ++t) {
        const int sl = snap_slots[b * T + t];
        if (sl >= 0 && sl < num_snap)
          store_window<TT>(qkwin, snap_conv + (size_t)sl * H * C + qkch, t + 4 - H, H, C);
      }
  }
  if (tid == 0 && sp == 0 && snap_slots && kh == 0) check_snap_rows(snap_slots, num_snap, b, T);
}

// ======================================================================= large batches
constexpr int WS_RW = 12;                    // row warps
constexpr int WS_PW = 4;                     // prologue warps
constexpr int WS_MAXNB = 5;                  // row buffers per row warp (at most)
constexpr int WS_THREADS = (WS_RW + WS_PW) * 32;
constexpr int WS_RT = WS_RW * 32, WS_PT = WS_PW * 32;
constexpr uint32_t WS_BAR_PRO = 2;           // named barrier of the prologue warps

// The staging area of an item's inputs (input type), byte offsets: x [T][ch_all] (without a
// conv: q, k, v), conv state [H][ch_all], conv weights [ch_all][W], bias [ch_all], with
// ch_all = (2 + r) D local channels (q, k, then the r value heads' v).  Every part is a
// multiple of 256 bytes.
struct MpStage {
  int x, cs, w, bias, bytes;
  __host__ __device__ MpStage(int T, int r, int W, bool has_bias, int esz) {
    const int ch = (2 + r) * D;
    x = 0;
    cs = x + T * ch * esz;
    w = cs + (W > 1 ? W - 1 : 0) * ch * esz;
    bias = w + W * ch * esz;
    bytes = bias + (W > 0 && has_bias ? ch * esz : 0);
  }
};

// shared memory of the warp-specialised kernel (bytes): two prologue buffers, two output
// buffers [T][r][D] (output type), the staging area, nb row buffers per row warp, the mbarriers
// (staged, ready[2], free[2]), the abort flag and the row warps' per-buffer done counts
struct WsLayout {
  ProOffsets pro;
  MpStage stg;
  int nb, pb, ost, stage, rows, bars, total;
  __host__ __device__ WsLayout(int T, int TM, int r, int W, bool has_bias, int esz, int osz,
                               int nb_)
      : pro(T, TM, r, D), stg(T, r, W, has_bias, esz), nb(nb_) {
    pb = 0;
    ost = pb + 2 * pro.total * 4;
    stage = ost + ((2 * T * r * D * osz + 15) & ~15);
    rows = stage + stg.bytes;
    bars = rows + WS_RW * nb * 4 * rows_per_lane(TM) * D * 4;
    total = bars + 7 * 8;
  }
};

// Bulk copies of an item's inputs into the staging area (warp-wide; lane i issues copies i,
// i + 32, ...): three runs (q, k, v channels) per token, per conv-state row, of the weights
// and of the bias.  Sources and sizes are multiples of 16 bytes (the launcher checks the
// base pointers).
template <typename Tin>
__device__ __forceinline__ void stage_item(const GdnLayerArgs& p, int T, int r, int b, int kh,
                                           int slot, uint8_t* stage, const MpStage& sl,
                                           uint32_t bar, int lane) {
  constexpr int E = sizeof(Tin);
  const int W = p.W, H = W > 0 ? W - 1 : 0, C = p.C_conv, ch = (2 + r) * D;
  // (the -DGDN_BOUNDS_CHECK build: an item outside the batch or the slot range is recorded and
  // replaced by item 0 of slot 0, so that the staged byte count stays what the barrier expects)
  if (!in_bounds(&g_err_multi, b >= 0 && b < p.B && kh >= 0 && kh < p.Hk && slot >= 0 &&
                                   slot < p.num_slots))
    b = kh = slot = 0;
  const int nx = 3 * T, ncs = nx + 3 * H, nw = ncs + (W > 0 ? 3 : 0);
  const int n = nw + (W > 0 && p.conv_b ? 3 : 0);
  if (lane == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)sl.bytes);
  __syncwarp();
  for (int i = lane; i < n; i += 32) {
    const int run = i % 3;                              // q, k, v channels
    const int lch = run * D;                            // first local channel
    const int gch = run == 0 ? kh * D : run == 1 ? (p.Hk + kh) * D : (2 * p.Hk + kh * r) * D;
    int len = run == 2 ? r * D : D;                     // elements
    const Tin* src;
    int dst;
    if (i < nx) {
      const int t = i / 3;
      if (W > 0) {
        src = (const Tin*)p.x + ((size_t)b * T + t) * C + gch;
      } else {
        src = run == 0   ? (const Tin*)p.q + (((size_t)b * T + t) * p.Hk + kh) * D
              : run == 1 ? (const Tin*)p.k + (((size_t)b * T + t) * p.Hk + kh) * D
                         : (const Tin*)p.v + (((size_t)b * T + t) * p.Hv + kh * r) * D;
      }
      dst = sl.x + (t * ch + lch) * E;
    } else if (i < ncs) {
      const int j = (i - nx) / 3;
      src = (const Tin*)p.conv_state + ((size_t)slot * H + j) * C + gch;
      dst = sl.cs + (j * ch + lch) * E;
    } else if (i < nw) {
      src = (const Tin*)p.conv_w + (size_t)gch * W;
      dst = sl.w + lch * W * E;
      len *= W;
    } else {
      src = (const Tin*)p.conv_b + gch;
      dst = sl.bias + lch * E;
    }
    ptx::bulk_load(ptx::smem_addr(stage + dst), src, (uint32_t)(len * E), bar);
  }
}

// four consecutive elements (an 8-byte bf16 / 16-byte fp32 load; the callers' offsets are
// multiples of four elements from 16-byte aligned bases)
__device__ __forceinline__ void ld4(const __nv_bfloat16* src, float (&o)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(src);
  o[0] = __uint_as_float(u.x << 16);
  o[1] = __uint_as_float(u.x & 0xffff0000u);
  o[2] = __uint_as_float(u.y << 16);
  o[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void ld4(const float* src, float (&o)[4]) {
  const float4 f = *reinterpret_cast<const float4*>(src);
  o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
}
__device__ __forceinline__ void st4(float* dst, const float (&v)[4]) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// Bulk stores of an item's new conv state, and of its conv state after every token, straight
// from the staged rows (warp-wide; lane i issues stores i, i + 32, ...; one commit group a
// lane): window position pos (conv-state rows at 3 - H .. 2, inputs at 3 .. 3 + T - 1) is
// staged conv-state row pos - (3 - H) below 3 and staged input row pos - 3 from 3 on; the
// conv state after token t is window positions t + 4 - H .. t + 3, the new one T + 3 - H ...
template <typename Tin>
__device__ __forceinline__ void store_conv_rows(const GdnLayerArgs& p, int T, int r,
                                                const RowItem& it, const uint8_t* stage,
                                                const MpStage& sl, const int32_t* snap_slots,
                                                int num_snap, Tin* snap_conv, int lane) {
  constexpr int E = sizeof(Tin);
  const int W = p.W, H = W > 0 ? W - 1 : 0, C = p.C_conv, ch = (2 + r) * D;
  const int njobs = 1 + (snap_conv && snap_slots ? T : 0), total = njobs * H * 3;
  for (int i = lane; i < total; i += 32) {
    const int job = i / (3 * H), rem = i - job * 3 * H, row = rem / 3, run = rem - row * 3;
    Tin* base;
    int shift;
    if (job == 0) {
      base = (Tin*)p.conv_state + (size_t)it.slot * H * C;
      shift = T + 3 - H;
    } else {
      const int s = snap_slots[it.b * T + job - 1];
      if (s < 0 || s >= num_snap) continue;
      base = snap_conv + (size_t)s * H * C;
      shift = job + 3 - H;                              // token t = job - 1: t + 4 - H
    }
    const int pos = shift + row, lch = run * D, len = run == 2 ? r * D : D;
    const int gch = run == 0   ? it.kh * D
                    : run == 1 ? (p.Hk + it.kh) * D
                               : (2 * p.Hk + it.kh * r) * D;
    const uint8_t* src = pos < 3 ? stage + sl.cs + ((pos - (3 - H)) * ch + lch) * E
                                 : stage + sl.x + ((pos - 3) * ch + lch) * E;
    ptx::bulk_store(base + (size_t)row * C + gch, ptx::smem_addr(src), (uint32_t)(len * E));
  }
  ptx::tma_store_commit();
}

// ---- 1+2. (staged, prologue warps) the conv (+SiLU) of an item's channels over the T tokens
//      (or its plain inputs), four channels a thread, and the L2 norms of q_t and k_t: the 128
//      channels of q (of k) are the four of each lane of prologue warp 0 (1), so that a norm
//      is one warp reduction.
template <typename Tin, int TM>
__device__ __forceinline__ void pro_conv_norm(const GdnLayerArgs& p, const ProView& v,
                                              const uint8_t* stage, const MpStage& sl,
                                              int T, int r, int pt, int nt) {
  const int W = p.W, H = W > 0 ? W - 1 : 0, ch_all = (2 + r) * D;
  const Tin* xs = reinterpret_cast<const Tin*>(stage + sl.x);
  const Tin* css = reinterpret_cast<const Tin*>(stage + sl.cs);
  const Tin* ws = reinterpret_cast<const Tin*>(stage + sl.w);
  const Tin* bs = reinterpret_cast<const Tin*>(stage + sl.bias);
  for (int cl = 4 * pt; cl < ch_all; cl += 4 * nt) {
    // window [3 + TM][4]: conv-state entries at 3 - H .. 2, inputs at 3 .. 3 + T - 1; after
    // the conv, entry t holds the output of token t
    float w[3 + TM][4];
    if (W > 0) {
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        if (j >= 3 - H) ld4(css + (j - 3 + H) * ch_all + cl, w[j]);
        else w[j][0] = w[j][1] = w[j][2] = w[j][3] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < T) ld4(xs + t * ch_all + cl, w[3 + t]);
        else w[3 + t][0] = w[3 + t][1] = w[3 + t][2] = w[3 + t][3] = 0.f;
      }
      float wt[4][4], bias[4] = {0.f, 0.f, 0.f, 0.f};   // taps right-aligned (zeros below 4 - W)
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) wt[c][j] = 0.f;
      if (W == 4) {                                    // a channel's taps: one 4-element load
#pragma unroll
        for (int c = 0; c < 4; ++c) ld4(ws + (cl + c) * 4, wt[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j >= 4 - W) wt[c][j] = ld_elem(ws + (cl + c) * W + j - 4 + W);
      }
      if (p.conv_b) ld4(bs + cl, bias);
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < T) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float y = bias[c];
#pragma unroll
            for (int j = 0; j < 4; ++j) y = fmaf(wt[c][j], w[t + j][c], y);
            w[t][c] = p.silu ? silu_gate(y) : y;
          }
        }
      }
    } else {
#pragma unroll
      for (int t = 0; t < TM; ++t)
        if (t < T) ld4(xs + t * ch_all + cl, w[t]);
    }
    float* dst;
    int stride;
    if (cl < 2 * D) {                                  // q (warp 0) or k (warp 1): the norms
      const bool isq = cl < D;
      float ss[TM];
#pragma unroll
      for (int t = 0; t < TM; ++t)
        ss[t] = fmaf(w[t][0], w[t][0], fmaf(w[t][1], w[t][1], fmaf(w[t][2], w[t][2],
                                                                  w[t][3] * w[t][3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int t = 0; t < TM; ++t)
          if (t < T) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        if (t < T) {
          const float inv =
              (p.l2norm ? 1.0f / sqrtf(ss[t] + p.eps) : 1.0f) * (isq ? p.scale : 1.0f);
#pragma unroll
          for (int c = 0; c < 4; ++c) w[t][c] *= inv;
        }
      }
      dst = (isq ? v.qh + cl : v.kh + cl - D);
      stride = D;
    } else {
      dst = v.vv + cl - 2 * D;
      stride = r * D;
    }
#pragma unroll
    for (int t = 0; t < TM; ++t)
      if (t < T) st4(dst + t * stride, w[t]);
  }
}

// ---- 3. (prologue warps) KK_ts = k_t . k_s and QK_ts = q_t . k_s: four lanes a pair (32
//      elements each), reduced over the four; each group starts at its own quarter of the
//      vectors, so that a warp's eight groups read different banks
__device__ __forceinline__ void pro_dots(const ProView& v, int T, int w0, int nw, int lane) {
  const int np = 2 * T * T, g4 = lane & 3, grp = lane >> 2;
  for (int base = w0 * 8; base < np; base += nw * 8) {
    const int pr = base + grp;
    const bool on = pr < np;
    const int which = pr / (T * T), t = (pr / T) % T, s2 = pr % T;
    float d = 0.f;
    if (on) {
      const float4* a4 = reinterpret_cast<const float4*>((which ? v.qh : v.kh) + t * D);
      const float4* k4 = reinterpret_cast<const float4*>(v.kh + s2 * D);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int i = g4 + 4 * ((m + grp) & 7);
        d = fma4(a4[i], k4[i], d);
      }
    }
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    if (on && g4 == 0) (which ? v.qk : v.kk)[t * T + s2] = d;
  }
}

// ---- 4. (prologue warps) per value head hh and column j (thread hh TM + j): the prefix
//      sums G_t from the gates, column j of (I + A)^{-1} by forward substitution and of
//      P (I + A)^{-1}, every A / P entry formed where it is used (no cross-lane steps); entry j
//      of e^{G_t}, beta_t, e^{G_{T-1} - G_t}, e^{g_t}.  Tokens T .. TM-1 give zeros.
template <int TM>
__device__ __forceinline__ void pro_mats(const ProView& v, int T, int r, int pt) {
  constexpr int HB = 3 * TM * TM + 4 * TM;
  if (pt >= r * TM) return;
  const int hh = pt / TM, j = pt - hh * TM;
  float* Mt = v.mats + hh * HB;
  float* eG = Mt + 3 * TM * TM;
  float* bt = eG + TM;
  float* dk = bt + TM;
  float* eg = dk + TM;
  const float* gb = v.gb + hh * TM * 2;
  float G[TM], beta[TM];
  float acc = 0.f, GT = 0.f, Gj = 0.f, gj = 0.f, bj = 0.f;
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    const float g = t < T ? gb[2 * t] : 0.f;
    beta[t] = t < T ? gb[2 * t + 1] : 0.f;
    acc += g;
    G[t] = acc;
    if (t == T - 1) GT = acc;
    if (t == j) { Gj = acc; gj = g; bj = beta[t]; }
  }
  const bool on = j < T;
  eG[j] = on ? expf(Gj) : 0.f;
  bt[j] = on ? bj : 0.f;
  dk[j] = on ? expf(GT - Gj) : 0.f;
  eg[j] = on ? expf(gj) : 1.f;
  float col[TM], pcol[TM];
#pragma unroll
  for (int t = 0; t < TM; ++t) col[t] = (t == j && on) ? 1.f : 0.f;
#pragma unroll
  for (int t = 1; t < TM; ++t) {
    if (t > j && t < T) {
      float a = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < TM; ++s2)
        if (s2 >= j && s2 < t)
          a = fmaf(beta[t] * expf(G[t] - G[s2]) * v.kk[t * T + s2], col[s2], a);
      col[t] = -a;
    }
  }
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    float a = 0.f;
    if (t < T && on) {
#pragma unroll
      for (int s2 = 0; s2 <= t; ++s2)
        if (s2 >= j) a = fmaf(expf(G[t] - G[s2]) * v.qk[t * T + s2], col[s2], a);
    }
    pcol[t] = a;
  }
#pragma unroll
  for (int t = 0; t < TM; ++t) {
    Mt[j * 2 * TM + t] = col[t];
    Mt[j * 2 * TM + TM + t] = pcol[t];
  }
}

// the slot of item `item`'s sequence, or -1 to skip it (a padded row, or an out-of-range slot,
// which thread 0 reports)
__device__ __forceinline__ int item_slot(const GdnLayerArgs& p, int item) {
  const int b = item / p.Hk;
  const int slot = p.slots ? p.slots[b] : b;
  if (slot >= p.num_slots) {
    if (threadIdx.x == 0 && item % p.Hk == 0) atomicOr(&g_err_multi, kErrIndex);
    return -1;
  }
  return slot;
}

// the first item at or after `item` (stepping by the grid) whose sequence has a state slot
__device__ __forceinline__ int next_item(const GdnLayerArgs& p, int item, int nitems,
                                         int& slot) {
  for (; item < nitems; item += gridDim.x)
    if ((slot = item_slot(p, item)) >= 0) return item;
  return nitems;
}

// a bounded wait on an mbarrier phase that also gives up once the other role has aborted;
// false (and the abort flag set) on a time-out
__device__ __forceinline__ bool ws_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (ptx::mbar_wait_or_abort(bar, parity, abort)) return true;
  if (!*abort) atomicOr(&g_err_multi, kErrTimeout);
  *abort = 1;
  return false;
}

template <typename Tin, typename Tout, int TM>
__global__ void __launch_bounds__(WS_THREADS, 1)
    gdn_decode_multi_ws_kernel(GdnLayerArgs p, int T, int nb, float* snap_state, int num_snap,
                               const int32_t* snap_slots, Tin* snap_conv) {
  extern __shared__ __align__(16) uint8_t wsm[];
  constexpr int SBUF = RowGeo<TM>::SBUF;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = p.Hv / p.Hk, nitems = p.B * p.Hk;
  const WsLayout lay(T, TM, r, p.W, p.conv_b != nullptr, (int)sizeof(Tin), (int)sizeof(Tout),
                     nb);
  const uint32_t bars = ptx::smem_addr(wsm + lay.bars);
  const uint32_t staged = bars, ready0 = bars + 8, free0 = bars + 24;
  volatile int* abort = reinterpret_cast<volatile int*>(wsm + lay.bars + 40);
  int* done = reinterpret_cast<int*>(wsm + lay.bars + 48);    // [2]
  auto pro_view = [&](int i) {
    return ProView(reinterpret_cast<float*>(wsm + lay.pb) + i * lay.pro.total, lay.pro);
  };
  const bool per_token = snap_state && snap_slots;
  if (tid == 0) {
    ptx::mbar_init(staged, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ready0 + 8 * i, 1);
      ptx::mbar_init(free0 + 8 * i, 1);
    }
    *abort = 0;
    done[0] = done[1] = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // ---- the first item's prologue, by every warp (no rows stream yet); the prologue warps then
  //      prepare the items after it
  const int pt = tid - WS_RT, pw = warp - WS_RW;       // (prologue warps)
  uint8_t* stage = wsm + lay.stage;
  int slot0 = -1;
  const int item0 = next_item(p, blockIdx.x, nitems, slot0);
  int nslot0 = -1;
  const int item1 = item0 < nitems ? next_item(p, item0 + gridDim.x, nitems, nslot0) : nitems;
  int pending = -1;                                  // ordinal of a staged, unconsumed item
  GateRaw graw{0.f, 0.f, 0.f, 0.f};
  if (item0 < nitems) {
    if (pw == 0) stage_item<Tin>(p, T, r, item0 / p.Hk, item0 % p.Hk, slot0, stage, lay.stg,
                                 staged, lane);
    pending = 0;
    if (warp >= WS_RW) graw = load_gate_raw<Tin>(p, item0 / p.Hk, T, item0 % p.Hk, r, pt);
  }
  // the row warps' copies start once the staging copies are issued (two passes ahead)
  const int NQ = r * (D / (4 * RowGeo<TM>::RL));       // passes per item (>= 16 > WS_RW)
  float4* buf = reinterpret_cast<float4*>(wsm + lay.rows) + (warp < WS_RW ? warp : 0) * nb * SBUF;
  int cs = slot0, ci = item0, cq = warp;               // copy cursor (row warps)
  auto issue = [&](int into) {
    prefetch_pass<TM>(p, RowItem{ci / p.Hk, ci % p.Hk, cs, 0, D}, r, cq, buf + into * SBUF,
                      lane, ci < nitems);
    if (ci < nitems && (cq += WS_RW) >= NQ) {
      cq = warp;
      ci = next_item(p, ci + gridDim.x, nitems, cs);
    }
  };
  // (the staged inputs go first: the rows' copies queue behind them)
  __syncthreads();
  if (warp < WS_RW)
    for (int j = 0; j < nb - 1; ++j) issue(j);
  bool ok0 = true;
  if (item0 < nitems) {
    const RowItem it{item0 / p.Hk, item0 % p.Hk, slot0, 0, D};
    const ProView v = pro_view(0);
    ok0 = ptx::mbar_wait_bounded(staged, 0);
    if (__syncthreads_and(ok0)) {
      pending = -1;
      if (pw == 0)
        store_conv_rows<Tin>(p, T, r, it, stage, lay.stg, snap_slots, num_snap, snap_conv, lane);
      if (warp >= WS_RW) store_gate<TM>(p, graw, v.gb, T, r, pt);
      if (tid < TM) v.ssl[tid] = (per_token && tid < T) ? snap_slots[it.b * T + tid] : -1;
      pro_conv_norm<Tin, TM>(p, v, stage, lay.stg, T, r, tid, WS_THREADS);
      __syncthreads();
      if (item1 < nitems) {
        if (pw == 0) {
          ptx::tma_store_wait_read();
          __syncwarp();
          stage_item<Tin>(p, T, r, item1 / p.Hk, item1 % p.Hk, nslot0, stage, lay.stg, staged,
                          lane);
        }
        pending = 1;
        if (warp >= WS_RW) graw = load_gate_raw<Tin>(p, item1 / p.Hk, T, item1 % p.Hk, r, pt);
      }
      pro_dots(v, T, warp, WS_THREADS / 32, lane);
      __syncthreads();
      pro_mats<TM>(v, T, r, tid);
      __syncthreads();
      if (tid == 0) ptx::mbar_arrive(ready0);          // (the first item's buffer is ready)
    } else if (tid == 0) {
      atomicOr(&g_err_multi, kErrTimeout);
    }
  }
  if (warp < WS_RW) {
    // ---------------------------------------------------------------- row warps
    const int rw = warp;
    int slot = slot0, pk = 0;
    int item = ok0 ? item0 : nitems;
    for (int n = 0; item < nitems; ++n) {
      const RowItem it{item / p.Hk, item % p.Hk, slot, 0, D};
      if (!ws_wait(ready0 + 8 * (n & 1), (n >> 1) & 1, abort)) break;
      const ProView v = pro_view(n & 1);
      Tout* ost = reinterpret_cast<Tout*>(wsm + lay.ost) + (n & 1) * T * r * D;
      for (int q = rw; q < NQ; q += WS_RW) {
        float4 st[RowGeo<TM>::RL][4];
        cp_async_wait_upto(nb - 2);
        read_pass<TM>(buf + pk * SBUF, st, lane);
        issue(pk == 0 ? nb - 1 : pk - 1);              // the buffer read a pass ago
        pk = pk + 1 == nb ? 0 : pk + 1;
        mt_pass<TM, 1>(p, v, ost, it, T, r, q, per_token ? snap_state : nullptr, num_snap, st,
                       lane);
      }
      // this warp's share of the item is done; the last row warp to finish it sends the
      // outputs (a bulk store per token row of the item's heads) and, once they have read
      // ost, hands the prologue buffer back (so that ost is free again when the item two on
      // is released to the row warps)
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&done[n & 1], 1) == WS_RW - 1) {
          done[n & 1] = 0;
          __threadfence_block();
          for (int t = 0; t < T; ++t)
            ptx::bulk_store((Tout*)p.out + (((size_t)it.b * T + t) * p.Hv + it.kh * r) * D,
                            ptx::smem_addr(ost + t * r * D), (uint32_t)(r * D * sizeof(Tout)));
          ptx::tma_store_commit();
          ptx::tma_store_wait_read();
          ptx::mbar_arrive(free0 + 8 * (n & 1));
        }
      }
      int ns = -1;
      item = next_item(p, item + gridDim.x, nitems, ns);
      slot = ns;
    }
    cp_async_wait_all();
    if (lane == 0) ptx::tma_store_wait_all();
  } else {
    // ---------------------------------------------------------------- prologue warps
    int item = ok0 ? item1 : nitems, slot = nslot0;
    for (int m = 1; item < nitems; ++m) {
      const RowItem it{item / p.Hk, item % p.Hk, slot, 0, D};
      int nslot = -1;
      const int next = next_item(p, item + gridDim.x, nitems, nslot);
      bool ok = m < 2 || ws_wait(free0 + 8 * (m & 1), ((m >> 1) + 1) & 1, abort);
      ok = ok && ws_wait(staged, m & 1, abort);
      if (ptx::named_bar_sync_or(WS_BAR_PRO, WS_PT, !ok)) break;
      pending = -1;
      const ProView v = pro_view(m & 1);
      // the new conv state (and the per-token ones) leave straight from the staged rows
      if (pw == 0)
        store_conv_rows<Tin>(p, T, r, it, stage, lay.stg, snap_slots, num_snap, snap_conv, lane);
      store_gate<TM>(p, graw, v.gb, T, r, pt);
      if (pt < TM) v.ssl[pt] = (per_token && pt < T) ? snap_slots[it.b * T + pt] : -1;
      pro_conv_norm<Tin, TM>(p, v, stage, lay.stg, T, r, pt, WS_PT);
      ptx::named_bar_sync(WS_BAR_PRO, WS_PT);
      // the staging area is read (by the conv, and by the stores once they report it): the
      // next item's inputs into it, its gates into registers
      if (next < nitems) {
        if (pw == 0) {
          ptx::tma_store_wait_read();
          __syncwarp();
          stage_item<Tin>(p, T, r, next / p.Hk, next % p.Hk, nslot, stage, lay.stg, staged,
                          lane);
        }
        pending = m + 1;
        graw = load_gate_raw<Tin>(p, next / p.Hk, T, next % p.Hk, r, pt);
      }
      pro_dots(v, T, pw, WS_PW, lane);
      ptx::named_bar_sync(WS_BAR_PRO, WS_PT);
      pro_mats<TM>(v, T, r, pt);
      ptx::named_bar_sync(WS_BAR_PRO, WS_PT);
      if (pt == 0) {
        ptx::mbar_arrive(ready0 + 8 * (m & 1));
        if (snap_slots && it.kh == 0) check_snap_rows(snap_slots, num_snap, it.b, T);
      }
      item = next;
      slot = nslot;
    }
    if (pt == 0 && item0 < nitems && snap_slots && item0 % p.Hk == 0)
      check_snap_rows(snap_slots, num_snap, item0 / p.Hk, T);
    // after an abort, staged copies still in flight must land before the CTA leaves; the
    // conv-state stores must have completed
    if (pending >= 0 && pt == 0) ptx::mbar_wait_bounded(staged, pending & 1, 1u << 16);
    if (pw == 0) ptx::tma_store_wait_all();
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// the warp-specialised kernel's inputs can be bulk-copied (16-byte aligned runs)
bool stageable(const GdnLayerArgs& p) {
  if (p.W > 0)
    return aligned16(p.x) && aligned16(p.conv_w) && (!p.conv_b || aligned16(p.conv_b)) &&
           (p.W == 1 || aligned16(p.conv_state));
  return aligned16(p.q) && aligned16(p.k) && aligned16(p.v);
}

constexpr int kMaxDynSmem = 227 * 1024;

// Raises a kernel's dynamic shared-memory limit to at least `bytes`: on the first call to
// `initial` (at least what the common shapes need), so that later launches, e.g. under
// CUDA-graph capture, make no attribute calls; later only for a larger request.
template <typename K>
cudaError_t ensure_smem(K kernel, int bytes, int initial, int* have) {
  if (bytes <= *have) return cudaSuccess;
  const int want = bytes > initial ? bytes : initial;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
  if (e == cudaSuccess) *have = want;
  return e;
}

template <typename Tin, typename Tout, int TM, int TT>
cudaError_t launch_multi_tm(const GdnLayerArgs& p, int T, float* snap_state, int num_snap,
                            const int32_t* snap_slots, void* snap_conv, cudaStream_t stream) {
  const int r = p.Hv / p.Hk;
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int nitems = p.B * p.Hk;
  // large batches of up to four tokens: the warp-specialised kernel, with as many row buffers
  // per warp as fit (up to five), when the inputs can be staged (at eight tokens and more the
  // per-item kernel below measured faster: 317.5 against 324 us at 16/48 heads, B = 128,
  // T = 8)
  if constexpr (TM == 4) {
    if (nitems > sms && T * r <= WS_PT && stageable(p) && aligned16(p.out)) {
      auto kern = gdn_decode_multi_ws_kernel<Tin, Tout, TM>;
      const bool hb = p.conv_b != nullptr;
      int nb = WS_MAXNB;
      const int isz = (int)sizeof(Tin), osz = (int)sizeof(Tout);
      size_t smem = WsLayout(T, TM, r, p.W, hb, isz, osz, nb).total;
      while (nb > 2 && smem > (size_t)kMaxDynSmem)
        smem = WsLayout(T, TM, r, p.W, hb, isz, osz, --nb).total;
      static int have[32] = {};
      if (smem <= (size_t)kMaxDynSmem &&
          ensure_smem(kern, (int)smem, kMaxDynSmem, &have[dev & 31]) == cudaSuccess) {
        const int grid = nitems < sms ? nitems : sms;
        return launch_pdl(false, kern, dim3(grid), dim3(WS_THREADS), smem, stream, p, T, nb,
                          snap_state, num_snap, snap_slots, static_cast<Tin*>(snap_conv));
      }
      (void)cudaGetLastError();        // (a refused size: the per-item kernel below)
    }
  }
  // rows of each value head split over a cluster of nsplit CTAs when the (sequence, key head)
  // items alone would leave most SMs idle
  int nsplit = 1;
  while (nsplit < 8 && nitems * nsplit * 2 <= 2 * sms) nsplit *= 2;
  const size_t smem = sizeof(float) * MtLayout(T, TM, r, D / nsplit).total;
  const int top = (int)(sizeof(float) * MtLayout(TT, TM, 8, D).total);
  static int have_c[32] = {};
  if ((e = ensure_smem(gdn_decode_multi_kernel<Tin, Tout, TM, TT>, (int)smem,
                       top < kMaxDynSmem ? top : kMaxDynSmem, &have_c[dev & 31])) !=
      cudaSuccess)
    return e;
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
  return cudaLaunchKernelEx(&cfg, gdn_decode_multi_kernel<Tin, Tout, TM, TT>, p, T, snap_state,
                            num_snap, snap_slots, static_cast<Tin*>(snap_conv), nsplit);
}

template <typename Tin, typename Tout>
cudaError_t launch_multi_t(const GdnLayerArgs& p, int T, float* snap_state, int num_snap,
                           const int32_t* snap_slots, void* snap_conv, cudaStream_t stream) {
  // up to 4 tokens: one chunk of 4; up to 8: one chunk of 8; up to 16: chunks of 8
  if (T <= 4)
    return launch_multi_tm<Tin, Tout, 4, 4>(p, T, snap_state, num_snap, snap_slots, snap_conv,
                                            stream);
  if (T <= 8)
    return launch_multi_tm<Tin, Tout, 8, 8>(p, T, snap_state, num_snap, snap_slots, snap_conv,
                                            stream);
  return launch_multi_tm<Tin, Tout, 8, 16>(p, T, snap_state, num_snap, snap_slots, snap_conv,
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
