// Chunked gated-delta-rule prefill on the fp32 FMA pipes: the all-fp32 mode.
//
// Chunked WY/UT form with a direct triangular solve (PR #164 "Fused DeltaNet Direct-Solve
// Follow-Up": the Neumann power-doubling solve is replaced by a direct solve of the lower-
// triangular causal system).  Per chunk of C = 64 tokens with entering state S0 [v][k] and
// in-chunk cumulative log-decay G_r:
//   A[r][s] = beta_r e^{G_r - G_s} (k_r . k_s), s < r      T = (I + A)^{-1}
//   W  = T diag(beta e^G) K,     U = T diag(beta) V - W S0^T
//   P[r][s] = e^{G_r - G_s} (q_r . k_s), s <= r
//   O  = diag(e^G) Q S0^T + P U
//   S  = e^{G_last} S0 + U^T diag(e^{G_last - G}) K
// which unrolls the per-token recurrence of the model card "Qwen3.5 Gated Delta Net NKI
// Kernel for AWS Neuron" ("How It Works") exactly.  Exponentials are only taken of
// G_r - G_s with r >= s (<= 0), so strong decay underflows to zero instead of overflowing.
//
// Grid: (4 row blocks of 32 state rows, Hv, B); the rows of S are independent, so a CTA owns
// a 32 x 128 slice of the state for the whole sequence and recomputes the chunk-local
// quantities (A, T, W, P) that all row blocks share.  A last chunk shorter than C is padded
// with q = k = v = 0, g = 0, beta = 0 (identity steps).
#include "common.cuh"

using namespace gdn;

static __device__ unsigned int g_err_simt;

unsigned gdn_take_error_prefill_simt() {
  unsigned v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_simt, sizeof(v));
  cudaMemcpyToSymbol(g_err_simt, &z, sizeof(z));
  return v;
}

namespace {
constexpr int C = kChunk, D = kHeadDim, R = 32, NSPLIT = D / R;
constexpr int LD = D + 4;     // padded row stride of [*, D] tiles
constexpr int LT = C + 1;     // padded row stride of [C, C] tiles
constexpr int LV = R + 1;     // padded row stride of [C, R] tiles
constexpr int SMEM_FLOATS = 3 * C * LD + 3 * C * LT + 2 * C * LV + R * LD + 8 * C;
constexpr int THREADS = 256;
}  // namespace

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(THREADS) gdn_prefill_simt_kernel(GdnLayerArgs p) {
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;              // [C][LD]  q-hat (scaled)
  float* Ks = Qs + C * LD;       // [C][LD]  k-hat
  float* Ws = Ks + C * LD;       // [C][LD]  W
  float* As = Ws + C * LD;       // [C][LT]  A (strictly lower)
  float* Ps = As + C * LT;       // [C][LT]  P (lower incl. diagonal)
  float* Ts = Ps + C * LT;       // [C][LT]  T = (I + A)^{-1}
  float* Vs = Ts + C * LT;       // [C][LV]  v slice
  float* Us = Vs + C * LV;       // [C][LV]  U slice
  float* Ss = Us + C * LV;       // [R][LD]  state slice S0 / S
  float* Gs = Ss + R * LD;       // [C] cumulative log-decay
  float* Bs = Gs + C;            // [C] beta
  float* Nq = Bs + C;            // [C] 1/||q||
  float* Nk = Nq + C;            // [C] 1/||k||
  float* Eg = Nk + C;            // [C] e^{G_r}
  float* BEg = Eg + C;           // [C] beta_r e^{G_r}
  float* Dk = BEg + C;           // [C] e^{G_last - G_r}

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r = p.Hv / p.Hk, kh = h / r, r0 = sp * R;
  const int slot = p.slots ? p.slots[b] : b;
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (tid == 0 && sp == 0) atomicOr(&g_err_simt, kErrIndex);
    return;
  }
  // tokens of sequence b: [tokb, tokb + Tb) of its own row, or of the packed axis
  const long long tokb = p.cu ? p.cu[b] : (long long)b * p.T;
  const int Tb = p.cu ? p.cu[b + 1] - p.cu[b] : p.T;
  const Tin* qg = (const Tin*)p.q + (size_t)tokb * p.q_tok_stride + kh * D;
  const Tin* kg = (const Tin*)p.k + (size_t)tokb * p.k_tok_stride + kh * D;
  const Tin* vg = (const Tin*)p.v + (size_t)tokb * p.v_tok_stride + h * D + r0;
  float* Sg = p.state + (((size_t)slot * p.Hv + h) * D + r0) * D;

  for (int idx = tid; idx < R * D; idx += THREADS) Ss[(idx / D) * LD + idx % D] = Sg[idx];

  // in-call snapshot j (the state after token (j + 1) snap_every) of this block's rows
  auto snapshot = [&](int j) {
    const int sl = p.snap_slots[(size_t)b * p.n_snap + j];
    if (sl < 0) return;
    if (sl >= p.num_snap_slots) {
      if (tid == 0) atomicOr(&g_err_simt, kErrIndex);
      return;
    }
    float* dst = p.snap_state + (((size_t)sl * p.Hv + h) * D + r0) * D;
    for (int idx = tid; idx < R * D; idx += THREADS) dst[idx] = Ss[(idx / D) * LD + idx % D];
  };

  for (int t0 = 0; t0 < Tb; t0 += C) {
    const int n = min(C, Tb - t0);
    if (p.snap_every > 0 && t0 > 0 && t0 % p.snap_every == 0) snapshot(t0 / p.snap_every - 1);
    // ---- load the chunk (zero padded)
    for (int idx = tid; idx < C * D; idx += THREADS) {
      const int rr = idx / D, j = idx % D;
      float qv = 0.f, kv = 0.f;
      if (rr < n) {
        qv = ld_elem(qg + (size_t)(t0 + rr) * p.q_tok_stride + j);
        kv = ld_elem(kg + (size_t)(t0 + rr) * p.k_tok_stride + j);
      }
      Qs[rr * LD + j] = qv;
      Ks[rr * LD + j] = kv;
    }
    for (int idx = tid; idx < C * R; idx += THREADS) {
      const int rr = idx / R, i = idx % R;
      Vs[rr * LV + i] = rr < n ? ld_elem(vg + (size_t)(t0 + rr) * p.v_tok_stride + i) : 0.f;
    }
    if (tid < C) {
      float g = 0.f, beta = 0.f;
      if (tid < n) {
        const size_t gi = ((size_t)tokb + t0 + tid) * p.Hv + h;
        if (p.gates_pre) {
          g = ((const float*)p.a)[gi];
          beta = ((const float*)p.b)[gi];
        } else {
          g = gate_g(ld_elem((const Tin*)p.a + gi), p.A_log[h], p.dt_bias ? p.dt_bias[h] : 0.f);
          beta = sigmoid_f(ld_elem((const Tin*)p.b + gi));
        }
      }
      Gs[tid] = g;
      Bs[tid] = beta;
    }
    __syncthreads();
    // ---- norms (one warp per row) and the prefix sum of g
    for (int rr = warp; rr < C; rr += THREADS / 32) {
      float sq = 0.f, sk = 0.f;
      for (int j = lane; j < D; j += 32) {
        const float a = Qs[rr * LD + j], c = Ks[rr * LD + j];
        sq = fmaf(a, a, sq);
        sk = fmaf(c, c, sk);
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      if (lane == 0) {
        Nq[rr] = (p.l2norm ? 1.0f / sqrtf(sq + p.eps) : 1.0f) * p.scale;
        Nk[rr] = p.l2norm ? 1.0f / sqrtf(sk + p.eps) : 1.0f;
      }
    }
    if (tid == 0) {
      float acc = 0.f;
      for (int rr = 0; rr < C; ++rr) { acc += Gs[rr]; Gs[rr] = acc; }
    }
    __syncthreads();
    for (int idx = tid; idx < C * D; idx += THREADS) {
      const int rr = idx / D, j = idx % D;
      Qs[rr * LD + j] *= Nq[rr];
      Ks[rr * LD + j] *= Nk[rr];
    }
    if (tid < C) {
      const float Gl = Gs[C - 1];
      Eg[tid] = expf(Gs[tid]);
      BEg[tid] = Bs[tid] * expf(Gs[tid]);
      Dk[tid] = expf(Gl - Gs[tid]);
    }
    __syncthreads();
    // ---- A and P
    for (int idx = tid; idx < C * C; idx += THREADS) {
      const int rr = idx / C, s = idx % C;
      float a = 0.f, pp = 0.f;
      if (s <= rr) {
        float dk = 0.f, dq = 0.f;
        const float4* kr = reinterpret_cast<const float4*>(Ks + rr * LD);
        const float4* qr = reinterpret_cast<const float4*>(Qs + rr * LD);
        const float4* ks = reinterpret_cast<const float4*>(Ks + s * LD);
#pragma unroll 8
        for (int j = 0; j < D / 4; ++j) {
          const float4 x = ks[j], y = kr[j], z = qr[j];
          dk = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, dk))));
          dq = fmaf(x.x, z.x, fmaf(x.y, z.y, fmaf(x.z, z.z, fmaf(x.w, z.w, dq))));
        }
        const float e = expf(Gs[rr] - Gs[s]);
        if (s < rr) a = Bs[rr] * e * dk;
        pp = e * dq;
      }
      As[rr * LT + s] = a;
      Ps[rr * LT + s] = pp;
    }
    __syncthreads();
    // ---- T = (I + A)^{-1}: one thread per column, forward substitution down the rows
    if (tid < C) {
      const int j = tid;
      for (int rr = 0; rr <= j; ++rr) Ts[rr * LT + j] = (rr == j) ? 1.f : 0.f;
      for (int rr = j + 1; rr < C; ++rr) {
        float acc = 0.f;
        for (int s = j; s < rr; ++s) acc = fmaf(As[rr * LT + s], Ts[s * LT + j], acc);
        Ts[rr * LT + j] = -acc;
      }
    }
    __syncthreads();
    // ---- W = T diag(beta e^G) K,  U' = T diag(beta) V
    for (int idx = tid; idx < C * D; idx += THREADS) {
      const int rr = idx / D, j = idx % D;
      float acc = 0.f;
      for (int s = 0; s <= rr; ++s) acc = fmaf(Ts[rr * LT + s] * BEg[s], Ks[s * LD + j], acc);
      Ws[rr * LD + j] = acc;
    }
    for (int idx = tid; idx < C * R; idx += THREADS) {
      const int rr = idx / R, i = idx % R;
      float acc = 0.f;
      for (int s = 0; s <= rr; ++s) acc = fmaf(Ts[rr * LT + s] * Bs[s], Vs[s * LV + i], acc);
      Us[rr * LV + i] = acc;
    }
    __syncthreads();
    // ---- U = U' - W S0^T
    for (int idx = tid; idx < C * R; idx += THREADS) {
      const int rr = idx / R, i = idx % R;
      float acc = 0.f;
      const float4* w4 = reinterpret_cast<const float4*>(Ws + rr * LD);
      const float4* s4 = reinterpret_cast<const float4*>(Ss + i * LD);
#pragma unroll 8
      for (int j = 0; j < D / 4; ++j) {
        const float4 x = w4[j], y = s4[j];
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
      }
      Us[rr * LV + i] -= acc;
    }
    __syncthreads();
    // ---- O = diag(e^G) Q S0^T + P U
    for (int idx = tid; idx < C * R; idx += THREADS) {
      const int rr = idx / R, i = idx % R;
      if (rr >= n) continue;
      float inter = 0.f;
      const float4* q4 = reinterpret_cast<const float4*>(Qs + rr * LD);
      const float4* s4 = reinterpret_cast<const float4*>(Ss + i * LD);
#pragma unroll 8
      for (int j = 0; j < D / 4; ++j) {
        const float4 x = q4[j], y = s4[j];
        inter = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, inter))));
      }
      float intra = 0.f;
      for (int s = 0; s <= rr; ++s) intra = fmaf(Ps[rr * LT + s], Us[s * LV + i], intra);
      const float o = fmaf(Eg[rr], inter, intra);
      Tout* og = (Tout*)p.out + (((size_t)tokb + t0 + rr) * p.Hv + h) * D + r0 + i;
      *og = from_float<Tout>(o);
    }
    __syncthreads();
    // ---- S = e^{G_last} S0 + U^T diag(e^{G_last - G}) K
    {
      const float eGl = expf(Gs[C - 1]);
      for (int idx = tid; idx < R * D; idx += THREADS) {
        const int i = idx / D, j = idx % D;
        float acc = eGl * Ss[i * LD + j];
        for (int rr = 0; rr < n; ++rr)
          acc = fmaf(Us[rr * LV + i] * Dk[rr], Ks[rr * LD + j], acc);
        Ss[i * LD + j] = acc;
      }
    }
    __syncthreads();
  }
  for (int idx = tid; idx < R * D; idx += THREADS) Sg[idx] = Ss[(idx / D) * LD + idx % D];
  if (p.snap_every > 0 && p.T % p.snap_every == 0) snapshot(p.T / p.snap_every - 1);
}

template <typename Tin, typename Tout>
static cudaError_t launch_simt_t(const GdnLayerArgs& p, cudaStream_t stream) {
  const size_t smem = sizeof(float) * SMEM_FLOATS;
  static unsigned done = 0;
  cudaError_t e = set_smem_once(gdn_prefill_simt_kernel<Tin, Tout>, (int)smem, &done);
  if (e != cudaSuccess) return e;
  dim3 grid(NSPLIT, (unsigned)p.Hv, (unsigned)p.B);
  gdn_prefill_simt_kernel<Tin, Tout><<<grid, THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t gdn_launch_prefill_simt(const GdnLayerArgs& p, cudaStream_t stream) {
  if (p.B == 0 || p.T == 0) return cudaSuccess;
  if (p.in_bf16) {
    if (p.out_bf16) return launch_simt_t<__nv_bfloat16, __nv_bfloat16>(p, stream);
    return launch_simt_t<__nv_bfloat16, float>(p, stream);
  }
  return launch_simt_t<float, float>(p, stream);
}

// ======================================================================= gated output norm
// out_i = w_i * o_i / sqrt(mean(o^2) + eps) * silu(z_i) per (token, value head) vector of 128,
// in place: one warp per vector, four channels per lane.
__global__ void __launch_bounds__(256) gdn_gated_norm_f32_kernel(
    float* out, const float* __restrict__ z, const float* __restrict__ w, float eps,
    long long rows, long long rows_per_seq, const int32_t* slots, int num_slots,
    const int32_t* cu, int nseq, int Hv) {
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  if (slots) {
    long long seq = r / rows_per_seq;
    if (cu) {                                      // packed batch: the sequence of the token
      const long long tok = r / Hv;
      int lo = 0, hi = nseq;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= tok) lo = mid; else hi = mid;
      }
      seq = lo;
    }
    const int s = slots[seq];
    if (s < 0 || s >= num_slots) return;           // a skipped batch entry keeps its rows
  }
  float4* o4 = reinterpret_cast<float4*>(out + r * D) + lane;
  const float4 o = *o4;
  const float4 zz = reinterpret_cast<const float4*>(z + r * D)[lane];
  const float4 ww = reinterpret_cast<const float4*>(w)[lane];
  const float ss = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
  const float inv = rsqrtf(ss * (1.0f / D) + eps);
  float4 y;
  y.x = ww.x * (o.x * inv) * silu_gate(zz.x);
  y.y = ww.y * (o.y * inv) * silu_gate(zz.y);
  y.z = ww.z * (o.z * inv) * silu_gate(zz.z);
  y.w = ww.w * (o.w * inv) * silu_gate(zz.w);
  *o4 = y;
}

cudaError_t gdn_launch_gated_norm_f32(float* out, const float* z, const float* w, float eps,
                                      int B, long long rows_per_seq, const int32_t* slots,
                                      int num_slots, cudaStream_t stream, const int32_t* cu,
                                      int Hv) {
  // (a packed batch passes B = 1, rows_per_seq = T Hv and its B sequences' offsets in cu)
  const long long rows = (long long)(cu ? 1 : B) * rows_per_seq;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  gdn_gated_norm_f32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      out, z, w, eps, rows, rows_per_seq, slots, num_slots, cu, B, Hv);
  return cudaGetLastError();
}
