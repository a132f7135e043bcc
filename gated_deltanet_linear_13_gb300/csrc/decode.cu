// Batched single-token decode of the gated delta rule: one fused kernel.
//
// Per (sequence b, value head h) the step is the model card's "How It Works" loop for one
// token (decay, read, delta, write, output) on the fp32 state S[v][k] already in HBM, with
// the causal conv update (+SiLU), the L2 norm of q and k and the gates fused in front.
//
// Row independence: row i of S only needs v_i, and the output o_i only needs row i:
//     alpha = s_i . k,  gamma = s_i . q,  delta_i = beta (v_i - e^g alpha),
//     s_i <- e^g s_i + delta_i k,        o_i = e^g gamma + delta_i (k . q)
// (o = S_new q = e^g S q + delta (k . q)), so each row is streamed through once.  A CTA's
// R contiguous state rows (R * 512 bytes) move HBM -> shared memory with one TMA bulk copy
// issued before the conv / norm / gates prologue, and back with one bulk store: the bytes in
// flight do not depend on registers or occupancy.  In shared memory one warp handles a
// 512-byte row with 128-bit accesses and two warp-wide dot products.
//
// Work split: a thread-block cluster per (b, key head); its CTAs are the r = Hv/Hk value
// heads of that key head times `nsplit` row blocks of R = 128/nsplit rows.  Every CTA
// recomputes the conv of the shared q/k channels; the cluster barrier orders all CTAs'
// reads of the old q/k conv state before the one CTA that writes the new one.  The v
// channels of rows [r0, r0+R) belong to one CTA only.
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

// Conv of one channel: window = [old state (W-1 values, oldest first), new input].
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

template <typename Tin, typename Tout, int R>
__global__ void __launch_bounds__(256) gdn_decode_kernel(GdnLayerArgs p, int nsplit) {
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
  if (tid < R) {
    Tout* o = (Tout*)p.out + ((size_t)b * p.Hv + h) * D + r0 + tid;
    *o = from_float<Tout>(so[tid]);
    if (p.W > 1) conv_store_state<Tin>(p, slot, chv, winv);
  }
  cluster_wait_acquire();
  if (p.W > 1 && hh == 0 && sp == 0) conv_store_state<Tin>(p, slot, ch, win);
  if (tid == 0) tma_store_wait_all();     // the bulk store has read shared memory and landed
}

template <typename Tin, typename Tout, int R>
static cudaError_t launch_decode_t(const GdnLayerArgs& p, int nsplit, cudaStream_t stream) {
  static unsigned done = 0;
  cudaError_t e = set_smem_once(gdn_decode_kernel<Tin, Tout, R>, R * kHeadDim * 4, &done);
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
  return cudaLaunchKernelEx(&cfg, gdn_decode_kernel<Tin, Tout, R>, p, nsplit);
}

cudaError_t gdn_launch_decode(const GdnLayerArgs& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  const int r = p.Hv / p.Hk;
  int nsplit = 8 / r;           // cluster of r * nsplit <= 8 CTAs
  if (nsplit >= 8) nsplit = 8;
  else if (nsplit >= 4) nsplit = 4;
  else if (nsplit >= 2) nsplit = 2;
  else nsplit = 1;
  const int R = kHeadDim / nsplit;
#define GDN_DEC(TI, TO)                                                         \
  switch (R) {                                                                  \
    case 16: return launch_decode_t<TI, TO, 16>(p, nsplit, stream);             \
    case 32: return launch_decode_t<TI, TO, 32>(p, nsplit, stream);             \
    case 64: return launch_decode_t<TI, TO, 64>(p, nsplit, stream);             \
    default: return launch_decode_t<TI, TO, 128>(p, nsplit, stream);            \
  }
  if (p.in_bf16) {
    if (p.out_bf16) { GDN_DEC(__nv_bfloat16, __nv_bfloat16) }
    GDN_DEC(__nv_bfloat16, float)
  }
  GDN_DEC(float, float)
#undef GDN_DEC
}
