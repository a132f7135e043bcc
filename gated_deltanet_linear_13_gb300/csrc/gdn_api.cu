// The C ABI of libgdn.so: host-side validation, workspace sizing, kernel dispatch, status.
// Every argument is checked before any CUDA call; see include/gdn.h for the contract.
#include <math.h>
#include <string.h>

#include "common.cuh"

namespace {

constexpr int32_t kVersion = 104;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
size_t elem_bytes(gdn_dtype t) { return t == GDN_BF16 ? 2 : 4; }

struct Checked {
  int B, T, Hk, Hv, W, Cc, num_slots;
  size_t in_elem;
};

gdn_status check_dims(const gdn_dims* d, const gdn_opts* o, bool decode, Checked* out) {
  if (!d || !o) return GDN_ERR_INVALID_ARGUMENT;
  if (d->batch < 0 || d->seqlen < 0 || d->num_k_heads < 1 || d->num_v_heads < 1 ||
      d->num_slots < 0 || d->conv_width < 0 || d->chunk_size < 0)
    return GDN_ERR_INVALID_ARGUMENT;
  if (d->num_v_heads % d->num_k_heads != 0) return GDN_ERR_INVALID_ARGUMENT;
  if (d->head_dim != gdn::kHeadDim) return GDN_ERR_UNSUPPORTED;
  if (d->chunk_size != 0 && d->chunk_size != gdn::kChunk) return GDN_ERR_UNSUPPORTED;
  if (d->conv_width > 4) return GDN_ERR_UNSUPPORTED;
  if ((o->in_dtype != GDN_F32 && o->in_dtype != GDN_BF16) ||
      (o->out_dtype != GDN_F32 && o->out_dtype != GDN_BF16))
    return GDN_ERR_INVALID_ARGUMENT;
  if (o->in_dtype == GDN_F32 && o->out_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
  if (!(o->l2_eps >= 0.0f) || !isfinite(o->l2_eps) || !isfinite(o->scale))
    return GDN_ERR_INVALID_ARGUMENT;
  if (decode) {
    if (d->seqlen != 1) return GDN_ERR_INVALID_ARGUMENT;
    if (d->num_v_heads / d->num_k_heads > 8) return GDN_ERR_UNSUPPORTED;
  }
  // grid limits: batch rides on gridDim.z / gridDim.x
  if (d->batch > 65535) return GDN_ERR_UNSUPPORTED;
  if ((long long)d->num_v_heads * d->head_dim > (1 << 20)) return GDN_ERR_UNSUPPORTED;
  out->B = d->batch;
  out->T = d->seqlen;
  out->Hk = d->num_k_heads;
  out->Hv = d->num_v_heads;
  out->W = d->conv_width;
  out->Cc = (2 * d->num_k_heads + d->num_v_heads) * d->head_dim;
  out->num_slots = d->num_slots ? d->num_slots : d->batch;
  out->in_elem = elem_bytes(o->in_dtype);
  return GDN_OK;
}

// Pointer checks shared by prefill and decode.  Fills the kernel argument block.
gdn_status check_layer_ptrs(const Checked& c, const gdn_opts* o, const void* q, const void* k,
                            const void* v, const void* a, const void* b, const float* A_log,
                            const float* dt_bias, const void* conv_weight,
                            const void* conv_bias, float* state, void* conv_state,
                            const int32_t* slots, void* out, GdnLayerArgs* L) {
  if (!q || !a || !b || !state || !out) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(state) || !aligned16(out)) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned4(a) || !aligned4(b)) return GDN_ERR_INVALID_ARGUMENT;
  if (!o->gates_precomputed && (!A_log || !aligned4(A_log))) return GDN_ERR_INVALID_ARGUMENT;
  if (dt_bias && !aligned4(dt_bias)) return GDN_ERR_INVALID_ARGUMENT;
  if (slots && !aligned4(slots)) return GDN_ERR_INVALID_ARGUMENT;
  if (!slots && c.num_slots < c.B) return GDN_ERR_INVALID_ARGUMENT;
  if (c.W > 0) {
    if (k || v) return GDN_ERR_INVALID_ARGUMENT;       // x arrives in q
    if (!conv_weight || !aligned4(conv_weight)) return GDN_ERR_INVALID_ARGUMENT;
    if (conv_bias && !aligned4(conv_bias)) return GDN_ERR_INVALID_ARGUMENT;
    if (c.W > 1 && (!conv_state || !aligned16(conv_state))) return GDN_ERR_INVALID_ARGUMENT;
  } else {
    if (!k || !v || !aligned16(k) || !aligned16(v)) return GDN_ERR_INVALID_ARGUMENT;
  }
  memset(L, 0, sizeof(*L));
  L->B = c.B; L->T = c.T; L->Hk = c.Hk; L->Hv = c.Hv; L->W = c.W; L->C_conv = c.Cc;
  L->num_slots = c.num_slots;
  L->in_bf16 = o->in_dtype == GDN_BF16;
  L->out_bf16 = o->out_dtype == GDN_BF16;
  L->l2norm = o->qk_l2norm != 0;
  L->silu = o->conv_silu != 0;
  L->gates_pre = o->gates_precomputed != 0;
  L->eps = o->l2_eps;
  L->scale = o->scale;
  L->a = a; L->b = b; L->A_log = A_log; L->dt_bias = dt_bias;
  L->conv_w = conv_weight; L->conv_b = conv_bias;
  L->state = state; L->conv_state = conv_state; L->slots = slots; L->out = out;
  if (c.W > 0) {
    L->x = q;
  } else {
    L->q = q; L->k = k; L->v = v;
    L->q_tok_stride = (long long)c.Hk * gdn::kHeadDim;
    L->k_tok_stride = (long long)c.Hk * gdn::kHeadDim;
    L->v_tok_stride = (long long)c.Hv * gdn::kHeadDim;
  }
  return GDN_OK;
}

// The tensor-core prefill with conv width 4 runs the conv of the q and k channels inside its
// chunk-local kernel (and that of the v channels as its first launch).
bool conv_fused(const Checked& c, const gdn_opts* o) { return o->in_dtype == GDN_BF16 && c.W == 4; }

size_t round_kb(size_t n) { return (n + 1023) & ~(size_t)1023; }
// the call's conv tail [B][W-1][C_conv], at offset 0 of a fused call's workspace, where a
// call that continues this one reads it
size_t tail_bytes_for(const Checked& c) {
  return round_kb((size_t)c.B * (size_t)(c.W - 1) * (size_t)c.Cc * c.in_elem);
}

// Workspace: [conv_width > 0, fused: the conv tail, then the post-conv v channels
// [B][T][Hv d] | conv_width > 0, not fused: the post-conv activations [B][T][C_conv]]
// [tensor-core prefill tiles, bf16].
size_t conv_bytes_for(const Checked& c, const gdn_opts* o) {
  if (c.W == 0) return 0;
  if (conv_fused(c, o))
    return tail_bytes_for(c) +
           round_kb((size_t)c.B * (size_t)c.T * (size_t)c.Hv * gdn::kHeadDim * c.in_elem);
  return round_kb((size_t)c.B * (size_t)c.T * (size_t)c.Cc * c.in_elem);
}

size_t workspace_bytes_for(const Checked& c, const gdn_opts* o) {
  size_t n = conv_bytes_for(c, o);
  if (o->in_dtype == GDN_BF16) n += gdn_prefill_tc_scratch_bytes(c.B, c.T, c.Hv);
  return n;
}

// Workspace of a packed variable-length call: [post-conv activations of the T tokens]
// [validated offsets, chunk offsets (N+1 int32 each), chunk table (U int4)][tensor-core
// tiles for a slice of U chunks], U = ceil(T / 64) + N bounding the chunk count.
struct VarlenLayout {
  size_t cu_ok, ccs, ctab, tc, total;
  int U;
};
VarlenLayout varlen_layout(const Checked& c, const gdn_opts* o) {
  auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  VarlenLayout v;
  v.U = (c.T + gdn::kChunk - 1) / gdn::kChunk + c.B;
  size_t off = 0;
  if (c.W > 0) off = ((size_t)c.T * c.Cc * c.in_elem + 1023) & ~(size_t)1023;
  v.cu_ok = off;
  off += up(sizeof(int32_t) * ((size_t)c.B + 1));
  v.ccs = off;
  off += up(sizeof(int32_t) * ((size_t)c.B + 1));
  v.ctab = off;
  off += up((size_t)16 * v.U);
  v.tc = off;
  if (o->in_dtype == GDN_BF16) off += gdn_prefill_tc_scratch_bytes(1, v.U * gdn::kChunk, c.Hv);
  v.total = off;
  return v;
}

// Copies a valid output gate into L (gate may be NULL: no norm).
gdn_status set_gate(const gdn_out_gate* gate, bool required, GdnLayerArgs* L) {
  if (!gate) return required ? GDN_ERR_INVALID_ARGUMENT : GDN_OK;
  if (!gate->z || !aligned16(gate->z) || !gate->weight || !aligned4(gate->weight) ||
      !(gate->eps >= 0.0f) || !(gate->eps < 3.0e38f))
    return GDN_ERR_INVALID_ARGUMENT;
  L->gate = 1;
  L->gate_z = gate->z;
  L->gate_w = gate->weight;
  L->gate_eps = gate->eps;
  return GDN_OK;
}

}  // namespace

extern "C" {

int32_t gdn_version(void) { return kVersion; }

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARGUMENT: return "GDN_ERR_INVALID_ARGUMENT";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT";
    case GDN_ERR_DEVICE_INDEX: return "GDN_ERR_DEVICE_INDEX";
  }
  return "GDN_UNKNOWN_STATUS";
}

size_t gdn_prefill_workspace_size(const gdn_dims* dims, const gdn_opts* opts) {
  Checked c;
  if (check_dims(dims, opts, false, &c) != GDN_OK) return 0;
  return workspace_bytes_for(c, opts);
}

// gdn_chunk_prefill, with in-call snapshots when snap_every > 0
static gdn_status prefill_impl(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                               const void* k, const void* v, const void* a, const void* b,
                               const float* A_log, const float* dt_bias,
                               const void* conv_weight, const void* conv_bias, float* state,
                               void* conv_state, const int32_t* state_slots, void* out,
                               int32_t snap_every, float* snap_state, void* snap_conv_state,
                               int32_t num_snap_slots, const int32_t* snap_slots,
                               const gdn_out_gate* gate, bool gated, const void* prev_ws,
                               void* workspace, size_t workspace_bytes, void* stream) {
  Checked c;
  gdn_status st = check_dims(dims, opts, false, &c);
  if (st != GDN_OK) return st;
  if (snap_every < 0 || snap_every % gdn::kChunk != 0) return GDN_ERR_INVALID_ARGUMENT;
  if (c.B == 0 || c.T == 0) return GDN_OK;
  GdnLayerArgs L;
  st = check_layer_ptrs(c, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                        conv_state, state_slots, out, &L);
  if (st != GDN_OK) return st;
  st = set_gate(gate, gated, &L);
  if (st != GDN_OK) return st;
  const int n_snap = snap_every > 0 ? c.T / snap_every : 0;
  if (n_snap > 0) {
    if (num_snap_slots <= 0 || !snap_state || !aligned16(snap_state) || !snap_slots ||
        !aligned4(snap_slots))
      return GDN_ERR_INVALID_ARGUMENT;
    if (c.W > 1 && (!snap_conv_state || !aligned16(snap_conv_state)))
      return GDN_ERR_INVALID_ARGUMENT;
    if ((long long)c.B * n_snap > 0x7fffffffLL) return GDN_ERR_INVALID_ARGUMENT;
    L.snap_every = snap_every;
    L.n_snap = n_snap;
    L.num_snap_slots = num_snap_slots;
    L.snap_state = snap_state;
    L.snap_slots = snap_slots;
    L.snap_conv_state = snap_conv_state;
  }
  const size_t need = workspace_bytes_for(c, opts);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return GDN_ERR_WORKSPACE;
  const bool fuse = conv_fused(c, opts);
  if (fuse && (!aligned16(conv_weight) || (conv_bias && !aligned16(conv_bias))))
    return GDN_ERR_INVALID_ARGUMENT;
  // a continuing call (the tensor-core path with the conv fused, or without a conv): the
  // previous call's workspace must not overlap this one's
  const bool chain = prev_ws && L.in_bf16 && (fuse || c.W == 0);
  if (chain) {
    const char* pw = static_cast<const char*>(prev_ws);
    const char* w0 = static_cast<const char*>(workspace);
    const size_t prev_bytes = fuse ? tail_bytes_for(c) : 1;
    if (!aligned16(prev_ws) || !(pw + prev_bytes <= w0 || pw >= w0 + need))
      return GDN_ERR_INVALID_ARGUMENT;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t conv_bytes = conv_bytes_for(c, opts);
  L.scratch = need > conv_bytes ? static_cast<char*>(workspace) + conv_bytes : nullptr;
  L.scratch_bytes = need - conv_bytes;
  L.chained = chain;
  if (fuse) {
    L.fuse = 1;
    L.tail = workspace;
    L.prev_tail = chain ? prev_ws : nullptr;
    L.v = static_cast<char*>(workspace) + tail_bytes_for(c);
    L.v_tok_stride = (long long)c.Hv * gdn::kHeadDim;
  } else if (c.W > 0) {
    // conv (+SiLU) into the workspace, conv state updated in place.  The tensor-core prefill
    // needs only the q / k channels before its chunk-local kernel: the value channels are
    // convolved by a second launch that runs beside that kernel (see vconv_pending).
    const int c_hi = L.in_bf16 ? 2 * c.Hk * gdn::kHeadDim : c.Cc;
    L.vconv_pending = c_hi < c.Cc;
    cudaError_t e = gdn_launch_conv(c.B, c.T, c.Cc, c.W, L.in_bf16, q, c.Cc, conv_weight,
                                    conv_bias, conv_state, c.num_slots, state_slots,
                                    L.silu, workspace, c.Cc, s, 0, c_hi);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    const char* y = static_cast<const char*>(workspace);
    L.q = y;
    L.k = y + (size_t)c.Hk * gdn::kHeadDim * c.in_elem;
    L.v = y + (size_t)2 * c.Hk * gdn::kHeadDim * c.in_elem;
    L.q_tok_stride = L.k_tok_stride = L.v_tok_stride = c.Cc;
  }
  cudaError_t e = L.in_bf16 ? gdn_launch_prefill_tc(L, s) : gdn_launch_prefill_simt(L, s);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  if (L.gate && !L.in_bf16) {
    // the FMA-pipe path (fp32 in and out) applies the norm as a pass of its own
    e = gdn_launch_gated_norm_f32(static_cast<float*>(out), static_cast<const float*>(L.gate_z),
                                  L.gate_w, L.gate_eps, c.B, (long long)c.T * c.Hv, state_slots,
                                  c.num_slots, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
  }
  if (n_snap > 0 && c.W > 1 && !L.fuse) {
    // the conv state at each boundary: W-1 rows of the call's pre-conv input (with the conv
    // fused, the state-chain kernels copy them)
    e = gdn_launch_conv_snapshots(c.B, c.T, c.Cc * c.in_elem, (long long)c.Cc * c.in_elem,
                                  c.W - 1, q, snap_every, n_snap, snap_conv_state,
                                  num_snap_slots, snap_slots, state_slots, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

gdn_status gdn_chunk_prefill(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                             const void* k, const void* v, const void* a, const void* b,
                             const float* A_log, const float* dt_bias, const void* conv_weight,
                             const void* conv_bias, float* state, void* conv_state,
                             const int32_t* state_slots, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return prefill_impl(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                      conv_state, state_slots, out, 0, nullptr, nullptr, 0, nullptr, nullptr,
                      false, nullptr, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_prefill_gated(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                   const void* k, const void* v, const void* a, const void* b,
                                   const float* A_log, const float* dt_bias,
                                   const void* conv_weight, const void* conv_bias, float* state,
                                   void* conv_state, const int32_t* state_slots, void* out,
                                   const gdn_out_gate* gate, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return prefill_impl(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                      conv_state, state_slots, out, 0, nullptr, nullptr, 0, nullptr, gate, true,
                      nullptr, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_prefill_ex(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                const void* k, const void* v, const void* a, const void* b,
                                const float* A_log, const float* dt_bias,
                                const void* conv_weight, const void* conv_bias, float* state,
                                void* conv_state, const int32_t* state_slots, void* out,
                                const gdn_prefill_ext* ext, void* workspace,
                                size_t workspace_bytes, void* stream) {
  static const gdn_prefill_ext none = {};
  const gdn_prefill_ext& e = ext ? *ext : none;
  return prefill_impl(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                      conv_state, state_slots, out, e.snap_every, e.snap_state,
                      e.snap_conv_state, e.num_snap_slots, e.snap_slots, e.gate, false,
                      e.prev_workspace, workspace, workspace_bytes, stream);
}

gdn_status gdn_chunk_prefill_snapshots(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                       const void* k, const void* v, const void* a,
                                       const void* b, const float* A_log, const float* dt_bias,
                                       const void* conv_weight, const void* conv_bias,
                                       float* state, void* conv_state,
                                       const int32_t* state_slots, void* out,
                                       int32_t snap_every, float* snap_state,
                                       void* snap_conv_state, int32_t num_snap_slots,
                                       const int32_t* snap_slots, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (snap_every <= 0) return GDN_ERR_INVALID_ARGUMENT;
  return prefill_impl(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                      conv_state, state_slots, out, snap_every, snap_state, snap_conv_state,
                      num_snap_slots, snap_slots, nullptr, false, nullptr, workspace,
                      workspace_bytes, stream);
}

size_t gdn_prefill_varlen_workspace_size(const gdn_dims* dims, const gdn_opts* opts) {
  Checked c;
  if (check_dims(dims, opts, false, &c) != GDN_OK) return 0;
  return varlen_layout(c, opts).total;
}

gdn_status gdn_chunk_prefill_varlen(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                    const void* k, const void* v, const void* a, const void* b,
                                    const float* A_log, const float* dt_bias,
                                    const void* conv_weight, const void* conv_bias,
                                    float* state, void* conv_state, const int32_t* state_slots,
                                    const int32_t* cu_seqlens, void* out,
                                    const gdn_out_gate* gate, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  Checked c;
  gdn_status st = check_dims(dims, opts, false, &c);
  if (st != GDN_OK) return st;
  if (!cu_seqlens || !aligned4(cu_seqlens)) return GDN_ERR_INVALID_ARGUMENT;
  if (c.B == 0 || c.T == 0) return GDN_OK;
  GdnLayerArgs L;
  st = check_layer_ptrs(c, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                        conv_state, state_slots, out, &L);
  if (st != GDN_OK) return st;
  st = set_gate(gate, false, &L);
  if (st != GDN_OK) return st;
  const VarlenLayout lay = varlen_layout(c, opts);
  if (!workspace || workspace_bytes < lay.total || !aligned16(workspace))
    return GDN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* cu_ok = reinterpret_cast<int32_t*>(ws + lay.cu_ok);
  int32_t* ccs = reinterpret_cast<int32_t*>(ws + lay.ccs);
  cudaError_t e = gdn_launch_varlen_prep(cu_seqlens, c.B, c.T, lay.U, cu_ok, ccs, ws + lay.ctab, s);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  if (c.W > 0) {
    // conv (+SiLU) of the packed tokens into the workspace, every sequence's conv state
    e = gdn_launch_conv_varlen(c.B, c.T, c.Cc, c.W, L.in_bf16, cu_ok, q, c.Cc, conv_weight,
                               conv_bias, conv_state, c.num_slots, state_slots, L.silu, ws,
                               c.Cc, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    L.q = ws;
    L.k = ws + (size_t)c.Hk * gdn::kHeadDim * c.in_elem;
    L.v = ws + (size_t)2 * c.Hk * gdn::kHeadDim * c.in_elem;
    L.q_tok_stride = L.k_tok_stride = L.v_tok_stride = c.Cc;
  }
  L.cu = cu_ok;
  L.ccs = ccs;
  L.ctab = ws + lay.ctab;
  L.n_chunks = lay.U;
  L.scratch = L.in_bf16 ? ws + lay.tc : nullptr;
  L.scratch_bytes = lay.total - lay.tc;
  e = L.in_bf16 ? gdn_launch_prefill_tc(L, s) : gdn_launch_prefill_simt(L, s);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  if (L.gate && !L.in_bf16) {
    e = gdn_launch_gated_norm_f32(static_cast<float*>(out), static_cast<const float*>(L.gate_z),
                                  L.gate_w, L.gate_eps, c.B, (long long)c.T * c.Hv, state_slots,
                                  c.num_slots, s, cu_ok, c.Hv);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
  }
  return GDN_OK;
}

gdn_status gdn_decode_multi(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                            const void* k, const void* v, const void* a, const void* b,
                            const float* A_log, const float* dt_bias, const void* conv_weight,
                            const void* conv_bias, float* state, void* conv_state,
                            const int32_t* state_slots, void* out, float* snap_state,
                            void* snap_conv_state, int32_t num_snap_slots,
                            const int32_t* snap_slots, void* stream) {
  Checked c;
  gdn_status st = check_dims(dims, opts, false, &c);
  if (st != GDN_OK) return st;
  if (c.T > 16) return GDN_ERR_UNSUPPORTED;
  if (c.B == 0 || c.T == 0) return GDN_OK;
  GdnLayerArgs L;
  st = check_layer_ptrs(c, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                        conv_state, state_slots, out, &L);
  if (st != GDN_OK) return st;
  if (snap_slots) {
    if (!aligned4(snap_slots) || num_snap_slots <= 0 || !snap_state || !aligned16(snap_state))
      return GDN_ERR_INVALID_ARGUMENT;
    if (c.W > 1 && (!snap_conv_state || !aligned16(snap_conv_state)))
      return GDN_ERR_INVALID_ARGUMENT;
  }
  cudaError_t e = gdn_launch_decode_multi(L, snap_slots ? snap_state : nullptr,
                                          snap_slots ? num_snap_slots : 0, snap_slots,
                                          (snap_slots && c.W > 1) ? snap_conv_state : nullptr,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// gdn_decode_step, with the output gate when `gated`
static gdn_status decode_impl(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                              const void* k, const void* v, const void* a, const void* b,
                              const float* A_log, const float* dt_bias, const void* conv_weight,
                              const void* conv_bias, float* state, void* conv_state,
                              const int32_t* state_slots, void* out, const gdn_out_gate* gate,
                              bool gated, void* stream) {
  Checked c;
  gdn_status st = check_dims(dims, opts, true, &c);
  if (st != GDN_OK) return st;
  if (c.B == 0) return GDN_OK;
  GdnLayerArgs L;
  st = check_layer_ptrs(c, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                        conv_state, state_slots, out, &L);
  if (st != GDN_OK) return st;
  st = set_gate(gate, gated, &L);
  if (st != GDN_OK) return st;
  cudaError_t e = gdn_launch_decode(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_decode_step(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                           const void* k, const void* v, const void* a, const void* b,
                           const float* A_log, const float* dt_bias, const void* conv_weight,
                           const void* conv_bias, float* state, void* conv_state,
                           const int32_t* state_slots, void* out, void* stream) {
  return decode_impl(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                     conv_state, state_slots, out, nullptr, false, stream);
}

gdn_status gdn_decode_step_gated(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                 const void* k, const void* v, const void* a, const void* b,
                                 const float* A_log, const float* dt_bias,
                                 const void* conv_weight, const void* conv_bias, float* state,
                                 void* conv_state, const int32_t* state_slots, void* out,
                                 const gdn_out_gate* gate, void* stream) {
  return decode_impl(dims, opts, q, k, v, a, b, A_log, dt_bias, conv_weight, conv_bias, state,
                     conv_state, state_slots, out, gate, true, stream);
}

gdn_status causal_conv1d_update(int32_t batch, int32_t seqlen, int32_t channels, int32_t width,
                                gdn_dtype dtype, const void* x, const void* weight,
                                const void* bias, void* conv_state, int32_t num_slots,
                                const int32_t* state_slots, int32_t silu, void* y,
                                void* stream) {
  if (batch < 0 || seqlen < 0 || channels < 0 || num_slots < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (width < 2 || width > 4) return GDN_ERR_UNSUPPORTED;
  if (channels % 8 != 0) return GDN_ERR_UNSUPPORTED;
  if (batch > 65535) return GDN_ERR_UNSUPPORTED;
  if (batch == 0 || seqlen == 0 || channels == 0) return GDN_OK;
  const int ns = num_slots ? num_slots : batch;
  if (!state_slots && ns < batch) return GDN_ERR_INVALID_ARGUMENT;
  if (!x || !weight || !conv_state || !y) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(y) || !aligned16(conv_state) || !aligned4(weight))
    return GDN_ERR_INVALID_ARGUMENT;
  if ((bias && !aligned4(bias)) || (state_slots && !aligned4(state_slots)))
    return GDN_ERR_INVALID_ARGUMENT;
  if (x == y) return GDN_ERR_INVALID_ARGUMENT;
  cudaError_t e = gdn_launch_conv(batch, seqlen, channels, width, dtype == GDN_BF16, x, channels,
                                  weight, bias, conv_state, ns, state_slots, silu != 0, y,
                                  channels, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_state_checkpoint(int32_t op, const gdn_dims* dims, gdn_dtype conv_dtype,
                                float* state, void* conv_state, float* slot_state,
                                void* slot_conv_state, int32_t num_bank_slots,
                                const int32_t* rows, const int32_t* slots, int32_t n,
                                void* stream) {
  if (op != 0 && op != 1) return GDN_ERR_INVALID_ARGUMENT;
  if (!dims || n < 0 || num_bank_slots < 0) return GDN_ERR_INVALID_ARGUMENT;
  if (dims->num_k_heads < 1 || dims->num_v_heads < 1 || dims->conv_width < 0 ||
      dims->num_slots < 0 || dims->batch < 0)
    return GDN_ERR_INVALID_ARGUMENT;
  if (dims->head_dim != gdn::kHeadDim) return GDN_ERR_UNSUPPORTED;
  if (dims->conv_width > 4) return GDN_ERR_UNSUPPORTED;
  if (conv_dtype != GDN_F32 && conv_dtype != GDN_BF16) return GDN_ERR_INVALID_ARGUMENT;
  if (n > 65535) return GDN_ERR_UNSUPPORTED;
  if (n == 0) return GDN_OK;
  const int num_rows = dims->num_slots ? dims->num_slots : dims->batch;
  if (!state || !slot_state || !rows || !slots) return GDN_ERR_INVALID_ARGUMENT;
  if (!aligned16(state) || !aligned16(slot_state) || !aligned4(rows) || !aligned4(slots))
    return GDN_ERR_INVALID_ARGUMENT;
  const int Cc = (2 * dims->num_k_heads + dims->num_v_heads) * dims->head_dim;
  const int conv_elems = dims->conv_width > 1 ? (dims->conv_width - 1) * Cc : 0;
  if (conv_elems > 0 && (!conv_state || !slot_conv_state || !aligned16(conv_state) ||
                         !aligned16(slot_conv_state)))
    return GDN_ERR_INVALID_ARGUMENT;
  cudaError_t e = gdn_launch_checkpoint(op, dims->num_v_heads, dims->head_dim, conv_elems,
                                        (int)elem_bytes(conv_dtype), state, conv_state,
                                        num_rows, slot_state, slot_conv_state, num_bank_slots,
                                        rows, slots, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_selftest_device_timeout(uint32_t max_iters, void* stream) {
  if (max_iters == 0 || max_iters > (1u << 20)) return GDN_ERR_INVALID_ARGUMENT;
  return gdn_launch_selftest_wait(max_iters, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

gdn_status gdn_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
  unsigned bits = gdn_take_error_decode() | gdn_take_error_conv() | gdn_take_error_checkpoint() |
                  gdn_take_error_prefill_simt() | gdn_take_error_prefill_tc() |
                  gdn_take_error_varlen() | gdn_take_error_decode_multi();
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  if (bits & gdn::kErrTimeout) return GDN_ERR_DEVICE_TIMEOUT;
  if (bits & gdn::kErrIndex) return GDN_ERR_DEVICE_INDEX;
  return GDN_OK;
}

}  // extern "C"
