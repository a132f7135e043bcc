/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule library, libgdn.so.
 *
 * The operation (Gated DeltaNet linear attention), per value head, token by token:
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t
 * with a 128 x 128 fp32 state S[v][k], L2-normalised q and k, and a short causal depthwise
 * conv in front.  Defined by the model card "Qwen3.5 Gated Delta Net NKI Kernel for AWS
 * Neuron", section "How It Works" (the five per-token steps: decay, read, delta, write,
 * output; the card stores state[k][v] = S^T) and section "Correctness Contract" (the gate
 * g = -exp(A_log) * softplus(a + dt_bias) <= 0, d_k = d_v = 128, each (batch, head)
 * independent).  The chunked prefill form with a direct triangular solve of (I + A) follows
 * PR #164 "Fused DeltaNet Direct-Solve Follow-Up" ("Why This Exists", "Implementation
 * Details"); decode with conv state + recurrent state caching follows the model card's
 * "Notice"; checkpoint slots with restore/commit masks follow PR #164 "Hybrid APC Runtime".
 *
 * Conventions shared by every entry point
 *   - Memory: every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     allocates nothing; the only global state is the device error word (see
 *     gdn_get_device_error).  Arrays are dense, row-major, in the layouts stated below.
 *     q/k/v (or x), state, conv state, out, y, workspace and the checkpoint bank must be
 *     16-byte aligned; a, b, A_log, dt_bias, conv weight / bias and the int32 index arrays
 *     4-byte aligned.
 *   - Validation: arguments are checked on the host before any CUDA call; a bad argument
 *     returns GDN_ERR_INVALID_ARGUMENT or GDN_ERR_UNSUPPORTED and launches nothing.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns immediately.  A failed launch returns GDN_ERR_CUDA.  Conditions
 *     found on the device (an out-of-range slot index, a bounded wait that gave up) are
 *     recorded in the error word and reported by gdn_get_device_error.
 *   - The library never aborts, exits, prints or traps.  Calls on different streams with
 *     disjoint buffers may run concurrently.
 *   - Slots: state arrays hold `num_slots` rows.  `state_slots[b]` (device int32, may be
 *     NULL = identity) names the row that batch entry b reads and updates in place; a
 *     negative entry skips batch entry b entirely (its outputs are left untouched), as for
 *     padded rows of a prefix-cache bucket.  An entry >= num_slots is skipped and recorded
 *     as GDN_ERR_DEVICE_INDEX.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARGUMENT = 1,  /* null / misaligned pointer, bad size, bad enum */
  GDN_ERR_UNSUPPORTED = 2,       /* valid but not implemented (head_dim != 128, ...) */
  GDN_ERR_WORKSPACE = 3,         /* workspace missing or smaller than required */
  GDN_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
  GDN_ERR_DEVICE_TIMEOUT = 5,    /* a bounded device-side wait gave up */
  GDN_ERR_DEVICE_INDEX = 6       /* a device-side slot/row index was out of range (skipped) */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Problem geometry. */
typedef struct {
  int32_t batch;        /* B >= 0: sequences in this call */
  int32_t seqlen;       /* T >= 0: tokens per sequence (gdn_decode_step: must be 1) */
  int32_t num_k_heads;  /* Hk >= 1 */
  int32_t num_v_heads;  /* Hv, a multiple of Hk with Hv / Hk <= 8; value head h reads key
                           head h / (Hv / Hk) */
  int32_t head_dim;     /* d = d_k = d_v; must be 128 */
  int32_t chunk_size;   /* prefill chunk length C; 0 or 64 (64 is the only one built) */
  int32_t conv_width;   /* W: 0 = q, k, v arrive post-conv; 2..4 = causal depthwise conv of
                           width W over the concatenated q|k|v channels first */
  int32_t num_slots;    /* rows of the state / conv-state arrays; 0 means `batch` */
} gdn_dims;

/* Numerical options. */
typedef struct {
  gdn_dtype in_dtype;         /* q/k/v (or x), a, b, conv weight / bias, conv state */
  gdn_dtype out_dtype;        /* out */
  int32_t qk_l2norm;          /* 1: q, k <- x / sqrt(sum x^2 + l2_eps) per head vector */
  float l2_eps;               /* epsilon inside the square root (1e-6 typical) */
  float scale;                /* factor applied to q after normalisation (1.0 typical) */
  int32_t conv_silu;          /* 1: SiLU after the conv (ignored when conv_width == 0) */
  int32_t gates_precomputed;  /* 0: a, b are raw gate inputs in in_dtype and
                                    g = -exp(A_log[h]) softplus(a + dt_bias[h]),
                                    beta = sigmoid(b);
                                 1: a holds g and b holds beta, both fp32 */
} gdn_opts;

/*
 * Precision modes.  in_dtype = GDN_BF16: bf16 operands on the tensor cores (tcgen05) with
 * fp32 accumulation and an fp32 state; out_dtype GDN_BF16 or GDN_F32.  in_dtype = GDN_F32
 * with out_dtype = GDN_F32 is the all-fp32 mode (fp32 FMA throughout).  Other combinations
 * return GDN_ERR_UNSUPPORTED.
 */

/*
 * Bytes of device workspace gdn_chunk_prefill needs for these dims/opts (0 when none): for
 * bf16 inputs with conv_width 4, the call's conv tail (its last W-1 pre-conv inputs,
 * [B][W-1][C_conv], at offset 0), else the post-conv activations when conv_width > 0; plus,
 * for bf16 inputs, the per-chunk operand tiles the tensor-core prefill passes from its
 * chunk-local kernel to its state-chain kernel (80 KB per chunk and value head, 96 KB when
 * the conv runs in the chunk-local kernel, for a slice of at most ~96 MB; twice that when the
 * call spans several slices, so that one slice's tiles are written while the previous
 * slice's are read).  Returns 0 for invalid dims.
 */
size_t gdn_prefill_workspace_size(const gdn_dims* dims, const gdn_opts* opts);

/*
 * gdn_chunk_prefill -- chunked context encoding of B sequences of T tokens.
 * Definition: the recurrence above, computed per chunk of C = 64 tokens in WY/UT form with a
 * direct (forward-substitution) solve of (I + A), A strictly lower triangular, carrying the
 * fp32 state across chunks (PR #164 "Fused DeltaNet Direct-Solve Follow-Up").  A last chunk
 * shorter than C is handled as a shorter chunk.  Results equal the token-by-token recurrence
 * up to rounding.
 *
 *   q, k, v      conv_width == 0: q [B,T,Hk,d], k [B,T,Hk,d], v [B,T,Hv,d] in in_dtype.
 *                conv_width  > 0: q points to the pre-conv activation x [B,T,C_conv] in
 *                in_dtype with channels ordered q | k | v, C_conv = (2 Hk + Hv) d; k and v
 *                must be NULL.
 *   a, b         [B,T,Hv] gate inputs (in_dtype), or g and beta (fp32) when
 *                gates_precomputed.
 *   A_log        [Hv] fp32 (ignored when gates_precomputed).
 *   dt_bias      [Hv] fp32 or NULL (= 0).
 *   conv_weight  [C_conv, W] in in_dtype (required when conv_width > 0, else ignored);
 *                16-byte aligned when in_dtype is bf16 and W = 4 (the conv then runs inside
 *                the chunk-local kernel, 16 bytes of taps at a time), else 4-byte aligned.
 *   conv_bias    [C_conv] in in_dtype or NULL (= 0); aligned as conv_weight.
 *   state        [num_slots, Hv, d, d] fp32, S[v][k]; read and written in place.
 *   conv_state   [num_slots, W-1, C_conv] in in_dtype: the last W-1 pre-conv inputs, oldest
 *                first; read and written in place (ignored when conv_width == 0).
 *   state_slots  [B] device int32 or NULL; see "Slots" above.
 *   out          [B,T,Hv,d] in out_dtype.
 *   workspace    device scratch of at least gdn_prefill_workspace_size() bytes (may be NULL
 *                when that is 0); contents are not preserved between calls.
 * T == 0 or B == 0 is a no-op returning GDN_OK.
 */
gdn_status gdn_chunk_prefill(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                             const void* k, const void* v, const void* a, const void* b,
                             const float* A_log, const float* dt_bias, const void* conv_weight,
                             const void* conv_bias, float* state, void* conv_state,
                             const int32_t* state_slots, void* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * gdn_decode_step -- one new token for each of B sequences (batched token generation).
 * Definition: one step of the recurrence (model card "How It Works") on the state already
 * resident in HBM, with the conv update, SiLU, L2 norm and gates fused, as in the model
 * card's "Notice" on conv-state + recurrent-state caching.  One kernel launch.
 * Arguments as gdn_chunk_prefill with T = 1 (dims->seqlen must be 1); no workspace.
 * Requires Hv / Hk <= 8.
 */
gdn_status gdn_decode_step(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                           const void* k, const void* v, const void* a, const void* b,
                           const float* A_log, const float* dt_bias, const void* conv_weight,
                           const void* conv_bias, float* state, void* conv_state,
                           const int32_t* state_slots, void* out, void* stream);

/*
 * causal_conv1d_update -- the short causal depthwise conv with a carried state, standalone
 * (model card "How It Works": the causal conv1d around the recurrence; "Notice": conv state
 * caching).  y[b,t,c] = bias[c] + sum_{j<W} w[c][j] * x[b, t-W+1+j, c], where positions
 * before the sequence start read conv_state[slot, W-1+(t-W+1+j), c]; then SiLU when `silu`.
 * conv_state[slot] becomes the last W-1 inputs (oldest first).
 *   x, y         [B,T,channels] in `dtype` (y may not alias x).
 *   weight       [channels, W]; bias [channels] or NULL.
 *   conv_state   [num_slots, W-1, channels] in place; state_slots as above (num_slots 0 = B).
 * 2 <= W <= 4.  channels must be a multiple of 8.
 */
gdn_status causal_conv1d_update(int32_t batch, int32_t seqlen, int32_t channels, int32_t width,
                                gdn_dtype dtype, const void* x, const void* weight,
                                const void* bias, void* conv_state, int32_t num_slots,
                                const int32_t* state_slots, int32_t silu, void* y,
                                void* stream);

/*
 * gdn_state_checkpoint -- copy recurrent + conv state between live rows and a slot bank
 * (PR #164 "Hybrid APC Runtime": checkpoint-slot lifecycle, restore and commit masks; the
 * reusable prefix of "Why this is larger than a normal contrib model").  A bit copy, so a
 * run resumed from a checkpoint continues exactly as the uninterrupted run.
 *   op           0 = SAVE (live row rows[i] -> bank slot slots[i]),
 *                1 = RESTORE (bank slot slots[i] -> live row rows[i]).
 *   dims         uses num_v_heads, head_dim, conv_width, num_k_heads, num_slots (live rows).
 *   state        [num_slots, Hv, d, d] fp32; conv_state [num_slots, W-1, C_conv] in conv_dtype
 *                (may be NULL when conv_width == 0).
 *   slot_state   [num_bank_slots, Hv, d, d] fp32; slot_conv_state [num_bank_slots, W-1,
 *                C_conv] (NULL when conv_width == 0).
 *   rows, slots  [n] device int32.  A negative entry in either masks pair i out (no copy);
 *                an entry past its array is skipped and recorded as GDN_ERR_DEVICE_INDEX.
 * Pairs must not write the same destination twice in one call.
 */
gdn_status gdn_state_checkpoint(int32_t op, const gdn_dims* dims, gdn_dtype conv_dtype,
                                float* state, void* conv_state, float* slot_state,
                                void* slot_conv_state, int32_t num_bank_slots,
                                const int32_t* rows, const int32_t* slots, int32_t n,
                                void* stream);

/*
 * Optional gated RMS norm fused into the output of gdn_chunk_prefill_gated and
 * gdn_decode_step_gated.  Definition: the model card (section "How It Works") lists an RMS norm
 * among the operations that run around the kernel, without a formula; this is the gated form
 * these layers use, per (token, value head) output vector o of length d:
 *     out_i = weight_i * o_i / sqrt(mean_j(o_j^2) + eps) * silu(z_i),  silu(z) = z sigmoid(z),
 * computed in fp32 and rounded once to out_dtype.  `weight` is the effective per-channel
 * factor: a checkpoint storing weight - 1 (the "RMSNorm +1 conversion" of PR #164 "Add
 * Qwen3.6-27B contrib model with vLLM APC baseline", "Unit Coverage") is converted by the
 * caller.
 */
typedef struct {
  const void* z;          /* [B, T, Hv, d] in in_dtype, 16-byte aligned: the output gate */
  const float* weight;    /* [d] fp32 */
  float eps;              /* >= 0, inside the square root (e.g. 1e-6) */
} gdn_out_gate;

/*
 * gdn_chunk_prefill_gated / gdn_decode_step_gated -- gdn_chunk_prefill / gdn_decode_step with
 * the gated RMS norm above applied to every output vector before it is stored (the plain
 * output is never written).  All other arguments, layouts, workspace and errors are those of
 * the plain calls.  `gate` must be non-NULL with non-NULL z and weight, z 16-byte aligned and
 * eps >= 0, else GDN_ERR_INVALID_ARGUMENT.  (For the decode step T = 1: z is [B, Hv, d].)
 */
gdn_status gdn_chunk_prefill_gated(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                   const void* k, const void* v, const void* a, const void* b,
                                   const float* A_log, const float* dt_bias,
                                   const void* conv_weight, const void* conv_bias, float* state,
                                   void* conv_state, const int32_t* state_slots, void* out,
                                   const gdn_out_gate* gate, void* workspace,
                                   size_t workspace_bytes, void* stream);
gdn_status gdn_decode_step_gated(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                 const void* k, const void* v, const void* a, const void* b,
                                 const float* A_log, const float* dt_bias,
                                 const void* conv_weight, const void* conv_bias, float* state,
                                 void* conv_state, const int32_t* state_slots, void* out,
                                 const gdn_out_gate* gate, void* stream);

/*
 * gdn_chunk_prefill_ex -- gdn_chunk_prefill with any of its optional parts, and the one call
 * form that can continue the previous call.  `ext` NULL (or zero-initialised) is the plain
 * call; each field adds one part:
 *   gate            non-NULL: the gated output norm, as gdn_chunk_prefill_gated.
 *   snap_every ...  snap_every > 0: in-call snapshots, as gdn_chunk_prefill_snapshots (same
 *                   fields, same errors); 0: none.
 *   prev_workspace  non-NULL: this call continues the sequences of the previous prefill call
 *                   enqueued on the same stream -- the next bucket of a long context prefilled
 *                   in fixed-size calls (the chunked form carries the state across calls
 *                   exactly; PR #164 "Fused DeltaNet Direct-Solve Follow-Up").  It is the
 *                   workspace that call used, whose first (W-1) * C_conv * B elements hold that
 *                   call's last W-1 pre-conv inputs per sequence (every call of the tensor-core
 *                   path with conv_width 4 leaves them there): the inputs before this call's
 *                   first token, read instead of conv_state.  16-byte aligned and not
 *                   overlapping `workspace` (else GDN_ERR_INVALID_ARGUMENT): alternate two
 *                   workspaces.  This call's first kernels may then start while the previous
 *                   call's state chain is still running (until it has finished they read only
 *                   this call's inputs and that conv tail); the results are those of the plain
 *                   call.  The caller guarantees that the previous call was a prefill of the
 *                   same sequences (same dims, state, conv_state and state_slots), that nothing
 *                   but gdn_state_checkpoint saves was enqueued on `stream` after it, and that
 *                   it wrote no input of this call.  The overlap applies to the tensor-core
 *                   path (in_dtype bf16) with conv_width 4 or 0; other calls ignore
 *                   prev_workspace and run as ordinary calls.
 * Errors: those of gdn_chunk_prefill and of the parts used.
 */
typedef struct {
  const gdn_out_gate* gate;
  int32_t snap_every;
  float* snap_state;
  void* snap_conv_state;
  int32_t num_snap_slots;
  const int32_t* snap_slots;
  const void* prev_workspace;
} gdn_prefill_ext;

gdn_status gdn_chunk_prefill_ex(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                const void* k, const void* v, const void* a, const void* b,
                                const float* A_log, const float* dt_bias,
                                const void* conv_weight, const void* conv_bias, float* state,
                                void* conv_state, const int32_t* state_slots, void* out,
                                const gdn_prefill_ext* ext, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_prefill_varlen -- gdn_chunk_prefill for a packed variable-length batch: N
 * sequences back to back on one token axis, sequence n on tokens [cu_seqlens[n],
 * cu_seqlens[n+1]).  Each sequence is its own recurrence (its own state and conv-state row,
 * its own chunk grid starting at its first token), so the results equal one
 * gdn_chunk_prefill call per sequence, bit for bit.  This is the packed-prefill half of the
 * mixed batches of PR #164 ("Hybrid APC Runtime": prefill and decode rows addressed through
 * state slots); a decode row is a sequence of length 1.
 *   dims         batch = N (>= 0), seqlen = T = the packed token count.
 *   q, k, v, x, a, b, out, gate->z   as gdn_chunk_prefill with B = 1: [1, T, ...].
 *   state_slots  [N] device int32 or NULL (identity, num_slots >= N): sequence n's row.
 *   cu_seqlens   [N+1] device int32: 0 = cu[0] <= cu[1] <= ... <= cu[N] = T.  Offsets that
 *                break this are reported as GDN_ERR_DEVICE_INDEX and nothing is computed
 *                (checked on the device: the host never reads them).  Empty sequences are
 *                allowed and leave their rows untouched.
 *   gate         NULL, or the gated output norm as for gdn_chunk_prefill_gated.
 *   workspace    at least gdn_prefill_varlen_workspace_size(dims, opts) bytes.
 */
size_t gdn_prefill_varlen_workspace_size(const gdn_dims* dims, const gdn_opts* opts);
gdn_status gdn_chunk_prefill_varlen(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                    const void* k, const void* v, const void* a, const void* b,
                                    const float* A_log, const float* dt_bias,
                                    const void* conv_weight, const void* conv_bias,
                                    float* state, void* conv_state, const int32_t* state_slots,
                                    const int32_t* cu_seqlens, void* out,
                                    const gdn_out_gate* gate, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * gdn_decode_multi -- a decode step over T = 1 .. 16 new tokens per sequence: speculative
 * multi-token verification and short prefills on the state already in HBM.  Definition: the
 * recurrence of gdn_chunk_prefill over the T tokens (the model card's "How It Works" loop);
 * computed as one T-token chunk of the WY/UT form per (sequence, value head), streaming every
 * state row once.  The model card's performance tables ("Performance") cover this 2-16 token
 * regime; PR #164 lists native multi-token (MTP) speculative decoding as a follow-up ("Known
 * limitations and follow-ups").
 *   all arguments but the ones below: as gdn_chunk_prefill with seqlen = T <= 16 (T > 16
 *                returns GDN_ERR_UNSUPPORTED; use gdn_chunk_prefill).
 *   snap_slots   [B, T] device int32 or NULL: the bank row that receives the state (and conv
 *                state) after token t of sequence b; negative = not recorded; >= num_snap_slots
 *                is skipped and recorded as GDN_ERR_DEVICE_INDEX.  With it, a verifier that
 *                accepts the first a tokens restores row snap_slots[b, a-1].
 *   snap_state   [num_snap_slots, Hv, d, d] fp32 (required with snap_slots).
 *   snap_conv_state  [num_snap_slots, W-1, C_conv] in in_dtype (required with snap_slots when
 *                conv_width > 1).
 */
gdn_status gdn_decode_multi(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                            const void* k, const void* v, const void* a, const void* b,
                            const float* A_log, const float* dt_bias, const void* conv_weight,
                            const void* conv_bias, float* state, void* conv_state,
                            const int32_t* state_slots, void* out, float* snap_state,
                            void* snap_conv_state, int32_t num_snap_slots,
                            const int32_t* snap_slots, void* stream);

/*
 * gdn_chunk_prefill_snapshots -- gdn_chunk_prefill over a whole prompt in one call that also
 * records the recurrent and conv state every `snap_every` tokens, in-kernel.
 * Definition: the prefix checkpoints of hybrid automatic prefix caching (PR #164 "Hybrid APC
 * Runtime": the state at fixed token boundaries is kept in checkpoint slots so that a later
 * request sharing the prefix resumes from it).  Snapshot j of row b (j = 0 .. n_snap-1,
 * n_snap = T / snap_every rounded down) is the state after token (j + 1) * snap_every of this
 * call: exactly what gdn_state_checkpoint(SAVE) would copy after gdn_chunk_prefill calls
 * over tokens [0, (j + 1) * snap_every) in buckets of snap_every tokens, bit for bit (the
 * chunk grid starts at the call start, so chunk boundaries and results are the same).
 *   all arguments but the ones below: as gdn_chunk_prefill, with the same workspace size
 *                (gdn_prefill_workspace_size); the live state and conv state end as after
 *                gdn_chunk_prefill.
 *   snap_every       tokens between snapshots: a positive multiple of the chunk (64), else
 *                    GDN_ERR_INVALID_ARGUMENT.
 *   snap_state       [num_snap_slots, Hv, d, d] fp32 bank, the layout of `state`.
 *   snap_conv_state  [num_snap_slots, W-1, C_conv] in in_dtype, the layout of `conv_state`
 *                    (the W-1 pre-conv inputs ending at the boundary, oldest first); ignored
 *                    (may be NULL) when conv_width <= 1.
 *   num_snap_slots   rows of the banks.
 *   snap_slots       [B, n_snap] device int32: the bank row receiving snapshot j of row b; a
 *                    negative entry records nothing; an entry >= num_snap_slots records
 *                    nothing and sets GDN_ERR_DEVICE_INDEX.  Rows that state_slots skips
 *                    record nothing.  No two entries may name the same bank row.
 * The banks are written only at the recorded rows.  With n_snap == 0 (T < snap_every) this
 * is gdn_chunk_prefill and the snapshot pointers are not read.
 */
gdn_status gdn_chunk_prefill_snapshots(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                       const void* k, const void* v, const void* a,
                                       const void* b, const float* A_log, const float* dt_bias,
                                       const void* conv_weight, const void* conv_bias,
                                       float* state, void* conv_state,
                                       const int32_t* state_slots, void* out,
                                       int32_t snap_every, float* snap_state,
                                       void* snap_conv_state, int32_t num_snap_slots,
                                       const int32_t* snap_slots, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_prefill_noalloc -- gdn_chunk_prefill for callers that cannot allocate device
 * memory.  The pages have no counterpart of this call; it is a convenience of this library.
 *
 * The prefill needs scratch memory (post-conv activations, the tensor-core path's chunk
 * tiles), which gdn_chunk_prefill takes from a caller-provided workspace.  Some callers
 * cannot provide one: code recorded into a CUDA graph that must not call cudaMalloc, plug-ins
 * that a host framework hands only input and output pointers, services whose allocator
 * forbids allocations after start-up.  This variant takes the same arguments minus the
 * workspace and uses a file-scope device array of GDN_NOALLOC_SCRATCH_BYTES bytes instead;
 * every GPU that loads the library holds that array until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: if gdn_prefill_workspace_size() of the call exceeds GDN_NOALLOC_SCRATCH_BYTES
 *     (64 MiB: e.g. one 512-token call of the 27B shape, 16/48 heads with the conv), it
 *     returns GDN_ERR_WORKSPACE and launches nothing.
 *   - Set-up: the first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream capture.
 *   - Device reset: the cached address belongs to the device context of that first call.
 *     cudaDeviceReset (or anything else that destroys the device's primary context) makes it
 *     stale, and the library is not told: after such a reset do not call this entry point on
 *     that device again in the same process.
 *   - Sharing: all calls share the one array and it keeps the last call's contents (nothing
 *     in it has to start at zero: each call writes every byte it reads).  Calls that overlap
 *     on the GPU (different streams, concurrent graph replays) race on it: serialise them.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_chunk_prefill_noalloc(const gdn_dims* dims, const gdn_opts* opts, const void* q,
                                     const void* k, const void* v, const void* a, const void* b,
                                     const float* A_log, const float* dt_bias,
                                     const void* conv_weight, const void* conv_bias,
                                     float* state, void* conv_state,
                                     const int32_t* state_slots, void* out, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device error word: GDN_OK, or the
 * first condition recorded by a kernel since the last call (GDN_ERR_DEVICE_INDEX,
 * GDN_ERR_DEVICE_TIMEOUT), or GDN_ERR_CUDA if the synchronisation itself failed.
 */
gdn_status gdn_get_device_error(void* stream);

/*
 * gdn_selftest_device_timeout -- exercises the failure-detection path of the kernels without
 * faulting or hanging anything.  The pages have no counterpart of this call.  Every wait of
 * the library's copy / tensor-core pipelines is bounded: when a copy or MMA never completes,
 * the CTA gives up, records the condition in the device error word and returns, and the next
 * gdn_get_device_error reports GDN_ERR_DEVICE_TIMEOUT.  This call enqueues one CTA on `stream`
 * that waits on an mbarrier that nothing ever arrives at (no copy, MMA or TMEM in flight),
 * with the given poll limit, through the same bounded wait and the same error word as the
 * prefill kernels.
 *   max_iters: polls before giving up, 1 .. 2^20 (each poll may suspend for a short,
 *     hardware-chosen time; 2^10 ends in well under a millisecond).
 * Returns GDN_OK once enqueued (the timeout is then reported by the next
 * gdn_get_device_error), GDN_ERR_INVALID_ARGUMENT for a limit out of range, GDN_ERR_CUDA if the
 * launch failed.
 */
gdn_status gdn_selftest_device_timeout(uint32_t max_iters, void* stream);

/* Static text for a status code (never NULL). */
const char* gdn_status_string(gdn_status status);

/* Library ABI version (major * 100 + minor). */
int32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
