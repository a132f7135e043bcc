/*
 * gdn_oracle.c -- fp64 CPU oracle of the gated delta rule (Gated DeltaNet).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file:
 * only the tests, the smoke check and the bench's CPU-baseline leg do.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes, and where that is defined:
 *   - The recurrence itself, token by token, from the Hugging Face model card
 *     "Qwen3.5 Gated Delta Net NKI Kernel for AWS Neuron" (jburtoft/qwen35-deltanet-neuron-
 *     kernels), section "How It Works": decay the state by exp(g_t), read the memory with
 *     k_t, form delta = beta_t (v_t - read), write outer(k_t, delta), read out with q_t.
 *     The card stores state[k][v]; this file stores S = state^T, i.e. S[v][k], so the read
 *     is S k and the output S q.  Written out, that is
 *         S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
 *   - The gate, same card, section "Correctness Contract":
 *         g = -exp(A_log) * softplus(a + dt_bias)    (never positive)
 *     and beta = sigmoid(b) (the usual Gated DeltaNet write strength).
 *   - The short causal depthwise conv over the concatenated q|k|v channels with a carried
 *     conv state (same card, "How It Works", the surrounding "causal conv1d"; and its
 *     "Notice" on conv state + recurrent state caching for decode).
 *   - The chunked WY/UT form with a direct triangular solve of (I + A) (PR #164 follow-up
 *     "Fused DeltaNet Direct-Solve Follow-Up", sections "Why This Exists" and "Implementation
 *     Details"), used here only to check the algebra that the GPU prefill relies on.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - L2 normalisation x / sqrt(sum x^2 + eps), eps = 1e-6, q additionally times `scale`.
 *   - Conv: y_t[c] = bias[c] + sum_{j=0}^{W-1} w[c][j] * x_{t-W+1+j}[c]; tap W-1 is the
 *     current token; indices before the sequence start come from the conv state (the last
 *     W-1 pre-conv inputs, oldest first); optional SiLU after the conv.
 *   - softplus(x) = max(x,0) + log1p(exp(-|x|)) (the exact function, no threshold).
 *   - GQA: value head h reads key head h / (Hv/Hk) (contiguous groups).
 *   - The gated output norm (gdn_oracle_gated_rmsnorm): the card lists an "RMS norm" among
 *     the operations around the kernel and gives no formula.  Read as the gated RMS norm of
 *     these layers, per (token, value head) output vector o of length n:
 *         y_i = w_i * o_i / sqrt((1/n) sum_j o_j^2 + eps) * silu(z_i),  silu(z) = z / (1 + e^-z),
 *     with w the effective per-channel weight (a checkpoint that stores w - 1, the
 *     "RMSNorm +1 conversion" of PR #164 "Add Qwen3.6-27B contrib model with vLLM APC
 *     baseline", "Unit Coverage", is converted by the caller).
 *
 * Everything is IEEE double, no fast-math, straight loops in the order the definitions give.
 * Work units (batch row, value head) are independent and spread over pthreads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int batch, seqlen, num_k_heads, num_v_heads, dk, dv, conv_width;
  int qk_l2norm;          /* 1: L2-normalise q and k per head vector */
  double l2_eps;          /* eps inside the square root */
  double scale;           /* extra factor on q (after normalisation) */
  int conv_silu;          /* 1: SiLU after the conv */
  int gates_precomputed;  /* 1: a holds g, b holds beta */
  int erase;              /* 1: the delta rule; 0: erase term off (gated linear attention) */
} gdn_oracle_cfg;

/* ---------------------------------------------------------------- elementwise prologue */

double gdn_oracle_softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

double gdn_oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Gate of the model card's correctness contract: g = -exp(A_log) * softplus(a + dt_bias). */
double gdn_oracle_gate(double a, double A_log, double dt_bias) {
  return -exp(A_log) * gdn_oracle_softplus(a + dt_bias);
}

/* y = scale * x / sqrt(sum x^2 + eps) over one vector of length n. */
void gdn_oracle_l2norm(int n, const double* x, double eps, double scale, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = scale / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv;
}

/* ---------------------------------------------------------------- gated output norm */

/* rows vectors of length n: o, z, y [rows][n] (y may alias o), w [n].  The mean of squares,
 * its root with eps inside, the per-channel weight, then the SiLU gate of z, in that order. */
void gdn_oracle_gated_rmsnorm(int rows, int n, const double* o, const double* z,
                              const double* w, double eps, double* y) {
  for (int r = 0; r < rows; ++r) {
    const double* orow = o + (size_t)r * n;
    const double* zrow = z + (size_t)r * n;
    double ms = 0.0;
    for (int i = 0; i < n; ++i) ms += orow[i] * orow[i];
    ms /= (double)n;
    double inv = 1.0 / sqrt(ms + eps);
    for (int i = 0; i < n; ++i) {
      double gate = zrow[i] * gdn_oracle_sigmoid(zrow[i]);
      y[(size_t)r * n + i] = w[i] * (orow[i] * inv) * gate;
    }
  }
}

/* ---------------------------------------------------------------- causal depthwise conv */

/* Pre-conv input of channel c at token tau of one sequence: x for tau >= 0, the conv state
 * (W-1 entries, oldest first) for tau in [-(W-1), -1]. */
static double conv_input(int T, int C, int W, const double* x_b, const double* state_b,
                         int tau, int c) {
  (void)T;
  if (tau >= 0) return x_b[(size_t)tau * C + c];
  int idx = (W - 1) + tau;
  return state_b ? state_b[(size_t)idx * C + c] : 0.0;
}

static double conv_at(int T, int C, int W, const double* x_b, const double* w,
                      const double* bias, const double* state_b, int silu, int t, int c) {
  double y = bias ? bias[c] : 0.0;
  for (int j = 0; j < W; ++j)
    y += w[(size_t)c * W + j] * conv_input(T, C, W, x_b, state_b, t - (W - 1) + j, c);
  if (silu) y = y * gdn_oracle_sigmoid(y);
  return y;
}

/* Final conv state of one sequence: the last W-1 pre-conv inputs (oldest first). */
static void conv_state_after(int T, int C, int W, const double* x_b, const double* state_b,
                             double* out_b) {
  for (int i = 0; i < W - 1; ++i)
    for (int c = 0; c < C; ++c)
      out_b[(size_t)i * C + c] = conv_input(T, C, W, x_b, state_b, T - (W - 1) + i, c);
}

/* x, y: [B][T][C]; w: [C][W]; bias: [C] or NULL; state_in/state_out: [B][W-1][C]
 * (state_in NULL = zeros).  state_out may alias state_in. */
void gdn_oracle_conv1d(int B, int T, int C, int W, const double* x, const double* w,
                       const double* bias, const double* state_in, int silu, double* y,
                       double* state_out) {
  size_t sw = (size_t)(W > 1 ? W - 1 : 0) * C;
  double* tmp = state_out ? (double*)malloc(sizeof(double) * (sw ? sw : 1)) : NULL;
  for (int b = 0; b < B; ++b) {
    const double* x_b = x + (size_t)b * T * C;
    const double* s_b = state_in ? state_in + (size_t)b * sw : NULL;
    for (int t = 0; t < T; ++t)
      for (int c = 0; c < C; ++c)
        y[((size_t)b * T + t) * C + c] = conv_at(T, C, W, x_b, w, bias, s_b, silu, t, c);
    if (state_out && sw) {
      conv_state_after(T, C, W, x_b, s_b, tmp);
      memcpy(state_out + (size_t)b * sw, tmp, sizeof(double) * sw);
    }
  }
  free(tmp);
}

/* ---------------------------------------------------------------- the recurrence */

/* One token of the model card's "How It Works" loop, with S[v][k] = state^T:
 *   S <- exp(g) S ; kv = S k ; delta = beta (v - kv) ; S <- S + delta k^T ; o = S q.
 * With erase == 0 the read is skipped (delta = beta v): gated linear attention. */
static void recurrence_step(int dk, int dv, double* S, const double* q, const double* k,
                            const double* v, double g, double beta, int erase, double* o) {
  double decay = exp(g);
  for (int i = 0; i < dv; ++i) {
    double* s = S + (size_t)i * dk;
    for (int j = 0; j < dk; ++j) s[j] *= decay;                 /* 1. decay */
    double kv = 0.0;
    if (erase)
      for (int j = 0; j < dk; ++j) kv += s[j] * k[j];           /* 2. read */
    double delta = beta * (v[i] - kv);                          /* 3. update */
    for (int j = 0; j < dk; ++j) s[j] += delta * k[j];          /* 4. write */
    double acc = 0.0;
    for (int j = 0; j < dk; ++j) acc += s[j] * q[j];            /* 5. output */
    o[i] = acc;
  }
}

/* One (batch, head) unit over T tokens.  q, k: [T][dk] (already normalised / scaled),
 * v: [T][dv], g, beta: [T], S: [dv][dk] in/out, o: [T][dv]. */
void gdn_oracle_recurrence(int T, int dk, int dv, const double* q, const double* k,
                           const double* v, const double* g, const double* beta, int erase,
                           double* S, double* o) {
  for (int t = 0; t < T; ++t)
    recurrence_step(dk, dv, S, q + (size_t)t * dk, k + (size_t)t * dk, v + (size_t)t * dv,
                    g[t], beta[t], erase, o + (size_t)t * dv);
}

/* ---------------------------------------------------------------- chunked WY/UT form */

/* T = (I + A)^{-1} for strictly lower-triangular A [n][n] (upper part ignored), by plain
 * forward substitution row by row: row r of T is e_r - sum_{s<r} A[r][s] * (row s of T). */
void gdn_oracle_unit_lower_inverse(int n, const double* A, double* T) {
  for (int r = 0; r < n; ++r) {
    double* tr = T + (size_t)r * n;
    for (int c = 0; c < n; ++c) tr[c] = (r == c) ? 1.0 : 0.0;
    for (int s = 0; s < r; ++s) {
      double a = A[(size_t)r * n + s];
      const double* ts = T + (size_t)s * n;
      for (int c = 0; c <= s; ++c) tr[c] -= a * ts[c];
    }
  }
}

/* Chunked form of the same recurrence, chunk length C (last chunk may be shorter).
 * Within a chunk with entering state S0 and local cumulative log-decay G_r = sum_{s<=r} g_s:
 *   A[r][s] = beta_r exp(G_r - G_s) (k_r . k_s) for s < r         (0 with erase off)
 *   T       = (I + A)^{-1}                                       (direct solve)
 *   W       = T diag(beta exp(G)) K,   U' = T diag(beta) V
 *   U       = U' - W S0^T              (rows: per-token write vectors u_r)
 *   P[r][s] = exp(G_r - G_s) (q_r . k_s) for s <= r
 *   O       = diag(exp(G)) Q S0^T + P U
 *   S_end   = exp(G_last) S0 + U^T diag(exp(G_last - G)) K
 * Exponentials are only ever taken of G_r - G_s with r >= s (never positive). */
void gdn_oracle_chunked(int T, int dk, int dv, int C, const double* q, const double* k,
                        const double* v, const double* g, const double* beta, int erase,
                        double* S, double* o) {
  double* G = (double*)malloc(sizeof(double) * C);
  double* A = (double*)malloc(sizeof(double) * C * C);
  double* Tm = (double*)malloc(sizeof(double) * C * C);
  double* Wm = (double*)malloc(sizeof(double) * C * dk);
  double* U = (double*)malloc(sizeof(double) * C * dv);
  double* Up = (double*)malloc(sizeof(double) * C * dv);
  double* rhsK = (double*)malloc(sizeof(double) * C * dk);
  double* rhsV = (double*)malloc(sizeof(double) * C * dv);
  double* S0 = (double*)malloc(sizeof(double) * dv * dk);
  for (int t0 = 0; t0 < T; t0 += C) {
    int n = (T - t0 < C) ? (T - t0) : C;
    const double* Q = q + (size_t)t0 * dk;
    const double* K = k + (size_t)t0 * dk;
    const double* V = v + (size_t)t0 * dv;
    const double* gg = g + t0;
    const double* bb = beta + t0;
    memcpy(S0, S, sizeof(double) * dv * dk);
    double acc = 0.0;
    for (int r = 0; r < n; ++r) { acc += gg[r]; G[r] = acc; }
    /* A, then T by forward substitution */
    for (int r = 0; r < n; ++r)
      for (int s = 0; s < n; ++s) {
        double val = 0.0;
        if (erase && s < r) {
          double kk = 0.0;
          for (int j = 0; j < dk; ++j) kk += K[(size_t)r * dk + j] * K[(size_t)s * dk + j];
          val = bb[r] * exp(G[r] - G[s]) * kk;
        }
        A[(size_t)r * n + s] = val;
      }
    gdn_oracle_unit_lower_inverse(n, A, Tm);
    /* right-hand sides diag(beta exp(G)) K and diag(beta) V */
    for (int r = 0; r < n; ++r) {
      for (int j = 0; j < dk; ++j) rhsK[(size_t)r * dk + j] = bb[r] * exp(G[r]) * K[(size_t)r * dk + j];
      for (int i = 0; i < dv; ++i) rhsV[(size_t)r * dv + i] = bb[r] * V[(size_t)r * dv + i];
    }
    /* W = T rhsK, U' = T rhsV */
    for (int r = 0; r < n; ++r) {
      for (int j = 0; j < dk; ++j) {
        double s_ = 0.0;
        for (int s = 0; s < n; ++s) s_ += Tm[(size_t)r * n + s] * rhsK[(size_t)s * dk + j];
        Wm[(size_t)r * dk + j] = erase ? s_ : 0.0;
      }
      for (int i = 0; i < dv; ++i) {
        double s_ = 0.0;
        for (int s = 0; s < n; ++s) s_ += Tm[(size_t)r * n + s] * rhsV[(size_t)s * dv + i];
        Up[(size_t)r * dv + i] = s_;
      }
    }
    /* U = U' - W S0^T */
    for (int r = 0; r < n; ++r)
      for (int i = 0; i < dv; ++i) {
        double s_ = 0.0;
        for (int j = 0; j < dk; ++j) s_ += Wm[(size_t)r * dk + j] * S0[(size_t)i * dk + j];
        U[(size_t)r * dv + i] = Up[(size_t)r * dv + i] - s_;
      }
    /* O = diag(exp(G)) Q S0^T + P U */
    for (int r = 0; r < n; ++r)
      for (int i = 0; i < dv; ++i) {
        double inter = 0.0;
        for (int j = 0; j < dk; ++j) inter += Q[(size_t)r * dk + j] * S0[(size_t)i * dk + j];
        double intra = 0.0;
        for (int s = 0; s <= r; ++s) {
          double qk = 0.0;
          for (int j = 0; j < dk; ++j) qk += Q[(size_t)r * dk + j] * K[(size_t)s * dk + j];
          intra += exp(G[r] - G[s]) * qk * U[(size_t)s * dv + i];
        }
        o[(size_t)(t0 + r) * dv + i] = exp(G[r]) * inter + intra;
      }
    /* S_end = exp(G_last) S0 + U^T diag(exp(G_last - G)) K */
    double Gl = G[n - 1];
    for (int i = 0; i < dv; ++i)
      for (int j = 0; j < dk; ++j) {
        double s_ = exp(Gl) * S0[(size_t)i * dk + j];
        for (int r = 0; r < n; ++r)
          s_ += U[(size_t)r * dv + i] * exp(Gl - G[r]) * K[(size_t)r * dk + j];
        S[(size_t)i * dk + j] = s_;
      }
  }
  free(G); free(A); free(Tm); free(Wm); free(U); free(Up); free(rhsK); free(rhsV); free(S0);
}

/* ---------------------------------------------------------------- the whole layer */

typedef struct {
  const gdn_oracle_cfg* cfg;
  const double *q, *k, *v, *x, *a, *b, *A_log, *dt_bias, *conv_w, *conv_b, *conv_state_in;
  double *state, *out;
  int nthreads, tid;
} layer_job;

static void run_unit(const layer_job* J, int bidx, int h) {
  const gdn_oracle_cfg* c = J->cfg;
  int T = c->seqlen, Hk = c->num_k_heads, Hv = c->num_v_heads, dk = c->dk, dv = c->dv;
  int W = c->conv_width, r = Hv / Hk, kh = h / r;
  int Cc = 2 * Hk * dk + Hv * dv;
  double* qr = (double*)malloc(sizeof(double) * dk);
  double* kr = (double*)malloc(sizeof(double) * dk);
  double* vr = (double*)malloc(sizeof(double) * dv);
  double* qn = (double*)malloc(sizeof(double) * dk);
  double* kn = (double*)malloc(sizeof(double) * dk);
  double* S = J->state + ((size_t)bidx * Hv + h) * dv * dk;
  const double* x_b = W > 0 ? J->x + (size_t)bidx * T * Cc : NULL;
  const double* s_b = (W > 0 && J->conv_state_in) ? J->conv_state_in + (size_t)bidx * (W - 1) * Cc : NULL;
  for (int t = 0; t < T; ++t) {
    /* 1. raw q, k, v of this unit (conv + optional SiLU first when W > 0) */
    if (W > 0) {
      for (int j = 0; j < dk; ++j) {
        qr[j] = conv_at(T, Cc, W, x_b, J->conv_w, J->conv_b, s_b, c->conv_silu, t, kh * dk + j);
        kr[j] = conv_at(T, Cc, W, x_b, J->conv_w, J->conv_b, s_b, c->conv_silu, t, Hk * dk + kh * dk + j);
      }
      for (int i = 0; i < dv; ++i)
        vr[i] = conv_at(T, Cc, W, x_b, J->conv_w, J->conv_b, s_b, c->conv_silu, t, 2 * Hk * dk + h * dv + i);
    } else {
      size_t tk = ((size_t)bidx * T + t) * Hk + kh;
      memcpy(qr, J->q + tk * dk, sizeof(double) * dk);
      memcpy(kr, J->k + tk * dk, sizeof(double) * dk);
      memcpy(vr, J->v + (((size_t)bidx * T + t) * Hv + h) * dv, sizeof(double) * dv);
    }
    /* 2. normalise */
    if (c->qk_l2norm) {
      gdn_oracle_l2norm(dk, qr, c->l2_eps, c->scale, qn);
      gdn_oracle_l2norm(dk, kr, c->l2_eps, 1.0, kn);
    } else {
      for (int j = 0; j < dk; ++j) { qn[j] = qr[j] * c->scale; kn[j] = kr[j]; }
    }
    /* 3. gates */
    size_t ti = ((size_t)bidx * T + t) * Hv + h;
    double g, beta;
    if (c->gates_precomputed) {
      g = J->a[ti];
      beta = J->b[ti];
    } else {
      g = gdn_oracle_gate(J->a[ti], J->A_log[h], J->dt_bias ? J->dt_bias[h] : 0.0);
      beta = gdn_oracle_sigmoid(J->b[ti]);
    }
    /* 4. recurrence */
    recurrence_step(dk, dv, S, qn, kn, vr, g, beta, c->erase, J->out + ti * dv);
  }
  free(qr); free(kr); free(vr); free(qn); free(kn);
}

static void* layer_worker(void* arg) {
  const layer_job* J = (const layer_job*)arg;
  int units = J->cfg->batch * J->cfg->num_v_heads;
  for (int u = J->tid; u < units; u += J->nthreads)
    run_unit(J, u / J->cfg->num_v_heads, u % J->cfg->num_v_heads);
  return NULL;
}

/* Full layer: optional conv (+SiLU) over x [B][T][C_conv] (channels q | k | v, C_conv =
 * 2*Hk*dk + Hv*dv) or q [B][T][Hk][dk], k [B][T][Hk][dk], v [B][T][Hv][dv] directly; L2 norm;
 * gates from a, b [B][T][Hv]; the recurrence on state [B][Hv][dv][dk] (in/out); out
 * [B][T][Hv][dv]; conv_state [B][W-1][C_conv] (in/out, may be NULL for zeros in / no out).
 * Returns 0, or 1 on an invalid configuration. */
int gdn_oracle_layer(const gdn_oracle_cfg* cfg, const double* q, const double* k,
                     const double* v, const double* x, const double* a, const double* b,
                     const double* A_log, const double* dt_bias, const double* conv_w,
                     const double* conv_b, double* state, double* conv_state, double* out,
                     int nthreads) {
  if (!cfg || cfg->batch < 0 || cfg->seqlen < 0 || cfg->num_k_heads <= 0 ||
      cfg->num_v_heads <= 0 || cfg->num_v_heads % cfg->num_k_heads != 0 || cfg->dk <= 0 ||
      cfg->dv <= 0 || cfg->conv_width < 0)
    return 1;
  if (cfg->conv_width > 0 && (!x || !conv_w)) return 1;
  if (cfg->conv_width == 0 && (!q || !k || !v)) return 1;
  if (!cfg->gates_precomputed && !A_log) return 1;
  if (nthreads < 1) nthreads = 1;
  int Cc = 2 * cfg->num_k_heads * cfg->dk + cfg->num_v_heads * cfg->dv;
  int W = cfg->conv_width, T = cfg->seqlen;
  /* the conv state entering the call, kept aside: the units read it, the layer rewrites it */
  double* cs_in = NULL;
  if (W > 1 && conv_state) {
    size_t n = (size_t)cfg->batch * (W - 1) * Cc;
    cs_in = (double*)malloc(sizeof(double) * (n ? n : 1));
    memcpy(cs_in, conv_state, sizeof(double) * n);
  }
  layer_job* jobs = (layer_job*)calloc((size_t)nthreads, sizeof(layer_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int i = 0; i < nthreads; ++i) {
    layer_job J = {cfg, q, k, v, x, a, b, A_log, dt_bias, conv_w, conv_b, cs_in, state, out,
                   nthreads, i};
    jobs[i] = J;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, layer_worker, &jobs[i]);
  layer_worker(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
  if (W > 1 && conv_state)
    for (int bi = 0; bi < cfg->batch; ++bi)
      conv_state_after(T, Cc, W, x + (size_t)bi * T * Cc, cs_in + (size_t)bi * (W - 1) * Cc,
                       conv_state + (size_t)bi * (W - 1) * Cc);
  free(cs_in); free(jobs); free(th);
  return 0;
}
