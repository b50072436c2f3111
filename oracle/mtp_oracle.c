/*
 * CPU ORACLE — test infrastructure only.
 *
 * A plain, slow, obviously correct restatement of what one step of
 * multi-token-prediction (MTP) self-speculative decoding computes. Only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg may
 * load this library; the product path never does. It shares no source with
 * the CUDA path.
 *
 * Arithmetic: every dot product, norm, softmax and cumulative sum is formed in
 * double from the stored fp32/bf16 values, and rounded once to fp32 where the
 * method stores a tensor (hidden states, logits, probabilities, KV entries,
 * which are further rounded to bf16 when the cache is bf16). Decisions that
 * turn floating point into an integer (argmax, accept test, thresholds) are
 * taken on those fp32 values, as the kernels take them.
 *
 * Sources (page title, section):
 *  - "support the qwen3_5_mtp drafter" issue, section "Upstream contract to
 *    port": module shape (fc 2H->H, two pre-fc RMSNorms, one decoder layer,
 *    final norm), the forward concat order [norm_e(embed) ; norm_h(hidden)],
 *    borrowed tied lm_head, separate draft KV, block_size = depth + 2.
 *  - same page, section "Where the MTP weights actually live": the fifteen
 *    tensors, including self_attn.{q,k}_norm and mlp.{gate,up,down}_proj.
 *  - Ollama MLX-runner commit log, commit "unify the MTP decode paths":
 *    greedy is the temperature-0 point mass, verify is rejection sampling
 *    ("leviathan/chen sampling" in the DFlash commit).
 *  - same log, sampler commit: temperature, repetition penalty over a ring
 *    history, top-k, top-p, min-p.
 * Where the pages are silent the readings are stated beside the code.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Threads of the parallel loops below (the CPU baseline runs on all host
 * cores, then on one). No arithmetic depends on it: every reduction is a
 * sequential loop inside one thread. */
void orc_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
int orc_threads(void) { return omp_get_max_threads(); }

/* ---------------------------------------------------------------- storage */

static inline double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* fp32 -> bf16 bits, round to nearest even; a NaN stays a quiet NaN (the
   rounding add would carry an all-ones payload into the sign bit) */
static inline uint16_t float_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* the oracle's bf16 rounding over n values (the rounding the bf16 KV cache
   stores with), exposed so that it can be pinned */
void orc_bf16_round(const float* x, long n, uint16_t* out) {
  for (long i = 0; i < n; ++i) out[i] = float_to_bf16(x[i]);
}

/* element i of a weight/KV/hidden array stored as fp32 (dt=0) or bf16 (dt=1) */
static inline double get(const void* p, int dt, size_t i) {
  return dt ? bf16_to_double(((const uint16_t*)p)[i]) : (double)((const float*)p)[i];
}

/* store an fp32 value into an fp32 or bf16 array */
static inline void put(void* p, int dt, size_t i, float v) {
  if (dt) ((uint16_t*)p)[i] = float_to_bf16(v);
  else ((float*)p)[i] = v;
}

/* ------------------------------------------------------------------ model */

typedef struct {
  int H, nq, nkv, dh, I, V;
  double eps, theta;
  int wdt; /* 0 = fp32, 1 = bf16: weights and the draft KV cache */
  const void *E, *lm, *fc, *wq, *wk, *wv, *wo, *wg, *wu, *wd;
  /* the seven RMSNorm weights, already carrying the layout's +1.0 shift */
  const double *n_emb, *n_hid, *n_in, *n_post, *n_qn, *n_kn, *n_fin;
  /* optional fp8 draft head: e4m3 codes [V][H] and one scale per row; when
   * set, the logits use them instead of lm (the embedding gather keeps E) */
  const uint8_t* lmq;
  const float* lmq_scale;
} orc_model;

/* y[n] = sum_k W[n,k] x[k];  W row-major [N,K] (a Linear's weight). */
static void matvec(const void* W, int dt, int N, int K, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    size_t base = (size_t)n * (size_t)K;
    for (int k = 0; k < K; ++k) acc += get(W, dt, base + k) * x[k];
    y[n] = acc;
  }
}

/* ---------------------------------------------------------- fp8 e4m3
 * The 8-bit float with 1 sign bit, 4 exponent bits (bias 7) and 3 mantissa
 * bits, no infinities, the all-ones magnitude pattern NaN, largest finite 448.
 * A draft-only quantised copy of the tied output head ("Ollama qwen3_5 MTP
 * loader and SelfDraft path", Facts: the draft's tied output head quantized;
 * format unstated, read as e4m3 with one fp32 scale per row). */
float orc_e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, mant = c & 7;
  double v;
  if (e == 15 && mant == 7) return NAN;
  if (e == 0) v = ldexp((double)mant, -9);          /* subnormal: m/8 * 2^-6 */
  else v = ldexp(1.0 + mant / 8.0, e - 7);
  return (float)(s ? -v : v);
}

/* Round to nearest (ties to even), saturating finite values beyond 448 to
 * 448; NaN -> the NaN code. */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  const int s = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  uint8_t c;
  if (a < ldexp(1.0, -6)) {                 /* subnormal range: steps of 2^-9 */
    const double m = rint(a * 512.0);       /* m == 8 lands on the smallest normal */
    c = (uint8_t)(m >= 8.0 ? (1 << 3) : (int)m);
  } else {
    int e;
    frexp(a, &e);
    e -= 1;                                 /* 2^e <= a < 2^(e+1) */
    double m = rint((ldexp(a, -e) - 1.0) * 8.0);
    if (m >= 8.0) { m = 0.0; e += 1; }
    if (e > 8 || (e == 8 && m > 6.0)) { e = 8; m = 6.0; }   /* 448 */
    c = (uint8_t)(((e + 7) << 3) | (int)m);
  }
  return (uint8_t)((s << 7) | c);
}

/* Per-row quantisation, the decisions in fp32: scale = max|w| / 448 (1 for an
 * all-zero row), code = e4m3(w / scale). */
void orc_quantize_rows_e4m3(const float* w, int rows, int cols, uint8_t* q, float* scale) {
  for (int r = 0; r < rows; ++r) {
    const float* row = w + (size_t)r * cols;
    float amax = 0.0f;
    for (int k = 0; k < cols; ++k) amax = fabsf(row[k]) > amax ? fabsf(row[k]) : amax;
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    scale[r] = sc;
    for (int k = 0; k < cols; ++k) q[(size_t)r * cols + k] = orc_e4m3_encode(row[k] / sc);
  }
}

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * w.  The pages name nn.RMSNorm with
 * rms_norm_eps and give no formula; this is the standard one, eps inside the
 * square root. */
static void rmsnorm(const double* x, int n, const double* w, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * r * w[i];
}

/* Rotary embedding, rotate-half convention over the full head: pairs
 * (i, i + dh/2) turn by pos * theta^(-2i/dh).  Reading: the pages say only
 * that RoPE runs at the drafter's own absolute offset. */
static void rope(double* x, int dh, int pos, double theta) {
  int half = dh / 2;
  for (int i = 0; i < half; ++i) {
    double inv = pow(theta, -2.0 * (double)i / (double)dh);
    double a = (double)pos * inv;
    double c = cos(a), s = sin(a);
    double x0 = x[i], x1 = x[i + half];
    x[i] = x0 * c - x1 * s;
    x[i + half] = x1 * c + x0 * s;
  }
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/*
 * One drafter position (the MTP head forward for one (token, hidden) pair).
 *
 *   x   = [ RMSNorm_e(E[tok]) ; RMSNorm_h(hid) ]          (2H, embedding first)
 *   h0  = W_fc x
 *   b   = RMSNorm_in(h0);  q = W_q b, k = W_k b, v = W_v b
 *   per head: q_norm / k_norm over head_dim, then RoPE at position `slot`
 *   cache[slot] <- (k, v)   (rounded to the cache dtype)
 *   o_j = softmax_t(q_j . K_g[t] / sqrt(dh)) V_g[t],  t = 0..slot, g = j / (nq/nkv)
 *   h1  = h0 + W_o o
 *   h2  = h1 + W_d( silu(W_g c) * (W_u c) ),  c = RMSNorm_post(h1)
 *   logits = E_lm . RMSNorm_final(h2)
 *
 * Kc/Vc: this row's cache, [nkv][cap][dh] in the model's dtype.  Slots below
 * `slot` must already hold valid entries.  hid_dt: 0 fp32, 1 bf16.
 * mode 1 stops after the cache write (the K/V of a slot depend only on its own
 * pair).  h2_out / logits_out may be NULL.  Returns 0, or -1 on a bad slot.
 */
int orc_step(const orc_model* m, int tok, const void* hid, int hid_dt, void* Kc, void* Vc,
             int cap, int slot, int mode, float* h2_out, float* logits_out) {
  if (slot < 0 || slot >= cap || tok < 0 || tok >= m->V) return -1;
  const int H = m->H, dh = m->dh, nq = m->nq, nkv = m->nkv, I = m->I;
  const int qw = nq * dh, kw = nkv * dh;
  double* e = malloc(sizeof(double) * H);
  double* hh = malloc(sizeof(double) * H);
  double* x = malloc(sizeof(double) * 2 * H);
  double* h0 = malloc(sizeof(double) * H);
  double* b = malloc(sizeof(double) * H);
  double* q = malloc(sizeof(double) * qw);
  double* k = malloc(sizeof(double) * kw);
  double* v = malloc(sizeof(double) * kw);
  double* o = malloc(sizeof(double) * qw);
  double* h1 = malloc(sizeof(double) * H);
  double* c = malloc(sizeof(double) * H);
  double* g = malloc(sizeof(double) * I);
  double* u = malloc(sizeof(double) * I);
  double* h2 = malloc(sizeof(double) * H);
  double* tmp = malloc(sizeof(double) * (size_t)(H > dh ? H : dh));

  for (int i = 0; i < H; ++i) e[i] = get(m->E, m->wdt, (size_t)tok * H + i);
  for (int i = 0; i < H; ++i) hh[i] = get(hid, hid_dt, i);
  rmsnorm(e, H, m->n_emb, m->eps, x);
  rmsnorm(hh, H, m->n_hid, m->eps, x + H);
  matvec(m->fc, m->wdt, H, 2 * H, x, h0);

  rmsnorm(h0, H, m->n_in, m->eps, b);
  matvec(m->wq, m->wdt, qw, H, b, q);
  matvec(m->wk, m->wdt, kw, H, b, k);
  matvec(m->wv, m->wdt, kw, H, b, v);
  for (int j = 0; j < nq; ++j) {
    rmsnorm(q + j * dh, dh, m->n_qn, m->eps, tmp);
    rope(tmp, dh, slot, m->theta);
    memcpy(q + j * dh, tmp, sizeof(double) * dh);
  }
  for (int j = 0; j < nkv; ++j) {
    rmsnorm(k + j * dh, dh, m->n_kn, m->eps, tmp);
    rope(tmp, dh, slot, m->theta);
    memcpy(k + j * dh, tmp, sizeof(double) * dh);
  }
  for (int gk = 0; gk < nkv; ++gk)
    for (int i = 0; i < dh; ++i) {
      size_t off = ((size_t)gk * cap + slot) * dh + i;
      put(Kc, m->wdt, off, (float)k[gk * dh + i]);
      put(Vc, m->wdt, off, (float)v[gk * dh + i]);
    }
  int rc = 0;
  if (mode == 1) goto done;

  {
    const int group = nq / nkv;
    const double scale = 1.0 / sqrt((double)dh);
#pragma omp parallel for schedule(static)
    for (int j = 0; j < nq; ++j) {
      int gk = j / group;
      double* sc = malloc(sizeof(double) * (size_t)(slot + 1));
      double mx = -INFINITY;
      for (int t = 0; t <= slot; ++t) {
        double dot = 0.0;
        size_t off = ((size_t)gk * cap + t) * dh;
        for (int i = 0; i < dh; ++i) dot += q[j * dh + i] * get(Kc, m->wdt, off + i);
        sc[t] = dot * scale;
        if (sc[t] > mx) mx = sc[t];
      }
      double den = 0.0;
      for (int t = 0; t <= slot; ++t) { sc[t] = exp(sc[t] - mx); den += sc[t]; }
      for (int i = 0; i < dh; ++i) {
        double acc = 0.0;
        for (int t = 0; t <= slot; ++t) acc += sc[t] * get(Vc, m->wdt, ((size_t)gk * cap + t) * dh + i);
        o[j * dh + i] = acc / den;
      }
      free(sc);
    }
  }
  matvec(m->wo, m->wdt, H, qw, o, h1);
  for (int i = 0; i < H; ++i) h1[i] += h0[i];

  rmsnorm(h1, H, m->n_post, m->eps, c);
  matvec(m->wg, m->wdt, I, H, c, g);
  matvec(m->wu, m->wdt, I, H, c, u);
  for (int i = 0; i < I; ++i) g[i] = silu(g[i]) * u[i];
  matvec(m->wd, m->wdt, H, I, g, h2);
  for (int i = 0; i < H; ++i) h2[i] += h1[i];

  if (h2_out)
    for (int i = 0; i < H; ++i) h2_out[i] = (float)h2[i];
  if (logits_out) {
    /* the next step chains the fp32-stored hidden; the head reads it too */
    for (int i = 0; i < H; ++i) h2[i] = (double)(float)h2[i];
    rmsnorm(h2, H, m->n_fin, m->eps, c);
    double* lg = malloc(sizeof(double) * m->V);
    if (m->lmq) {
      /* logits[v] = scale[v] * sum_k e4m3(q[v,k]) * x[k] */
#pragma omp parallel for schedule(static)
      for (int n = 0; n < m->V; ++n) {
        double acc = 0.0;
        const uint8_t* row = m->lmq + (size_t)n * H;
        for (int k = 0; k < H; ++k) acc += (double)orc_e4m3_decode(row[k]) * c[k];
        lg[n] = (double)m->lmq_scale[n] * acc;
      }
    } else {
      matvec(m->lm, m->wdt, m->V, H, c, lg);
    }
    for (int i = 0; i < m->V; ++i) logits_out[i] = (float)lg[i];
    free(lg);
  }
done:
  free(e); free(hh); free(x); free(h0); free(b); free(q); free(k); free(v); free(o);
  free(h1); free(c); free(g); free(u); free(h2); free(tmp);
  return rc;
}

/* ------------------------------------------------------------- sampling */

typedef struct {
  float temperature, rep_penalty, top_p, min_p;
  int top_k, reserved;
} orc_params;

typedef struct {
  int argmax;        /* of the penalised logits, lowest id on ties */
  int kept;          /* support size of the final distribution */
  double top2_gap;   /* z[argmax] - next largest z (greedy near-tie measure) */
  double topp_margin;/* distance of the nearest cumulative mass to top_p*S, / S */
  double minp_margin;/* relative distance of the nearest exp(z-zmax) to min_p */
} orc_tinfo;

typedef struct { float z; int id; } zid;

static int cmp_zid(const void* a, const void* b) {
  const zid* x = a;
  const zid* y = b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

static int is_greedy(const orc_params* p) { return p->temperature <= 0.0f || p->top_k == 1; }

/*
 * The sampler's transform chain for one row of logits.  The commit log names
 * the transforms (temperature, repetition penalty over a ring history seeded
 * from the prompt, top-k, top-p, min-p) but prints no formulas; readings:
 *  1. repetition penalty r over the DISTINCT valid tokens of the window:
 *     z <- z / r if z > 0 else z * r;
 *  2. greedy (temperature 0, or top_k 1): point mass at argmax z, lowest id on
 *     ties -- the temperature-0 sampler "yields a point mass";
 *  3. z <- z / T;
 *  4. order tokens by (z desc, id asc); top-k keeps the first k;
 *  5. e = exp(z - zmax) over the kept tokens, S = sum e;
 *  6. top-p keeps the shortest prefix whose cumulative e reaches top_p * S;
 *  7. min-p keeps e >= min_p, i.e. p >= min_p * p_max;
 *  8. the kept set is the shortest of the three prefixes (at least one token),
 *     renormalised: probs = e / sum_kept e.  Steps 6 and 7 both read the
 *     step-5 softmax, so their order does not matter.
 * probs: [V] output, zero outside the kept set.
 */
int orc_transform(const float* logits, int V, const orc_params* p, const int* win, int nw,
                  float* probs, orc_tinfo* info) {
  float* z = malloc(sizeof(float) * V);
  memcpy(z, logits, sizeof(float) * V);
  if (p->rep_penalty != 1.0f) {
    char* seen = calloc((size_t)V, 1);
    for (int i = 0; i < nw; ++i) {
      int t = win[i];
      if (t < 0 || t >= V || seen[t]) continue;
      seen[t] = 1;
      z[t] = z[t] > 0.0f ? z[t] / p->rep_penalty : z[t] * p->rep_penalty;
    }
    free(seen);
  }
  int am = 0;
  for (int i = 1; i < V; ++i)
    if (z[i] > z[am]) am = i;
  double second = -INFINITY;
  for (int i = 0; i < V; ++i)
    if (i != am && (double)z[i] > second) second = z[i];
  info->argmax = am;
  info->top2_gap = (double)z[am] - second;
  info->topp_margin = INFINITY;
  info->minp_margin = INFINITY;
  for (int i = 0; i < V; ++i) probs[i] = 0.0f;
  if (is_greedy(p)) {
    probs[am] = 1.0f;
    info->kept = 1;
    free(z);
    return 0;
  }
  zid* s = malloc(sizeof(zid) * V);
  for (int i = 0; i < V; ++i) { s[i].z = z[i] / p->temperature; s[i].id = i; }
  qsort(s, V, sizeof(zid), cmp_zid);
  int K = (p->top_k > 0 && p->top_k < V) ? p->top_k : V;
  double* e = malloc(sizeof(double) * K);
  double S = 0.0;
  for (int j = 0; j < K; ++j) { e[j] = exp((double)s[j].z - (double)s[0].z); S += e[j]; }
  int Kp = K;
  if (p->top_p > 0.0f && p->top_p < 1.0f) {
    double thr = (double)p->top_p * S, cum = 0.0, prev = 0.0;
    for (int j = 0; j < K; ++j) {
      prev = cum;
      cum += e[j];
      if (cum >= thr) {
        Kp = j + 1;
        double d1 = fabs(cum - thr), d0 = j > 0 ? fabs(thr - prev) : INFINITY;
        info->topp_margin = (d1 < d0 ? d1 : d0) / S;
        break;
      }
    }
  }
  int Km = K;
  if (p->min_p > 0.0f) {
    Km = 0;
    while (Km < K && e[Km] >= (double)p->min_p) ++Km;
    if (Km < 1) Km = 1;
    double best = INFINITY;
    if (Km < K) best = fabs(e[Km] - p->min_p);
    if (Km > 1 && fabs(e[Km - 1] - p->min_p) < best) best = fabs(e[Km - 1] - p->min_p);
    info->minp_margin = best / p->min_p;
  }
  int Kf = K;
  if (Kp < Kf) Kf = Kp;
  if (Km < Kf) Kf = Km;
  if (Kf < 1) Kf = 1;
  double Sk = 0.0;
  for (int j = 0; j < Kf; ++j) Sk += e[j];
  for (int j = 0; j < Kf; ++j) probs[s[j].id] = (float)(e[j] / Sk);
  info->kept = Kf;
  free(e); free(s); free(z);
  return 0;
}

/*
 * Inverse-CDF draw from non-negative weights w[0..V-1] (not necessarily
 * normalised) with a pre-drawn u in [0,1): the smallest id whose cumulative
 * weight, in ascending id order, exceeds u * sum(w).  If rounding leaves no
 * such id, the last id with positive weight.  *margin: distance of the nearest
 * cumulative sum to the threshold, divided by the total.
 */
int orc_draw(const float* w, int V, float u, double* margin) {
  double S = 0.0;
  for (int i = 0; i < V; ++i) S += w[i];
  double thr = (double)u * S, cum = 0.0;
  int last = -1;
  for (int i = 0; i < V; ++i) {
    if (w[i] > 0.0f) last = i;
    double prev = cum;
    cum += w[i];
    if (w[i] > 0.0f && cum > thr) {
      if (margin) {
        double d1 = fabs(cum - thr), d0 = fabs(thr - prev);
        *margin = (d1 < d0 ? d1 : d0) / S;
      }
      return i;
    }
  }
  if (margin) *margin = 0.0;
  return last;
}

/*
 * Rejection-sampling verify of one row (Leviathan et al. / Chen et al.; the
 * commit log: at temperature 0 acceptance reduces to argmax-match, one path).
 *
 *   logits [d+1][V]: target rows; row i is the distribution after x_1..x_i
 *   drafts [d]:      x_1..x_d
 *   q      [d][V]:   the draft distributions x_i was drawn from (ignored for
 *                    greedy rows, whose q is the point mass at x_i)
 *   hist   [W]:      the penalty window through the last committed token,
 *                    oldest first, negative = empty
 *   u      [d+1]:    u[0..d-1] accept uniforms, u[d] the one draw uniform
 *
 * Row i uses the window "last W of hist ++ x_1..x_i" (reading: the drafts are
 * part of the sequence the target row conditions on).
 *   accept x_i  iff  q_i(x_i) > 0 and u[i-1] < p_{i-1}(x_i) / q_i(x_i)
 *   first reject at i: y ~ norm(max(p_{i-1} - q_i, 0)) (p_{i-1} if that is 0)
 *   all accepted:      y ~ p_d (the bonus token)
 * out_tok[0..n-1] = accepted drafts, out_tok[n] = y, rest -1.
 * margins[i-1]: accept-test margin |p/q - u| (greedy: top-2 gap of row i-1);
 * margins[d]: margin of the final draw (greedy: top-2 gap of the argmax row).
 */
int orc_verify_row(int V, int d, const float* logits, const int* drafts, const float* q,
                   const orc_params* p, const int* hist, int W, const float* u,
                   int* out_tok, int* n_acc, double* margins) {
  float* probs = malloc(sizeof(float) * (size_t)V * (d + 1));
  orc_tinfo* info = malloc(sizeof(orc_tinfo) * (d + 1));
  int* win = malloc(sizeof(int) * (size_t)(W + d + 1));
  for (int i = 0; i <= d; ++i) {
    int nw = 0;
    int drop = i < W ? i : W;
    for (int t = drop; t < W; ++t) win[nw++] = hist[t];
    int first = i > W ? i - W : 0;
    for (int t = first; t < i; ++t) win[nw++] = drafts[t];
    orc_transform(logits + (size_t)i * V, V, p, win, nw, probs + (size_t)i * V, &info[i]);
  }
  int greedy = is_greedy(p);
  int n = 0;
  for (int i = 1; i <= d; ++i) {
    int x = drafts[i - 1];
    int acc;
    if (greedy) {
      acc = (x == info[i - 1].argmax);
      margins[i - 1] = info[i - 1].top2_gap;
    } else {
      float pv = probs[(size_t)(i - 1) * V + x];
      float qv = q[(size_t)(i - 1) * V + x];
      float r = qv > 0.0f ? pv / qv : 0.0f;
      acc = qv > 0.0f && u[i - 1] < r;
      margins[i - 1] = fabs((double)r - (double)u[i - 1]);
    }
    if (!acc) break;
    n = i;
  }
  for (int i = n + 1; i < d; ++i) margins[i] = INFINITY;
  int y;
  if (greedy) {
    y = info[n].argmax;
    margins[d] = info[n].top2_gap;
  } else if (n < d) {
    float* res = malloc(sizeof(float) * V);
    const float* pn = probs + (size_t)n * V;
    const float* qn = q + (size_t)n * V;
    double tot = 0.0;
    for (int v = 0; v < V; ++v) {
      float r = pn[v] - qn[v];
      res[v] = r > 0.0f ? r : 0.0f;
      tot += res[v];
    }
    y = orc_draw(tot > 0.0 ? res : pn, V, u[d], &margins[d]);
    free(res);
  } else {
    y = orc_draw(probs + (size_t)d * V, V, u[d], &margins[d]);
  }
  for (int i = 0; i <= d; ++i) out_tok[i] = -1;
  for (int i = 0; i < n; ++i) out_tok[i] = drafts[i];
  out_tok[n] = y;
  *n_acc = n;
  free(probs); free(info); free(win);
  return 0;
}
