/*
 * ORACLE -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load or run this code. It shares nothing with the CUDA path.
 *
 * A plain, slow CPU implementation of one eager decode step of a decoder-only
 * transformer trunk split into N contiguous layer stages:
 *
 *   - stage map: fence = [0, c1, .., cN-1, n_layers], stage s runs layers
 *     [fence[s], fence[s+1]) (memra_engine::pp module docs, "Door" and pp_cuts);
 *   - the f32 hidden state [n_embd] is the only tensor that crosses a stage
 *     boundary; each stage owns the KV cache of its layers; the position is a
 *     per-step scalar; the embedding lives with stage 0 and the final norm and
 *     LM head with the last stage (memra_engine::pp, "Ownership across a
 *     boundary");
 *   - the split changes scheduling, not math (memra_engine::pp, "M2 increment
 *     3"; ninfer pipeline-stages.md, "Verification": split output equals one
 *     device byte for byte), so the step itself is the plain decoder below.
 *
 * The pages take the decoder's formulas as known. Readings used here, where
 * they are silent: the standard forms of a decoder-only trunk (the pages name
 * RMSNorm, RoPE, GQA and SwiGLU without defining them) --
 *   RMSNorm  xn_i = h_i * g_i / sqrt(mean(h^2) + eps), eps = 1e-5
 *   RoPE     rotate-half pairs (i, i + hd/2), angle pos * theta^(-2i/hd)
 *   attention over cache rows [0, pos] (the current row included), scale
 *            1/sqrt(hd), max-subtracted softmax; q head h reads kv head
 *            h / (nq / nkv) ("TP3 support via zero-padded dummy heads",
 *            Implementation status item 2: GQA is part of the trained weights)
 *   MLP      a = silu(W_g xn) * (W_u xn), silu(z) = z / (1 + exp(-z))
 *   no biases, no q/k norm, untied LM head.
 *
 * Precision: the residual stream h is an f32 vector (the hidden state that
 * crosses a boundary is f32) and the KV cache stores bf16 (round to nearest,
 * ties to even), as the workloads fix; everything else -- normalised inputs,
 * q/k/v, scores, softmax, attention outputs, MLP activations, every dot
 * product -- is computed in fp64, summing in index order. Weights are read as
 * bf16, or as int8 with one fp32 scale per output row and dequantised as
 * (double)q * (double)s. Logits are returned as f32.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

typedef struct orc_desc {
  int n_layers, n_embd, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int weight_int8; /* 0: bf16 weights; 1: int8 weights, one fp32 scale per output row */
  int max_ctx, batch;
  double rope_theta, rms_eps;
} orc_desc;

/* A weight matrix [rows, cols], row-major: bf16 bit patterns, or int8 + row scales. */
typedef struct orc_mat {
  const void* w;
  const float* s;
  int rows, cols;
} orc_mat;

typedef struct orc_layer {
  const float* attn_norm;
  orc_mat wq, wk, wv, wo;
  const float* ffn_norm;
  orc_mat wg, wu, wd;
} orc_layer;

typedef struct orc_model {
  orc_desc d;
  int n_stages;
  int* fence;
  orc_layer* layers;
  orc_mat embed, head;
  const float* out_norm;
  uint16_t* kcache; /* [L][B][nkv][max_ctx][hd] bf16 bit patterns */
  uint16_t* vcache;
  int* filled;      /* [B]: cache rows [0, filled) hold valid entries */
  double* attn_out; /* [L][B][nq*hd]: attention outputs of the latest step (for invariants) */
  float* boundary;  /* [n_stages][n_embd]: the hidden state handed to each stage */
} orc_model;

/* ------------------------------------------------------------------------- */
/* number formats                                                            */
/* ------------------------------------------------------------------------- */

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even. */
uint16_t orc_bf16_round(double x) {
  double r = 0.0;
  if (x != 0.0 && isfinite(x)) {
    int e;
    double m = frexp(x, &e);                 /* x = m * 2^e, 0.5 <= |m| < 1 */
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8); /* keep 8 significant bits */
  } else {
    r = x;
  }
  float f = (float)r; /* exact: r has 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Element (r, k) of a weight matrix, dequantised to double. */
static double w_at(const orc_mat* m, int int8, long r, long k) {
  long i = r * (long)m->cols + k;
  if (int8) return (double)((const int8_t*)m->w)[i] * (double)m->s[r];
  return bf16_value(((const uint16_t*)m->w)[i]);
}

/* ------------------------------------------------------------------------- */
/* building blocks                                                           */
/* ------------------------------------------------------------------------- */

/* y[r] = sum_k W[r, k] x[k], k ascending. */
void orc_matvec(const orc_mat* m, int int8, const double* x, double* y) {
  long rows = m->rows, cols = m->cols;
#pragma omp parallel for schedule(static)
  for (long r = 0; r < rows; ++r) {
    double acc = 0.0;
    for (long k = 0; k < cols; ++k) acc += w_at(m, int8, r, k) * x[k];
    y[r] = acc;
  }
}

/* xn_i = h_i * g_i / sqrt(mean(h^2) + eps). */
void orc_rmsnorm(const float* h, const float* g, int n, double eps, double* xn) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += (double)h[i] * (double)h[i];
  double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) xn[i] = (double)h[i] * inv * (double)g[i];
}

/* Rotate one head vector x[hd] to position pos: pair (i, i + hd/2) turns by
 * pos * theta^(-2i/hd). */
void orc_rope(double* x, int hd, int pos, double theta) {
  int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    double ang = (double)pos * pow(theta, -2.0 * i / hd);
    double c = cos(ang), s = sin(ang);
    double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = a * s + b * c;
  }
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One head's attention over cache rows [0, pos]: o = softmax(q.K^T / sqrt(hd)) V,
 * K and V given as bf16 rows [max_ctx][hd]. */
void orc_attend_head(const double* q, const uint16_t* K, const uint16_t* V, int pos, int hd, double* o) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(pos + 1));
  double scale = 1.0 / sqrt((double)hd);
  double m = -INFINITY;
  for (int t = 0; t <= pos; ++t) {
    double acc = 0.0;
    for (int i = 0; i < hd; ++i) acc += q[i] * bf16_value(K[(long)t * hd + i]);
    s[t] = acc * scale;
    if (s[t] > m) m = s[t];
  }
  double l = 0.0;
  for (int t = 0; t <= pos; ++t) {
    s[t] = exp(s[t] - m);
    l += s[t];
  }
  for (int i = 0; i < hd; ++i) o[i] = 0.0;
  for (int t = 0; t <= pos; ++t)
    for (int i = 0; i < hd; ++i) o[i] += s[t] * bf16_value(V[(long)t * hd + i]);
  for (int i = 0; i < hd; ++i) o[i] /= l;
  free(s);
}

/* ------------------------------------------------------------------------- */
/* model                                                                     */
/* ------------------------------------------------------------------------- */

static size_t kv_index(const orc_desc* d, int l, int b, int g, int t) {
  return ((((size_t)l * d->batch + b) * d->n_kv_heads + g) * (size_t)d->max_ctx + t) * d->head_dim;
}

orc_model* orc_create(const orc_desc* d, const int* fence, int n_stages) {
  if (!d || !fence || n_stages < 1) return NULL;
  if (d->n_q_heads % d->n_kv_heads || d->head_dim % 2) return NULL;
  if (fence[0] != 0 || fence[n_stages] != d->n_layers) return NULL;
  for (int s = 0; s < n_stages; ++s)
    if (fence[s + 1] <= fence[s]) return NULL;
  orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
  if (!m) return NULL;
  m->d = *d;
  m->n_stages = n_stages;
  m->fence = (int*)malloc(sizeof(int) * (n_stages + 1));
  m->layers = (orc_layer*)calloc(d->n_layers, sizeof(orc_layer));
  size_t kv = (size_t)d->n_layers * d->batch * d->n_kv_heads * (size_t)d->max_ctx * d->head_dim;
  m->kcache = (uint16_t*)calloc(kv ? kv : 1, 2);
  m->vcache = (uint16_t*)calloc(kv ? kv : 1, 2);
  m->filled = (int*)calloc(d->batch, sizeof(int));
  m->attn_out = (double*)calloc((size_t)d->n_layers * d->batch * d->n_q_heads * d->head_dim, sizeof(double));
  m->boundary = (float*)calloc((size_t)n_stages * d->n_embd, sizeof(float));
  if (!m->fence || !m->layers || !m->kcache || !m->vcache || !m->filled || !m->attn_out || !m->boundary) {
    free(m->fence); free(m->layers); free(m->kcache); free(m->vcache); free(m->filled);
    free(m->attn_out); free(m->boundary); free(m);
    return NULL;
  }
  memcpy(m->fence, fence, sizeof(int) * (n_stages + 1));
  return m;
}

void orc_destroy(orc_model* m) {
  if (!m) return;
  free(m->fence); free(m->layers); free(m->kcache); free(m->vcache); free(m->filled);
  free(m->attn_out); free(m->boundary); free(m);
}

static orc_mat mat(const void* w, const float* s, int rows, int cols) {
  orc_mat x = {w, s, rows, cols};
  return x;
}

/* Weight pointers are borrowed (not copied); they must outlive the model. */
void orc_set_layer(orc_model* m, int l, const float* attn_norm, const void* wq, const float* wq_s,
                   const void* wk, const float* wk_s, const void* wv, const float* wv_s, const void* wo,
                   const float* wo_s, const float* ffn_norm, const void* wg, const float* wg_s,
                   const void* wu, const float* wu_s, const void* wd, const float* wd_s) {
  const orc_desc* d = &m->d;
  int qw = d->n_q_heads * d->head_dim, kw = d->n_kv_heads * d->head_dim;
  orc_layer* L = &m->layers[l];
  L->attn_norm = attn_norm;
  L->wq = mat(wq, wq_s, qw, d->n_embd);
  L->wk = mat(wk, wk_s, kw, d->n_embd);
  L->wv = mat(wv, wv_s, kw, d->n_embd);
  L->wo = mat(wo, wo_s, d->n_embd, qw);
  L->ffn_norm = ffn_norm;
  L->wg = mat(wg, wg_s, d->ffn, d->n_embd);
  L->wu = mat(wu, wu_s, d->ffn, d->n_embd);
  L->wd = mat(wd, wd_s, d->n_embd, d->ffn);
}

void orc_set_global(orc_model* m, const void* embed, const float* embed_s, const float* out_norm,
                    const void* head, const float* head_s) {
  m->embed = mat(embed, embed_s, m->d.vocab, m->d.n_embd);
  m->out_norm = out_norm;
  m->head = mat(head, head_s, m->d.vocab, m->d.n_embd);
}

/* One layer for sequence b at position pos; h (f32 [n_embd]) is updated in place. */
static void layer_step(orc_model* m, int l, int b, int pos, float* h) {
  const orc_desc* d = &m->d;
  const orc_layer* L = &m->layers[l];
  int E = d->n_embd, hd = d->head_dim, nq = d->n_q_heads, nkv = d->n_kv_heads, F = d->ffn;
  int int8 = d->weight_int8;
  double* xn = (double*)malloc(sizeof(double) * E);
  double* q = (double*)malloc(sizeof(double) * nq * hd);
  double* k = (double*)malloc(sizeof(double) * nkv * hd);
  double* v = (double*)malloc(sizeof(double) * nkv * hd);
  double* o = m->attn_out + ((size_t)l * d->batch + b) * nq * hd;
  double* y = (double*)malloc(sizeof(double) * E);
  double* g = (double*)malloc(sizeof(double) * F);
  double* u = (double*)malloc(sizeof(double) * F);

  /* attention block */
  orc_rmsnorm(h, L->attn_norm, E, d->rms_eps, xn);
  orc_matvec(&L->wq, int8, xn, q);
  orc_matvec(&L->wk, int8, xn, k);
  orc_matvec(&L->wv, int8, xn, v);
  for (int hh = 0; hh < nq; ++hh) orc_rope(q + (size_t)hh * hd, hd, pos, d->rope_theta);
  for (int kh = 0; kh < nkv; ++kh) orc_rope(k + (size_t)kh * hd, hd, pos, d->rope_theta);
  for (int kh = 0; kh < nkv; ++kh)
    for (int i = 0; i < hd; ++i) {
      m->kcache[kv_index(d, l, b, kh, pos) + i] = orc_bf16_round(k[(size_t)kh * hd + i]);
      m->vcache[kv_index(d, l, b, kh, pos) + i] = orc_bf16_round(v[(size_t)kh * hd + i]);
    }
  int group = nq / nkv;
#pragma omp parallel for schedule(static)
  for (int hh = 0; hh < nq; ++hh) {
    int kh = hh / group;
    orc_attend_head(q + (size_t)hh * hd, m->kcache + kv_index(d, l, b, kh, 0),
                    m->vcache + kv_index(d, l, b, kh, 0), pos, hd, o + (size_t)hh * hd);
  }
  orc_matvec(&L->wo, int8, o, y);
  for (int i = 0; i < E; ++i) h[i] = (float)((double)h[i] + y[i]);

  /* MLP block */
  orc_rmsnorm(h, L->ffn_norm, E, d->rms_eps, xn);
  orc_matvec(&L->wg, int8, xn, g);
  orc_matvec(&L->wu, int8, xn, u);
  for (int i = 0; i < F; ++i) g[i] = silu(g[i]) * u[i];
  orc_matvec(&L->wd, int8, g, y);
  for (int i = 0; i < E; ++i) h[i] = (float)((double)h[i] + y[i]);

  free(xn); free(q); free(k); free(v); free(y); free(g); free(u);
}

/* One decode step for every sequence: token tokens[b] at position pos[b]
 * (0 <= pos[b] <= filled[b] < max_ctx; rewinding is allowed, holes are not).
 * Writes logits [batch][vocab]. */
int orc_decode_step(orc_model* m, const int* tokens, const int* pos, float* logits) {
  const orc_desc* d = &m->d;
  int E = d->n_embd;
  for (int b = 0; b < d->batch; ++b) {
    if (tokens[b] < 0 || tokens[b] >= d->vocab) return ORC_EINVAL;
    if (pos[b] < 0 || pos[b] >= d->max_ctx || pos[b] > m->filled[b]) return ORC_EINVAL;
  }
  float* h = (float*)malloc(sizeof(float) * E);
  double* xn = (double*)malloc(sizeof(double) * E);
  double* z = (double*)malloc(sizeof(double) * d->vocab);
  for (int b = 0; b < d->batch; ++b) {
    /* stage 0 owns the embedding */
    for (int i = 0; i < E; ++i) h[i] = (float)w_at(&m->embed, d->weight_int8, tokens[b], i);
    for (int s = 0; s < m->n_stages; ++s) {
      /* the boundary: stage s receives the f32 hidden state and nothing else */
      float* hs = m->boundary + (size_t)s * E;
      memcpy(hs, h, sizeof(float) * E);
      for (int l = m->fence[s]; l < m->fence[s + 1]; ++l) layer_step(m, l, b, pos[b], hs);
      memcpy(h, hs, sizeof(float) * E);
    }
    /* the last stage owns the final norm and the LM head */
    orc_rmsnorm(h, m->out_norm, E, d->rms_eps, xn);
    orc_matvec(&m->head, d->weight_int8, xn, z);
    for (int v = 0; v < d->vocab; ++v) logits[(size_t)b * d->vocab + v] = (float)z[v];
    m->filled[b] = pos[b] + 1;
  }
  free(h); free(xn); free(z);
  return ORC_OK;
}

/* Cache rows of (layer, sequence): K and V as bf16 [nkv][max_ctx][hd]. */
int orc_kv_export(const orc_model* m, int l, int b, uint16_t* k, uint16_t* v) {
  const orc_desc* d = &m->d;
  if (l < 0 || l >= d->n_layers || b < 0 || b >= d->batch) return ORC_EINVAL;
  size_t n = (size_t)d->n_kv_heads * d->max_ctx * d->head_dim;
  memcpy(k, m->kcache + kv_index(d, l, b, 0, 0), n * 2);
  memcpy(v, m->vcache + kv_index(d, l, b, 0, 0), n * 2);
  return ORC_OK;
}

/* Replace the cache rows of (layer, sequence) and declare rows [0, filled) valid. */
int orc_kv_import(orc_model* m, int l, int b, const uint16_t* k, const uint16_t* v, int filled) {
  const orc_desc* d = &m->d;
  if (l < 0 || l >= d->n_layers || b < 0 || b >= d->batch || filled < 0 || filled > d->max_ctx)
    return ORC_EINVAL;
  size_t n = (size_t)d->n_kv_heads * d->max_ctx * d->head_dim;
  memcpy(m->kcache + kv_index(d, l, b, 0, 0), k, n * 2);
  memcpy(m->vcache + kv_index(d, l, b, 0, 0), v, n * 2);
  m->filled[b] = filled;
  return ORC_OK;
}

/* Attention outputs of the latest step: [nq*hd] doubles for (layer, sequence). */
int orc_attn_out(const orc_model* m, int l, int b, double* out) {
  const orc_desc* d = &m->d;
  if (l < 0 || l >= d->n_layers || b < 0 || b >= d->batch) return ORC_EINVAL;
  size_t n = (size_t)d->n_q_heads * d->head_dim;
  memcpy(out, m->attn_out + ((size_t)l * d->batch + b) * n, n * sizeof(double));
  return ORC_OK;
}

/* The hidden state the given stage received in the latest step (last sequence). */
int orc_boundary(const orc_model* m, int s, float* out) {
  if (s < 0 || s >= m->n_stages) return ORC_EINVAL;
  memcpy(out, m->boundary + (size_t)s * m->d.n_embd, sizeof(float) * m->d.n_embd);
  return ORC_OK;
}

void orc_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}

int orc_get_threads(void) { return omp_get_max_threads(); }
