/*
 * CPU oracle for GPT-2 single-token decode.  TEST INFRASTRUCTURE ONLY: only
 * tests, the smoke check and the benchmark's CPU-baseline / reference legs
 * use it.  It shares no code with the CUDA library.  See gpt2_oracle.h for
 * the sources and the precision rules (fp32, -ffp-contract=off).
 */
#include "gpt2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* The CPU baseline's multi-core build (-fopenmp) splits the outputs of each
 * matrix product between threads, as [P1] "Inner Workings" splits the rows of
 * each matrix product between its -j workers; each output is still computed
 * by one thread with the same operations in the same order, so both builds
 * give the same bits.  Without OpenMP the loops run on one thread. */
#ifdef _OPENMP
#include <omp.h>
#define ORC_PARALLEL _Pragma("omp parallel")
#define ORC_PARALLEL_FOR _Pragma("omp parallel for schedule(static)")
static void orc_share(int32_t n, int32_t *lo, int32_t *hi)
{
    const int64_t t = omp_get_thread_num(), nt = omp_get_num_threads();
    *lo = (int32_t)(n * t / nt);
    *hi = (int32_t)(n * (t + 1) / nt);
}
#else
#define ORC_PARALLEL
#define ORC_PARALLEL_FOR
static void orc_share(int32_t n, int32_t *lo, int32_t *hi)
{
    *lo = 0;
    *hi = n;
}
#endif

/* ======================================================================== */
/* Scalar math: [P2] "Step 5: Math without a math library".                */
/* ======================================================================== */

/* x = k*ln2 + r with k the nearest whole number to x/ln2, so |r| <= ln2/2
 * (< 0.35, as Step 5 states).  The reduction is done in double so that r is
 * the correctly rounded float of the exact remainder; the pages leave the
 * precision of this step open. */
void orc_expf_reduce(float x, int32_t *k, float *r)
{
    const double ln2 = 0.69314718055994530942;
    double kd = nearbyint((double)x / ln2);
    *k = (int32_t)kd;
    *r = (float)((double)x - kd * ln2);
}

/* e^x = 2^k * e^r, e^r from the degree-6 Taylor polynomial
 * 1 + r + r^2/2 + ... + r^6/720, and 2^k built by writing k+127 into the
 * exponent field of a float (Step 5, items 1-3).  Results below the smallest
 * normal float are flushed to 0; above FLT_MAX give +inf. */
float orc_expf(float x)
{
    if (x != x) return x;
    if (x > 88.72283935546875f) return INFINITY;
    if (x < -87.33654475f) return 0.0f;
    int32_t k;
    float r;
    orc_expf_reduce(x, &k, &r);
    float p = 1.0f / 720.0f;
    p = p * r + 1.0f / 120.0f;
    p = p * r + 1.0f / 24.0f;
    p = p * r + 1.0f / 6.0f;
    p = p * r + 0.5f;
    p = p * r + 1.0f;
    p = p * r + 1.0f;
    if (k > 127) { p = p * 2.0f; k -= 1; }   /* 2^128 is not a float */
    if (k < -126) return 0.0f;
    uint32_t bits = (uint32_t)(k + 127) << 23;
    float two_k;
    memcpy(&two_k, &bits, sizeof two_k);
    return p * two_k;
}

/* tanh(z) = 1 - 2 / (e^(2z) + 1)  (Step 5). */
float orc_tanhf(float z)
{
    return 1.0f - 2.0f / (orc_expf(2.0f * z) + 1.0f);
}

/* gelu_new(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 * The graph file writes the same function as
 * x * sigmoid(2 sqrt(2/pi) (x + 0.044715 x^3)) ([P3] comment above
 * g2.gelu_new); [P2] Step 5 evaluates it through tanh written with exp. */
float orc_gelu_new(float x)
{
    const float c = 0.7978845608028654f;     /* sqrt(2/pi) */
    float x3 = x * x * x;
    float u = c * (x + 0.044715f * x3);
    return 0.5f * x * (1.0f + orc_tanhf(u));
}

void orc_gelu_new_vec(const float *x, float *y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = orc_gelu_new(x[i]);
}

void orc_expf_vec(const float *x, float *y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = orc_expf(x[i]);
}

/* ======================================================================== */
/* Vector kernels.                                                          */
/* ======================================================================== */

/* LayerNorm over one row ([P3] kernel g2.layernorm): mean, then the biased
 * variance (both divided by n), then (x - mean) * (1/sqrt(var + eps)) * gamma
 * + beta; the square root is the IEEE one ([P2] Step 5: fsqrt). */
void orc_layernorm(const float *x, const float *gamma, const float *beta,
                   int32_t n, float eps, float *y)
{
    float sum = 0.0f;
    for (int32_t i = 0; i < n; ++i) sum += x[i];
    float mean = sum / (float)n;
    float ss = 0.0f;
    for (int32_t i = 0; i < n; ++i) {
        float d = x[i] - mean;
        ss += d * d;
    }
    float var = ss / (float)n;
    float rstd = 1.0f / sqrtf(var + eps);
    for (int32_t i = 0; i < n; ++i)
        y[i] = (x[i] - mean) * rstd * gamma[i] + beta[i];
}

/* Softmax with the maximum subtracted, then divided by the sum, so the
 * weights add up to 1 ([P2] "Step 6": step 2; [P3] g2.attn_decode). */
void orc_softmax(float *s, int32_t n)
{
    float m = s[0];
    for (int32_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    float sum = 0.0f;
    for (int32_t j = 0; j < n; ++j) {
        s[j] = orc_expf(s[j] - m);
        sum += s[j];
    }
    for (int32_t j = 0; j < n; ++j) s[j] = s[j] / sum;
}

/* HF Conv1D linear on the checkpoint's [input][output] layout ([P2] Step 1;
 * [P3] header): every output is one dot product over the inputs taken in
 * ascending order ([P2] Step 4), then the bias is added (the graph file's
 * separate *_bias g2.add node). */
void orc_linear(const float *x, const float *W, const float *b,
                int32_t in, int32_t out, float *y)
{
    ORC_PARALLEL
    {
        int32_t o0, o1;   /* this thread's outputs (all of them on one thread) */
        orc_share(out, &o0, &o1);
        for (int32_t o = o0; o < o1; ++o) y[o] = 0.0f;
        for (int32_t i = 0; i < in; ++i) {
            const float xi = x[i];
            const float *row = W + (size_t)i * (size_t)out;
            for (int32_t o = o0; o < o1; ++o) y[o] += xi * row[o];
        }
        if (b)
            for (int32_t o = o0; o < o1; ++o) y[o] = y[o] + b[o];
    }
}

/* Multiply by the transpose of a stored [out][in] matrix: the tied output
 * head reads wte [vocab][n_embd] this way ([P3] node head, fir.linear_t;
 * [P1] "Inner Workings": the head uses wte). */
void orc_linear_t(const float *x, const float *W, int32_t in, int32_t out,
                  float *y)
{
    ORC_PARALLEL_FOR
    for (int32_t o = 0; o < out; ++o) {
        const float *row = W + (size_t)o * (size_t)in;
        float acc = 0.0f;
        for (int32_t i = 0; i < in; ++i) acc += row[i] * x[i];
        y[o] = acc;
    }
}

/* Decode attention for one layer ([P3] kernel g2.attn_decode; [P2] Step 6):
 * write this token's k and v into the cache at pos, then for every head score
 * positions 0..pos with q.k * (1/sqrt(head_dim)), softmax, and sum the
 * values with those weights.  The cache is [head][position][head_dim]
 * ([P1] "Inner Workings": the KV cache is stored by head). */
void orc_attn_decode(const float *qkv, int32_t pos, int32_t n_head,
                     int32_t head_dim, int32_t n_positions,
                     float *k_cache, float *v_cache, float *out)
{
    const int32_t E = n_head * head_dim;
    const float scale = (float)(1.0 / sqrt((double)head_dim));
    float *s = (float *)malloc(sizeof(float) * (size_t)(pos + 1));
    for (int32_t h = 0; h < n_head; ++h) {
        const float *q = qkv + h * head_dim;
        const float *k = qkv + E + h * head_dim;
        const float *v = qkv + 2 * E + h * head_dim;
        float *kh = k_cache + (size_t)h * n_positions * head_dim;
        float *vh = v_cache + (size_t)h * n_positions * head_dim;
        memcpy(kh + (size_t)pos * head_dim, k, sizeof(float) * head_dim);
        memcpy(vh + (size_t)pos * head_dim, v, sizeof(float) * head_dim);
        for (int32_t j = 0; j <= pos; ++j) {
            float dot = 0.0f;
            for (int32_t d = 0; d < head_dim; ++d)
                dot += q[d] * kh[(size_t)j * head_dim + d];
            s[j] = dot * scale;
        }
        orc_softmax(s, pos + 1);
        for (int32_t d = 0; d < head_dim; ++d) {
            float acc = 0.0f;
            for (int32_t j = 0; j <= pos; ++j)
                acc += s[j] * vh[(size_t)j * head_dim + d];
            out[h * head_dim + d] = acc;
        }
    }
    free(s);
}

/* Greedy choice: the highest score ([P2] "Step 7"); among exact ties the
 * lowest index (the pages do not say; the scan keeps the first maximum). */
int32_t orc_argmax(const float *v, int32_t n)
{
    int32_t best = 0;
    for (int32_t i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* ======================================================================== */
/* Temperature sampling ([P2] "Step 7": divide the scores by a temperature, */
/* apply softmax and draw at random; [P1] Options: -t, 0 means greedy).    */
/* ======================================================================== */

/* Output k of a counter-based SplitMix64 generator (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014): the state
 * seed + (k + 1) * gamma, gamma = 0x9E3779B97F4A7C15, through the generator's
 * output mixer. */
uint64_t orc_splitmix64(uint64_t seed, uint64_t k)
{
    uint64_t z = seed + (k + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* A uniform float in the open interval (0, 1) from 64 random bits: the top
 * 23 bits m, as (m + 1/2) * 2^-23.  2m + 1 < 2^24, so m + 1/2 is exact in
 * fp32 and the largest value is 1 - 2^-24 < 1 (with 24 bits, m + 1/2 for
 * m = 2^24 - 1 rounds to 2^24 and the draw would be exactly 1). */
float orc_uniform_bits(uint64_t z)
{
    return ((float)(z >> 41) + 0.5f) * 1.1920928955078125e-7f;
}

/* Uniform number k of the generator with this seed. */
float orc_uniform(uint64_t seed, uint64_t k)
{
    return orc_uniform_bits(orc_splitmix64(seed, k));
}

/* The Gumbel-max form of a draw from softmax(s / T): score i is
 * s_i / T - log(-log u_i), u_i = uniform(seed, pos * n + i), in fp32 (the
 * logarithms correctly rounded from double); the draw is the highest score.
 * The pages draw one uniform number per token and walk the softmax
 * distribution; this is the same distribution, with one number per score. */
void orc_sample_scores(const float *s, int32_t n, float T, uint64_t seed, int32_t pos, float *out)
{
    for (int32_t i = 0; i < n; ++i) {
        const float u = orc_uniform(seed, (uint64_t)pos * (uint64_t)n + (uint64_t)i);
        const float e = (float)(-log((double)u));        /* -log u > 0 */
        const float g = -(float)log((double)e);          /* Gumbel noise */
        out[i] = s[i] / T + g;
    }
}

/* The token the pass at position `pos` chooses: greedy when T == 0, else the
 * draw above (exact ties to the lowest id, as for greedy). */
int32_t orc_sample(const float *s, int32_t n, float T, uint64_t seed, int32_t pos)
{
    if (!(T > 0.f)) return orc_argmax(s, n);
    float *v = (float *)malloc(sizeof(float) * (size_t)n);
    if (!v) return -1;
    orc_sample_scores(s, n, T, seed, pos, v);
    const int32_t id = orc_argmax(v, n);
    free(v);
    return id;
}

/* ======================================================================== */
/* The model: one token's forward pass ([P1] model.s description; [P3]     */
/* node list: token, positional, embeddings, repeat layers { ln1, qkv,     */
/* attention, out-projection, residual, ln2, fc, gelu, proj, residual },   */
/* final_norm, head).                                                       */
/* ======================================================================== */

struct orc_model {
    orc_config cfg;
    orc_weights w;
    float *k_cache, *v_cache;     /* [L][H][P][D] each */
    int32_t cached;               /* rows 0..cached-1 of the cache are valid */
    int32_t kv_bf16;              /* the cache holds k, v rounded to bf16 */
    uint16_t *kv16;               /* [2E] scratch for that rounding */
    float *x, *norm, *qkv, *attn, *mix, *fc, *act;
};

static int cfg_ok(const orc_config *c)
{
    if (!c) return 0;
    if (c->n_layer <= 0 || c->n_embd <= 0 || c->n_head <= 0) return 0;
    if (c->n_positions <= 0 || c->vocab_size <= 0) return 0;
    if (c->n_embd % c->n_head) return 0;   /* [P3] require hidden = nheads*headdim */
    return 1;
}

orc_model *orc_create(const orc_config *cfg, const orc_weights *w)
{
    if (!cfg_ok(cfg) || !w) return NULL;
    orc_model *m = (orc_model *)calloc(1, sizeof *m);
    if (!m) return NULL;
    m->cfg = *cfg;
    m->w = *w;
    const size_t E = (size_t)cfg->n_embd, F = 4 * E;   /* [P3] sym mlp = 4*hidden */
    const size_t kv = (size_t)cfg->n_layer * cfg->n_positions * E;
    m->k_cache = (float *)calloc(kv, sizeof(float));
    m->v_cache = (float *)calloc(kv, sizeof(float));
    m->x = (float *)calloc(E, sizeof(float));
    m->norm = (float *)calloc(E, sizeof(float));
    m->qkv = (float *)calloc(3 * E, sizeof(float));
    m->attn = (float *)calloc(E, sizeof(float));
    m->mix = (float *)calloc(E, sizeof(float));
    m->fc = (float *)calloc(F, sizeof(float));
    m->act = (float *)calloc(F, sizeof(float));
    m->kv16 = (uint16_t *)calloc(2 * E, sizeof(uint16_t));
    if (!m->k_cache || !m->v_cache || !m->x || !m->norm || !m->qkv ||
        !m->attn || !m->mix || !m->fc || !m->act || !m->kv16) {
        orc_destroy(m);
        return NULL;
    }
    return m;
}

void orc_destroy(orc_model *m)
{
    if (!m) return;
    free(m->k_cache); free(m->v_cache); free(m->x); free(m->norm);
    free(m->qkv); free(m->attn); free(m->mix); free(m->fc); free(m->act);
    free(m->kv16);
    free(m);
}

void orc_reset(orc_model *m)
{
    if (m) m->cached = 0;
}

/* The batched configuration's KV variant: every k and v row is rounded to
 * bf16 (round to nearest even) when it enters the cache, and attention reads
 * the cached values, this position's included.  q stays fp32. */
void orc_set_kv_bf16(orc_model *m, int32_t on)
{
    if (m) m->kv_bf16 = on ? 1 : 0;
}

/* Copies the cached K and V rows 0..n_rows-1 of one layer, [H][n_rows][D]
 * each (a copy of the cache the decode passes fill, for inspection). */
int32_t orc_export_kv(const orc_model *m, int32_t layer, int32_t n_rows, float *k, float *v)
{
    const orc_config *c = &m->cfg;
    const int32_t H = c->n_head, D = c->n_embd / H, P = c->n_positions;
    if (layer < 0 || layer >= c->n_layer || n_rows < 0 || n_rows > m->cached) return -1;
    for (int32_t h = 0; h < H; ++h) {
        const size_t src = ((size_t)layer * H + h) * P * D, dst = (size_t)h * n_rows * D;
        memcpy(k + dst, m->k_cache + src, sizeof(float) * (size_t)n_rows * D);
        memcpy(v + dst, m->v_cache + src, sizeof(float) * (size_t)n_rows * D);
    }
    return 0;
}

int32_t orc_forward(orc_model *m, int32_t token, int32_t pos, float *logits)
{
    const orc_config *c = &m->cfg;
    if (token < 0 || token >= c->vocab_size) return -1;
    if (pos < 0 || pos >= c->n_positions || pos > m->cached) return -1;
    m->cached = pos + 1;
    const int32_t E = c->n_embd, F = 4 * E, H = c->n_head, D = E / H;
    const int32_t P = c->n_positions;
    const float eps = c->ln_eps;

    /* token + positional embeddings, then g2.add */
    for (int32_t e = 0; e < E; ++e)
        m->x[e] = m->w.wte[(size_t)token * E + e] + m->w.wpe[(size_t)pos * E + e];

    for (int32_t l = 0; l < c->n_layer; ++l) {
        const orc_layer *L = &m->w.layers[l];
        float *kc = m->k_cache + (size_t)l * H * P * D;
        float *vc = m->v_cache + (size_t)l * H * P * D;
        orc_layernorm(m->x, L->ln1_w, L->ln1_b, E, eps, m->norm);
        orc_linear(m->norm, L->attn_w, L->attn_b, E, 3 * E, m->qkv);
        if (m->kv_bf16) {   /* k | v as the cache will hold them */
            orc_f32_to_bf16(m->qkv + E, m->kv16, 2 * (size_t)E);
            orc_bf16_to_f32(m->kv16, m->qkv + E, 2 * (size_t)E);
        }
        orc_attn_decode(m->qkv, pos, H, D, P, kc, vc, m->attn);
        orc_linear(m->attn, L->proj_w, L->proj_b, E, E, m->mix);
        for (int32_t e = 0; e < E; ++e) m->x[e] = m->x[e] + m->mix[e];
        orc_layernorm(m->x, L->ln2_w, L->ln2_b, E, eps, m->norm);
        orc_linear(m->norm, L->fc_w, L->fc_b, E, F, m->fc);
        for (int32_t f = 0; f < F; ++f) m->act[f] = orc_gelu_new(m->fc[f]);
        orc_linear(m->act, L->mlp_proj_w, L->mlp_proj_b, F, E, m->mix);
        for (int32_t e = 0; e < E; ++e) m->x[e] = m->x[e] + m->mix[e];
    }
    orc_layernorm(m->x, m->w.lnf_w, m->w.lnf_b, E, eps, m->norm);
    orc_linear_t(m->norm, m->w.head ? m->w.head : m->w.wte, E, c->vocab_size, logits);
    return orc_argmax(logits, c->vocab_size);
}

/* Whole-sequence evaluation with no cache: every layer runs over all n
 * positions at once, and position t attends to positions 0..t through an
 * explicit causal mask.  Used to pin the cached decode. */
int32_t orc_forward_full(const orc_config *c, const orc_weights *w,
                         const int32_t *tokens, int32_t n, float *logits_all)
{
    if (!cfg_ok(c) || !w || n <= 0 || n > c->n_positions) return -1;
    for (int32_t t = 0; t < n; ++t)
        if (tokens[t] < 0 || tokens[t] >= c->vocab_size) return -1;
    const int32_t E = c->n_embd, F = 4 * E, H = c->n_head, D = E / H;
    const float eps = c->ln_eps;
    const float scale = (float)(1.0 / sqrt((double)D));
    float *X = (float *)calloc((size_t)n * E, sizeof(float));
    float *N = (float *)calloc((size_t)n * E, sizeof(float));
    float *QKV = (float *)calloc((size_t)n * 3 * E, sizeof(float));
    float *O = (float *)calloc((size_t)n * E, sizeof(float));
    float *M = (float *)calloc((size_t)n * E, sizeof(float));
    float *Fh = (float *)calloc((size_t)n * F, sizeof(float));
    float *S = (float *)calloc((size_t)n, sizeof(float));
    if (!X || !N || !QKV || !O || !M || !Fh || !S) {
        free(X); free(N); free(QKV); free(O); free(M); free(Fh); free(S);
        return -1;
    }
    for (int32_t t = 0; t < n; ++t)
        for (int32_t e = 0; e < E; ++e)
            X[(size_t)t * E + e] = w->wte[(size_t)tokens[t] * E + e] +
                                   w->wpe[(size_t)t * E + e];
    for (int32_t l = 0; l < c->n_layer; ++l) {
        const orc_layer *L = &w->layers[l];
        for (int32_t t = 0; t < n; ++t) {
            orc_layernorm(X + (size_t)t * E, L->ln1_w, L->ln1_b, E, eps, N + (size_t)t * E);
            orc_linear(N + (size_t)t * E, L->attn_w, L->attn_b, E, 3 * E, QKV + (size_t)t * 3 * E);
        }
        for (int32_t t = 0; t < n; ++t) {
            for (int32_t h = 0; h < H; ++h) {
                const float *q = QKV + (size_t)t * 3 * E + h * D;
                for (int32_t j = 0; j < n; ++j) {
                    if (j > t) { S[j] = -INFINITY; continue; }   /* causal mask */
                    const float *k = QKV + (size_t)j * 3 * E + E + h * D;
                    float dot = 0.0f;
                    for (int32_t d = 0; d < D; ++d) dot += q[d] * k[d];
                    S[j] = dot * scale;
                }
                orc_softmax(S, t + 1);   /* masked entries lie past t */
                for (int32_t d = 0; d < D; ++d) {
                    float acc = 0.0f;
                    for (int32_t j = 0; j <= t; ++j)
                        acc += S[j] * QKV[(size_t)j * 3 * E + 2 * E + h * D + d];
                    O[(size_t)t * E + h * D + d] = acc;
                }
            }
        }
        for (int32_t t = 0; t < n; ++t) {
            float *x = X + (size_t)t * E;
            orc_linear(O + (size_t)t * E, L->proj_w, L->proj_b, E, E, M + (size_t)t * E);
            for (int32_t e = 0; e < E; ++e) x[e] = x[e] + M[(size_t)t * E + e];
            orc_layernorm(x, L->ln2_w, L->ln2_b, E, eps, N + (size_t)t * E);
            orc_linear(N + (size_t)t * E, L->fc_w, L->fc_b, E, F, Fh + (size_t)t * F);
            for (int32_t f = 0; f < F; ++f)
                Fh[(size_t)t * F + f] = orc_gelu_new(Fh[(size_t)t * F + f]);
            orc_linear(Fh + (size_t)t * F, L->mlp_proj_w, L->mlp_proj_b, F, E, M + (size_t)t * E);
            for (int32_t e = 0; e < E; ++e) x[e] = x[e] + M[(size_t)t * E + e];
        }
    }
    for (int32_t t = 0; t < n; ++t) {
        orc_layernorm(X + (size_t)t * E, w->lnf_w, w->lnf_b, E, eps, N + (size_t)t * E);
        orc_linear_t(N + (size_t)t * E, w->head ? w->head : w->wte, E, c->vocab_size,
                     logits_all + (size_t)t * c->vocab_size);
    }
    free(X); free(N); free(QKV); free(O); free(M); free(Fh); free(S);
    return 0;
}

/* ======================================================================== */
/* Stored-weight formats.                                                   */
/* ======================================================================== */

/* Round the integer m right by `shift` bits, to nearest, ties to even. */
static uint32_t shift_rne(uint32_t m, int shift)
{
    if (shift <= 0) return m;
    if (shift >= 32) return 0;
    uint32_t q = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return q;
}

/* fp32 -> IEEE binary16 by round-to-nearest-even on the bit fields: the fp16
 * mode of [P1] "Options" (-h) stores the block matrices this way; the pages
 * do not name the rounding, round-to-nearest-even is the IEEE default. */
static uint16_t f32_to_f16_1(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    int32_t exp = (int32_t)((x >> 23) & 0xFFu);
    uint32_t man = x & 0x7FFFFFu;
    if (exp == 0xFF) return (uint16_t)(sign | (man ? 0x7E00u : 0x7C00u));
    int32_t e = exp - 127 + 15;
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    if (e <= 0) {
        if (e < -10) return (uint16_t)sign;
        uint32_t mm = man | 0x800000u;
        return (uint16_t)(sign | shift_rne(mm, 14 - e));
    }
    uint32_t h = ((uint32_t)e << 10) | (man >> 13);
    uint32_t rem = man & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;  /* may carry into exp */
    return (uint16_t)(sign | h);
}

static float f16_to_f32_1(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t man = (uint32_t)h & 0x3FFu;
    uint32_t bits;
    if (exp == 0) {
        float v = (float)man * (1.0f / 16777216.0f);   /* man * 2^-24, exact */
        memcpy(&bits, &v, 4);
        bits |= sign;
    } else if (exp == 31) {
        bits = sign | 0x7F800000u | (man << 13);
    } else {
        bits = sign | ((exp - 15 + 127) << 23) | (man << 13);
    }
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

void orc_f32_to_f16(const float *in, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; ++i) out[i] = f32_to_f16_1(in[i]);
}

void orc_f16_to_f32(const uint16_t *in, float *out, size_t n)
{
    for (size_t i = 0; i < n; ++i) out[i] = f16_to_f32_1(in[i]);
}

void orc_f32_to_bf16(const float *in, uint16_t *out, size_t n)
{
    for (size_t i = 0; i < n; ++i) {
        uint32_t x;
        memcpy(&x, &in[i], 4);
        if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu)) {
            out[i] = (uint16_t)((x >> 16) | 0x40u);          /* quiet NaN */
            continue;
        }
        out[i] = (uint16_t)(shift_rne(x & 0x7FFFFFFFu, 16) | ((x >> 16) & 0x8000u));
    }
}

void orc_bf16_to_f32(const uint16_t *in, float *out, size_t n)
{
    for (size_t i = 0; i < n; ++i) {
        uint32_t x = (uint32_t)in[i] << 16;
        memcpy(&out[i], &x, 4);
    }
}

/* Grouped asymmetric int4 ([P3] header: transpose to [output,input], then
 * grouped asymmetric int4).  The pages give no more than that; this is the
 * plainest reading: per group of 32 inputs of one output row the range
 * [min(0, min w), max(0, max w)] is split into 15 steps, s = range / 15
 * (s = 1 if the range is empty), zero point z = rint(-min / s) clamped to
 * 0..15, code q = rint(w / s) + z clamped to 0..15, rint rounding half to
 * even; a weight is stored back as (q - z) * s. */
void orc_quant_int4(const float *W, int32_t in, int32_t out,
                    uint8_t *codes, float *scales, uint8_t *zeros)
{
    const int32_t G = in / 32;
    memset(codes, 0, (size_t)out * (size_t)(in / 2));
    memset(zeros, 0, (size_t)out * (size_t)(in / 64));
    for (int32_t o = 0; o < out; ++o) {
        for (int32_t g = 0; g < G; ++g) {
            float mn = 0.0f, mx = 0.0f;
            for (int32_t i = 32 * g; i < 32 * g + 32; ++i) {
                float v = W[(size_t)i * out + o];
                if (v < mn) mn = v;
                if (v > mx) mx = v;
            }
            float s = (mx - mn) / 15.0f;
            if (s == 0.0f) s = 1.0f;
            float zf = rintf(-mn / s);
            int32_t z = zf < 0.0f ? 0 : (zf > 15.0f ? 15 : (int32_t)zf);
            scales[(size_t)o * G + g] = s;
            zeros[(size_t)o * (in / 64) + g / 2] |= (uint8_t)(z << (4 * (g & 1)));
            for (int32_t i = 32 * g; i < 32 * g + 32; ++i) {
                float qf = rintf(W[(size_t)i * out + o] / s) + (float)z;
                int32_t q = qf < 0.0f ? 0 : (qf > 15.0f ? 15 : (int32_t)qf);
                codes[(size_t)o * (in / 2) + i / 2] |= (uint8_t)(q << (4 * (i & 1)));
            }
        }
    }
}

void orc_dequant_int4(const uint8_t *codes, const float *scales,
                      const uint8_t *zeros, int32_t in, int32_t out,
                      float *W_oi)
{
    const int32_t G = in / 32;
    for (int32_t o = 0; o < out; ++o) {
        for (int32_t i = 0; i < in; ++i) {
            int32_t g = i / 32;
            int32_t q = (codes[(size_t)o * (in / 2) + i / 2] >> (4 * (i & 1))) & 0xF;
            int32_t z = (zeros[(size_t)o * (in / 64) + g / 2] >> (4 * (g & 1))) & 0xF;
            W_oi[(size_t)o * in + i] = (float)(q - z) * scales[(size_t)o * G + g];
        }
    }
}

void orc_pack_nibbles(const uint8_t *vals, size_t n, uint8_t *packed)
{
    for (size_t k = 0; k < (n + 1) / 2; ++k) packed[k] = 0;
    for (size_t i = 0; i < n; ++i)
        packed[i / 2] |= (uint8_t)((vals[i] & 0xF) << (4 * (i & 1)));
}

void orc_unpack_nibbles(const uint8_t *packed, size_t n, uint8_t *vals)
{
    for (size_t i = 0; i < n; ++i)
        vals[i] = (uint8_t)((packed[i / 2] >> (4 * (i & 1))) & 0xF);
}
