/*
 * CPU oracle for GPT-2 single-token decode.  TEST INFRASTRUCTURE ONLY.
 *
 * This is a plain, slow, obviously-correct C implementation of what the
 * decode hot path computes.  It exists so that tests, the smoke check and the
 * benchmark's CPU-baseline leg can check the CUDA library against it.  The
 * product library never links, loads or calls anything here, and nothing here
 * includes or calls the product library.
 *
 * Sources (web pages on the subject; cited by page title and section):
 *   [P1] "gpt2.s" README, sections "Options", "Inner Workings", "Limitations".
 *   [P2] "Let's make GPT-2 in assembly", sections "Step 1: weights" .. "Step 7".
 *   [P3] "model.fir" (Resident GPT-2 decode graph file): the header comments,
 *        the config checks, the kernels g2.add, g2.gelu_new, g2.layernorm,
 *        g2.attn_decode and the per-token node list.
 *
 * Precision: fp32 storage and fp32 arithmetic, as the pages fix it ([P1]
 * "Benchmarks": one thread, fp32; [P2] "Does it work?": both sides use 32-bit
 * floats).  Build with -ffp-contract=off and without -ffast-math so that every
 * multiply and add rounds separately and the results are identical on x86-64
 * and AArch64.
 *
 * Parity status of each function is stated beside it; every function here is
 * pinned by tests under tests/test_oracle_*.py (see the pin named beside it).
 */
#ifndef GPT2_ORACLE_H
#define GPT2_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t n_layer;      /* number of transformer blocks                  */
    int32_t n_embd;       /* hidden size E                                 */
    int32_t n_head;       /* heads H; head dim D = E / H                   */
    int32_t n_positions;  /* context length P (KV cache rows)              */
    int32_t vocab_size;   /* V                                             */
    float   ln_eps;       /* LayerNorm epsilon                             */
} orc_config;

/* One block's tensors, in the checkpoint's (HF Conv1D) layout:
 * every matrix is [input][output] row-major. */
typedef struct {
    const float *ln1_w, *ln1_b;          /* [E]                 */
    const float *attn_w, *attn_b;        /* [E][3E], [3E]       */
    const float *proj_w, *proj_b;        /* [E][E],  [E]        */
    const float *ln2_w, *ln2_b;          /* [E]                 */
    const float *fc_w, *fc_b;            /* [E][4E], [4E]       */
    const float *mlp_proj_w, *mlp_proj_b;/* [4E][E], [E]        */
} orc_layer;

typedef struct {
    const float *wte;      /* [V][E]  token embedding, also the tied head */
    const float *wpe;      /* [P][E]  position embedding                  */
    const float *lnf_w, *lnf_b;          /* [E]                            */
    const orc_layer *layers;             /* n_layer entries                */
    const float *head;     /* [V][E] the output head as stored, or NULL: the
                              tied wte ("gpt2.s" README, Options: -h stores the
                              output head in fp16; its values widened here) */
} orc_weights;

/* ---- scalar math ([P2] "Step 5: Math without a math library") ---------- */
float orc_expf(float x);
float orc_tanhf(float z);
float orc_gelu_new(float x);
/* exposes the range reduction of orc_expf: x = k*ln2 + r */
void  orc_expf_reduce(float x, int32_t *k, float *r);

/* ---- vector kernels ------------------------------------------------------ */
void orc_layernorm(const float *x, const float *gamma, const float *beta,
                   int32_t n, float eps, float *y);
void orc_softmax(float *s, int32_t n);
/* y[o] = sum_i x[i] * W[i][o] + b[o]; W is [in][out] (HF Conv1D). b may be NULL */
void orc_linear(const float *x, const float *W, const float *b,
                int32_t in, int32_t out, float *y);
/* y[o] = sum_i W[o][i] * x[i]; W is [out][in] (the tied head's wte) */
void orc_linear_t(const float *x, const float *W, int32_t in, int32_t out,
                  float *y);
/* One layer's decode attention at position pos over a cache laid out
 * [H][P][D] for this layer; appends this token's k,v first. */
void orc_attn_decode(const float *qkv, int32_t pos, int32_t n_head,
                     int32_t head_dim, int32_t n_positions,
                     float *k_cache, float *v_cache, float *out);
int32_t orc_argmax(const float *v, int32_t n);
/* elementwise fp32 -> fp32 map of gelu_new over an array (test helper) */
void orc_gelu_new_vec(const float *x, float *y, size_t n);
void orc_expf_vec(const float *x, float *y, size_t n);

/* ---- the model ----------------------------------------------------------- */
typedef struct orc_model orc_model;
orc_model *orc_create(const orc_config *cfg, const orc_weights *w);
void       orc_destroy(orc_model *m);
void       orc_reset(orc_model *m);
/* One decode step: token at position pos (pos must be <= cached length).
 * Writes V logits and returns the greedy argmax. Returns -1 on bad input. */
int32_t    orc_forward(orc_model *m, int32_t token, int32_t pos, float *logits);
/* Cache k, v rounded to bf16 (RNE) from now on (0: fp32, the default). */
void       orc_set_kv_bf16(orc_model *m, int32_t on);
/* The same model evaluated from scratch for a whole sequence with a causal
 * mask and no cache: logits_all is [n][V]. Returns 0, or -1 on bad input. */
int32_t    orc_forward_full(const orc_config *cfg, const orc_weights *w,
                            const int32_t *tokens, int32_t n, float *logits_all);

/* ---- stored-weight formats ---------------------------------------------- */
/* fp32 -> IEEE binary16, round to nearest even (handles subnormals, inf) */
void orc_f32_to_f16(const float *in, uint16_t *out, size_t n);
void orc_f16_to_f32(const uint16_t *in, float *out, size_t n);
/* fp32 -> bfloat16, round to nearest even */
void orc_f32_to_bf16(const float *in, uint16_t *out, size_t n);
void orc_bf16_to_f32(const uint16_t *in, float *out, size_t n);

/* Grouped asymmetric int4 of one HF matrix W[in][out], quantised per output
 * row o over groups of 32 consecutive inputs (after the transpose to
 * [out][in] that the graph file's header describes).
 *   codes : [out][in/2]   byte k holds input 2k (low nibble), 2k+1 (high)
 *   scales: [out][in/32]  fp32
 *   zeros : [out][in/64]  4-bit zero points, group 2j low nibble, 2j+1 high
 * in must be a multiple of 64. */
void orc_quant_int4(const float *W, int32_t in, int32_t out,
                    uint8_t *codes, float *scales, uint8_t *zeros);
/* Dequantised weights as [out][in]: w = (float)(q - z) * s */
void orc_dequant_int4(const uint8_t *codes, const float *scales,
                      const uint8_t *zeros, int32_t in, int32_t out,
                      float *W_oi);
/* Temperature sampling ("Let's make GPT-2 in assembly", Step 7; "gpt2.s"
 * README, Options -t): counter-based SplitMix64 output k, a uniform float in
 * (0, 1) from it, the Gumbel-max scores s_i / T - log(-log u_i) with
 * u_i = uniform(seed, pos * n + i), and the chosen token (greedy if T == 0). */
uint64_t orc_splitmix64(uint64_t seed, uint64_t k);
float orc_uniform_bits(uint64_t z);   /* top 23 bits of z -> (0, 1) */
float orc_uniform(uint64_t seed, uint64_t k);
void orc_sample_scores(const float *s, int32_t n, float T, uint64_t seed, int32_t pos, float *out);
int32_t orc_sample(const float *s, int32_t n, float T, uint64_t seed, int32_t pos);

/* The cached K and V rows 0..n_rows-1 of one layer, [H][n_rows][D] each. */
int32_t orc_export_kv(const orc_model *m, int32_t layer, int32_t n_rows, float *k, float *v);

/* nibble helpers (for the round-trip pin) */
void orc_pack_nibbles(const uint8_t *vals, size_t n, uint8_t *packed);
void orc_unpack_nibbles(const uint8_t *packed, size_t n, uint8_t *vals);

#ifdef __cplusplus
}
#endif
#endif
