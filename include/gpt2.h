/*
 * gpt2.h — C ABI of libgpt2.so: GPT-2 single-token (batch 1) decode on one
 * GB300 (sm_103a).
 *
 * What it computes.  One forward pass per token, as the node list of the
 * "model.fir" graph file (Resident GPT-2 decode) and the model.s description
 * of the "gpt2.s" README ("Inner Workings") lay it out:
 *   x = wte[token] + wpe[position]
 *   for each of n_layer blocks:
 *     qkv  = LayerNorm1(x) . W_attn + b_attn          (fused QKV linear)
 *     attn = causal attention of q over the cached k, v of positions
 *            0..position, after appending this token's k, v
 *     x   += attn . W_proj + b_proj
 *     x   += gelu_new(LayerNorm2(x) . W_fc + b_fc) . W_mlp_proj + b_mlp_proj
 *   logits = wte . LayerNorm_f(x)                      (tied output head)
 *   token' = argmax(logits)                            (greedy choice,
 *            "Let's make GPT-2 in assembly", Step 7; exact ties -> lowest id)
 *
 * Conventions shared by every call.
 *   - Every call returns an int status: GPT2_OK (0) or a negative GPT2_ERR_*
 *     code; gpt2_strerror() names it.  No call throws, aborts or traps, and no
 *     kernel traps: a device-side problem is recorded in a device error word
 *     and returned by the next call that synchronises (gpt2_argmax,
 *     gpt2_generate, gpt2_copy_logits, gpt2_sync).
 *   - "stream" arguments are a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  All of a model's work is ordered on its stream.
 *   - Device pointers must come from the CUDA device that is current when the
 *     call is made; host pointers may be pageable.
 *   - A model is not thread-safe: serialise calls on one model.
 */
#ifndef GPT2_H
#define GPT2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define GPT2_OK                      0
#define GPT2_ERR_INVALID_ARG        -1  /* NULL pointer, bad enum, bad shape  */
#define GPT2_ERR_UNSUPPORTED_DEVICE -2  /* current device is not cc 10.3      */
#define GPT2_ERR_TOKEN_RANGE        -3  /* token outside [0, vocab_size)      */
#define GPT2_ERR_POSITION_RANGE     -4  /* position >= n_positions, or past
                                           the cached length (see decode_step) */
#define GPT2_ERR_NOT_READY          -5  /* e.g. argmax before any step        */
#define GPT2_ERR_CUDA               -6  /* a CUDA runtime call failed         */
#define GPT2_ERR_TIMEOUT            -7  /* a bounded device wait gave up      */
#define GPT2_ERR_DEVICE_STATE       -8  /* a kernel rejected its inputs       */
#define GPT2_ERR_OUT_OF_MEMORY      -9  /* device allocation failed           */
#define GPT2_ERR_RANGE             -10  /* an activation left the range of the
                                           cluster kernel's fixed-point residual
                                           sums (|value| > 65000, or NaN)      */

/* ---- configuration ------------------------------------------------------- */
/* Model shape, as the graph file's config checks and symbols define it
 * ("model.fir": sym hidden = n_embd, nheads = n_head, headdim = hidden/nheads,
 * mlp = 4*hidden, positions = n_positions, vocab = vocab_size; epsilon
 * layer_norm_epsilon).  Accepted: n_embd % 32 == 0, n_embd % n_head == 0,
 * head_dim in {32, 64, 128}; GPT2_INT4 also needs n_embd % 128 == 0. */
typedef struct gpt2_config {
    int32_t n_layer;
    int32_t n_embd;
    int32_t n_head;
    int32_t n_positions;
    int32_t vocab_size;
    float   ln_eps;            /* GPT-2 uses 1e-5 */
} gpt2_config;

/* How the 48 (4 * n_layer) block matrices are stored on the device.  The
 * embeddings, biases, LayerNorm parameters, the tied head and the KV cache
 * are fp32 in every mode ("gpt2.s" README, Options: -h; "model.fir" header:
 * wte/lm_head stays tied fp32).
 *   GPT2_F32 : fp32, transposed to [out][in].
 *   GPT2_F16 : IEEE fp16 (round to nearest even), [out][in]; widened to fp32
 *              inside the kernels, products and sums in fp32.
 *   GPT2_INT4: grouped asymmetric int4 of the [out][in] matrix, groups of 32
 *              consecutive inputs, fp32 scale s and 4-bit zero point z per
 *              group, s = (max(0,max w) - min(0,min w)) / 15 (1 if that is 0),
 *              z = clamp(rint(-min/s), 0, 15), q = clamp(rint(w/s) + z, 0, 15),
 *              dequantised weight (q - z) * s.  Layout: codes [out][in/2]
 *              (input 2k in the low nibble of byte k), scales [out][in/32] f32,
 *              zeros [out][in/64] (group 2j in the low nibble of byte j). */
typedef enum gpt2_wdtype {
    GPT2_F32  = 0,
    GPT2_F16  = 1,
    GPT2_INT4 = 2,
    GPT2_BF16 = 3     /* batched models only (gpt2_create_batch)          */
} gpt2_wdtype;

/* One block's tensors, DEVICE pointers to fp32, in the checkpoint's HF
 * Conv1D layout (matrices [input][output], row-major): names and shapes as
 * the graph file's weight lines give them. */
typedef struct gpt2_layer_weights {
    const float *ln1_w, *ln1_b;            /* [E]                  */
    const float *attn_w, *attn_b;          /* [E][3E], [3E]        */
    const float *proj_w, *proj_b;          /* [E][E],  [E]         */
    const float *ln2_w, *ln2_b;            /* [E]                  */
    const float *fc_w, *fc_b;              /* [E][4E], [4E]        */
    const float *mlp_proj_w, *mlp_proj_b;  /* [4E][E], [E]         */
} gpt2_layer_weights;

/* All 4 + 12 * n_layer tensors (148 for GPT-2 small).  Tensor pointers are
 * DEVICE pointers; `layers` itself is a HOST array of n_layer entries. */
typedef struct gpt2_weights {
    const float *wte;                      /* [V][E] token embedding = head */
    const float *wpe;                      /* [P][E]                        */
    const float *ln_f_w, *ln_f_b;          /* [E]                           */
    const gpt2_layer_weights *layers;      /* host array, n_layer entries   */
} gpt2_weights;

typedef struct gpt2_model gpt2_model;

/* ---- model lifecycle ------------------------------------------------------ */

/* Validates cfg (the graph file's `require` checks: hidden = nheads*headdim,
 * mlp = 4*hidden) and the device (compute capability 10.3), allocates every
 * device buffer the model needs (weights in the chosen format, the fp32 KV
 * cache [n_layer][n_head][n_positions][head_dim] — "stored by head", as the
 * "gpt2.s" README's Inner Workings puts it — activations, logits), repacks
 * the weights on the device (transpose to [out][in]; fp16 rounding; int4
 * quantisation) and prepares the decode path (gpt2_create_ex: the cluster
 * kernel's tiled copies and launch shape, or, on the per-kernel path, one
 * decode pass captured into a CUDA graph).
 * The caller keeps ownership of `w`'s tensors and may free them once this
 * returns.  On success *out owns everything and must be released with
 * gpt2_destroy.  Errors: INVALID_ARG, UNSUPPORTED_DEVICE, OUT_OF_MEMORY, CUDA. */
int gpt2_create(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype,
                void *stream, gpt2_model **out);

/* gpt2_create with options.  flags = 0 is gpt2_create.  Two paths compute
 * the same pass (the node list of the "model.fir" graph file and the model.s
 * description of the "gpt2.s" README, "Inner Workings"; greedy choice as in
 * "Let's make GPT-2 in assembly", Step 7):
 *  - cluster (default): one cooperative launch per call of a kernel whose
 *    CTAs form clusters of 4.  One cluster per attention head computes that
 *    head's q, k, v, attention and its share of the output projection,
 *    trading values inside the cluster through distributed shared memory; the
 *    other CTAs own slices of the MLP.  Residual sums between the two groups
 *    are fixed-point integer atomics, so runs are bitwise reproducible; two
 *    GPU-wide exchanges per block.  Greedy steps never return to the host.
 *  - per-kernel (GPT2_FLAG_PER_KERNEL): the CUDA graph, captured at create
 *    time, of 5 * n_layer + 1 kernels per pass.
 * Where the cluster kernel cannot run (it needs n_embd a multiple of 64 and
 * at most 1024, vocab_size <= 131072, and enough co-resident clusters of 4
 * CTAs for one per head plus the MLP's), the per-kernel path is used;
 * gpt2_path reports which one a model uses. */
#define GPT2_FLAG_PER_KERNEL 1
/* GPT2_FLAG_HEAD_F16: the tied output head is also stored as fp16 (round to
 * nearest even), as the "gpt2.s" README's -h option stores it ("Options": the
 * 48 block matrices and the output head as fp16); the LM head reads that
 * copy (widened to fp32, products and sums in fp32) while the embedding
 * lookup still reads the fp32 wte.  Adds n_vocab * n_embd * 2 bytes of device
 * memory.  Cluster path only: with a flag or device that rules it out,
 * gpt2_create_ex returns GPT2_ERR_INVALID_ARG. */
#define GPT2_FLAG_HEAD_F16 4
/* GPT2_FLAG_HEAD_INT4: the output head stored as grouped asymmetric int4 of
 * wte's rows (the GPT2_INT4 scheme and layout, groups of 32 along n_embd),
 * the "next" variant for the int4 mode, where the fp32 head is three quarters
 * of the bytes; the embedding still reads the fp32 wte.  Cluster path only,
 * n_embd % 64 == 0; not together with GPT2_FLAG_HEAD_F16. */
#define GPT2_FLAG_HEAD_INT4 8
/* Prompts (gpt2_prefill, gpt2_generate) on the cluster path run, by default,
 * on the tensor cores: the prompt's positions become the rows of one batched
 * step (see gpt2_create_batch), up to 64 positions per step, with the stored
 * block matrices and head held again as bf16 hi + lo planes (about 16 bits of
 * each weight, fp32 sums; greedy choice; 340 MB more for GPT-2 small's block
 * matrices, plus the head's planes).  Prompts of fewer than 5 tokens (where
 * single-token passes are faster), or a model with a sampling temperature,
 * use single-token passes.  GPT2_FLAG_NO_TC_PREFILL keeps every prompt on
 * single-token passes. */
#define GPT2_FLAG_NO_TC_PREFILL 16
int gpt2_create_ex(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype,
                   int32_t flags, void *stream, gpt2_model **out);

#define GPT2_PATH_PER_KERNEL 0
#define GPT2_PATH_CLUSTER 2
int gpt2_path(const gpt2_model *m, int32_t *path);

/* Frees every device buffer and the graph.  NULL is accepted. */
void gpt2_destroy(gpt2_model *m);

/* Forget the cached tokens (cached length 0). */
int gpt2_reset(gpt2_model *m);

/* ---- decoding ------------------------------------------------------------ */

/* One forward pass for `token` at `position` ("gpt2.s" README, Inner
 * Workings: model.s, the forward pass for one token; the KV cache gains one
 * row per token, "Let's make GPT-2 in assembly" Step 6).  `position` must be
 * < n_positions and <= the cached length: equal appends; smaller rewinds the
 * cache to `position` first.  On success the cached length is position + 1
 * and, if dev_logits is not NULL, *dev_logits points at the model's device
 * buffer of vocab_size fp32 logits, valid until the next decoding call.
 * Asynchronous: returns once the work is queued on the model's stream.
 * Errors: INVALID_ARG, TOKEN_RANGE, POSITION_RANGE, CUDA. */
int gpt2_decode_step(gpt2_model *m, int32_t token, int32_t position,
                     const float **dev_logits);

/* Resets the cache, then runs decode steps for ids[0..n-1] at positions
 * 0..n-1 (the prompt is consumed one token at a time, as in "gpt2.s").
 * host_ids is a host array.  Afterwards the last step's logits and argmax are
 * available.  Errors: as gpt2_decode_step; n must be in [1, n_positions]. */
int gpt2_prefill(gpt2_model *m, const int32_t *host_ids, int32_t n);

/* Greedy choice of the last step's logits: the highest logit, exact ties to
 * the lowest id ("Let's make GPT-2 in assembly", Step 7).  Synchronises the
 * model's stream and copies 4 bytes to the host.
 * Errors: NOT_READY (no step yet), DEVICE_STATE / TIMEOUT (reported by a
 * kernel), CUDA. */
int gpt2_argmax(gpt2_model *m, int32_t *token_out);

/* How the following passes choose their token ("Let's make GPT-2 in
 * assembly", Step 7: divide the scores by a temperature, apply softmax, draw
 * at random; "gpt2.s" README, Options: -t, 0 means greedy).  temperature 0
 * (the default) is greedy.  temperature > 0 draws each pass's token from
 * softmax(logits / temperature), in the Gumbel-max form: the token with the
 * highest logit / temperature - log(-log u), u the uniform number of counter
 * position * vocab_size + id from a counter-based SplitMix64 generator with
 * this seed (u = (top 23 bits of the output + 0.5) * 2^-23, strictly inside
 * (0, 1)).  The same seed,
 * prompt and weights give the same tokens.  The drawn token is what
 * gpt2_argmax returns and what gpt2_decode_greedy / gpt2_generate feed to the
 * next pass; the logits stay the plain ones.  Takes effect from the next
 * call.  Errors: INVALID_ARG (temperature negative or not finite, or
 * temperature > 0 on a model that does not use the cluster kernel). */
int gpt2_set_sampling(gpt2_model *m, float temperature, uint64_t seed);

/* Device-resident greedy decoding: n_steps more decode passes, each fed the
 * previous pass's argmax without a round trip to the host (token and
 * position live in device memory).  Needs a previous step; the cached length
 * grows by n_steps and must stay <= n_positions.  Asynchronous.
 * Errors: NOT_READY, POSITION_RANGE, INVALID_ARG, CUDA. */
int gpt2_decode_greedy(gpt2_model *m, int32_t n_steps);

/* Whole greedy generation from host to host: prefill(host_prompt, n_prompt),
 * then n_steps device-resident decode passes; host_out receives n_steps + 1
 * ids: the argmax after the last prompt token, then the argmax after each
 * decode pass (the pass i input is host_out[i]).  Synchronises.
 * Errors: as prefill and decode_greedy; n_prompt + n_steps <= n_positions. */
int gpt2_generate(gpt2_model *m, const int32_t *host_prompt, int32_t n_prompt,
                  int32_t n_steps, int32_t *host_out);

/* Copies the last step's vocab_size logits to dst (host or device memory)
 * and synchronises.  Errors: NOT_READY, INVALID_ARG, CUDA, DEVICE_STATE. */
int gpt2_copy_logits(gpt2_model *m, float *dst);

/* Waits for the model's queued work; returns a recorded device error if any
 * (and clears it, with the cluster kernel's exchange state, so the model
 * stays usable). */
int gpt2_sync(gpt2_model *m);

/* Time limit of every wait inside the cluster kernel (for a weight stage, a
 * peer CTA, a GPU-wide sum or the previous pass's token), in nanoseconds of
 * the GPU's global timer; default 2e9 (2 s).  When a wait runs out the kernel
 * records GPT2_ERR_TIMEOUT, every CTA skips its remaining work and returns,
 * and the next synchronising call reports the error ("gpt2.s" README,
 * Limitations: a worker that stops ends the program with an error instead of
 * hanging it).  A test hook: a tiny limit makes the first wait that does not
 * succeed at once give up.  Takes effect from the next call.
 * Errors: INVALID_ARG (NULL model, or a model on the per-kernel path). */
int gpt2_set_wait_limit(gpt2_model *m, uint64_t ns);

/* ---- inspection (for parity tests and tools) ---------------------------- */

/* Selects one stored block matrix. */
#define GPT2_MAT_ATTN      0   /* c_attn   [3E][E] after the transpose */
#define GPT2_MAT_PROJ      1   /* c_proj   [E][E]                      */
#define GPT2_MAT_FC        2   /* c_fc     [4E][E]                     */
#define GPT2_MAT_MLP_PROJ  3   /* mlp proj [E][4E]                     */

/* Byte sizes of a stored matrix's parts: main (fp32/fp16 values or int4
 * codes), scales and zeros (0 unless GPT2_INT4).  Any out pointer may be NULL. */
int gpt2_matrix_bytes(const gpt2_model *m, int32_t which, size_t *main_bytes,
                      size_t *scale_bytes, size_t *zero_bytes);

/* Copies a stored matrix's bytes, in the layout gpt2_wdtype describes, to
 * host or device memory.  Any destination may be NULL to skip that part. */
int gpt2_export_matrix(gpt2_model *m, int32_t layer, int32_t which,
                       void *dst_main, void *dst_scales, void *dst_zeros);

/* Writes the matrix as the kernels see it, widened to fp32 in [out][in]
 * (fp16 widened, int4 dequantised as (q - z) * s), to DEVICE memory dst. */
int gpt2_export_dequant(gpt2_model *m, int32_t layer, int32_t which, float *dst);

/* Copies the cached K and V rows 0..n_rows-1 of one layer, laid out
 * [n_head][n_rows][head_dim] fp32 each, to host or device memory. */
int gpt2_export_kv(gpt2_model *m, int32_t layer, int32_t n_rows,
                   float *dst_k, float *dst_v);

/* Kernel launches per decode pass: 5 * n_layer + 1 on the per-kernel path,
 * 1 on the cluster path (where one launch runs every pass of a call). */
int gpt2_kernels_per_step(const gpt2_model *m, int32_t *count);

/* Total kernel launches this model has issued so far (graph kernels and the
 * small state-setting kernel included), for launch accounting. */
int gpt2_launch_count(const gpt2_model *m, uint64_t *count);

/* ---- stand-alone operations on caller buffers --------------------------- */

/* Warp-per-row LayerNorm of `rows` rows of n fp32 values ("model.fir" kernel
 * g2.layernorm: mean, biased variance, (x-mean)*rsqrt(var+eps)*gamma+beta).
 * x, gamma, beta, y are DEVICE pointers; y may equal x.  n % 4 == 0. */
int gpt2_op_layernorm(const float *x, const float *gamma, const float *beta,
                      int32_t rows, int32_t n, float eps, float *y, void *stream);

/* Final LayerNorm + tied head + greedy argmax on caller buffers (the
 * graph file's final_norm and head nodes, then "Let's make GPT-2 in
 * assembly" Step 7): logits[v] = sum_e wte[v][e] * LN(x)[e];
 * *dev_token = argmax.  All pointers are DEVICE pointers; wte is [V][E] with
 * E % 4 == 0.  The kernel combines per-block maxima in `workspace`, which must
 * hold gpt2_op_head_argmax_workspace(V, E) bytes, be 16-byte aligned, and not
 * be used by another call in flight.  The call zeroes what it needs.
 * Asynchronous on `stream`.  Errors: INVALID_ARG, CUDA. */
size_t gpt2_op_head_argmax_workspace(int32_t vocab, int32_t n_embd);
int gpt2_op_head_argmax(const float *x, const float *ln_w, const float *ln_b,
                        float eps, const float *wte, int32_t vocab,
                        int32_t n_embd, float *logits, int32_t *dev_token,
                        void *workspace, size_t workspace_bytes, void *stream);

/* The same final LayerNorm + tied head + argmax for callers that cannot
 * allocate device memory (no counterpart on the pages: it exists for hosts
 * that own all device memory through their own pools, or whose steady-state
 * loop must never call the CUDA allocator).  It takes no workspace: the
 * per-CTA maxima and the arrival counter live in a fixed 4112-byte array in
 * the library's device memory, one copy per GPU that loads the library, kept
 * until the process exits.  It allocates nothing and calls no allocating
 * routine.
 *   - vocab must be <= GPT2_NOALLOC_MAX_VOCAB (131072); larger vocabularies
 *     return GPT2_ERR_INVALID_ARG (the array holds one key per 256 rows).
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture begins.  The address is kept with the device's context: after
 *     cudaDeviceReset the next call looks it up again (again a first call).
 *   - All calls on a device share the array: calls whose kernels can overlap
 *     on the GPU (different streams, different threads) race and must be
 *     serialised by the caller.  Each call clears the counter it needs.
 * Arguments, layouts and results are those of gpt2_op_head_argmax; outputs
 * match it.  Asynchronous on `stream`.  Errors: INVALID_ARG, CUDA. */
#define GPT2_NOALLOC_MAX_VOCAB 131072
int gpt2_op_head_argmax_noalloc(const float *x, const float *ln_w, const float *ln_b,
                                float eps, const float *wte, int32_t vocab,
                                int32_t n_embd, float *logits, int32_t *dev_token,
                                void *stream);

/* ---- batched decoding ------------------------------------------------------ */

/* A batched model decodes up to max_batch independent sequences together,
 * one token of each per step.  Each step is, for every sequence of the batch,
 * the decode pass above (the graph file's node list; the model.s description
 * of the "gpt2.s" README, "Inner Workings"; greedy choice as in "Let's make
 * GPT-2 in assembly", Step 7) over that sequence's own KV cache; with many
 * sequences the linears become dense matrix products, which run on the tensor
 * cores (tcgen05, bf16 operands, fp32 accumulators in tensor memory).
 *   - Weights: GPT2_BF16 only.  The 48 block matrices are stored as bf16
 *     [out][in] (round to nearest even) and the tied head as a bf16 copy of
 *     wte; embeddings, biases, LayerNorm parameters and the KV cache stay
 *     fp32 (the cache: bf16 with GPT2_BATCH_KV_BF16).  Activations enter each product as two bf16 parts (x = hi + lo,
 *     lo = bf16(x - hi)), so products use about 16 bits of x; sums are fp32.
 *   - Cache: [n_layer][max_batch][n_head][n_positions][head_dim] fp32, one
 *     slot per sequence; sequences have independent lengths (ragged).
 *   - One step is a CUDA graph of 8 * n_layer + 4 kernels captured at create
 *     time; steps are asynchronous on the model's stream.
 * Errors as for the single-sequence calls. */
typedef struct gpt2_batch gpt2_batch;

/* max_batch in [1, 64].  Same weights argument and ownership as gpt2_create.
 * Errors: INVALID_ARG (wdtype other than GPT2_BF16, shapes: n_embd % 64,
 * n_embd <= 1024, head_dim in {32, 64, 128}), UNSUPPORTED_DEVICE,
 * OUT_OF_MEMORY, CUDA. */
int gpt2_create_batch(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype,
                      int32_t max_batch, void *stream, gpt2_batch **out);
/* GPT2_BATCH_KV_BF16: the cache holds k and v rounded to bf16 (round to
 * nearest even) when they are written, [n_layer][max_batch][n_head]
 * [n_positions][head_dim] bf16; attention reads the cached values, the
 * current position's included (q, the scores and the softmax stay fp32).
 * Halves the cache's memory and the bytes a step reads from it. */
#define GPT2_BATCH_KV_BF16 1u
/* gpt2_create_batch with options: flags is 0 or GPT2_BATCH_KV_BF16 (other
 * bits: INVALID_ARG). */
int gpt2_create_batch_ex(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype,
                         int32_t max_batch, uint32_t flags, void *stream, gpt2_batch **out);
void gpt2_destroy_batch(gpt2_batch *m);

/* One step: sequence b (b < n) consumes host tokens[b] at host positions[b]
 * (append at its cached length, or rewind to a smaller position, as in
 * gpt2_decode_step); positions[b] == -1 leaves sequence b out of this step
 * (its cache is untouched).  If dev_logits is not NULL it receives the
 * model's device buffer of [max_batch][vocab_size] fp32 logits (rows of
 * sequences left out are not meaningful), valid until the next step. */
int gpt2_decode_batch(gpt2_batch *m, const int32_t *tokens, const int32_t *positions,
                      int32_t n, const float **dev_logits);

/* Resets every sequence, then consumes the ragged prompts: sequence b's
 * lens[b] ids follow one another in the host array ids (sequence 0 first).
 * Every position but each sequence's last runs in prompt steps of max_batch
 * (sequence, position) rows packed sequence by sequence (the blocks only:
 * they fill the cache); the last positions then run as one decode step, so
 * each sequence's greedy choice after its prompt (gpt2_argmax_batch) and
 * its logits (gpt2_copy_logits_batch) are available afterwards.  The ids
 * chosen at prompt positions other than the last are not recorded
 * (gpt2_batch_ids). */
int gpt2_prefill_batch(gpt2_batch *m, const int32_t *ids, const int32_t *lens, int32_t n);

/* n_steps device-resident greedy steps for every sequence with a cached
 * prefix: each continues at its own length with its last choice; the host is
 * not involved between steps.  Errors: NOT_READY, POSITION_RANGE (a sequence
 * would pass n_positions), INVALID_ARG. */
int gpt2_decode_batch_greedy(gpt2_batch *m, int32_t n_steps);

/* The greedy choice of the last step for sequences 0..n-1 (synchronises). */
int gpt2_argmax_batch(gpt2_batch *m, int32_t *host_ids, int32_t n);

/* The tokens chosen by the passes at positions first_pos .. first_pos +
 * n_pos - 1, [n_pos][max_batch] int32, copied to host memory (an entry of a
 * sequence that never ran that position is not meaningful); synchronises. */
int gpt2_batch_ids(gpt2_batch *m, int32_t first_pos, int32_t n_pos, int32_t *host_ids);

/* Copies the logits of sequences 0..n-1 ([n][vocab_size] fp32) of the last
 * step to host or device memory; synchronises. */
int gpt2_copy_logits_batch(gpt2_batch *m, int32_t n, float *dst);

/* Copies the cached K and V rows 0..n_rows-1 of one layer and sequence,
 * [n_head][n_rows][head_dim] fp32 each (a bf16 cache widened exactly), to
 * host or device memory; synchronises. */
int gpt2_export_kv_batch(gpt2_batch *m, int32_t layer, int32_t seq, int32_t n_rows,
                         float *dst_k, float *dst_v);

/* Kernels per step and kernel launches so far (any pointer may be NULL). */
int gpt2_batch_info(const gpt2_batch *m, int32_t *kernels_per_step, uint64_t *launches);

/* Waits for the model's queued work; returns (and clears) a recorded device
 * error. */
int gpt2_sync_batch(gpt2_batch *m);

/* The batched path's tensor-core linear on caller buffers: Y[r][o] =
 * sum_k W[o][k] * X[r][k] for r < n, W a DEVICE bf16 [M][K] matrix (16-byte
 * aligned), X DEVICE fp32 [n][K], Y DEVICE fp32 [n][M]; n <= 64, K % 64 == 0.
 * X enters as hi + lo bf16 parts, sums are fp32 (the graph file's linear node
 * with bf16 weights).  workspace (DEVICE, 256-byte aligned) holds
 * gpt2_op_linear_bf16_workspace(M, n, K) bytes and may not be used by another
 * call in flight.  Asynchronous on `stream`.  Errors: INVALID_ARG,
 * UNSUPPORTED_DEVICE, CUDA. */
size_t gpt2_op_linear_bf16_workspace(int32_t M, int32_t n, int32_t K);
int gpt2_op_linear_bf16(const void *W, const float *X, int32_t M, int32_t n, int32_t K,
                        float *Y, void *workspace, size_t workspace_bytes, void *stream);

/* ---- errors ------------------------------------------------------------- */
const char *gpt2_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_H */
