// Host-visible launch interface of the decode kernels.  Internal to
// libgpt2.so; the public surface is include/gpt2.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gpt2 {

struct DeviceState;

enum WeightType : int { kWF32 = 0, kWF16 = 1, kWI4 = 2 };

// What a row-GEMV launch does around its dot products.
enum GemvMode : int {
    kModeLnBias = 0,       // y = W . LN(x) + b                  (QKV)
    kModeEmbLnBias = 1,    // x = wte[tok] + wpe[pos]; then as 0  (layer-0 QKV)
    kModeBiasRes = 2,      // y += W . v + b  (y is the residual stream x)
    kModeLnBiasGelu = 3,   // y = gelu_new(W . LN(x) + b)        (MLP fc)
    kModeHead = 4,         // logits = W . LN(x); argmax         (tied head)
};

struct GemvArgs {
    // weights, [out][in]; for int4 also scales [out][in/32], zeros [out][in/64]
    const void *W;
    const float *scales;
    const uint8_t *zeros;
    int32_t in, out;
    // work split: CTA b owns rows [b*rows_per_cta, min(out, (b+1)*rows_per_cta)),
    // streamed through shared memory in chunks of chunk_rows rows, n_stages
    // chunks in flight, each stage stage_bytes long
    int32_t rows_per_cta, chunk_rows, n_stages;
    uint32_t stage_bytes;
    uint32_t stage_scale_off, stage_zero_off;   // int4 sub-offsets in a stage
    int32_t evict_first;                        // weights read once: L2 evict-first hint
    // input vector and prologue
    const float *xin;                           // x (LN modes) or attn / mlp activations
    const float *ln_w, *ln_b;
    float eps;
    const float *wte, *wpe;                     // kModeEmbLnBias
    float *x_out;                               // kModeEmbLnBias: where x is stored
    int32_t vocab, n_positions;
    // epilogue
    const float *bias;
    float *y;
    // kModeHead: per-CTA maxima, arrival counter, appended ids / single token
    unsigned long long *partials;
    unsigned int *counter;
    int32_t *out_ids;
    int32_t out_cap;
    int32_t *dev_token;
    DeviceState *st;
};

// Shared memory a GEMV launch needs.
size_t gemv_smem_bytes(const GemvArgs &a);
// Fills the chunking fields of `a` for `ctas` CTAs and returns the grid size.
int gemv_plan(GemvArgs &a, int wtype, int ctas, size_t stage_budget_bytes, int max_stages);
cudaError_t launch_gemv(int wtype, int mode, const GemvArgs &a, int grid, cudaStream_t s, bool pdl);
// Raises the dynamic shared-memory limit of every GEMV instantiation on the
// current device (once per device; call before any stream capture).
cudaError_t gemv_init();

struct AttnArgs {
    const float *qkv;       // [3E]: q | k | v, head h at [h*D, (h+1)*D) of each
    float *k_cache;         // this layer's [H][P][D]
    float *v_cache;
    float *out;             // [E]
    int32_t n_head, head_dim, n_positions;
    float scale;            // 1/sqrt(head_dim)
    DeviceState *st;
};
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s, bool pdl);

cudaError_t launch_layernorm_rows(const float *x, const float *g, const float *b, int rows, int n,
                                  float eps, float *y, cudaStream_t s);

cudaError_t launch_set_state(DeviceState *st, int32_t tok, int32_t pos, int32_t flags, int32_t *out_ids,
                             cudaStream_t s);
enum : int32_t { kSetTokPos = 1, kResetOut = 2, kSeedOutWithNext = 4, kClearErr = 8 };

// ---- one-time repacking -----------------------------------------------------
// src is HF [in][out] fp32; writes dst [out][in] in the chosen format.
cudaError_t repack_f32(const float *src, int in, int out, float *dst, cudaStream_t s);
cudaError_t repack_f16(const float *src, int in, int out, void *dst, cudaStream_t s);
// src HF [in][out] fp32 -> dst [out][in] bf16 (round to nearest even).
cudaError_t repack_bf16(const float *src, int in, int out, void *dst, cudaStream_t s);
// Elementwise split of n fp32 values into bf16 hi = bf16(v), lo = bf16(v - hi)
// (lo may be null), layout unchanged.
cudaError_t split_bf16(const float *src, size_t n, void *hi, void *lo, cudaStream_t s);
// Elementwise fp32 -> fp16 (round to nearest even) of n values, layout unchanged.
cudaError_t convert_f16(const float *src, size_t n, void *dst, cudaStream_t s);
// tmp must hold out*in floats.
// Grouped int4 of a matrix already in [out][in] layout (the second step of repack_int4).
cudaError_t quant_int4_rows(const float *Wt, int in, int out, uint8_t *codes, float *scales, uint8_t *zeros,
                            cudaStream_t s);
cudaError_t repack_int4(const float *src, int in, int out, float *tmp, uint8_t *codes, float *scales,
                        uint8_t *zeros, cudaStream_t s);
// c1[r] = sum_i W[r][i] gamma[i], c2[r] = sum_i W[r][i] beta[i] for W [out][in]
cudaError_t ln_fold(const float *W, const float *gamma, const float *beta, int in, int out, float *c1, float *c2,
                    cudaStream_t s);
// Widen a stored matrix to fp32 [out][in].
cudaError_t dequant_to_f32(int wtype, const void *W, const float *scales, const uint8_t *zeros, int in,
                           int out, float *dst, cudaStream_t s);

}  // namespace gpt2
