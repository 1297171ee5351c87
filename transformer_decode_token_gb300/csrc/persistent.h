// Host-visible interface of the persistent decode kernel (persistent.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kernels.h"

namespace gpt2 {

enum PhaseType : int32_t { kPhGemv = 0, kPhAttn = 1, kPhHead = 2 };
// tagged activation buffers: x before LN1 (after the MLP residual), x before
// LN2 (after the attention residual), qkv, attention output, MLP hidden
enum LLBuf : int32_t { kBufXA = 0, kBufXB = 1, kBufQKV = 2, kBufATT = 3, kBufH = 4, kNumLL = 5 };
constexpr int kMaxRing = 16;
constexpr int kMaxPhases = 63;        // epochs keep the phase index in 6 bits
constexpr int kMaxBlockRows = 32;     // rows of a block phase one CTA holds at once
constexpr uint32_t kKvWindowBytes = 24576;   // attention: cached K/V rows held in shared memory

// One phase of the pass (device table, one entry per phase, in order).
struct PPhase {
    int32_t type, mode, layer;
    int32_t in, out;             // GEMV: in / out features (head: E / V)
    int32_t rpc, chunk_rows;     // rows per CTA, rows per ring stage
    uint32_t stage_scale_off, stage_zero_off;
    int32_t in_buf, in_src;      // input buffer and the phase (same pass) that wrote it
    int32_t out_buf;
    const void *W;
    const float *scales;
    const uint8_t *zeros;
    const float *ln_w, *ln_b, *bias;
    // LayerNorm folded into the matrix (block phases with an LN prologue):
    // W.LN(x) = rstd * (W.(gamma*x) - mean * c1) + c2, c1 = W.gamma, c2 = W.beta
    const float *c1, *c2;
};
// copied word by word into shared memory, followed by float4-read vectors
static_assert(sizeof(PPhase) % 16 == 0, "PPhase keeps the shared-memory layout 16-byte aligned");

struct PersistArgs {
    const PPhase *phases;
    int32_t n_phases;
    int32_t n_steps;             // passes in this launch
    const int32_t *prompt;       // pass s < n_prompt consumes prompt[s] (or tok_first)
    int32_t n_prompt, tok_first;
    int32_t pos0;                // position of pass 0
    uint64_t *ll[kNumLL];
    uint64_t *ll_tok;
    float *kcache, *vcache;      // [L][H][P][D]
    float *logits;
    unsigned long long *partials;
    unsigned int *counter;
    int32_t *out_ids;
    int32_t out_cap;
    DeviceState *st;
    const float *wte, *wpe;
    int32_t E, H, D, P, V;
    float scale, eps;
    int32_t n_stages, max_rows;
    uint32_t stage_bytes, ring_offset;
    float head_l2_frac;          // share of each CTA's head rows kept in L2 (evict-last)
    int32_t block_mode;          // block matrices: 0 = resident slice, inputs consumed as they arrive
                                 // (LayerNorm folded); 1 = streamed rows after a LayerNorm prologue
};

cudaError_t launch_persistent(int wtype, const PersistArgs &a, int grid, size_t smem, cudaStream_t s);
// Shared memory before the ring (barriers, vectors, scratch).
size_t persistent_fixed_smem(int E, int D, int max_rows);
// c1[r] = sum_i W[r][i] gamma[i], c2[r] = sum_i W[r][i] beta[i] for W [out][in]
cudaError_t ln_fold(const float *W, const float *gamma, const float *beta, int in, int out, float *c1, float *c2,
                    cudaStream_t s);
int persistent_threads();
// Raises the kernel's dynamic shared-memory limit to `limit` and returns how
// many CTAs of `smem` bytes fit on one SM (call before the first launch).
cudaError_t persistent_blocks_per_sm(int wtype, int D, size_t smem, size_t limit, int *blocks);

}  // namespace gpt2
