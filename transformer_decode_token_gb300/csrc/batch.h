// Internal interface of the batched engine (batch.cu) used by the
// single-sequence model: the prompt of one sequence run as the rows of one
// batched step (prefill on the tensor cores).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <functional>

#include "../../include/gpt2.h"

namespace gpt2 {

struct DeviceState;

// A prefill engine for one sequence: rows are consecutive positions of the
// sequence and share its KV cache (kc, vc: [L][H][P][D], owned by the
// caller); the matrices are held as two bf16 planes (hi + lo) of the fp32
// values `matrix(l, k, dst)` writes ([out][in]: QKV, out-projection, fc, MLP
// projection) and the head as two planes of the [V][E] values `head(dst)`
// writes; wte, wpe and the small parameters of `layers` are read in place
// for the embedding (wte, wpe) or copied (the rest).
struct PrefillSrc {
    const float *wte, *wpe, *lnf_w, *lnf_b;
    const float *const *params;   // [L][8]: ln1_w, ln1_b, attn_b, proj_b, ln2_w, ln2_b, fc_b, mlp_proj_b
    std::function<cudaError_t(int layer, int which, float *dst, cudaStream_t s)> matrix;
    std::function<cudaError_t(float *dst, cudaStream_t s)> head;
    float *kc, *vc;
};
int prefill_engine_create(const gpt2_config &cfg, const PrefillSrc &src, cudaStream_t s, int sms, gpt2_batch **out);
// Runs positions 0..n-1 of ids (host) through the engine, in steps of up to
// 64 positions, on stream s; then leaves in the single model's device state
// what its own prefill leaves: the greedy choice after the last position as
// the next token (st->tok, st->next_tok, appended to out_ids), st->pos = n,
// and that position's logits in `logits`; adds the kernels it launched to
// *launches.
int prefill_engine_run(gpt2_batch *e, const int32_t *ids, int n, DeviceState *st, int32_t *out_ids, int out_cap,
                       float *logits, cudaStream_t s, unsigned long long *launches);
void prefill_engine_destroy(gpt2_batch *e);

}  // namespace gpt2
