// Host-visible interface of the cluster decode kernel (cluster.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kernels.h"

namespace gpt2 {

constexpr int kClusterSize = 4;
constexpr int kClusterRing = 16;   // ring stages of the weight stream (a power of two)
// Words between consecutive elements of a residual sum (1: contiguous; 4: one
// element per 32-byte sector, spreading the atomics over more L2 lines).
#ifndef GPT2_ACC_STRIDE
#define GPT2_ACC_STRIDE 1
#endif
constexpr int kClusterAccStride = GPT2_ACC_STRIDE;

// Weights of one layer as the cluster kernel reads them.  The fc matrix is
// the canonical [out][in] copy; the QKV matrix is a copy with its rows
// grouped by (head, rank) (cluster_gather_qkv); the two matrices consumed by
// column slices are re-tiled so that one CTA's slice is contiguous:
//   Wo_t: [H][4 ranks][E/4 rows][D cols] (head h's columns, rank's rows)
//   Wp_t: [nfc][E rows][fr cols]         (fc CTA f's columns fr = F / nfc)
// Tiles store 16-byte units of a row swizzled by (row & (units - 1)) (units a
// power of two, at most 8) so that threads reading consecutive rows hit
// different shared-memory banks.  int4 tiles: codes [rows][cols/2], scales
// [rows][cols/32] f32, zero points [rows][cols/32] one byte each.
struct CLayer {
    const void *Wqkv;
    const float *qkv_s;
    const uint8_t *qkv_z;
    const float *ln1_w, *ln1_b, *attn_b;
    const void *Wo_t;
    const float *o_s;
    const uint8_t *o_z;
    const float *proj_b;
    const void *Wfc;
    const float *fc_s;
    const uint8_t *fc_z;
    const float *ln2_w, *ln2_b, *fc_b;
    const void *Wp_t;
    const float *p_s;
    const uint8_t *p_z;
    const float *mlp_proj_b;
    // LayerNorm folded into the rows that follow it:
    //   W.LN(x) + b = rstd * (W.(gamma*(x-s)) - (mean-s) * c1) + cb  (s = x[0]),
    //   c1 = W.gamma, cb = W.beta + b (from the weights as stored)
    const float *q_c1, *q_cb;    // [3E], in the gathered QKV row order
    const float *f_c1, *f_cb;    // [F]
};

struct ClusterArgs {
    const CLayer *layers;
    int32_t L;
    int32_t n_steps;
    const int32_t *prompt;
    int32_t n_prompt, tok_first, pos0;
    int32_t E, H, D, F, P, V;
    float eps, scale;
    int32_t nfc, fr;             // fc CTAs, fc rows (= mlp-proj columns) per fc CTA
    int32_t head_rpc;            // LM-head rows per CTA (a multiple of 4)
    const void *head_w;          // the LM head's rows [V][E]: the fp32 wte, or its fp16 / int4 copy
    const float *head_s;         // int4 head: scales [Vp][E/32] (Vp = head_rpc * grid, padding rows zero)
    const uint8_t *head_z;       // int4 head: zero points [Vp][E/64]
    int32_t head_wt;             // their type (kWF32, kWF16 or kWI4)
    float temperature;           // token choice: 0 = greedy, > 0 = a draw from softmax(logits / T)
    unsigned long long seed;     // sampling: seed of the counter-based generator
    int32_t pr_rows;             // row slots of the parameter area (a multiple of 4)
    const float *h_c1, *h_cb;    // LM head: wte.gamma_f, wte.beta_f, padded to head_rpc * grid
    // residual-stream sums, one 64-bit word per element holding the biased
    // fixed-point sum and the number of contributions (double-buffered by
    // pass parity; the other parity is zeroed during a pass)
    long long *acc_new;          // [2 parity][L][E][kClusterAccStride]  x after the attention block
    long long *acc_next;         // [2 parity][L][E][kClusterAccStride]  x after the MLP block
    float *kcache, *vcache;      // [L][H][P][D]
    float *logits;
    unsigned long long *partials;  // [grid] each CTA's best LM-head key, tagged with its pass
    int32_t *out_ids;
    int32_t out_cap;
    DeviceState *st;
    const float *wte, *wpe, *lnf_w, *lnf_b;
    int32_t wtype;
    int32_t n_stages;
    uint32_t stage_bytes, ring_offset;
    unsigned long long wait_ns;  // every device wait gives up after this long (GPT2_ERR_TIMEOUT)
};

// Dynamic shared memory before the ring.
size_t cluster_fixed_smem(int E, int D, int fr, int L, int pr_rows);
cudaError_t launch_cluster(int wtype, const ClusterArgs &a, int n_clusters, size_t smem, cudaStream_t s);
// Co-resident clusters of kClusterSize CTAs with `smem` bytes each (sets the
// kernel's shared-memory limit to `limit` first).
cudaError_t cluster_max_active(int wtype, int D, size_t smem, size_t limit, int *clusters);
// Writes the tiled copy of a stored [out][in] matrix: T tiles of rows x cols;
// tile t, row i = canonical row (t % rdiv) * rows + i, columns
// (t / rdiv) * cols + [0, cols).  int4 also writes per-row scales and one
// zero-point byte per 32-column group.
cudaError_t cluster_tile(int wtype, const void *W, const float *scales, const uint8_t *zeros, int in, int T,
                         int rdiv, int rows, int cols, void *dW, float *dscales, uint8_t *dzeros, cudaStream_t s);
// Writes the copy of a stored QKV matrix [3E][E] whose rows are grouped by
// (head, rank): block h * 4 + r holds that CTA's D/4 q rows, then its D/4 k
// rows, then its D/4 v rows, in the canonical row format.
cudaError_t cluster_gather_qkv(int wtype, const void *W, const float *scales, const uint8_t *zeros, int E, int D,
                               void *dW, float *dscales, uint8_t *dzeros, cudaStream_t s);
// Stage bytes that `gran` rows of a segment need (sections 16-byte aligned).
uint32_t cluster_stage_need(int gran, uint32_t rb, uint32_t srb, uint32_t zrb);

}  // namespace gpt2
