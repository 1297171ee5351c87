// The tensor-core linear of the batched path (tc_gemm.cu): Y = X . W^T for a
// batch of activation rows against a stored bf16 weight matrix, on tcgen05
// with the accumulators in tensor memory.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gpt2 {

struct DeviceState;

// Tile: 128 weight rows (the MMA's M side: weights are the A operand, "swap
// AB") x 128 activation rows (N: the batch's hi parts in rows 0..63, its lo
// parts in rows 64..127) x 64 inputs (one 128-byte swizzle atom of bf16).
constexpr int kTcM = 128;
constexpr int kTcN = 128;
constexpr int kTcK = 64;
constexpr int kTcMaxRows = 64;          // activation rows (sequences or positions) per call
constexpr int kTcStages = 3;            // shared-memory pipeline depth (97 KB: two CTAs fit an SM)
constexpr int kTcThreads = 128;         // 4 warps: TMA producer, MMA issuer, then all four read TMEM
constexpr int kTcMaxSplits = 8;         // K splits of one linear (the consumers sum at most this many shares)

// Activations as the MMA's B operand: a bf16 [128][K] matrix whose row r < 64
// is bf16(x_r) and row 64 + r is bf16(x_r - bf16(x_r)), so that
// W.x = W.hi + W.lo carries about 16 bits of x (fp32 products, fp32 sums).
// Weights: `a_planes` stored bf16 planes of [M][K] (plane p at rows p*M..):
// one plane (bf16 weights), or two (an fp32 matrix split the same way).
struct TcGemmArgs {
    int32_t M, K;              // weight rows and inputs (K % 64 == 0)
    int32_t n_rows;            // activation rows that are stored (<= 64)
    int32_t a_planes;          // 1 or 2
    int32_t a_plane_rows;      // rows from one plane to the next (>= M, a multiple of 128 when a_planes > 1)
    int32_t chunks_per_split;  // 64-input chunks of K per CTA (grid.y = splits)
    float *partials;           // [splits][n_rows][M]: this split's share of Y (hi + lo summed)
    DeviceState *st;           // where a wait that runs out is recorded
    unsigned long long wait_ns;
};

// Tensor maps (TMA descriptors) of a bf16 [rows][K] row-major matrix, boxes of
// 128 rows x 64 inputs, 128-byte swizzle; rows past `rows` read as zero.
int tc_make_tmap(CUtensorMap *map, const void *base, uint64_t rows, uint64_t K);
size_t tc_gemm_smem_bytes();
// Launches grid (ceil(M / 128), splits); the caller checks the shapes.
cudaError_t tc_gemm_launch(const CUtensorMap &a_map, const CUtensorMap &b_map, const TcGemmArgs &a, int splits,
                           cudaStream_t s, bool pdl);
cudaError_t tc_gemm_init();   // raises the kernel's shared-memory limit (once per device)

}  // namespace gpt2
