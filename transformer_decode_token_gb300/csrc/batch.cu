// Batched decode: the decode pass for up to 64 independent sequences at once,
// one token each per step, with bf16 block matrices and head on the tensor
// cores.
//
// Every step is the per-token pass of the "model.fir" graph file's node list
// (and the model.s description of the "gpt2.s" README, "Inner Workings"),
// applied to each sequence of the batch: embedding, 12 pre-LN blocks, the
// final LayerNorm, the tied head and the greedy choice ("Let's make GPT-2 in
// assembly", Step 7).  With 64 sequences the four linears of a block and the
// head become dense contractions of the stored weights with 64 activation
// rows (tc_gemm.cu); attention stays per sequence over that sequence's own
// (ragged) KV cache.  One step is a CUDA graph of 8 kernels per block + 4,
// chained by programmatic dependent launch (each kernel lets the next one
// launch once it has passed its own wait, so the next one's CTAs are resident
// and the linears' weight tiles in flight before its input exists):
//   k_b_ln     residual add (the previous linear's split-K shares summed in a
//              fixed order, + bias), or the embedding; LayerNorm; the bf16
//              hi/lo B operand of the next linear
//   tc_gemm    QKV / out-projection / fc / MLP projection / head: fp32 shares
//              of the K splits
//   k_b_attn   q, k, v of one (sequence, head) from the QKV shares, k and v
//              appended at the sequence's position, softmax(q.k / sqrt(D))
//              over positions 0..pos, the weighted sum of v
//   k_b_gelu   fc shares + bias, gelu_new, the B operand of the MLP projection
//   k_b_argmax greedy choice per sequence; k_b_advance feeds it to the next step
// When the rows are positions of one sequence (a prompt on the tensor cores),
// k_b_append writes every row's k and v into the cache before the attention
// reads them (9 kernels per block).
// The KV cache and all activations are fp32; a sequence whose position is -1
// is inactive for the step (no cache row written, its outputs ignored).
#include "../../include/gpt2.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <new>
#include <vector>

#include "batch.h"
#include "common.cuh"
#include "kernels.h"
#include "tc_gemm.h"

using namespace gpt2;

namespace {

constexpr int kBT = 256;   // threads of the elementwise / attention kernels

__device__ __forceinline__ void put_hi_lo(__nv_bfloat16 *b_op, int row, int ld, int i, float y)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(y);
    b_op[size_t(row) * ld + i] = h;
    b_op[size_t(kTcMaxRows + row) * ld + i] = __float2bfloat16_rn(y - __bfloat162float(h));
}

// Sum of `v` over the CTA in a fixed order (warp butterflies, then the warps'
// sums in warp order): every run gives the same bits.
__device__ __forceinline__ float block_sum(float v, float *red)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) t += red[w];
    return t;
}
__device__ __forceinline__ float block_max(float v, float *red)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = red[0];
    for (int w = 1; w < int(blockDim.x >> 5); ++w) t = fmaxf(t, red[w]);
    return t;
}

// Sum of the K-split shares of element i of row b ([splits][rows][n]), in
// split order, with every share's load in flight at once.
__device__ __forceinline__ float sum_shares(const float *parts, int splits, int rows, int n, int b, int i)
{
    float v[kTcMaxSplits];
#pragma unroll
    for (int k = 0; k < kTcMaxSplits; ++k) v[k] = k < splits ? parts[(size_t(k) * rows + b) * n + i] : 0.f;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kTcMaxSplits; ++k)
        if (k < splits) s += v[k];
    return s;
}

struct BLnArgs {
    float *x;                       // [rows][E] residual stream
    const float *parts;             // [splits][rows][E] shares of the linear before (mode 1)
    int32_t splits;
    const float *bias;              // its bias [E]
    const int32_t *tok, *pos;       // mode 0: the embedding of tok at pos
    const float *wte, *wpe;
    const float *gamma, *beta;
    float eps;
    int32_t E, rows, V, P;
    __nv_bfloat16 *out;             // [128][E] hi/lo B operand
    int32_t mode;                   // 0: x = wte[tok] + wpe[pos]; 1: x += sum(parts) + bias
    DeviceState *st;
};

// One CTA per row: the residual stream update, then LayerNorm ("model.fir"
// kernel g2.layernorm: mean, biased variance, (x - mean) / sqrt(var + eps) *
// gamma + beta) into the next linear's B operand.  The row stays in
// registers (E <= kLnPer * kBT) and the statistics take one block reduction:
// s and q, the sums of v - K and (v - K)^2 with K a value near the row (the
// first element of the row's previous residual, or of its embedding), give
// mean = K + s/E and var = q/E - (s/E)^2 without cancelling when the row has
// a large common offset.  The residual is stored after the reduction (K was
// read by every thread before it).
constexpr int kLnPer = 4;
__global__ void __launch_bounds__(kBT) k_b_ln(const BLnArgs a)
{
    __shared__ float red[2][kBT / 32];
    const int b = blockIdx.x, E = a.E, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // gamma, beta and the bias are weights (no kernel of the step writes
    // them): loaded before the wait for the previous kernel
    float gm[kLnPer], bt[kLnPer], bi[kLnPer];
#pragma unroll
    for (int j = 0; j < kLnPer; ++j) {
        const int i = tid + j * kBT;
        gm[j] = i < E ? a.gamma[i] : 0.f;
        bt[j] = i < E ? a.beta[i] : 0.f;
        bi[j] = i < E && a.mode != 0 ? a.bias[i] : 0.f;
    }
    pdl_wait();
    pdl_launch_dependents();   // the next kernel's CTAs may start and park on their wait
    float v[kLnPer];
    float K;
    float *xr = a.x + size_t(b) * E;
    if (a.mode == 0) {
        int t = a.tok[b], p = a.pos[b];
        if (t < 0 || t >= a.V || p >= a.P) {
            if (tid == 0 && p >= 0) record_error(a.st, t < 0 || t >= a.V ? kDevErrBadToken : kDevErrBadPosition, b);
            t = min(max(t, 0), a.V - 1);
        }
        p = min(max(p, 0), a.P - 1);
        const float *we = a.wte + size_t(t) * E, *wp = a.wpe + size_t(p) * E;
        K = we[0] + wp[0];
#pragma unroll
        for (int j = 0; j < kLnPer; ++j) {
            const int i = tid + j * kBT;
            v[j] = i < E ? we[i] + wp[i] : 0.f;
        }
    } else {
        K = xr[0];
#pragma unroll
        for (int j = 0; j < kLnPer; ++j) {
            const int i = tid + j * kBT;
            v[j] = i < E ? xr[i] + (sum_shares(a.parts, a.splits, a.rows, E, b, i) + bi[j]) : 0.f;
        }
    }
    float s = 0.f, q = 0.f;
#pragma unroll
    for (int j = 0; j < kLnPer; ++j)
        if (tid + j * kBT < E) {
            const float d = v[j] - K;
            s += d;
            q = fmaf(d, d, q);
        }
    s = warp_sum(s);
    q = warp_sum(q);
    if (lane == 0) {
        red[0][warp] = s;
        red[1][warp] = q;
    }
    __syncthreads();
    float S = 0.f, Q = 0.f;
    for (int w = 0; w < kBT / 32; ++w) {
        S += red[0][w];
        Q += red[1][w];
    }
    const float ds = S / float(E);
    const float mean = K + ds;
    const float var = fmaxf(Q / float(E) - ds * ds, 0.f);
    const float rstd = 1.0f / sqrtf(var + a.eps);
#pragma unroll
    for (int j = 0; j < kLnPer; ++j) {
        const int i = tid + j * kBT;
        if (i < E) {
            xr[i] = v[j];
            put_hi_lo(a.out, b, E, i, (v[j] - mean) * rstd * gm[j] + bt[j]);
        }
    }
}

struct BAttnArgs {
    const float *parts;             // [splits][rows][3E] QKV shares
    int32_t splits;
    const float *bias;              // [3E]
    void *kc, *vc;                  // this layer's cache: [slots][H][P][D], fp32 or bf16
    const int32_t *pos;             // [rows]; -1: inactive
    int32_t E, H, P, rows, slots;
    int32_t append;                 // 1: this row's k, v are written at pos here
    float scale;
    __nv_bfloat16 *out;             // [128][E] hi/lo B operand of the output projection
    DeviceState *st;
    const int32_t *slot_of;         // [rows] cache slot of each row, or null: slot = row (or 0, one slot)
    const int32_t *order;           // [rows] rows by decreasing position: CTA x takes row order[x]
};

__device__ __forceinline__ int row_slot(const BAttnArgs &a, int b)
{
    return a.slot_of ? a.slot_of[b] : (a.slots == 1 ? 0 : b);
}

constexpr int kAttnStageB = 16384;  // bytes per stage (64 fp32 or 128 bf16 rows of 64 dimensions)
constexpr int kAttnStages = 2;

// Dynamic shared memory of k_b_attn: the stages, then the scores [P];
// es = bytes per cache element.
__host__ __device__ constexpr size_t attn_smem(int D, int P, int es)
{
    return size_t(kAttnStages) * kAttnStageB + size_t(P) * 4;
}

// A cache element from fp32, and 4 consecutive cache elements as fp32.
__device__ __forceinline__ void kv_put(float *p, float v) { *p = v; }
__device__ __forceinline__ void kv_put(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ float kv_round(float v, const float *) { return v; }
__device__ __forceinline__ float kv_round(float v, const __nv_bfloat16 *)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float4 kv_load4(const float *row, int l)
{
    return reinterpret_cast<const float4 *>(row)[l];
}
__device__ __forceinline__ float4 kv_load4(const __nv_bfloat16 *row, int l)
{
    const uint2 u = reinterpret_cast<const uint2 *>(row)[l];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// One CTA per (row, head).  The row's cached K rows, then its V rows, stream
// through a ring of shared-memory stages by bulk copies (thread 0 refills a
// stage once every thread is done with it), so each CTA keeps kAttnStages
// copies in flight.  Scores: D/4 threads per cached row (a float4 of the
// head dimension each), shuffles within the row's threads; softmax over
// positions 0..pos (max subtracted); the weighted sum of v with the same
// thread layout, the row groups' partial sums combined in a fixed order.
// When this kernel appends (decode), row pos is this token's k, v (from the
// shares, kept in shared memory as the cache holds them) and the cache
// supplies rows 0..pos-1.  KT: the cache's element type (fp32, or bf16 with
// k and v rounded to nearest even when written).
template <int D, typename KT>
__global__ void __launch_bounds__(kBT) k_b_attn(const BAttnArgs a)
{
    constexpr int LPR = D / 4;               // threads per row
    constexpr int RPP = kBT / LPR;           // rows per pass
    constexpr uint32_t kRowB = D * sizeof(KT), kStageB = kAttnStageB;
    constexpr int kAttnRows = kStageB / kRowB;          // cache rows per stage
    constexpr int NPS = kAttnRows / RPP;     // passes per stage
    static_assert(kAttnRows % RPP == 0 && kAttnRows * kRowB == kStageB && LPR <= 32, "thread layout");
    extern __shared__ __align__(128) uint8_t dyn[];   // [stages][kAttnRows][D] KT, then scores [P] fp32
    float *sc = reinterpret_cast<float *>(dyn + size_t(kAttnStages) * kStageB);
    __shared__ __align__(8) uint64_t full[kAttnStages];
    __shared__ float red[kBT / 32];
    __shared__ __align__(16) float qkv[3 * D];
    __shared__ __align__(16) float part[RPP][D];
    const int b = a.order[blockIdx.x], h = blockIdx.y, E = a.E;
    const int tid = threadIdx.x, g = tid / LPR, l = tid % LPR;
    if (tid == 0) {
        for (int i = 0; i < kAttnStages; ++i) mbar_init(&full[i], 1);
        mbar_init_fence();
    }
    // this thread's q, k, v bias elements (weights: loaded before the wait)
    constexpr int kQ = (3 * D + kBT - 1) / kBT;
    const int nq = a.append ? 3 * D : D;
    float bq[kQ];
#pragma unroll
    for (int u = 0; u < kQ; ++u) {
        const int t = tid + u * kBT;
        bq[u] = t < nq ? a.bias[(t / D) * E + h * D + t % D] : 0.f;
    }
    // the row's position is fixed for the whole step (uploaded by the host,
    // or advanced by the last kernel of the previous step, which has finished
    // before the kernel ahead of this one started)
    const int pos = a.pos[b];
    const bool active = pos >= 0 && pos < a.P;
    const int slot = active ? row_slot(a, b) : 0;
    KT *kh = static_cast<KT *>(a.kc) + (size_t(slot) * a.H + h) * a.P * D;
    KT *vh = static_cast<KT *>(a.vc) + (size_t(slot) * a.H + h) * a.P * D;
    const int n = pos + 1;
    const int nk = a.append ? pos : n;                                   // rows read from the cache
    const int m = active ? (nk + kAttnRows - 1) / kAttnRows : 0;         // stages of K, then as many of V
    // chunk q of the stream (K chunks 0..m-1, then V chunks) into stage q % kAttnStages
    auto issue = [&](int q) {
        const bool isv = q >= m;
        const int r0 = (isv ? q - m : q) * kAttnRows, rows = min(kAttnRows, nk - r0);
        uint64_t *bar = &full[q % kAttnStages];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after the stage's generic reads
        mbar_arrive_expect_tx(bar, uint32_t(rows) * kRowB);
        bulk_g2s(dyn + size_t(q % kAttnStages) * kStageB, (isv ? vh : kh) + size_t(r0) * D, uint32_t(rows) * kRowB,
                 bar);
    };
    // decode steps (append): rows 0..pos-1 were written by earlier steps, so
    // the first copies go out before the wait and stream while the QKV linear
    // runs; a prompt step's rows come from the append kernel just before this
    // one, so its copies wait for it
    if (a.append && tid == 0)
        for (int q = 0; q < min(kAttnStages, 2 * m); ++q) issue(q);
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();   // the next kernel's CTAs may start and park on their wait
    if (!active) {             // inactive row: zero output
        for (int d = tid; d < D; d += kBT) put_hi_lo(a.out, b, E, h * D + d, 0.f);
        return;
    }
    if (!a.append && tid == 0)
        for (int q = 0; q < min(kAttnStages, 2 * m); ++q) issue(q);
    bool good = true;   // (the copies always land; a wait that runs out is recorded)
    auto wait_chunk = [&](int q) {
        if (!mbar_wait_bounded(&full[q % kAttnStages], uint32_t(q / kAttnStages) & 1u) && good) {
            good = false;
            if (l == 0) record_error(a.st, kDevErrTimeout, 14000 + b);
        }
    };
    // q, k, v from the QKV shares; k and v appended to the cache
#pragma unroll
    for (int u = 0; u < kQ; ++u) {
        const int t = tid + u * kBT;
        if (t >= nq) break;
        const int part_ = t / D, d = t % D;
        const int j = part_ * E + h * D + d;
        const float v = sum_shares(a.parts, a.splits, a.rows, 3 * E, b, j) + bq[u];
        qkv[t] = part_ == 0 ? v : kv_round(v, kh);
        if (part_ == 1) kv_put(kh + size_t(pos) * D + d, v);
        if (part_ == 2) kv_put(vh + size_t(pos) * D + d, v);
    }
    __syncthreads();
    const float4 q4 = reinterpret_cast<const float4 *>(qkv)[l];
    auto dot_row = [&](const float4 k4) {
        float d = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, q4.w * k4.w)));
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        return d;
    };
    for (int c = 0; c < m; ++c) {
        wait_chunk(c);
        const KT *stg = reinterpret_cast<const KT *>(dyn + size_t(c % kAttnStages) * kStageB);
#pragma unroll
        for (int u = 0; u < NPS; ++u) {
            const int r = u * RPP + g, j = c * kAttnRows + r;
            const float d = dot_row(kv_load4(stg + r * D, l));
            if (l == 0 && j < nk) sc[j] = d * a.scale;
        }
        __syncthreads();   // the stage is free again
        if (tid == 0 && c + kAttnStages < 2 * m) issue(c + kAttnStages);
    }
    if (a.append && tid < 32) {   // row pos: this token's k (warp 0; group 0 holds the sum)
        const float d = dot_row(reinterpret_cast<const float4 *>(qkv + D)[l]);
        if (tid == 0) sc[pos] = d * a.scale;
    }
    __syncthreads();
    float mx = -INFINITY;
    for (int j = tid; j < n; j += kBT) mx = fmaxf(mx, sc[j]);
    mx = block_max(mx, red);
    float sum = 0.f;
    for (int j = tid; j < n; j += kBT) {
        const float p = expf(sc[j] - mx);
        sc[j] = p;
        sum += p;
    }
    sum = block_sum(sum, red);   // (its barriers also publish sc)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < m; ++c) {
        const int q = m + c;
        wait_chunk(q);
        const KT *stg = reinterpret_cast<const KT *>(dyn + size_t(q % kAttnStages) * kStageB);
#pragma unroll
        for (int u = 0; u < NPS; ++u) {
            const int r = u * RPP + g, j = c * kAttnRows + r;
            if (j < nk) {
                const float p = sc[j];
                const float4 v4 = kv_load4(stg + r * D, l);
                acc.x = fmaf(p, v4.x, acc.x);
                acc.y = fmaf(p, v4.y, acc.y);
                acc.z = fmaf(p, v4.z, acc.z);
                acc.w = fmaf(p, v4.w, acc.w);
            }
        }
        __syncthreads();
        if (tid == 0 && q + kAttnStages < 2 * m) issue(q + kAttnStages);
    }
    if (a.append && g == 0) {   // row pos: this token's v
        const float p = sc[pos];
        const float4 v4 = reinterpret_cast<const float4 *>(qkv + 2 * D)[l];
        acc.x = fmaf(p, v4.x, acc.x);
        acc.y = fmaf(p, v4.y, acc.y);
        acc.z = fmaf(p, v4.z, acc.z);
        acc.w = fmaf(p, v4.w, acc.w);
    }
    reinterpret_cast<float4 *>(part[g])[l] = acc;
    __syncthreads();
    for (int d = tid; d < D; d += kBT) {
        float o = 0.f;
        for (int r = 0; r < RPP; ++r) o += part[r][d];
        put_hi_lo(a.out, b, E, h * D + d, o / sum);
    }
}

struct BGeluArgs {
    const float *parts;             // [splits][rows][F]
    int32_t splits;
    const float *bias;              // [F]
    int32_t F, rows;
    __nv_bfloat16 *out;             // [128][F]
};

__global__ void __launch_bounds__(kBT) k_b_gelu(const BGeluArgs a)
{
    const int b = blockIdx.x, f = blockIdx.y * kBT + threadIdx.x;
    const float bf = f < a.F ? a.bias[f] : 0.f;   // a weight: loaded before the wait
    pdl_wait();
    pdl_launch_dependents();   // the next kernel's CTAs may start and park on their wait
    if (f < a.F) put_hi_lo(a.out, b, a.F, f, gelu_new(sum_shares(a.parts, a.splits, a.rows, a.F, b, f) + bf));
}

// k and v of every row (QKV shares + bias) into the cache at the row's
// position, before any row's attention reads them: the rows of one step are
// then positions of sequences, consecutive within each (prompts).
template <typename KT>
__global__ void __launch_bounds__(kBT) k_b_append(const BAttnArgs a, int D)
{
    const int b = blockIdx.x, E = a.E;
    pdl_wait();
    pdl_launch_dependents();   // the next kernel's CTAs may start and park on their wait
    const int pos = a.pos[b];
    if (pos >= 0 && pos < a.P) {
        const int slot = row_slot(a, b);
        for (int t = blockIdx.y * kBT + threadIdx.x; t < 2 * E; t += gridDim.y * kBT) {
            const int part_ = 1 + t / E, hd = t % E, h = hd / D, d = hd % D, j = part_ * E + hd;
            const float v = sum_shares(a.parts, a.splits, a.rows, 3 * E, b, j) + a.bias[j];
            kv_put(static_cast<KT *>(part_ == 1 ? a.kc : a.vc) + ((size_t(slot) * a.H + h) * a.P + pos) * D + d, v);
        }
    }
}

struct BArgmaxArgs {
    const float *logits;            // [rows][V]
    int32_t V, rows, P;
    const int32_t *pos;
    int32_t *next_tok;              // [rows]
    int32_t *out_ids;               // [P][rows]: the token chosen by the pass at each position
};

__global__ void __launch_bounds__(1024) k_b_argmax(const BArgmaxArgs a)
{
    __shared__ unsigned long long keys[32];
    const int b = blockIdx.x;
    pdl_wait();
    pdl_launch_dependents();   // the next kernel's CTAs may start and park on their wait
    // kArgLoads loads in flight per thread, so a row of 50,257 logits takes
    // two rounds (the maximum of the keys does not depend on the order they
    // are taken in)
    constexpr int kArgLoads = 25;
    const float *row = a.logits + size_t(b) * a.V;
    unsigned long long best = 0ull;
    for (int i0 = threadIdx.x; i0 < a.V; i0 += kArgLoads * 1024) {
        float v[kArgLoads];
#pragma unroll
        for (int u = 0; u < kArgLoads; ++u) {
            const int i = i0 + u * 1024;
            v[u] = i < a.V ? row[i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kArgLoads; ++u) {
            const int i = i0 + u * 1024;
            if (i < a.V) {
                const unsigned long long k = argmax_key(v[u], uint32_t(i));
                best = k > best ? k : best;
            }
        }
    }
    best = warp_max_u64(best);
    if ((threadIdx.x & 31) == 0) keys[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long m = 0ull;
        for (int w = 0; w < 32; ++w) m = keys[w] > m ? keys[w] : m;
        const int p = a.pos[b];
        if (p >= 0 && p < a.P) {
            const int32_t tok = argmax_key_index(m);
            a.next_tok[b] = tok;
            a.out_ids[size_t(p) * a.rows + b] = tok;
        }
    }
}

// Feeds each active row's choice to the next step, one position further.
__global__ void k_b_advance(int32_t *tok, int32_t *pos, const int32_t *next_tok, int rows, int P, DeviceState *st)
{
    pdl_wait();
    pdl_launch_dependents();   // the next kernel's CTAs may start and park on their wait
    const int b = threadIdx.x;
    if (b < rows && pos[b] >= 0) {
        tok[b] = next_tok[b];
        pos[b] = pos[b] + 1 < P ? pos[b] + 1 : -1;   // a full cache stops the row
    }
}

// X [n][K] fp32 -> the hi/lo B operand [128][K] (stand-alone linear).
__global__ void k_b_split_rows(const float *X, int n, int K, __nv_bfloat16 *out)
{
    const int r = blockIdx.x;
    for (int i = threadIdx.x; i < K; i += blockDim.x) put_hi_lo(out, r, K, i, X[size_t(r) * K + i]);
}

// Y [n][M] = sum over splits of the shares (stand-alone linear).
__global__ void k_b_sum_splits(const float *parts, int splits, int n, int M, float *Y)
{
    const size_t total = size_t(n) * M;
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
        float s = 0.f;
        for (int k = 0; k < splits; ++k) s += parts[size_t(k) * total + i];
        Y[i] = s;
    }
}

cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// K splits of a linear (the CTAs of one cluster, at most kTcMaxSplits): as
// many CTAs as the GPU has SMs, about, each with a whole number of 64-input
// chunks and every split non-empty.
void plan_splits(int M, int K, int sms, int *splits, int *cps)
{
    const int tiles = (M + kTcM - 1) / kTcM, chunks = K / kTcK;
    // (at most ~128 CTAs: the clusters of a launch then fit the GPU at once)
    const int cap = std::min(sms, 128);
    int want = std::max(1, std::min(std::min(chunks, kTcMaxSplits), cap / std::max(1, tiles)));
    int c = (chunks + want - 1) / want;
    *cps = c;
    *splits = (chunks + c - 1) / c;
}

struct Linear {
    CUtensorMap a_map;              // the stored weights [planes][plane_rows][K] bf16
    int M, K, splits, cps, plane_rows;
};

}  // namespace

struct gpt2_batch {
    gpt2_config cfg{};
    int wdtype = GPT2_BF16;
    int max_batch = 0;              // activation rows per step
    int planes = 1;                 // bf16 planes per stored matrix (2: hi + lo of fp32 weights)
    int slots = 1;                  // cache slots: one per row (sequences), or 1 (positions of one sequence)
    bool own_cache = true;
    cudaStream_t stream = nullptr;
    int num_sms = 0;
    uint8_t *arena = nullptr;       // weights
    uint8_t *work = nullptr;        // cache, activations, shares, state
    // weights
    float *wte = nullptr, *wpe = nullptr, *lnf_w = nullptr, *lnf_b = nullptr;
    struct Layer {
        float *ln1_w, *ln1_b, *attn_b, *proj_b, *ln2_w, *ln2_b, *fc_b, *mlp_proj_b;
        void *w[4];                 // bf16 [out][in]: QKV, out-projection, fc, MLP projection
        Linear lin[4];
    };
    std::vector<Layer> layers;
    void *head = nullptr;           // bf16 planes of the head [planes][Vp][E] (rows V..Vp zero)
    Linear head_lin{};
    // work
    void *kc = nullptr, *vc = nullptr;                    // [L][slots][H][P][D] fp32, or bf16 (kv_bf16)
    bool kv_bf16 = false;
    float *x = nullptr;                                   // [64][E]
    __nv_bfloat16 *b_e = nullptr, *b_a = nullptr, *b_f = nullptr;   // [128][E], [128][E], [128][F]
    CUtensorMap map_e{}, map_a{}, map_f{};
    float *p_qkv = nullptr, *p_o = nullptr, *p_fc = nullptr, *p_p = nullptr;   // K-split shares
    float *logits = nullptr;                                                  // [rows][V]
    int32_t *tok = nullptr, *pos = nullptr, *next_tok = nullptr, *out_ids = nullptr;
    DeviceState *st = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int kernels_per_step = 0;
    cudaGraph_t graph_p = nullptr;  // prompt steps of a batched model (packed rows)
    cudaGraphExec_t exec_p = nullptr;
    int kernels_per_prompt_step = 0;
    int32_t *slot_of = nullptr;     // [kTcMaxRows] cache slot of each row in a prompt step
    int32_t *order = nullptr;       // [kTcMaxRows] rows by decreasing position (the attention's CTA order)
    std::vector<int> cached;        // host view: cached length of each sequence
    bool has_step = false;
    unsigned long long launches = 0;
    unsigned long long wait_ns = kWaitLimitNs;
};

namespace {

int cuda_rc(cudaError_t e)
{
    if (e == cudaSuccess) return GPT2_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? GPT2_ERR_OUT_OF_MEMORY : GPT2_ERR_CUDA;
}
#define BTRY(expr)                                   \
    do {                                             \
        cudaError_t _e = (expr);                     \
        if (_e != cudaSuccess) return cuda_rc(_e);   \
    } while (0)

size_t a256(size_t v) { return (v + 255) / 256 * 256; }

bool dev_ptr(const void *p)
{
    if (!p) return false;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

cudaError_t run_linear(const gpt2_batch *m, const Linear &L, const CUtensorMap &b_map, float *parts, cudaStream_t s,
                       bool pdl)
{
    TcGemmArgs a;
    a.M = L.M;
    a.K = L.K;
    a.n_rows = m->max_batch;
    a.a_planes = m->planes;
    a.a_plane_rows = L.plane_rows;
    a.chunks_per_split = L.cps;
    a.partials = parts;
    a.st = m->st;
    a.wait_ns = m->wait_ns;
    return tc_gemm_launch(L.a_map, b_map, a, L.splits, s, pdl);
}

const void *attn_kernel(int D, bool bf16)
{
    if (bf16)
        return D == 32 ? reinterpret_cast<const void *>(k_b_attn<32, __nv_bfloat16>)
               : D == 64 ? reinterpret_cast<const void *>(k_b_attn<64, __nv_bfloat16>)
                         : reinterpret_cast<const void *>(k_b_attn<128, __nv_bfloat16>);
    return D == 32 ? reinterpret_cast<const void *>(k_b_attn<32, float>)
           : D == 64 ? reinterpret_cast<const void *>(k_b_attn<64, float>)
                     : reinterpret_cast<const void *>(k_b_attn<128, float>);
}

// Records one batched step on stream s (under capture).
// packed: a prompt step of the batched model: rows are (sequence, position)
// pairs (slot_of), every row's k, v appended first; only the blocks run (the
// cache is what a prompt step is for: no head, no choice).
int record_step(gpt2_batch *m, cudaStream_t s, bool packed = false)
{
    const gpt2_config &c = m->cfg;
    const int E = c.n_embd, H = c.n_head, D = E / H, F = 4 * E, R = m->max_batch, P = c.n_positions;
    const int V = c.vocab_size, L = c.n_layer, slots = m->slots;
    int kernels = 0;
    bool first = true;
    auto pdl = [&]() {
        const bool p = !first;
        first = false;
        return p;
    };
    const size_t ln_smem = 0;
    for (int l = 0; l < L; ++l) {
        const gpt2_batch::Layer &Ly = m->layers[l];
        BLnArgs ln{};
        ln.x = m->x;
        ln.E = E;
        ln.rows = R;
        ln.V = V;
        ln.P = P;
        ln.eps = c.ln_eps;
        ln.st = m->st;
        ln.out = m->b_e;
        ln.gamma = Ly.ln1_w;
        ln.beta = Ly.ln1_b;
        ln.tok = m->tok;
        ln.pos = m->pos;
        ln.wte = m->wte;
        ln.wpe = m->wpe;
        if (l == 0) {
            ln.mode = 0;
        } else {
            ln.mode = 1;
            ln.parts = m->p_p;
            ln.splits = m->layers[l - 1].lin[3].splits;
            ln.bias = m->layers[l - 1].mlp_proj_b;
        }
        void *a1[] = {&ln};
        BTRY(launch_pdl(reinterpret_cast<const void *>(k_b_ln), dim3(R), dim3(kBT), ln_smem, s, pdl(), a1));
        BTRY(run_linear(m, Ly.lin[0], m->map_e, m->p_qkv, s, pdl()));
        BAttnArgs at{};
        at.parts = m->p_qkv;
        at.splits = Ly.lin[0].splits;
        at.bias = Ly.attn_b;
        const size_t layer_bytes = size_t(slots) * H * P * D * (m->kv_bf16 ? 2 : 4);
        at.kc = static_cast<uint8_t *>(m->kc) + size_t(l) * layer_bytes;
        at.vc = static_cast<uint8_t *>(m->vc) + size_t(l) * layer_bytes;
        at.pos = m->pos;
        at.E = E;
        at.H = H;
        at.P = P;
        at.rows = R;
        at.slots = slots;
        const bool pre = slots == 1 || packed;   // rows of prompts: every row's k, v first (k_b_append)
        at.append = pre ? 0 : 1;
        at.slot_of = packed ? m->slot_of : nullptr;
        at.order = m->order;
        at.scale = float(1.0 / std::sqrt(double(D)));
        at.out = m->b_a;
        at.st = m->st;
        if (pre) {
            int dd = D;
            void *ap[] = {&at, &dd};
            const void *fn = m->kv_bf16 ? reinterpret_cast<const void *>(k_b_append<__nv_bfloat16>)
                                        : reinterpret_cast<const void *>(k_b_append<float>);
            BTRY(launch_pdl(fn, dim3(R, 2), dim3(kBT), 0, s, pdl(), ap));
            ++kernels;
        }
        void *a2[] = {&at};
        BTRY(launch_pdl(attn_kernel(D, m->kv_bf16), dim3(R, H), dim3(kBT), attn_smem(D, P, m->kv_bf16 ? 2 : 4), s,
                        pdl(), a2));
        BTRY(run_linear(m, Ly.lin[1], m->map_a, m->p_o, s, pdl()));
        ln.mode = 1;
        ln.parts = m->p_o;
        ln.splits = Ly.lin[1].splits;
        ln.bias = Ly.proj_b;
        ln.gamma = Ly.ln2_w;
        ln.beta = Ly.ln2_b;
        void *a3[] = {&ln};
        BTRY(launch_pdl(reinterpret_cast<const void *>(k_b_ln), dim3(R), dim3(kBT), ln_smem, s, pdl(), a3));
        BTRY(run_linear(m, Ly.lin[2], m->map_e, m->p_fc, s, pdl()));
        BGeluArgs ge{};
        ge.parts = m->p_fc;
        ge.splits = Ly.lin[2].splits;
        ge.bias = Ly.fc_b;
        ge.F = F;
        ge.rows = R;
        ge.out = m->b_f;
        void *a4[] = {&ge};
        BTRY(launch_pdl(reinterpret_cast<const void *>(k_b_gelu), dim3(R, (F + kBT - 1) / kBT), dim3(kBT), 0, s,
                        pdl(), a4));
        BTRY(run_linear(m, Ly.lin[3], m->map_f, m->p_p, s, pdl()));
        kernels += 8;
    }
    if (packed) {
        m->kernels_per_prompt_step = kernels;
        return GPT2_OK;
    }
    BLnArgs ln{};
    ln.x = m->x;
    ln.E = E;
    ln.rows = R;
    ln.V = V;
    ln.P = P;
    ln.eps = c.ln_eps;
    ln.st = m->st;
    ln.out = m->b_e;
    ln.mode = 1;
    ln.parts = m->p_p;
    ln.splits = m->layers[L - 1].lin[3].splits;
    ln.bias = m->layers[L - 1].mlp_proj_b;
    ln.gamma = m->lnf_w;
    ln.beta = m->lnf_b;
    void *a5[] = {&ln};
    BTRY(launch_pdl(reinterpret_cast<const void *>(k_b_ln), dim3(R), dim3(kBT), ln_smem, s, pdl(), a5));
    BTRY(run_linear(m, m->head_lin, m->map_e, m->logits, s, pdl()));
    BArgmaxArgs am{};
    am.logits = m->logits;
    am.V = V;
    am.rows = R;
    am.P = P;
    am.pos = m->pos;
    am.next_tok = m->next_tok;
    am.out_ids = m->out_ids;
    void *a6[] = {&am};
    BTRY(launch_pdl(reinterpret_cast<const void *>(k_b_argmax), dim3(R), dim3(1024), 0, s, pdl(), a6));
    int32_t *tk = m->tok, *ps = m->pos;
    const int32_t *nt = m->next_tok;
    int rows = R, pp = P;
    DeviceState *st = m->st;
    void *a7[] = {&tk, &ps, &nt, &rows, &pp, &st};
    BTRY(launch_pdl(reinterpret_cast<const void *>(k_b_advance), dim3(1), dim3(kTcMaxRows), 0, s, pdl(), a7));
    m->kernels_per_step = kernels + 4;   // + final LayerNorm, head, argmax, advance
    return GPT2_OK;
}

int capture_step(gpt2_batch *m, bool packed, cudaGraph_t *graph, cudaGraphExec_t *exec)
{
    cudaStream_t cs;
    BTRY(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(cs);
        return cuda_rc(e);
    }
    const int rc = record_step(m, cs, packed);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (rc != GPT2_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return cuda_rc(e);
    *graph = g;
    BTRY(cudaGraphInstantiate(exec, g, 0));
    return GPT2_OK;
}

// The decode step's graph, and for a batched model (one cache slot per
// sequence) the prompt step's.
int build_step_graph(gpt2_batch *m)
{
    int rc = capture_step(m, false, &m->graph, &m->exec);
    if (rc == GPT2_OK && m->slots > 1) rc = capture_step(m, true, &m->graph_p, &m->exec_p);
    return rc;
}

void free_batch(gpt2_batch *m)
{
    if (!m) return;
    if (m->exec) cudaGraphExecDestroy(m->exec);
    if (m->graph) cudaGraphDestroy(m->graph);
    if (m->exec_p) cudaGraphExecDestroy(m->exec_p);
    if (m->graph_p) cudaGraphDestroy(m->graph_p);
    if (m->arena) cudaFree(m->arena);
    if (m->work) cudaFree(m->work);
    delete m;
}

int read_batch_state(gpt2_batch *m)
{
    BTRY(cudaStreamSynchronize(m->stream));
    DeviceState hs;
    BTRY(cudaMemcpy(&hs, m->st, sizeof hs, cudaMemcpyDeviceToHost));
    if (hs.err != kDevErrNone) {
        BTRY(cudaMemset(&m->st->err, 0, 3 * sizeof(int32_t)));
        return hs.err == kDevErrTimeout ? GPT2_ERR_TIMEOUT : GPT2_ERR_DEVICE_STATE;
    }
    return GPT2_OK;
}

int set_linear(Linear &L, const void *w, int M, int K, int sms, int planes = 1, int plane_rows = 0)
{
    L.M = M;
    L.K = K;
    L.plane_rows = plane_rows > 0 ? plane_rows : M;
    plan_splits(M, K, sms, &L.splits, &L.cps);
    return tc_make_tmap(&L.a_map, w, uint64_t(L.plane_rows) * planes, uint64_t(K)) == 0 ? GPT2_OK : GPT2_ERR_CUDA;
}

// What an engine is built from (device pointers, read during the build only
// unless stated).  The block matrices come either in the checkpoint's HF
// [in][out] layout (hf = true) or as fp32 [out][in] (hf = false); a head
// source of [V][E].  borrow: wte and wpe are used in place for the embedding
// (their owner keeps them alive); kc, vc: an external cache (else own).
struct EngineSrc {
    const float *wte, *wpe, *lnf_w, *lnf_b, *head;
    struct Layer {
        const float *p[8];   // ln1_w, ln1_b, attn_b, proj_b, ln2_w, ln2_b, fc_b, mlp_proj_b
        const float *w[4];   // QKV, out-projection, fc, MLP projection
    };
    std::vector<Layer> layers;
    bool hf = true;
    bool borrow = false;
    float *kc = nullptr, *vc = nullptr;   // an fp32 cache of the caller's
    bool kv_bf16 = false;                 // an own cache of bf16 k, v (RNE)
    int planes = 1, slots = 1, rows = kTcMaxRows;
    // in place of w[] / head: write the fp32 [out][in] matrix (or the [V][E]
    // head) into dst
    std::function<cudaError_t(int, int, float *, cudaStream_t)> matrix;
    std::function<cudaError_t(float *, cudaStream_t)> head_fn;
};

// The attention's CTA order for a step's positions pos[kTcMaxRows]: rows by
// decreasing position (inactive rows, -1, last; ties by row), so that the
// longest rows start first and every SM gets a mix of lengths.
cudaError_t upload_order(gpt2_batch *m, const int32_t *pos, cudaStream_t s)
{
    int32_t ord[kTcMaxRows];
    for (int r = 0; r < kTcMaxRows; ++r) ord[r] = r;
    std::stable_sort(ord, ord + kTcMaxRows, [&](int x, int y) { return pos[x] > pos[y]; });
    return cudaMemcpyAsync(m->order, ord, sizeof ord, cudaMemcpyHostToDevice, s);
}

int engine_build(gpt2_batch *m, const gpt2_config &cfg, const EngineSrc &src, cudaStream_t stream, int sms)
{
    const int L = cfg.n_layer, E = cfg.n_embd, H = cfg.n_head, P = cfg.n_positions, V = cfg.vocab_size;
    const int D = E / H, F = 4 * E;
    BTRY(tc_gemm_init());
    {
        const bool kb = src.kv_bf16 && src.kc == nullptr;
        BTRY(cudaFuncSetAttribute(attn_kernel(D, kb), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(attn_smem(D, P, kb ? 2 : 4))));
    }
    m->cfg = cfg;
    m->max_batch = src.rows;
    m->planes = src.planes;
    m->slots = src.slots;
    m->own_cache = src.kc == nullptr;
    m->kv_bf16 = src.kv_bf16 && m->own_cache;
    m->stream = stream;
    m->num_sms = sms;
    m->cached.assign(src.rows, 0);
    const int mat_in[4] = {E, E, E, F}, mat_out[4] = {3 * E, E, F, E};
    const int pl = src.planes;
    // rows of one plane: a multiple of the tile height when there are two
    // planes (a tile never reads into the next plane; padding rows are zero)
    auto plane_rows = [&](int M) { return pl > 1 ? (M + kTcM - 1) / kTcM * kTcM : M; };
    const int Vp = plane_rows(V);
    // ---- weights ----
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += a256(bytes);
        return o;
    };
    const size_t o_wte = src.borrow ? 0 : take(size_t(V) * E * 4), o_wpe = src.borrow ? 0 : take(size_t(P) * E * 4);
    const size_t o_lnf_w = take(size_t(E) * 4), o_lnf_b = take(size_t(E) * 4);
    const size_t o_head = take(size_t(pl) * Vp * E * 2);
    struct LO {
        size_t p[8], w[4];
    };
    std::vector<LO> lo(L);
    const int psz[8] = {E, E, 3 * E, E, E, E, F, E};
    for (int l = 0; l < L; ++l) {
        for (int k = 0; k < 8; ++k) lo[l].p[k] = take(size_t(psz[k]) * 4);
        for (int k = 0; k < 4; ++k) lo[l].w[k] = take(size_t(pl) * plane_rows(mat_out[k]) * mat_in[k] * 2);
    }
    const size_t arena_bytes = off;
    // ---- work ----
    off = 0;
    const size_t kv = m->own_cache ? size_t(L) * src.slots * H * P * D * (m->kv_bf16 ? 2 : 4) : 0;
    const size_t o_k = m->own_cache ? take(kv) : 0, o_v = m->own_cache ? take(kv) : 0;
    const size_t o_x = take(size_t(kTcMaxRows) * E * 4);
    const size_t o_be = take(size_t(2 * kTcMaxRows) * E * 2), o_ba = take(size_t(2 * kTcMaxRows) * E * 2);
    const size_t o_bf = take(size_t(2 * kTcMaxRows) * F * 2);
    int sp[4], cps[4];
    for (int k = 0; k < 4; ++k) plan_splits(mat_out[k], mat_in[k], sms, &sp[k], &cps[k]);
    const size_t o_pq = take(size_t(sp[0]) * src.rows * 3 * E * 4), o_po = take(size_t(sp[1]) * src.rows * E * 4);
    const size_t o_pf = take(size_t(sp[2]) * src.rows * F * 4), o_pp = take(size_t(sp[3]) * src.rows * E * 4);
    const size_t o_lg = take(size_t(src.rows) * V * 4);
    const size_t o_tok = take(size_t(kTcMaxRows) * 4), o_pos = take(size_t(kTcMaxRows) * 4);
    const size_t o_nt = take(size_t(kTcMaxRows) * 4), o_ids = take(size_t(P) * src.rows * 4);
    const size_t o_slot = take(size_t(kTcMaxRows) * 4), o_order = take(size_t(kTcMaxRows) * 4);
    const size_t o_st = take(sizeof(DeviceState));
    const size_t work_bytes = off;
    const size_t tmp_elems = size_t(F) * E > size_t(Vp) * E ? size_t(F) * E : size_t(Vp) * E;
    float *tmp = nullptr;
    cudaError_t e = cudaMalloc(&m->arena, arena_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&m->work, work_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&tmp, tmp_elems * 4);
    if (e != cudaSuccess) {
        if (tmp) cudaFree(tmp);
        return cuda_rc(e);
    }
    uint8_t *A = m->arena, *W = m->work;
    cudaStream_t s = stream;
    // the bf16 planes of one fp32 [rows][K] matrix (rows of each plane padded
    // to prow, padding zero)
    auto planes_of = [&](const float *w_oi, int rows, int K, int prow, void *dst) -> cudaError_t {
        __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(dst);
        cudaError_t r = cudaSuccess;
        if (prow > rows) r = cudaMemsetAsync(d, 0, size_t(pl) * prow * K * 2, s);
        if (r == cudaSuccess)
            r = split_bf16(w_oi, size_t(rows) * K, d, pl > 1 ? d + size_t(prow) * K : nullptr, s);
        return r;
    };
    int rc = GPT2_OK;
#define ECK(expr)                        \
    do {                                 \
        cudaError_t _e2 = (expr);        \
        if (_e2 != cudaSuccess) {        \
            rc = cuda_rc(_e2);           \
            goto done;                   \
        }                                \
    } while (0)
    ECK(cudaMemsetAsync(m->work, 0, work_bytes, s));
    if (src.borrow) {
        m->wte = const_cast<float *>(src.wte);
        m->wpe = const_cast<float *>(src.wpe);
    } else {
        m->wte = reinterpret_cast<float *>(A + o_wte);
        m->wpe = reinterpret_cast<float *>(A + o_wpe);
        ECK(cudaMemcpyAsync(m->wte, src.wte, size_t(V) * E * 4, cudaMemcpyDeviceToDevice, s));
        ECK(cudaMemcpyAsync(m->wpe, src.wpe, size_t(P) * E * 4, cudaMemcpyDeviceToDevice, s));
    }
    m->lnf_w = reinterpret_cast<float *>(A + o_lnf_w);
    m->lnf_b = reinterpret_cast<float *>(A + o_lnf_b);
    ECK(cudaMemcpyAsync(m->lnf_w, src.lnf_w, size_t(E) * 4, cudaMemcpyDeviceToDevice, s));
    ECK(cudaMemcpyAsync(m->lnf_b, src.lnf_b, size_t(E) * 4, cudaMemcpyDeviceToDevice, s));
    m->head = A + o_head;
    if (src.head_fn) {
        ECK(src.head_fn(tmp, s));
        ECK(planes_of(tmp, V, E, Vp, m->head));
        ECK(cudaStreamSynchronize(s));
    } else {
        ECK(planes_of(src.head, V, E, Vp, m->head));   // the embedding reads the fp32 wte
    }
    m->layers.resize(L);
    for (int l = 0; l < L; ++l) {
        const EngineSrc::Layer &sl = src.layers[l];
        gpt2_batch::Layer &d = m->layers[l];
        float **pp[8] = {&d.ln1_w, &d.ln1_b, &d.attn_b, &d.proj_b, &d.ln2_w, &d.ln2_b, &d.fc_b, &d.mlp_proj_b};
        for (int k = 0; k < 8; ++k) {
            *pp[k] = reinterpret_cast<float *>(A + lo[l].p[k]);
            ECK(cudaMemcpyAsync(*pp[k], sl.p[k], size_t(psz[k]) * 4, cudaMemcpyDeviceToDevice, s));
        }
        for (int k = 0; k < 4; ++k) {
            d.w[k] = A + lo[l].w[k];
            const float *w_oi = sl.w[k];
            if (src.matrix) {
                ECK(src.matrix(l, k, tmp, s));
                w_oi = tmp;
            } else if (src.hf) {   // [in][out] -> [out][in]
                ECK(repack_f32(sl.w[k], mat_in[k], mat_out[k], tmp, s));
                w_oi = tmp;
            }
            ECK(planes_of(w_oi, mat_out[k], mat_in[k], plane_rows(mat_out[k]), d.w[k]));
            ECK(cudaStreamSynchronize(s));   // tmp is reused
            rc = set_linear(d.lin[k], d.w[k], mat_out[k], mat_in[k], sms, pl, plane_rows(mat_out[k]));
            if (rc != GPT2_OK) goto done;
        }
    }
    rc = set_linear(m->head_lin, m->head, V, E, sms, pl, Vp);
    if (rc != GPT2_OK) goto done;
    m->head_lin.splits = 1;                       // whole logits from one pass over K
    m->head_lin.cps = E / kTcK;
    m->kc = m->own_cache ? static_cast<void *>(W + o_k) : static_cast<void *>(src.kc);
    m->vc = m->own_cache ? static_cast<void *>(W + o_v) : static_cast<void *>(src.vc);
    m->x = reinterpret_cast<float *>(W + o_x);
    m->b_e = reinterpret_cast<__nv_bfloat16 *>(W + o_be);
    m->b_a = reinterpret_cast<__nv_bfloat16 *>(W + o_ba);
    m->b_f = reinterpret_cast<__nv_bfloat16 *>(W + o_bf);
    m->p_qkv = reinterpret_cast<float *>(W + o_pq);
    m->p_o = reinterpret_cast<float *>(W + o_po);
    m->p_fc = reinterpret_cast<float *>(W + o_pf);
    m->p_p = reinterpret_cast<float *>(W + o_pp);
    m->logits = reinterpret_cast<float *>(W + o_lg);
    m->tok = reinterpret_cast<int32_t *>(W + o_tok);
    m->pos = reinterpret_cast<int32_t *>(W + o_pos);
    m->next_tok = reinterpret_cast<int32_t *>(W + o_nt);
    m->out_ids = reinterpret_cast<int32_t *>(W + o_ids);
    m->slot_of = reinterpret_cast<int32_t *>(W + o_slot);
    m->order = reinterpret_cast<int32_t *>(W + o_order);
    m->st = reinterpret_cast<DeviceState *>(W + o_st);
    if (tc_make_tmap(&m->map_e, m->b_e, 2 * kTcMaxRows, uint64_t(E)) ||
        tc_make_tmap(&m->map_a, m->b_a, 2 * kTcMaxRows, uint64_t(E)) ||
        tc_make_tmap(&m->map_f, m->b_f, 2 * kTcMaxRows, uint64_t(F))) {
        rc = GPT2_ERR_CUDA;
        goto done;
    }
    {
        std::vector<int32_t> neg(kTcMaxRows, -1);   // every row inactive until a call feeds it
        ECK(cudaMemcpyAsync(m->pos, neg.data(), neg.size() * 4, cudaMemcpyHostToDevice, s));
        ECK(upload_order(m, neg.data(), s));
        ECK(cudaStreamSynchronize(s));
    }
    rc = build_step_graph(m);
done:
    cudaStreamSynchronize(s);
    cudaFree(tmp);
    return rc;
#undef ECK
}

// Shape checks common to every engine.
int engine_shape_ok(const gpt2_config *cfg)
{
    const int L = cfg->n_layer, E = cfg->n_embd, H = cfg->n_head, P = cfg->n_positions, V = cfg->vocab_size;
    if (L < 1 || H < 1 || P < 1 || V < 1 || E < 64 || E % 64 || E % H) return GPT2_ERR_INVALID_ARG;
    if (E > kLnPer * kBT) return GPT2_ERR_INVALID_ARG;   // a LayerNorm row in one CTA's registers
    const int D = E / H;
    if (D != 32 && D != 64 && D != 128) return GPT2_ERR_INVALID_ARG;
    if (!(cfg->ln_eps > 0.f) || !std::isfinite(cfg->ln_eps)) return GPT2_ERR_INVALID_ARG;
    if ((long long)V * E > (1ll << 31) - 1 || (long long)P * 4 > 48 * 1024) return GPT2_ERR_INVALID_ARG;
    return GPT2_OK;
}

// The single model's device state after a prefill through the engine (what
// its own prefill leaves): the choice after the last position is the next
// token, appended to the generated ids.
__global__ void k_seed_after_prefill(const int32_t *next_tok, int row, DeviceState *st, int32_t *out_ids,
                                     int out_cap, int n)
{
    const int32_t tok = next_tok[row];
    st->next_tok = tok;
    st->tok = tok;
    st->pos = n;
    const int32_t k = st->n_out;
    if (out_ids && k >= 0 && k < out_cap) out_ids[k] = tok;
    st->n_out = k + 1;
}

}  // namespace

namespace gpt2 {

int prefill_engine_create(const gpt2_config &cfg, const PrefillSrc &ps, cudaStream_t s, int sms, gpt2_batch **out)
{
    *out = nullptr;
    int rc = engine_shape_ok(&cfg);
    if (rc != GPT2_OK) return rc;
    EngineSrc src;
    src.wte = ps.wte;
    src.wpe = ps.wpe;
    src.lnf_w = ps.lnf_w;
    src.lnf_b = ps.lnf_b;
    src.head = nullptr;
    src.head_fn = ps.head;
    src.matrix = ps.matrix;
    src.layers.resize(cfg.n_layer);
    for (int l = 0; l < cfg.n_layer; ++l)
        for (int k = 0; k < 8; ++k) src.layers[l].p[k] = ps.params[l * 8 + k];
    src.hf = false;
    src.borrow = true;
    src.kc = ps.kc;
    src.vc = ps.vc;
    src.planes = 2;
    src.slots = 1;
    src.rows = kTcMaxRows;
    gpt2_batch *e = new (std::nothrow) gpt2_batch();
    if (!e) return GPT2_ERR_OUT_OF_MEMORY;
    rc = engine_build(e, cfg, src, s, sms);
    if (rc != GPT2_OK) {
        free_batch(e);
        return rc;
    }
    *out = e;
    return GPT2_OK;
}

int prefill_engine_run(gpt2_batch *e, const int32_t *ids, int n, DeviceState *st, int32_t *out_ids, int out_cap,
                       float *logits, cudaStream_t s, unsigned long long *launches)
{
    if (!e || n < 1 || n > e->cfg.n_positions) return GPT2_ERR_INVALID_ARG;
    std::vector<int32_t> t(kTcMaxRows), p(kTcMaxRows);
    int last = 0;
    for (int c0 = 0; c0 < n; c0 += kTcMaxRows) {
        const int rows = std::min(kTcMaxRows, n - c0);
        for (int r = 0; r < kTcMaxRows; ++r) {
            t[r] = r < rows ? ids[c0 + r] : 0;
            p[r] = r < rows ? c0 + r : -1;
        }
        BTRY(cudaMemcpyAsync(e->tok, t.data(), t.size() * 4, cudaMemcpyHostToDevice, s));
        BTRY(cudaMemcpyAsync(e->pos, p.data(), p.size() * 4, cudaMemcpyHostToDevice, s));
        BTRY(upload_order(e, p.data(), s));
        BTRY(cudaGraphLaunch(e->exec, s));
        e->launches += e->kernels_per_step;
        if (launches) *launches += e->kernels_per_step;
        last = rows - 1;
    }
    k_seed_after_prefill<<<1, 1, 0, s>>>(e->next_tok, last, st, out_ids, out_cap, n);
    BTRY(cudaGetLastError());
    if (launches) *launches += 1;
    BTRY(cudaMemcpyAsync(logits, e->logits + size_t(last) * e->cfg.vocab_size, size_t(e->cfg.vocab_size) * 4,
                         cudaMemcpyDeviceToDevice, s));
    return GPT2_OK;
}

void prefill_engine_destroy(gpt2_batch *e) { free_batch(e); }

}  // namespace gpt2

extern "C" {

int gpt2_create_batch(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype, int32_t max_batch, void *stream,
                      gpt2_batch **out)
{
    return gpt2_create_batch_ex(cfg, w, wdtype, max_batch, 0u, stream, out);
}

int gpt2_create_batch_ex(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype, int32_t max_batch,
                         uint32_t flags, void *stream, gpt2_batch **out)
{
    if (!out) return GPT2_ERR_INVALID_ARG;
    *out = nullptr;
    if (flags & ~uint32_t(GPT2_BATCH_KV_BF16)) return GPT2_ERR_INVALID_ARG;
    if (!cfg || !w || !w->layers) return GPT2_ERR_INVALID_ARG;
    if (wdtype != GPT2_BF16) return GPT2_ERR_INVALID_ARG;
    if (max_batch < 1 || max_batch > kTcMaxRows) return GPT2_ERR_INVALID_ARG;
    int rc = engine_shape_ok(cfg);
    if (rc != GPT2_OK) return rc;
    int dev;
    BTRY(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    BTRY(cudaGetDeviceProperties(&prop, dev));
    if (!(prop.major == 10 && prop.minor == 3)) return GPT2_ERR_UNSUPPORTED_DEVICE;
    const float *top[4] = {w->wte, w->wpe, w->ln_f_w, w->ln_f_b};
    for (const float *p : top)
        if (!dev_ptr(p)) return GPT2_ERR_INVALID_ARG;
    EngineSrc src;
    src.wte = w->wte;
    src.wpe = w->wpe;
    src.lnf_w = w->ln_f_w;
    src.lnf_b = w->ln_f_b;
    src.head = w->wte;                // the tied head, stored as its bf16 copy
    src.layers.resize(cfg->n_layer);
    for (int l = 0; l < cfg->n_layer; ++l) {
        const gpt2_layer_weights &Lw = w->layers[l];
        const float *ps[12] = {Lw.ln1_w, Lw.ln1_b, Lw.attn_w, Lw.attn_b, Lw.proj_w, Lw.proj_b,
                               Lw.ln2_w, Lw.ln2_b, Lw.fc_w,   Lw.fc_b,   Lw.mlp_proj_w, Lw.mlp_proj_b};
        for (const float *p : ps)
            if (!dev_ptr(p)) return GPT2_ERR_INVALID_ARG;
        EngineSrc::Layer &sl = src.layers[l];
        const float *pv[8] = {Lw.ln1_w, Lw.ln1_b, Lw.attn_b, Lw.proj_b, Lw.ln2_w, Lw.ln2_b, Lw.fc_b, Lw.mlp_proj_b};
        for (int k = 0; k < 8; ++k) sl.p[k] = pv[k];
        sl.w[0] = Lw.attn_w;
        sl.w[1] = Lw.proj_w;
        sl.w[2] = Lw.fc_w;
        sl.w[3] = Lw.mlp_proj_w;
    }
    src.hf = true;
    src.planes = 1;
    src.slots = max_batch;
    src.rows = max_batch;
    src.kv_bf16 = (flags & GPT2_BATCH_KV_BF16) != 0;
    gpt2_batch *m = new (std::nothrow) gpt2_batch();
    if (!m) return GPT2_ERR_OUT_OF_MEMORY;
    rc = engine_build(m, *cfg, src, static_cast<cudaStream_t>(stream), prop.multiProcessorCount);
    if (rc != GPT2_OK) {
        free_batch(m);
        return rc;
    }
    *out = m;
    return GPT2_OK;
}

void gpt2_destroy_batch(gpt2_batch *m)
{
    if (!m) return;
    cudaStreamSynchronize(m->stream);
    free_batch(m);
}

int gpt2_decode_batch(gpt2_batch *m, const int32_t *tokens, const int32_t *positions, int32_t n,
                      const float **dev_logits)
{
    if (!m || !tokens || !positions || n < 1 || n > m->max_batch) return GPT2_ERR_INVALID_ARG;
    const gpt2_config &c = m->cfg;
    std::vector<int32_t> t(kTcMaxRows, 0), p(kTcMaxRows, -1);
    for (int b = 0; b < n; ++b) {
        if (positions[b] == -1) continue;          // this sequence sits the step out
        if (tokens[b] < 0 || tokens[b] >= c.vocab_size) return GPT2_ERR_TOKEN_RANGE;
        if (positions[b] < 0 || positions[b] >= c.n_positions || positions[b] > m->cached[b])
            return GPT2_ERR_POSITION_RANGE;
        t[b] = tokens[b];
        p[b] = positions[b];
    }
    BTRY(cudaMemcpyAsync(m->tok, t.data(), t.size() * 4, cudaMemcpyHostToDevice, m->stream));
    BTRY(cudaMemcpyAsync(m->pos, p.data(), p.size() * 4, cudaMemcpyHostToDevice, m->stream));
    BTRY(upload_order(m, p.data(), m->stream));
    BTRY(cudaGraphLaunch(m->exec, m->stream));
    m->launches += m->kernels_per_step;
    for (int b = 0; b < n; ++b)
        if (p[b] >= 0) m->cached[b] = p[b] + 1;
    m->has_step = true;
    if (dev_logits) *dev_logits = m->logits;
    return GPT2_OK;
}

int gpt2_prefill_batch(gpt2_batch *m, const int32_t *ids, const int32_t *lens, int32_t n)
{
    if (!m || !ids || !lens || n < 1 || n > m->max_batch) return GPT2_ERR_INVALID_ARG;
    size_t total = 0;
    for (int b = 0; b < n; ++b) {
        if (lens[b] < 1 || lens[b] > m->cfg.n_positions) return GPT2_ERR_POSITION_RANGE;
        total += size_t(lens[b]);
    }
    for (size_t i = 0; i < total; ++i)
        if (ids[i] < 0 || ids[i] >= m->cfg.vocab_size) return GPT2_ERR_TOKEN_RANGE;
    std::fill(m->cached.begin(), m->cached.end(), 0);
    std::vector<size_t> start(n, 0);
    for (int b = 1; b < n; ++b) start[b] = start[b - 1] + size_t(lens[b - 1]);
    // prompt steps: every position but each sequence's last, max_batch rows
    // per step (the rows a step's kernels process) taken sequence by sequence
    // (a sequence's rows in a step are consecutive positions; the step appends
    // all their k, v before any attention reads the cache)
    std::vector<int32_t> t(kTcMaxRows), p(kTcMaxRows), sl(kTcMaxRows);
    const int rows = m->max_batch;
    int r = 0;
    auto flush = [&]() -> int {
        if (r == 0) return GPT2_OK;
        for (int i = r; i < kTcMaxRows; ++i) {
            t[i] = 0;
            p[i] = -1;
            sl[i] = 0;
        }
        BTRY(cudaMemcpyAsync(m->tok, t.data(), t.size() * 4, cudaMemcpyHostToDevice, m->stream));
        BTRY(cudaMemcpyAsync(m->pos, p.data(), p.size() * 4, cudaMemcpyHostToDevice, m->stream));
        BTRY(cudaMemcpyAsync(m->slot_of, sl.data(), sl.size() * 4, cudaMemcpyHostToDevice, m->stream));
        BTRY(upload_order(m, p.data(), m->stream));
        BTRY(cudaGraphLaunch(m->exec_p, m->stream));
        m->launches += m->kernels_per_prompt_step;
        r = 0;
        return GPT2_OK;
    };
    if (!m->exec_p) {
        // a model of one sequence (no prompt-step graph): a decode step per position
        for (int q = 0; q + 1 < lens[0]; ++q) {
            const int32_t tq = ids[q], pq = q;
            m->cached[0] = q;
            const int rc = gpt2_decode_batch(m, &tq, &pq, 1, nullptr);
            if (rc != GPT2_OK) return rc;
        }
    } else {
        for (int b = 0; b < n; ++b)
            for (int q = 0; q + 1 < lens[b]; ++q) {
                t[r] = ids[start[b] + q];
                p[r] = q;
                sl[r] = b;
                if (++r == rows) {
                    const int rc = flush();
                    if (rc != GPT2_OK) return rc;
                }
            }
        const int rc = flush();
        if (rc != GPT2_OK) return rc;
    }
    // each sequence's last prompt token: one decode step, which leaves the
    // choice after the prompt and its logits by sequence
    std::vector<int32_t> tl(n), pl(n);
    for (int b = 0; b < n; ++b) {
        m->cached[b] = lens[b] - 1;
        tl[b] = ids[start[b] + lens[b] - 1];
        pl[b] = lens[b] - 1;
    }
    return gpt2_decode_batch(m, tl.data(), pl.data(), n, nullptr);
}

int gpt2_decode_batch_greedy(gpt2_batch *m, int32_t n_steps)
{
    if (!m || n_steps < 0) return GPT2_ERR_INVALID_ARG;
    if (!m->has_step) return GPT2_ERR_NOT_READY;
    for (int b = 0; b < m->max_batch; ++b)
        if (m->cached[b] > 0 && m->cached[b] + n_steps > m->cfg.n_positions) return GPT2_ERR_POSITION_RANGE;
    if (n_steps == 0) return GPT2_OK;
    // every sequence with a cached prefix continues from its own length with
    // its last choice
    std::vector<int32_t> p(kTcMaxRows, -1);
    for (int b = 0; b < m->max_batch; ++b)
        if (m->cached[b] > 0) p[b] = m->cached[b];
    BTRY(cudaMemcpyAsync(m->pos, p.data(), p.size() * 4, cudaMemcpyHostToDevice, m->stream));
    BTRY(upload_order(m, p.data(), m->stream));
    BTRY(cudaMemcpyAsync(m->tok, m->next_tok, size_t(kTcMaxRows) * 4, cudaMemcpyDeviceToDevice, m->stream));
    for (int i = 0; i < n_steps; ++i) BTRY(cudaGraphLaunch(m->exec, m->stream));
    m->launches += (unsigned long long)n_steps * m->kernels_per_step;
    for (int b = 0; b < m->max_batch; ++b)
        if (m->cached[b] > 0) m->cached[b] += n_steps;
    return GPT2_OK;
}

int gpt2_argmax_batch(gpt2_batch *m, int32_t *host_ids, int32_t n)
{
    if (!m || !host_ids || n < 1 || n > m->max_batch) return GPT2_ERR_INVALID_ARG;
    if (!m->has_step) return GPT2_ERR_NOT_READY;
    const int rc = read_batch_state(m);
    if (rc != GPT2_OK) return rc;
    BTRY(cudaMemcpy(host_ids, m->next_tok, size_t(n) * 4, cudaMemcpyDeviceToHost));
    return GPT2_OK;
}

int gpt2_batch_ids(gpt2_batch *m, int32_t first_pos, int32_t n_pos, int32_t *host_ids)
{
    if (!m || !host_ids || first_pos < 0 || n_pos < 0 || first_pos + n_pos > m->cfg.n_positions)
        return GPT2_ERR_INVALID_ARG;
    const int rc = read_batch_state(m);
    if (rc != GPT2_OK) return rc;
    BTRY(cudaMemcpy(host_ids, m->out_ids + size_t(first_pos) * m->max_batch, size_t(n_pos) * m->max_batch * 4,
                    cudaMemcpyDeviceToHost));
    return GPT2_OK;
}

int gpt2_copy_logits_batch(gpt2_batch *m, int32_t n, float *dst)
{
    if (!m || !dst || n < 1 || n > m->max_batch) return GPT2_ERR_INVALID_ARG;
    if (!m->has_step) return GPT2_ERR_NOT_READY;
    BTRY(cudaMemcpyAsync(dst, m->logits, size_t(n) * m->cfg.vocab_size * 4, cudaMemcpyDefault, m->stream));
    return read_batch_state(m);
}

int gpt2_export_kv_batch(gpt2_batch *m, int32_t layer, int32_t seq, int32_t n_rows, float *dst_k, float *dst_v)
{
    if (!m || layer < 0 || layer >= m->cfg.n_layer || seq < 0 || seq >= m->max_batch) return GPT2_ERR_INVALID_ARG;
    const int H = m->cfg.n_head, D = m->cfg.n_embd / H, P = m->cfg.n_positions;
    if (n_rows < 0 || n_rows > P) return GPT2_ERR_INVALID_ARG;
    const size_t es = m->kv_bf16 ? 2 : 4, row_elems = size_t(n_rows) * D;
    // bf16 rows are widened to fp32 on the host on their way out
    std::vector<uint16_t> tmp16(m->kv_bf16 ? row_elems : 0);
    std::vector<float> tmp32(m->kv_bf16 ? row_elems : 0);
    for (int h = 0; h < H; ++h) {
        const size_t src = ((size_t(layer) * m->max_batch + seq) * H + h) * P * D * es;
        for (int part = 0; part < 2; ++part) {
            float *dst = part == 0 ? dst_k : dst_v;
            if (!dst) continue;
            const uint8_t *from = static_cast<const uint8_t *>(part == 0 ? m->kc : m->vc) + src;
            dst += size_t(h) * row_elems;
            if (!m->kv_bf16) {
                BTRY(cudaMemcpyAsync(dst, from, row_elems * 4, cudaMemcpyDefault, m->stream));
                continue;
            }
            BTRY(cudaMemcpyAsync(tmp16.data(), from, row_elems * 2, cudaMemcpyDeviceToHost, m->stream));
            BTRY(cudaStreamSynchronize(m->stream));
            for (size_t i = 0; i < row_elems; ++i) {
                const uint32_t bits = uint32_t(tmp16[i]) << 16;
                std::memcpy(&tmp32[i], &bits, 4);
            }
            BTRY(cudaMemcpy(dst, tmp32.data(), row_elems * 4, cudaMemcpyDefault));
        }
    }
    BTRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_batch_info(const gpt2_batch *m, int32_t *kernels_per_step, uint64_t *launches)
{
    if (!m) return GPT2_ERR_INVALID_ARG;
    if (kernels_per_step) *kernels_per_step = m->kernels_per_step;
    if (launches) *launches = m->launches;
    return GPT2_OK;
}

int gpt2_sync_batch(gpt2_batch *m)
{
    if (!m) return GPT2_ERR_INVALID_ARG;
    return read_batch_state(m);
}

// ---- the stand-alone tensor-core linear ------------------------------------

size_t gpt2_op_linear_bf16_workspace(int32_t M, int32_t n, int32_t K)
{
    if (M < 1 || K < kTcK || n < 1) return 0;
    // the hi/lo B operand, then the K splits' shares (at most kTcMaxSplits)
    return a256(size_t(2 * kTcMaxRows) * K * 2) + a256(size_t(kTcMaxSplits) * n * M * 4);
}

int gpt2_op_linear_bf16(const void *W, const float *X, int32_t M, int32_t n, int32_t K, float *Y, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    if (!W || !X || !Y || !workspace) return GPT2_ERR_INVALID_ARG;
    if (M < 1 || n < 1 || n > kTcMaxRows || K < kTcK || K % kTcK) return GPT2_ERR_INVALID_ARG;
    if ((long long)M * K > (1ll << 31) - 1) return GPT2_ERR_INVALID_ARG;
    if (workspace_bytes < gpt2_op_linear_bf16_workspace(M, n, K)) return GPT2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(W) % 16 || reinterpret_cast<uintptr_t>(workspace) % 256)
        return GPT2_ERR_INVALID_ARG;
    int dev, sms;
    BTRY(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    BTRY(cudaGetDeviceProperties(&prop, dev));
    if (!(prop.major == 10 && prop.minor == 3)) return GPT2_ERR_UNSUPPORTED_DEVICE;
    sms = prop.multiProcessorCount;
    BTRY(tc_gemm_init());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    __nv_bfloat16 *bop = static_cast<__nv_bfloat16 *>(workspace);
    float *parts = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + a256(size_t(2 * kTcMaxRows) * K * 2));
    Linear L;
    if (set_linear(L, W, M, K, sms) != GPT2_OK) return GPT2_ERR_CUDA;
    CUtensorMap bmap;
    if (tc_make_tmap(&bmap, bop, 2 * kTcMaxRows, uint64_t(K))) return GPT2_ERR_CUDA;
    BTRY(cudaMemsetAsync(bop, 0, size_t(2 * kTcMaxRows) * K * 2, s));
    k_b_split_rows<<<n, 256, 0, s>>>(X, n, K, bop);
    BTRY(cudaGetLastError());
    TcGemmArgs a;
    a.M = M;
    a.K = K;
    a.n_rows = n;
    a.a_planes = 1;
    a.a_plane_rows = M;
    a.chunks_per_split = L.cps;
    a.partials = parts;
    a.st = nullptr;
    a.wait_ns = kWaitLimitNs;
    BTRY(tc_gemm_launch(L.a_map, bmap, a, L.splits, s, false));
    k_b_sum_splits<<<std::min(4096, (n * M + 255) / 256), 256, 0, s>>>(parts, L.splits, n, M, Y);
    BTRY(cudaGetLastError());
    return GPT2_OK;
}

}  // extern "C"
