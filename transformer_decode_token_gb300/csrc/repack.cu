// One-time weight repacking on the device.
//
// The checkpoint stores the block matrices as [input][output]; the decode
// kernels want [output][input] so that one output is one contiguous row
// ("Let's make GPT-2 in assembly", Step 1: the transposed copy made the
// matrix kernel go from about 60 to about 100 tokens/s on its CPU).  The
// fp16 mode rounds each weight to nearest even; the int4 mode quantises each
// group of 32 consecutive inputs of an output row with an fp32 scale and a
// 4-bit zero point ("model.fir" header: transpose to [output,input], then
// grouped asymmetric int4).  Every decision that turns a float into an
// integer uses IEEE division and round-half-to-even, so the codes are the
// same bits on any IEEE machine.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace gpt2 {

template <typename T>
__device__ __forceinline__ T cvt_out(float v);
template <>
__device__ __forceinline__ float cvt_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half cvt_out<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// src [in][out] -> dst [out][in], 32x32 tiles through shared memory.
template <typename T>
__global__ void __launch_bounds__(256) k_transpose(const float *src, int in, int out, T *dst)
{
    __shared__ float tile[32][33];
    const int bo = blockIdx.x * 32, bi = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    for (int k = ty; k < 32; k += 8) {
        const int i = bi + k, o = bo + tx;
        if (i < in && o < out) tile[k][tx] = src[size_t(i) * out + o];
    }
    __syncthreads();
    for (int k = ty; k < 32; k += 8) {
        const int o = bo + k, i = bi + tx;
        if (o < out && i < in) dst[size_t(o) * in + i] = cvt_out<T>(tile[tx][k]);
    }
}

template <typename T>
static cudaError_t transpose(const float *src, int in, int out, T *dst, cudaStream_t s)
{
    dim3 grid((out + 31) / 32, (in + 31) / 32), block(32, 8);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    k_transpose<T><<<grid, block, 0, s>>>(src, in, out, dst);
    return cudaGetLastError();
}

cudaError_t repack_f32(const float *src, int in, int out, float *dst, cudaStream_t s)
{
    return transpose<float>(src, in, out, dst, s);
}

cudaError_t repack_f16(const float *src, int in, int out, void *dst, cudaStream_t s)
{
    return transpose<__half>(src, in, out, static_cast<__half *>(dst), s);
}

cudaError_t repack_bf16(const float *src, int in, int out, void *dst, cudaStream_t s)
{
    return transpose<__nv_bfloat16>(src, in, out, static_cast<__nv_bfloat16 *>(dst), s);
}

// Elementwise split of fp32 values into bf16 planes: hi = bf16(v) and
// lo = bf16(v - hi) (round to nearest even; v - hi is exact in fp32), so that
// hi + lo keeps about 16 bits of v.  lo may be null (hi only).
__global__ void __launch_bounds__(256) k_to_bf16(const float *src, size_t n, __nv_bfloat16 *hi, __nv_bfloat16 *lo)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
        const float v = src[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        hi[i] = h;
        if (lo) lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
    }
}

cudaError_t split_bf16(const float *src, size_t n, void *hi, void *lo, cudaStream_t s)
{
    const size_t blocks = std::min<size_t>((n + 255) / 256, 8192);
    if (blocks == 0) return cudaSuccess;
    k_to_bf16<<<unsigned(blocks), 256, 0, s>>>(src, n, static_cast<__nv_bfloat16 *>(hi),
                                                static_cast<__nv_bfloat16 *>(lo));
    return cudaGetLastError();
}

// Elementwise fp32 -> fp16 (round to nearest even), layout unchanged.
__global__ void __launch_bounds__(256) k_to_f16(const float *src, size_t n, __half *dst)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        dst[i] = __float2half_rn(src[i]);
}

cudaError_t convert_f16(const float *src, size_t n, void *dst, cudaStream_t s)
{
    const size_t blocks = std::min<size_t>((n + 255) / 256, 8192);
    if (blocks == 0) return cudaSuccess;
    k_to_f16<<<unsigned(blocks), 256, 0, s>>>(src, n, static_cast<__half *>(dst));
    return cudaGetLastError();
}

// One warp per pair of groups (64 inputs of one output row), lane = input.
__global__ void __launch_bounds__(256) k_quant_int4(const float *Wt, int in, int out, uint8_t *codes, float *scales,
                                                    uint8_t *zeros)
{
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int pairs = in / 64;
    if (gw >= out * pairs) return;
    const int o = gw / pairs, pj = gw % pairs;
    uint32_t zbyte = 0;
    for (int half = 0; half < 2; ++half) {
        const int g = 2 * pj + half;
        const float w = Wt[size_t(o) * in + g * 32 + lane];
        float mn = fminf(w, 0.0f), mx = fmaxf(w, 0.0f);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, d));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
        }
        float s = __fdiv_rn(mx - mn, 15.0f);
        if (s == 0.0f) s = 1.0f;
        const float zf = rintf(__fdiv_rn(-mn, s));
        const int z = zf < 0.0f ? 0 : (zf > 15.0f ? 15 : int(zf));
        const float qf = rintf(__fdiv_rn(w, s)) + float(z);
        const int q = qf < 0.0f ? 0 : (qf > 15.0f ? 15 : int(qf));
        const int qn = __shfl_down_sync(0xffffffffu, q, 1);
        if ((lane & 1) == 0)
            codes[size_t(o) * (in / 2) + (g * 32 + lane) / 2] = uint8_t(q | (qn << 4));
        if (lane == 0) scales[size_t(o) * (in / 32) + g] = s;
        zbyte |= uint32_t(z) << (4 * half);
    }
    if (lane == 0) zeros[size_t(o) * (in / 64) + pj] = uint8_t(zbyte);
}

cudaError_t quant_int4_rows(const float *Wt, int in, int out, uint8_t *codes, float *scales, uint8_t *zeros,
                            cudaStream_t s)
{
    if (in % 64) return cudaErrorInvalidValue;
    const long long warps = (long long)out * (in / 64);
    const long long blocks = (warps + 7) / 8;
    k_quant_int4<<<unsigned(blocks), 256, 0, s>>>(Wt, in, out, codes, scales, zeros);
    return cudaGetLastError();
}

cudaError_t repack_int4(const float *src, int in, int out, float *tmp, uint8_t *codes, float *scales,
                        uint8_t *zeros, cudaStream_t s)
{
    if (in % 64) return cudaErrorInvalidValue;
    cudaError_t e = transpose<float>(src, in, out, tmp, s);
    if (e != cudaSuccess) return e;
    const long long warps = (long long)out * (in / 64);
    const long long blocks = (warps + 7) / 8;
    k_quant_int4<<<unsigned(blocks), 256, 0, s>>>(tmp, in, out, codes, scales, zeros);
    return cudaGetLastError();
}

// The stored matrix as the GEMV kernels read it, widened to fp32 [out][in].
__global__ void __launch_bounds__(256) k_dequant(int wtype, const void *W, const float *scales, const uint8_t *zeros,
                                                 int in, int out, float *dst)
{
    const size_t idx = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= size_t(in) * out) return;
    const int o = int(idx / in), i = int(idx % in);
    float v;
    if (wtype == kWF32) {
        v = static_cast<const float *>(W)[idx];
    } else if (wtype == kWF16) {
        v = __half2float(static_cast<const __half *>(W)[idx]);
    } else {
        const uint8_t *c = static_cast<const uint8_t *>(W);
        const int q = (c[size_t(o) * (in / 2) + i / 2] >> (4 * (i & 1))) & 15;
        const int g = i / 32;
        const int z = (zeros[size_t(o) * (in / 64) + g / 2] >> (4 * (g & 1))) & 15;
        v = float(q - z) * scales[size_t(o) * (in / 32) + g];
    }
    dst[idx] = v;
}

cudaError_t dequant_to_f32(int wtype, const void *W, const float *scales, const uint8_t *zeros, int in, int out,
                           float *dst, cudaStream_t s)
{
    const size_t n = size_t(in) * out;
    const size_t blocks = (n + 255) / 256;
    k_dequant<<<unsigned(blocks), 256, 0, s>>>(wtype, W, scales, zeros, in, out, dst);
    return cudaGetLastError();
}

// LayerNorm folded into the rows that follow it (see CLayer in cluster.h):
// one warp per row of a stored [out][in] matrix, c1 = W.gamma, c2 = W.beta,
// fixed-order sums.
__global__ void __launch_bounds__(256) k_ln_fold(const float *W, const float *gamma, const float *beta, int in,
                                                 int out, float *c1, float *c2)
{
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (row >= out) return;
    float a = 0.f, b = 0.f;
    for (int i = lane; i < in; i += 32) {
        const float w = W[size_t(row) * in + i];
        a = fmaf(w, gamma[i], a);
        b = fmaf(w, beta[i], b);
    }
    a = warp_sum(a);
    b = warp_sum(b);
    if (lane == 0) {
        c1[row] = a;
        c2[row] = b;
    }
}

cudaError_t ln_fold(const float *W, const float *gamma, const float *beta, int in, int out, float *c1, float *c2,
                    cudaStream_t s)
{
    k_ln_fold<<<(out + 7) / 8, 256, 0, s>>>(W, gamma, beta, in, out, c1, c2);
    return cudaGetLastError();
}

}  // namespace gpt2
