// Device-side pieces shared by the decode kernels: stored-row layout and the
// row dot product.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace gpt2 {

inline __host__ __device__ uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

inline __host__ __device__ uint32_t row_bytes(int wtype, int in)
{
    return wtype == kWF32 ? uint32_t(in) * 4u : wtype == kWF16 ? uint32_t(in) * 2u : uint32_t(in) / 2u;
}

constexpr uint32_t kHdrBytes = 128;   // 8 mbarriers, then 8 per-warp argmax keys
constexpr int kMaxStages = 8;

inline __host__ __device__ uint32_t vec_region_bytes(int in)
{
    return align_up(uint32_t(in + in / 32) * 4u, 128u);   // x (in floats) + per-group sums
}

// Units a row is split into for the lanes: 16-byte vectors for fp32 / fp16,
// 32-bit words (8 codes) for int4.
template <int WT>
__host__ __device__ __forceinline__ int row_units(int in)
{
    return WT == kWF32 ? in >> 2 : in >> 3;
}

// Partial dot product over units [vb, ve) of one stored row; see row_dot.
template <int WT>
__device__ __forceinline__ float row_dot_range(const uint8_t *stg, int rl, int in, const float *xs,
                                               const float *xsum, uint32_t soff, uint32_t zoff, int lane, int vb,
                                               int ve)
{
    float acc = 0.f;
    const float4 *x4 = reinterpret_cast<const float4 *>(xs);
    if (WT == kWF32) {
        const float4 *w = reinterpret_cast<const float4 *>(stg + size_t(rl) * in * 4);
        const int nv = ve;
        for (int v = vb + lane; v < nv; v += 32) {
            const float4 a = w[v], b = x4[v];
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
            acc = fmaf(a.z, b.z, acc);
            acc = fmaf(a.w, b.w, acc);
        }
    } else if (WT == kWF16) {
        const uint4 *w = reinterpret_cast<const uint4 *>(stg + size_t(rl) * in * 2);
        const int nv = ve;
        for (int v = vb + lane; v < nv; v += 32) {
            const uint4 r = w[v];
            const float4 b0 = x4[2 * v], b1 = x4[2 * v + 1];
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
            const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&r.z));
            const float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&r.w));
            acc = fmaf(f0.x, b0.x, acc);
            acc = fmaf(f0.y, b0.y, acc);
            acc = fmaf(f1.x, b0.z, acc);
            acc = fmaf(f1.y, b0.w, acc);
            acc = fmaf(f2.x, b1.x, acc);
            acc = fmaf(f2.y, b1.y, acc);
            acc = fmaf(f3.x, b1.z, acc);
            acc = fmaf(f3.y, b1.w, acc);
        }
    } else {
        // One 32-bit word = 8 codes of one group; four lanes share a group.
        // sum_k (q_k - z) s x_k = s * (sum_k q_k x_k - z * sum_k x_k)
        const int G = in >> 5;
        const uint32_t *w = reinterpret_cast<const uint32_t *>(stg + size_t(rl) * (in >> 1));
        const float *sc = reinterpret_cast<const float *>(stg + soff) + size_t(rl) * G;
        const uint8_t *zp = stg + zoff + size_t(rl) * (in >> 6);
        const int nw = ve;
        for (int v = vb + lane; v < nw; v += 32) {
            const uint32_t q = w[v];
            const int g = v >> 2;
            const float4 b0 = x4[2 * v], b1 = x4[2 * v + 1];
            // exact small-integer -> float: 2^23 + q has q in its low mantissa bits
            auto nib = [&](int t) { return __uint_as_float(0x4B000000u | ((q >> (4 * t)) & 15u)) - 8388608.0f; };
            float part = nib(0) * b0.x;
            part = fmaf(nib(1), b0.y, part);
            part = fmaf(nib(2), b0.z, part);
            part = fmaf(nib(3), b0.w, part);
            part = fmaf(nib(4), b1.x, part);
            part = fmaf(nib(5), b1.y, part);
            part = fmaf(nib(6), b1.z, part);
            part = fmaf(nib(7), b1.w, part);
            const float s = sc[g];
            if ((v & 3) == 0) {
                const float z = float((zp[g >> 1] >> ((g & 1) * 4)) & 15);
                part = fmaf(-z, xsum[g], part);
            }
            acc = fmaf(s, part, acc);
        }
    }
    return acc;
}

template <int WT>
__device__ __forceinline__ float row_dot(const uint8_t *stg, int rl, int in, const float *xs, const float *xsum,
                                         uint32_t soff, uint32_t zoff, int lane)
{
    return row_dot_range<WT>(stg, rl, in, xs, xsum, soff, zoff, lane, 0, row_units<WT>(in));
}


}  // namespace gpt2
