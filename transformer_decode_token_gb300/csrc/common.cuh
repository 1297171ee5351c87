// Shared device helpers for the decode kernels (sm_103a).
//
// * 1-D bulk copies global -> shared (cp.async.bulk) completed on an mbarrier,
//   used to stage weight rows in shared memory before the data they multiply
//   exists (the copies are issued ahead of griddepcontrol.wait).
// * griddepcontrol (programmatic dependent launch) wrappers.
// * Bounded mbarrier waits: every wait gives up after a time limit, records
//   an error code in the device state word and returns false; kernels never
//   trap and never spin forever.
// * Warp reductions in a fixed order (results are bitwise reproducible).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gpt2 {

constexpr int kWarps = 8;                 // warps per CTA of the GEMV/head kernels
constexpr int kThreads = kWarps * 32;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

// Error codes a kernel can record (device state word `err`).
enum : int32_t {
    kDevErrNone = 0,
    kDevErrTimeout = 1,        // a bounded wait gave up
    kDevErrBadToken = 2,       // token outside [0, vocab)
    kDevErrBadPosition = 3,    // position outside [0, n_positions)
    kDevErrLaunchShape = 4,    // a kernel found a grid / cluster shape it was not built for
    kDevErrRange = 5,          // an activation outside the range of the fixed-point residual sums
};

// Per-model scalars that live in device memory so that a captured graph can
// be replayed for any token and position, and greedy decoding can feed each
// pass's argmax into the next without the host.
struct DeviceState {
    int32_t tok;        // token consumed by the next pass
    int32_t pos;        // its position
    int32_t next_tok;   // argmax of the last pass
    int32_t n_out;      // number of ids appended to out_ids
    int32_t err;        // first recorded kDevErr* code (0 = none)
    int32_t err_info;   // where it happened (kernel-specific)
    int32_t abort;      // cluster kernel: a CTA gave up, every CTA returns
    int32_t seq;        // cluster kernel: passes run so far + 1 (epoch base)
};

__device__ __forceinline__ void record_error(DeviceState *st, int32_t code, int32_t info)
{
    if (st && atomicCAS(&st->err, 0, code) == 0) st->err_info = info;
}

// ---- programmatic dependent launch ----------------------------------------
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- shared-memory barriers and bulk copies --------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of phase `parity`: true if it has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of `bar` to complete, for at most kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u) {
            unsigned long long t = global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > kWaitLimitNs) return false;
        }
    }
}

// L2 policy: stream once (evict first).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy: keep (evict last).
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
        "[%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// ---- reductions -----------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Argmax key: the float's bits mapped to an order-preserving unsigned value
// in the high word, the complement of the index in the low word, so the
// largest key is the largest value with the lowest index among exact ties.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx)
{
    uint32_t b = __float_as_uint(v);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (static_cast<unsigned long long>(b) << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ int32_t argmax_key_index(unsigned long long k)
{
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
}

// LayerNorm statistics of one row of n floats in shared memory, computed by
// one warp (every warp that calls it gets the same bits): mean, then the
// biased variance around it, then 1/sqrt(var + eps) with IEEE sqrt and
// division ("model.fir" kernel g2.layernorm).
__device__ __forceinline__ void warp_ln_stats(const float *row, int n, float eps, float &mean, float &rstd)
{
    const int lane = threadIdx.x & 31;
    float s = 0.f;
    for (int i = lane; i < n; i += 32) s += row[i];
    s = warp_sum(s);
    mean = s / static_cast<float>(n);
    float ss = 0.f;
    for (int i = lane; i < n; i += 32) {
        float d = row[i] - mean;
        ss = fmaf(d, d, ss);
    }
    ss = warp_sum(ss);
    const float var = ss / static_cast<float>(n);
    rstd = 1.0f / sqrtf(var + eps);
}

__device__ __forceinline__ float gelu_new(float v)
{
    // 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))  ("model.fir" g2.gelu_new)
    const float c = 0.7978845608028654f;
    float u = c * fmaf(0.044715f * v, v * v, v);
    return 0.5f * v * (1.0f + tanhf(u));
}

}  // namespace gpt2
