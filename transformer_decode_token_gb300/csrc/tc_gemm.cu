// Tensor-core linear of the batched decode path: Y = X . W^T on tcgen05.
//
// At batch 64 each of the block's four linears is a dense contraction of the
// stored weights with 64 activation rows: the MMA's M side takes 128 weight
// rows (swap AB: weights are the A operand, so no weight tile is wasted on a
// 64-row batch), its N side 128 activation rows (the batch's bf16 hi parts and
// lo parts, so the fp32 activations keep ~16 bits through the bf16 MMA), and
// K runs over 64-input chunks (one 128-byte swizzle atom).  One CTA per
// (128-row tile, K split):
//   warp 0, one lane: TMA loads of the weight and activation tiles into a
//       3-stage shared-memory ring (97 KB, so two CTAs share an SM;
//       cp.async.bulk.tensor, 128-byte swizzle,
//       mbarrier completion; the weight tiles of the first stages are issued
//       before the wait for the previous kernel, which writes the activations);
//   warp 1, one lane: tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M = 128,
//       N = 128, K = 16) into 128 TMEM columns, tcgen05.commit frees a stage;
//   all four warps: tcgen05.ld of their 32 TMEM lanes, hi + lo summed, the
//       split's share of Y written as fp32 (summed in a fixed order by the
//       consumer kernel, so results do not depend on timing).
// Every wait is bounded (the model's wait limit); a wait that runs out records
// GPT2_ERR_TIMEOUT, lets the copies in flight land and frees the TMEM.
#include "common.cuh"
#include "tc_gemm.h"

namespace gpt2 {

namespace {

constexpr uint32_t kTileA = kTcM * kTcK * 2;   // 16 KB
constexpr uint32_t kTileB = kTcN * kTcK * 2;   // 16 KB
constexpr uint32_t kStageBytes = kTileA + kTileB;
constexpr uint32_t kBarOff = kTcStages * kStageBytes;
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;   // barriers, TMEM slot, alignment slack
constexpr uint32_t kTmemCols = 128;                     // N fp32 accumulators per lane

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kTcN >> 3) << 17) |
                            (uint32_t(kTcM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// start address >> 4 (bits 0-13), leading offset (unused for this layout,
// 1), stride between 8-row groups 1024 bytes >> 4 (bits 32-45), descriptor
// version 1 (bits 46-47), swizzle mode 128 B = 2 (bits 61-63).  Tiles start on
// 1024-byte boundaries, so the base-offset field is 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, unsigned long long limit)
{
    if (mbar_test_wait(bar, parity)) return true;
    unsigned long long t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            const unsigned long long t = global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > limit) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kTcThreads, 1) k_tc_gemm(const __grid_constant__ CUtensorMap a_map,
                                                           const __grid_constant__ CUtensorMap b_map,
                                                           const TcGemmArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base: the 128-byte swizzle pattern repeats every 1024
    // bytes, and TMA and the MMA both apply it to the absolute address
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kBarOff);
    uint64_t *empty = full + kTcStages;
    uint64_t *done = empty + kTcStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTcM;
    const int n_chunks = a.K / kTcK;
    const int kc0 = blockIdx.y * a.chunks_per_split;
    const int nk = min(a.chunks_per_split, n_chunks - kc0);
    const int total = nk > 0 ? nk * a.a_planes : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        mbar_init_fence();
    }
    if (warp == 0) {   // the whole warp allocates the accumulator columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    int issued = 0;
    if (warp == 0 && lane == 0) {
        // producer: the weight tiles of the first stages go out before the
        // previous kernel has finished; activation tiles only after it
        const int pre = min(total, kTcStages);
        for (int i = 0; i < pre; ++i) {
            const int plane = i / nk, kc = kc0 + i % nk;
            const uint32_t st = base + uint32_t(i) * kStageBytes;
            mbar_arrive_expect_tx(&full[i], kStageBytes);
            tma_load_2d(st, &a_map, kc * kTcK, plane * a.a_plane_rows + m0, &full[i]);
        }
        pdl_wait();
        for (int i = 0; i < pre; ++i) {
            const int kc = kc0 + i % nk;
            tma_load_2d(base + uint32_t(i) * kStageBytes + kTileA, &b_map, kc * kTcK, 0, &full[i]);
        }
        issued = pre;
        for (int i = pre; i < total; ++i) {
            const int s = i % kTcStages;
            if (!wait_bar(&empty[s], uint32_t((i / kTcStages) - 1) & 1u, a.wait_ns)) {
                record_error(a.st, kDevErrTimeout, 11000 + int(blockIdx.x));
                ok = false;
                break;
            }
            const int plane = i / nk, kc = kc0 + i % nk;
            const uint32_t st = base + uint32_t(s) * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_2d(st, &a_map, kc * kTcK, plane * a.a_plane_rows + m0, &full[s]);
            tma_load_2d(st + kTileA, &b_map, kc * kTcK, 0, &full[s]);
            issued = i + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        for (int i = 0; i < total; ++i) {
            const int s = i % kTcStages;
            if (!wait_bar(&full[s], uint32_t(i / kTcStages) & 1u, a.wait_ns)) {
                record_error(a.st, kDevErrTimeout, 12000 + int(blockIdx.x));
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t st = base + uint32_t(s) * kStageBytes;
            const uint64_t da = smem_desc(st), db = smem_desc(st + kTileA);
#pragma unroll
            for (int kk = 0; kk < kTcK / 16; ++kk)   // +32 bytes along K per step: +2 in the address field
                mma_bf16(tmem, da + uint64_t(2 * kk), db + uint64_t(2 * kk), (i | kk) != 0 ? 1u : 0u);
            mma_commit(&empty[s]);
        }
        mma_commit(done);   // arrives once every MMA issued above has completed
    }
    pdl_wait();                 // every thread: the previous kernel's writes and reads are over
    pdl_launch_dependents();

    // epilogue: warp w reads TMEM lanes 32w..32w+31 (tile rows), columns c and
    // 64 + c (the hi and lo parts of activation row c)
    bool good = wait_bar(done, 0u, a.wait_ns);
    if (!good && threadIdx.x == 64) record_error(a.st, kDevErrTimeout, 13000 + int(blockIdx.x));
    good = __all_sync(0xffffffffu, good) && total > 0;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (good) {
        const int m = m0 + warp * 32 + lane;
        const uint32_t row_addr = tmem + (uint32_t(warp * 32) << 16);
        float *out = a.partials + size_t(blockIdx.y) * a.n_rows * a.M;
        for (int c0 = 0; c0 < kTcMaxRows && c0 < a.n_rows; c0 += 16) {
            float hi[16], lo[16];
            tmem_ld16(row_addr + uint32_t(c0), hi);
            tmem_ld16(row_addr + uint32_t(c0 + kTcMaxRows), lo);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (m < a.M) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < a.n_rows) out[size_t(c0 + j) * a.M + m] = hi[j] + lo[j];
            }
        }
    }
    // copies in flight land before the CTA leaves (after a wait that ran out)
    if (warp == 0 && lane == 0 && !ok) {
        for (int j = max(0, issued - kTcStages); j < issued; ++j)
            wait_bar(&full[j % kTcStages], uint32_t(j / kTcStages) & 1u, kWaitLimitNs);
    }
    if (!ok || !good) wait_bar(done, 0u, kWaitLimitNs);   // no MMA still writes the columns
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn()
{
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

}  // namespace

int tc_make_tmap(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t K)
{
    EncodeTiled fn = encode_fn();
    if (!fn) return 1;
    if (reinterpret_cast<uintptr_t>(ptr) % 16 || (K * 2) % 16 || K % kTcK) return 2;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {uint32_t(kTcK), uint32_t(kTcM)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 3;
}

size_t tc_gemm_smem_bytes() { return kSmemBytes; }

cudaError_t tc_gemm_init()
{
    return cudaFuncSetAttribute(k_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
}

cudaError_t tc_gemm_launch(const CUtensorMap &a_map, const CUtensorMap &b_map, const TcGemmArgs &a, int splits,
                           cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.M + kTcM - 1) / kTcM, splits);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_tc_gemm, a_map, b_map, a);
}

}  // namespace gpt2
