// Decode-pass kernels for sm_103a: row GEMV with fused prologue/epilogue
// (also the tied head + argmax), decode attention, warp-per-row LayerNorm.
//
// The GEMV is the pass's whole cost at batch 1: "about 124 million
// multiply-adds per token", every weight read once per token ("Let's make
// GPT-2 in assembly", Step 4).  Each CTA owns a contiguous range of output
// rows of a [out][in] matrix, so its weights are one contiguous byte range;
// one thread streams that range into shared memory with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier) in chunks, and all warps take
// dot products out of shared memory.  The first chunks are requested before
// griddepcontrol.wait, i.e. while the previous kernel of the pass is still
// running, because the weights never depend on it.
#include "gemv_dev.cuh"

namespace gpt2 {

size_t gemv_smem_bytes(const GemvArgs &a)
{
    return kHdrBytes + vec_region_bytes(a.in) + size_t(a.n_stages) * a.stage_bytes;
}

int gemv_plan(GemvArgs &a, int wtype, int ctas, size_t budget, int max_stages)
{
    const int gran = wtype == kWI4 ? 8 : 1;
    int rpc = (a.out + ctas - 1) / ctas;
    rpc = (rpc + gran - 1) / gran * gran;
    const int grid = (a.out + rpc - 1) / rpc;
    const uint32_t rb = row_bytes(wtype, a.in);
    const int G = a.in / 32;
    // bytes a row needs in a stage (int4: codes + scales + zero points)
    const uint32_t per_row = wtype == kWI4 ? rb + uint32_t(G) * 4u + uint32_t(a.in / 64) : rb;
    int chunk = kWarps;
    if (size_t(chunk) * per_row > budget) chunk = int(budget / per_row);
    chunk = chunk / gran * gran;
    if (chunk < gran) chunk = gran;
    if (chunk > rpc) chunk = rpc;
    uint32_t stage;
    if (wtype == kWI4) {
        a.stage_scale_off = align_up(uint32_t(chunk) * rb, 16u);
        a.stage_zero_off = a.stage_scale_off + align_up(uint32_t(chunk) * uint32_t(G) * 4u, 16u);
        stage = align_up(a.stage_zero_off + uint32_t(chunk) * uint32_t(a.in / 64), 128u);
    } else {
        a.stage_scale_off = a.stage_zero_off = 0;
        stage = align_up(uint32_t(chunk) * rb, 128u);
    }
    const int nchunks = (rpc + chunk - 1) / chunk;
    int ns = int(budget / stage);
    if (ns > max_stages) ns = max_stages;
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns > nchunks) ns = nchunks;
    if (ns < 1) ns = 1;
    a.rows_per_cta = rpc;
    a.chunk_rows = chunk;
    a.n_stages = ns;
    a.stage_bytes = stage;
    return grid;
}

template <int WT, int MODE>
__global__ void __launch_bounds__(kThreads) k_gemv(const GemvArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_flag;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned long long *wkeys = reinterpret_cast<unsigned long long *>(smem + 64);
    const int in = a.in;
    const int G = in >> 5;
    float *xs = reinterpret_cast<float *>(smem + kHdrBytes);
    float *xsum = xs + in;
    uint8_t *stages = smem + kHdrBytes + vec_region_bytes(in);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.x * a.rows_per_cta;
    const int r1 = min(a.out, r0 + a.rows_per_cta);
    const int nrows = max(0, r1 - r0);
    const int nchunks = (nrows + a.chunk_rows - 1) / a.chunk_rows;
    const uint32_t rb = row_bytes(WT, in);

    if (tid == 0) {
        for (int s = 0; s < a.n_stages; ++s) mbar_init(&bars[s], 1);
        mbar_init_fence();
        s_flag = 0;
    }
    __syncthreads();

    const uint64_t pol = a.evict_first ? l2_evict_first_policy() : 0ull;
    auto copy = [&](void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
        if (a.evict_first) bulk_g2s_hint(dst, src, bytes, bar, pol);
        else bulk_g2s(dst, src, bytes, bar);
    };
    auto issue = [&](int c) {   // thread 0 only
        const int s = c % a.n_stages;
        const int rs = r0 + c * a.chunk_rows;
        const int n = min(a.chunk_rows, r1 - rs);
        uint8_t *dst = stages + size_t(s) * a.stage_bytes;
        const uint32_t b0 = uint32_t(n) * rb;
        uint32_t total = b0;
        if (WT == kWI4) total += uint32_t(n) * uint32_t(G) * 4u + uint32_t(n) * uint32_t(in >> 6);
        mbar_arrive_expect_tx(&bars[s], total);
        copy(dst, static_cast<const uint8_t *>(a.W) + size_t(rs) * rb, b0, &bars[s]);
        if (WT == kWI4) {
            copy(dst + a.stage_scale_off, a.scales + size_t(rs) * G, uint32_t(n) * uint32_t(G) * 4u, &bars[s]);
            copy(dst + a.stage_zero_off, a.zeros + size_t(rs) * (in >> 6), uint32_t(n) * uint32_t(in >> 6),
                 &bars[s]);
        }
    };
    int issued = 0;
    if (tid == 0) {
        const int first = min(a.n_stages, nchunks);
        for (int c = 0; c < first; ++c) issue(c);
        issued = first;
    }

    pdl_launch_dependents();
    pdl_wait();   // everything below may read what the previous kernel wrote

    // ---- prologue: the input vector in shared memory --------------------
    if (MODE == kModeEmbLnBias) {
        int tok = __ldcg(&a.st->tok), pos = __ldcg(&a.st->pos);
        const bool tok_ok = tok >= 0 && tok < a.vocab, pos_ok = pos >= 0 && pos < a.n_positions;
        if (!(tok_ok && pos_ok)) {
            if (tid == 0 && blockIdx.x == 0)
                record_error(a.st, tok_ok ? kDevErrBadPosition : kDevErrBadToken, tok_ok ? pos : tok);
            tok = tok_ok ? tok : 0;
            pos = pos_ok ? pos : 0;
        }
        for (int i = tid; i < in; i += kThreads) {
            const float v = __ldg(a.wte + size_t(tok) * in + i) + __ldg(a.wpe + size_t(pos) * in + i);
            xs[i] = v;
            if (blockIdx.x == 0) a.x_out[i] = v;
        }
    } else {
        for (int i = tid; i < in; i += kThreads) xs[i] = __ldcg(a.xin + i);
    }
    __syncthreads();
    if (MODE == kModeLnBias || MODE == kModeEmbLnBias || MODE == kModeLnBiasGelu || MODE == kModeHead) {
        float mean, rstd;
        warp_ln_stats(xs, in, a.eps, mean, rstd);   // every warp, same bits
        __syncthreads();
        for (int i = tid; i < in; i += kThreads)
            xs[i] = (xs[i] - mean) * rstd * __ldg(a.ln_w + i) + __ldg(a.ln_b + i);
        __syncthreads();
    }
    if (WT == kWI4) {
        for (int g = warp; g < G; g += kWarps) {
            const float v = warp_sum(xs[g * 32 + lane]);
            if (lane == 0) xsum[g] = v;
        }
        __syncthreads();
    }

    // ---- rows ----------------------------------------------------------
    unsigned long long best = 0ull;
    int c = 0;
    for (; c < nchunks; ++c) {
        const int s = c % a.n_stages;
        const uint32_t par = uint32_t(c / a.n_stages) & 1u;
        const bool ok = mbar_wait_bounded(&bars[s], par);
        if (!ok) atomicOr(&s_flag, 1);
        const int rs = r0 + c * a.chunk_rows;
        const int n = min(a.chunk_rows, r1 - rs);
        const uint8_t *stg = stages + size_t(s) * a.stage_bytes;
        if (ok) {
            for (int rl = warp; rl < n; rl += kWarps) {
                float acc = row_dot<WT>(stg, rl, in, xs, xsum, a.stage_scale_off, a.stage_zero_off, lane);
                acc = warp_sum(acc);
                const int r = rs + rl;
                if (lane == 0) {
                    if (MODE == kModeLnBias || MODE == kModeEmbLnBias) {
                        a.y[r] = acc + __ldg(a.bias + r);
                    } else if (MODE == kModeLnBiasGelu) {
                        a.y[r] = gelu_new(acc + __ldg(a.bias + r));
                    } else if (MODE == kModeBiasRes) {
                        a.y[r] = __ldcg(a.y + r) + (acc + __ldg(a.bias + r));
                    } else {   // kModeHead
                        a.y[r] = acc;
                        const unsigned long long k = argmax_key(acc, uint32_t(r));
                        best = k > best ? k : best;
                    }
                }
            }
        }
        __syncthreads();
        if (s_flag) break;   // a copy never arrived: stop issuing, drain below
        if (tid == 0 && c + a.n_stages < nchunks) {
            issue(c + a.n_stages);
            ++issued;
        }
    }
    if (s_flag) {
        if (tid == 0) {
            record_error(a.st, kDevErrTimeout, blockIdx.x);
            // wait (bounded) for copies still in flight before the CTA exits
            for (int cc = c; cc < issued; ++cc)
                (void)mbar_wait_bounded(&bars[cc % a.n_stages], uint32_t(cc / a.n_stages) & 1u);
        }
        return;
    }

    if (MODE == kModeHead) {
        __shared__ int s_last;
        if (lane == 0) wkeys[warp] = best;
        __syncthreads();
        if (tid == 0) {
            unsigned long long b = 0ull;
            for (int w = 0; w < kWarps; ++w) b = wkeys[w] > b ? wkeys[w] : b;
            a.partials[blockIdx.x] = b;
            __threadfence();
            const unsigned int t = atomicAdd(a.counter, 1u);
            s_last = (t == gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (s_last && warp == 0) {
            __threadfence();
            unsigned long long b = 0ull;
            for (int i = lane; i < int(gridDim.x); i += 32) {
                const unsigned long long v = __ldcg(a.partials + i);
                b = v > b ? v : b;
            }
            b = warp_max_u64(b);
            if (lane == 0) {
                const int32_t tok = argmax_key_index(b);
                if (a.st) {
                    DeviceState *st = a.st;
                    st->next_tok = tok;
                    const int32_t n = st->n_out;
                    if (a.out_ids && n >= 0 && n < a.out_cap) a.out_ids[n] = tok;
                    st->n_out = n + 1;
                    st->tok = tok;           // greedy: the next pass consumes it
                    st->pos = st->pos + 1;
                }
                if (a.dev_token) *a.dev_token = tok;
                *a.counter = 0u;             // ready for the next launch
            }
        }
    }
}

template <int WT, int MODE>
static cudaError_t set_smem_attr()
{
    return cudaFuncSetAttribute(k_gemv<WT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
}

cudaError_t gemv_init()
{
    // once per device: the launches need more than 48 KB of dynamic shared
    // memory; done outside any stream capture
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    const cudaError_t r[] = {
        set_smem_attr<kWF32, kModeLnBias>(), set_smem_attr<kWF32, kModeEmbLnBias>(),
        set_smem_attr<kWF32, kModeBiasRes>(), set_smem_attr<kWF32, kModeLnBiasGelu>(),
        set_smem_attr<kWF16, kModeLnBias>(), set_smem_attr<kWF16, kModeEmbLnBias>(),
        set_smem_attr<kWF16, kModeBiasRes>(), set_smem_attr<kWF16, kModeLnBiasGelu>(),
        set_smem_attr<kWI4, kModeLnBias>(), set_smem_attr<kWI4, kModeEmbLnBias>(),
        set_smem_attr<kWI4, kModeBiasRes>(), set_smem_attr<kWI4, kModeLnBiasGelu>(),
        set_smem_attr<kWF32, kModeHead>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) return x;
    if (dev >= 0 && dev < 64) done[dev] = true;
    return cudaSuccess;
}

template <int WT, int MODE>
static cudaError_t launch_gemv_t(const GemvArgs &a, int grid, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes(a);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_gemv<WT, MODE>, a);
}

cudaError_t launch_gemv(int wtype, int mode, const GemvArgs &a, int grid, cudaStream_t s, bool pdl)
{
#define GPT2_GEMV_CASE(WT)                                                          \
    switch (mode) {                                                                 \
    case kModeLnBias: return launch_gemv_t<WT, kModeLnBias>(a, grid, s, pdl);       \
    case kModeEmbLnBias: return launch_gemv_t<WT, kModeEmbLnBias>(a, grid, s, pdl); \
    case kModeBiasRes: return launch_gemv_t<WT, kModeBiasRes>(a, grid, s, pdl);     \
    case kModeLnBiasGelu: return launch_gemv_t<WT, kModeLnBiasGelu>(a, grid, s, pdl); \
    default: return cudaErrorInvalidValue;                                          \
    }
    if (mode == kModeHead) {
        if (wtype != kWF32) return cudaErrorInvalidValue;
        return launch_gemv_t<kWF32, kModeHead>(a, grid, s, pdl);
    }
    switch (wtype) {
    case kWF32: GPT2_GEMV_CASE(kWF32)
    case kWF16: GPT2_GEMV_CASE(kWF16)
    case kWI4: GPT2_GEMV_CASE(kWI4)
    default: return cudaErrorInvalidValue;
    }
#undef GPT2_GEMV_CASE
}

// ---- decode attention ----------------------------------------------------
// One CTA per head ("model.fir" g2.attn_decode runs one lane per head; here a
// head gets a CTA).  Appends this token's k, v at `pos` of the head's cache,
// then its 4 warps each take a contiguous slice of positions 0..pos and run
// an online softmax over it in tiles of 32 positions (one position per lane
// for the scores, one head dimension per lane for the weighted values); the
// slices are merged at the end by rescaling to the common maximum.
template <int D>
__global__ void __launch_bounds__(128) k_attention(const AttnArgs a)
{
    constexpr int NW = 4;
    constexpr int DPL = D / 32;
    __shared__ __align__(16) float qs[D];
    __shared__ float wm[NW], wl[NW];
    __shared__ float wo[NW][D];
    pdl_launch_dependents();
    pdl_wait();
    const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.n_head * D;
    int pos = __ldcg(&a.st->pos);
    if (pos < 0 || pos >= a.n_positions) {
        if (tid == 0 && h == 0) record_error(a.st, kDevErrBadPosition, pos);
        for (int t = tid; t < D; t += 128) a.out[h * D + t] = 0.f;
        return;
    }
    float *kh = a.k_cache + size_t(h) * a.n_positions * D;
    float *vh = a.v_cache + size_t(h) * a.n_positions * D;
    for (int t = tid; t < D; t += 128) {
        qs[t] = __ldcg(a.qkv + h * D + t);
        kh[size_t(pos) * D + t] = __ldcg(a.qkv + E + h * D + t);
        vh[size_t(pos) * D + t] = __ldcg(a.qkv + 2 * E + h * D + t);
    }
    __syncthreads();

    const int n = pos + 1;
    const int per = (n + NW - 1) / NW;
    const int j0 = warp * per, j1 = min(n, j0 + per);
    float m = -INFINITY, l = 0.f;
    float o[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[k] = 0.f;
    const float4 *q4 = reinterpret_cast<const float4 *>(qs);
    for (int base = j0; base < j1; base += 32) {
        const int j = base + lane;
        const bool valid = j < j1;
        float sc = -INFINITY;
        if (valid) {
            const float4 *kr = reinterpret_cast<const float4 *>(kh + size_t(j) * D);
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < D / 4; ++i) {
                const float4 kv = kr[i], qv = q4[i];
                d = fmaf(qv.x, kv.x, d);
                d = fmaf(qv.y, kv.y, d);
                d = fmaf(qv.z, kv.z, d);
                d = fmaf(qv.w, kv.w, d);
            }
            sc = d * a.scale;
        }
        const float mn = fmaxf(m, warp_max(sc));
        const float corr = expf(m - mn);            // 0 on the first tile
        const float p = valid ? expf(sc - mn) : 0.f;
        l = fmaf(l, corr, warp_sum(p));
#pragma unroll
        for (int k = 0; k < DPL; ++k) o[k] *= corr;
        const int cnt = min(32, j1 - base);
        for (int i = 0; i < cnt; ++i) {
            const float pi = __shfl_sync(0xffffffffu, p, i);
            const float *vr = vh + size_t(base + i) * D;
#pragma unroll
            for (int k = 0; k < DPL; ++k) o[k] = fmaf(pi, vr[lane + 32 * k], o[k]);
        }
        m = mn;
    }
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
#pragma unroll
    for (int k = 0; k < DPL; ++k) wo[warp][lane + 32 * k] = o[k];
    __syncthreads();
    for (int t = tid; t < D; t += 128) {
        float M = -INFINITY;
        for (int w = 0; w < NW; ++w)
            if (wl[w] > 0.f) M = fmaxf(M, wm[w]);
        float L = 0.f, O = 0.f;
        for (int w = 0; w < NW; ++w) {
            if (wl[w] > 0.f) {
                const float e = expf(wm[w] - M);
                L = fmaf(wl[w], e, L);
                O = fmaf(wo[w][t], e, O);
            }
        }
        a.out[h * D + t] = O / L;
    }
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_head);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (a.head_dim) {
    case 32: return cudaLaunchKernelEx(&cfg, k_attention<32>, a);
    case 64: return cudaLaunchKernelEx(&cfg, k_attention<64>, a);
    case 128: return cudaLaunchKernelEx(&cfg, k_attention<128>, a);
    default: return cudaErrorInvalidValue;
    }
}

// ---- warp-per-row LayerNorm ------------------------------------------------
__global__ void __launch_bounds__(256) k_layernorm_rows(const float *x, const float *g, const float *b, int rows,
                                                        int n, float eps, float *y)
{
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *xr = x + size_t(row) * n;
    float mean, rstd;
    warp_ln_stats(xr, n, eps, mean, rstd);
    float *yr = y + size_t(row) * n;
    for (int i = lane; i < n; i += 32) yr[i] = (xr[i] - mean) * rstd * g[i] + b[i];
}

cudaError_t launch_layernorm_rows(const float *x, const float *g, const float *b, int rows, int n, float eps,
                                  float *y, cudaStream_t s)
{
    const int warps_per_block = 8;
    const int grid = (rows + warps_per_block - 1) / warps_per_block;
    k_layernorm_rows<<<grid, warps_per_block * 32, 0, s>>>(x, g, b, rows, n, eps, y);
    return cudaGetLastError();
}

// ---- device state --------------------------------------------------------
__global__ void k_set_state(DeviceState *st, int32_t tok, int32_t pos, int32_t flags, int32_t *out_ids)
{
    if (flags & kClearErr) {
        st->err = 0;
        st->err_info = 0;
        st->abort = 0;
    }
    if (flags & kSetTokPos) {
        st->tok = tok;
        st->pos = pos;
    }
    if (flags & kResetOut) st->n_out = 0;
    if (flags & kSeedOutWithNext) {
        out_ids[0] = st->next_tok;
        st->n_out = 1;
        st->tok = st->next_tok;
    }
}

cudaError_t launch_set_state(DeviceState *st, int32_t tok, int32_t pos, int32_t flags, int32_t *out_ids,
                             cudaStream_t s)
{
    k_set_state<<<1, 1, 0, s>>>(st, tok, pos, flags, out_ids);
    return cudaGetLastError();
}

}  // namespace gpt2
