// Persistent decode kernel: every pass of a launch (prompt tokens and greedy
// steps) in one cooperative grid of one CTA per SM.
//
// Why: at batch 1 a pass is 61 small dependent matrix-vector products and
// attentions; as separate kernels each one pays a launch/dependency release
// and several dependent memory round trips, and the GPU idles between them.
// Here
//   * one producer warp per CTA streams that CTA's share of every weight
//     matrix, phase after phase and token after token, into a ring of
//     shared-memory stages with 1-D bulk copies (cp.async.bulk).  It waits only
//     for free stages, never for activations, so HBM keeps streaming while the
//     consumers wait for their inputs;
//   * eight consumer warps run the phases in order: fused LayerNorm prologue,
//     row dot products out of the ring, bias / gelu_new / residual epilogue;
//   * activations move between CTAs as 64-bit words that carry the value and
//     an epoch (the pass and phase that wrote it); a consumer spins on the
//     words of its input vector until every epoch matches, so a phase boundary
//     costs one L2 round trip instead of a grid barrier plus a read.  Each
//     buffer is rewritten only after every CTA has consumed it (the data
//     dependences of the pass order all writes after all reads), so no other
//     synchronisation is needed;
//   * the tied head ends with a per-CTA argmax key and a last-arriving-CTA
//     reduction that publishes the next token as one more tagged word: greedy
//     decoding never leaves the GPU.
// Every spin is bounded (2 s of %globaltimer) and checks a grid-wide abort
// word; on timeout the kernel records GPT2_ERR_TIMEOUT and every CTA returns
// after draining its bulk copies.
#include "gemv_dev.cuh"
#include "persistent.h"

namespace gpt2 {

#ifdef GPT2_TRACE
// Debug builds only: SM-clock stamps of three CTAs (0, 13, last) at four
// points of every phase of the first 64 passes.
__device__ long long g_trace[3][64][64][5];
__device__ long long g_trace2[128][6];   // CTA 0, head phase of pass 20: stamps inside each chunk
#define GPT2_TRACE2(j, kk) ((void)0)
__device__ __forceinline__ void trace(int s, int i, int k)
{
    const int b = blockIdx.x == 0 ? 0 : blockIdx.x == 13 ? 1 : blockIdx.x == gridDim.x - 1 ? 2 : -1;
    if (b >= 0 && threadIdx.x == 0 && s < 64 && i < 64) g_trace[b][s][i][k] = clock64();
}
#define GPT2_TRACE_AT(s, i, k) trace(s, i, k)
#else
#define GPT2_TRACE_AT(s, i, k) ((void)0)
#define GPT2_TRACE2(j, kk) ((void)0)
#endif

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kPThreads = kConsumers + 32;     // + one producer warp
constexpr int kProducerWarp = kConsumerWarps;

// ---- tagged words ------------------------------------------------------------
__device__ __forceinline__ void ll_store(uint64_t *p, uint32_t bits, uint32_t epoch)
{
    const uint64_t w = (uint64_t(epoch) << 32) | bits;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ll_load(const uint64_t *p)
{
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ int ld_relaxed_int(const int *p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// Shared control block of a CTA.
struct Ctl {
    int abort;                         // this CTA saw a timeout / abort
    int last;                          // this CTA is the last arrival of a head phase
    unsigned long long keys[kConsumerWarps];
    float red[2][kConsumerWarps];      // LayerNorm: per-warp sums, sums of squares
    // block phases: reduction scratch, double-buffered by phase parity so a
    // phase can start without a barrier
    float rowred[2][kConsumerWarps][kMaxBlockRows];
    float stn[2][kConsumerWarps], stmean[2][kConsumerWarps], stm2[2][kConsumerWarps];
};

__device__ __forceinline__ bool abort_seen(const PersistArgs &a)
{
    return ld_relaxed_int(&a.st->abort) != 0;
}

__device__ __forceinline__ void raise_abort(const PersistArgs &a, int info)
{
    record_error(a.st, kDevErrTimeout, info);
    atomicExch(&a.st->abort, 1);
}

// Spins until word p carries `epoch`; returns its low 32 bits.  false on
// timeout or grid abort.
__device__ __forceinline__ bool ll_wait(const PersistArgs &a, const uint64_t *p, uint32_t epoch, uint32_t &bits)
{
    uint64_t w = ll_load(p);
    unsigned long long t0 = 0;
    uint32_t it = 0;
    while (uint32_t(w >> 32) != epoch) {
        if ((++it & 127u) == 0) {
            if (abort_seen(a)) return false;
            const unsigned long long t = global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > kWaitLimitNs) {
                raise_abort(a, 1000 + int(blockIdx.x));
                return false;
            }
        }
        w = ll_load(p);
    }
    bits = uint32_t(w);
    return true;
}

__device__ __forceinline__ void ll_load2(const uint64_t *p, uint64_t &w0, uint64_t &w1)
{
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
}

// All consumer threads: dst[i] = value of src[i] once tagged `epoch`, i < n
// (n even, src 16-byte aligned).  Each thread issues all of its 16-byte loads
// at once and re-polls only the pairs still carrying an old epoch, so a
// whole vector arrives in about one L2 round trip.
__device__ __forceinline__ bool ll_read_vec(const PersistArgs &a, const uint64_t *src, int n, uint32_t epoch,
                                            float *dst, int tid, float *psum = nullptr)
{
    float sum = 0.f;
    constexpr int kPer = 4;                      // pairs per thread per round
    const int npairs = n >> 1;
    for (int base = 0; base < npairs; base += kPer * kConsumers) {
        uint64_t w0[kPer], w1[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int p = base + tid + j * kConsumers;
            if (p < npairs) ll_load2(src + 2 * p, w0[j], w1[j]);
        }
        unsigned long long t0 = 0;
        for (uint32_t it = 0;; ++it) {
            bool all = true;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const int p = base + tid + j * kConsumers;
                if (p < npairs && (uint32_t(w0[j] >> 32) != epoch || uint32_t(w1[j] >> 32) != epoch)) {
                    all = false;
                    ll_load2(src + 2 * p, w0[j], w1[j]);
                }
            }
            if (all) break;
            if ((it & 63u) == 63u) {
                if (abort_seen(a)) return false;
                const unsigned long long t = global_ns();
                if (t0 == 0) t0 = t;
                else if (t - t0 > kWaitLimitNs) {
                    raise_abort(a, 1000 + int(blockIdx.x));
                    return false;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int p = base + tid + j * kConsumers;
            if (p < npairs) {
                const float v0 = __uint_as_float(uint32_t(w0[j])), v1 = __uint_as_float(uint32_t(w1[j]));
                dst[2 * p] = v0;
                dst[2 * p + 1] = v1;
                sum += v0 + v1;
            }
        }
    }
    if (psum) *psum = sum;
    return true;
}

__device__ __forceinline__ uint32_t epoch_of(uint32_t seq, int phase) { return (seq << 6) | uint32_t(phase + 1); }

// Rows [r0, r1) of this CTA in a GEMV phase.
__device__ __forceinline__ void cta_rows(const PPhase &ph, int &r0, int &r1)
{
    r0 = blockIdx.x * ph.rpc;
    r1 = min(ph.out, r0 + ph.rpc);
    if (r1 < r0) r1 = r0;
}

// ---- producer: stream every chunk of every GEMV phase, in consumer order ------
template <int WT>
__device__ void producer(const PersistArgs &a, const PPhase *sph, uint8_t *ring, uint64_t *full, uint64_t *empty)
{
    uint32_t k = 0;                    // chunk counter (ring position)
    const uint64_t pol = l2_evict_first_policy();
    uint64_t pol_keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
    // the head's leading rows of this CTA, kept in L2 across passes
    const PPhase &hp = sph[a.n_phases - 1];
    int h0, h1;
    cta_rows(hp, h0, h1);
    const int hkeep = h0 + int(float(h1 - h0) * a.head_l2_frac);
    const uint32_t hrb = uint32_t(hp.in) * 4u;
    bool ok = true;
    for (int s = 0; s < a.n_steps && ok; ++s) {
        // The blocks of a pass are latency-bound and leave HBM mostly idle:
        // pull the kept head rows into L2 now (a no-op when they stayed).
        for (int r = h0; r < hkeep; r += 64) {
            const uint32_t bytes = uint32_t(min(64, hkeep - r)) * hrb;
            asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(
                             static_cast<const uint8_t *>(hp.W) + size_t(r) * hrb),
                         "r"(bytes), "l"(pol_keep)
                         : "memory");
        }
        for (int i = 0; i < a.n_phases && ok; ++i) {
            const PPhase &ph = sph[i];
            if (ph.type == kPhAttn) continue;
            int r0, r1;
            cta_rows(ph, r0, r1);
            const int wt = ph.type == kPhHead ? int(kWF32) : WT;
            const uint32_t rb = row_bytes(wt, ph.in);
            const int G = ph.in >> 5;
            for (int rs = r0; rs < r1; rs += ph.chunk_rows) {
                const int n = min(ph.chunk_rows, r1 - rs);
                const uint32_t st = k % uint32_t(a.n_stages);
                if (k >= uint32_t(a.n_stages)) {
                    const uint32_t par = ((k / a.n_stages) - 1u) & 1u;
                    unsigned long long t0 = 0;
                    uint32_t it = 0;
                    while (!mbar_try_wait(&empty[st], par)) {
                        if ((++it & 255u) == 0) {
                            if (abort_seen(a)) { ok = false; break; }
                            const unsigned long long t = global_ns();
                            if (t0 == 0) t0 = t;
                            else if (t - t0 > kWaitLimitNs) { raise_abort(a, 2000 + int(blockIdx.x)); ok = false; break; }
                        }
                    }
                    if (!ok) break;
                }
                uint8_t *dst = ring + size_t(st) * a.stage_bytes;
                const uint32_t b0 = uint32_t(n) * rb;
                uint32_t total = b0;
                if (wt == kWI4) total += uint32_t(n) * uint32_t(G) * 4u + uint32_t(n) * uint32_t(ph.in >> 6);
                mbar_arrive_expect_tx(&full[st], total);
                const uint64_t cp = (ph.type == kPhHead && rs < hkeep) ? pol_keep : pol;
                bulk_g2s_hint(dst, static_cast<const uint8_t *>(ph.W) + size_t(rs) * rb, b0, &full[st], cp);
                if (wt == kWI4) {
                    bulk_g2s_hint(dst + ph.stage_scale_off, ph.scales + size_t(rs) * G, uint32_t(n) * uint32_t(G) * 4u,
                                  &full[st], pol);
                    bulk_g2s_hint(dst + ph.stage_zero_off, ph.zeros + size_t(rs) * (ph.in >> 6),
                                  uint32_t(n) * uint32_t(ph.in >> 6), &full[st], pol);
                }
                ++k;
            }
        }
    }
    // drain: the copies still in flight must land before the CTA exits
    const uint32_t first = k > uint32_t(a.n_stages) ? k - uint32_t(a.n_stages) : 0u;
    for (uint32_t j = first; j < k; ++j) {
        const uint32_t st = j % uint32_t(a.n_stages), par = (j / a.n_stages) & 1u;
        unsigned long long t0 = 0;
        uint32_t it = 0;
        while (!mbar_try_wait(&full[st], par)) {
            if ((++it & 255u) == 0) {
                const unsigned long long t = global_ns();
                if (t0 == 0) t0 = t;
                else if (t - t0 > kWaitLimitNs) break;
            }
        }
    }
}

// ---- consumers -------------------------------------------------------------

constexpr int kGroup = 4;       // rows a warp carries at once (independent chains)

// Contribution of one 4-input column `c` of stored row `rl` of a stage to the
// row's dot product with x (x4[c] = x[4c..4c+3]).  A column is 16 bytes of an
// fp32 row, 8 bytes of an fp16 row, 2 bytes (4 codes) of an int4 row; for
// int4, sum_k (q_k - z) s x_k = s (sum_k q_k x_k - z sum_k x_k) with the
// group's sum of x precomputed and the z term taken once per group
// (c % 8 == 0).
template <int WT>
__device__ __forceinline__ float col_dot(const uint8_t *stg, int rl, int in, int c, const float4 &x,
                                         const float *xsum, uint32_t soff, uint32_t zoff, float acc)
{
    const int cols = in >> 2;
    if (WT == kWF32) {
        const float4 v = reinterpret_cast<const float4 *>(stg)[size_t(rl) * cols + c];
        return fmaf(v.x, x.x, fmaf(v.y, x.y, fmaf(v.z, x.z, fmaf(v.w, x.w, acc))));
    } else if (WT == kWF16) {
        const uint2 u = reinterpret_cast<const uint2 *>(stg)[size_t(rl) * cols + c];
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        return fmaf(a.x, x.x, fmaf(a.y, x.y, fmaf(b.x, x.z, fmaf(b.y, x.w, acc))));
    } else {
        const int G = in >> 5, g = c >> 3;
        const uint32_t q = reinterpret_cast<const uint16_t *>(stg)[size_t(rl) * cols + c];
        // exact small integer -> float: 2^23 + q carries q in its low mantissa bits
        const float q0 = __uint_as_float(0x4B000000u | (q & 15u)) - 8388608.0f;
        const float q1 = __uint_as_float(0x4B000000u | ((q >> 4) & 15u)) - 8388608.0f;
        const float q2 = __uint_as_float(0x4B000000u | ((q >> 8) & 15u)) - 8388608.0f;
        const float q3 = __uint_as_float(0x4B000000u | ((q >> 12) & 15u)) - 8388608.0f;
        float d = fmaf(q0, x.x, fmaf(q1, x.y, fmaf(q2, x.z, q3 * x.w)));
        if ((c & 7) == 0) {
            const float z = float(((stg + zoff)[size_t(rl) * (in >> 6) + (g >> 1)] >> ((g & 1) * 4)) & 15);
            d = fmaf(-z, xsum[g], d);
        }
        return fmaf(reinterpret_cast<const float *>(stg + soff)[size_t(rl) * G + g], d, acc);
    }
}

// Sums 4 per-lane values over the warp in 6 shuffles; afterwards lane l holds
// the total of row ((l>>4)&1)*2 + ((l>>3)&1): lanes 0, 8, 16, 24 hold rows
// 0..3.  Fixed order: the result is reproducible bit for bit.
__device__ __forceinline__ float warp_sum4(float (&v)[kGroup], int lane)
{
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool hi = lane & 16;
        const float send = hi ? v[i] : v[i + 2], keep = hi ? v[i + 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    {
        const bool hi = lane & 8;
        const float send = hi ? v[0] : v[1], keep = hi ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 4);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    return v[0];
}
__device__ __forceinline__ int warp_sum4_row(int lane) { return ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1); }

// Bounded wait, by one warp, for stage `kk` of the ring (chunk counter kk).
__device__ __forceinline__ bool wait_chunk(const PersistArgs &a, uint64_t *full, uint32_t kk)
{
    const uint32_t st = kk % uint32_t(a.n_stages), par = (kk / a.n_stages) & 1u;
    if (mbar_test_wait(&full[st], par)) return true;      // usually landed long ago
    unsigned long long t0 = 0;
    uint32_t it = 0;
    while (!mbar_try_wait(&full[st], par)) {
        if ((++it & 255u) == 0) {
            if (abort_seen(a)) return false;
            const unsigned long long t = global_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > kWaitLimitNs) {
                raise_abort(a, 3000 + int(blockIdx.x));
                return false;
            }
        }
    }
    return true;
}


struct CSmem {
    float *x_raw;      // the residual stream as last read (E)
    float *vec;        // the phase's input vector, normalised for LN phases (max(4E, E))
    float *xsum;       // per-group sums of vec (int4)
    float *rowval;     // bias of this CTA's rows of the phase
    float *qs, *wm, *wl, *wo;   // attention scratch
    float *kv;                  // attention: this head's cached K then V rows, first kv_cap positions
    uint64_t *kv_bar;           // completion of the K/V bulk copies
    int kv_cap;
    uint32_t kv_uses;           // bulk copies issued so far (barrier parity)
};

template <int WT>
__device__ __forceinline__ bool gemv_phase(const PersistArgs &a, const PPhase &ph, int phase, int s, uint32_t seq,
                                           Ctl &ctl, CSmem &sm, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                           uint32_t &k, unsigned long long &best)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int in = ph.in;
    const bool ln = ph.mode == kModeLnBias || ph.mode == kModeEmbLnBias || ph.mode == kModeLnBiasGelu ||
                    ph.type == kPhHead;
    int r0, r1;
    cta_rows(ph, r0, r1);
    // Loads that do not depend on this pass, issued before waiting for the
    // input: LayerNorm gamma/beta for this thread's element pairs
    // (pair p = tid + j * kConsumers holds elements 2p, 2p+1) and this CTA's
    // biases.
    constexpr int kPairs = 8;                 // n_embd <= 2 * 8 * 256 = 4096
    const int npairs = in >> 1;
    float bias0 = 0.f, bias1 = 0.f;          // at most 2 * kConsumers rows (checked on the host)
    if (ph.bias) {
        if (tid < r1 - r0) bias0 = __ldg(ph.bias + r0 + tid);
        if (tid + kConsumers < r1 - r0) bias1 = __ldg(ph.bias + r0 + tid + kConsumers);
    }

    consumer_sync();   // the previous phase is done with vec / x_raw / rowval
    GPT2_TRACE_AT(s, phase, 0);
    if (ph.bias) {
        if (tid < r1 - r0) sm.rowval[tid] = bias0;
        if (tid + kConsumers < r1 - r0) sm.rowval[tid + kConsumers] = bias1;
    }
    bool ok = true;
    float psum = 0.f;
    if (ph.mode == kModeEmbLnBias) {
        const int pos = a.pos0 + s;
        int tok;
        if (s < a.n_prompt) {
            tok = a.prompt ? __ldg(a.prompt + s) : a.tok_first;
        } else if (s == 0) {
            tok = ld_relaxed_int(&a.st->tok);
        } else {
            uint32_t b = 0;
            ok = ll_wait(a, a.ll_tok, epoch_of(seq - 1, a.n_phases - 1), b);
            tok = int(b);
        }
        if (tok < 0 || tok >= a.V || pos < 0 || pos >= a.P) {
            if (tid == 0) record_error(a.st, tok < 0 || tok >= a.V ? kDevErrBadToken : kDevErrBadPosition, tok);
            tok = min(max(tok, 0), a.V - 1);
        }
        const int pp = min(max(pos, 0), a.P - 1);
        const float2 *te = reinterpret_cast<const float2 *>(a.wte + size_t(tok) * in);
        const float2 *pe = reinterpret_cast<const float2 *>(a.wpe + size_t(pp) * in);
        for (int p = tid; p < npairs; p += kConsumers) {
            const float2 t = __ldg(te + p), q = __ldg(pe + p);
            const float v0 = t.x + q.x, v1 = t.y + q.y;
            sm.x_raw[2 * p] = v0;
            sm.x_raw[2 * p + 1] = v1;
            psum += v0 + v1;
        }
    } else {
        ok = ll_read_vec(a, a.ll[ph.in_buf], in, epoch_of(seq, ph.in_src), ln ? sm.x_raw : sm.vec, tid, &psum);
    }
    if (!ok) atomicExch(&ctl.abort, 1);
    if (ln) {
        const float w = warp_sum(psum);
        if (lane == 0) ctl.red[0][warp] = w;
    }
    consumer_sync();
    GPT2_TRACE_AT(s, phase, 1);
    if (ln) {
        // mean, then the biased variance around it, each reduced over all
        // consumer threads in a fixed order ("model.fir" g2.layernorm)
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += ctl.red[0][w];
        const float mean = tot / float(in);
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            const int p = tid + j * kConsumers;
            if (p < npairs) {
                const float d0 = sm.x_raw[2 * p] - mean, d1 = sm.x_raw[2 * p + 1] - mean;
                sq = fmaf(d0, d0, fmaf(d1, d1, sq));
            }
        }
        sq = warp_sum(sq);
        if (lane == 0) ctl.red[1][warp] = sq;
        consumer_sync();
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) ss += ctl.red[1][w];
        const float rstd = 1.0f / sqrtf(ss / float(in) + a.eps);
        // (the head streams 154 MB; its gamma/beta loads need not be early)
#pragma unroll
        for (int j = 0; j < kPairs; ++j) {
            const int p = tid + j * kConsumers;
            if (p < npairs) {
                const float2 g2 = __ldg(reinterpret_cast<const float2 *>(ph.ln_w) + p);
                const float2 b2 = __ldg(reinterpret_cast<const float2 *>(ph.ln_b) + p);
                sm.vec[2 * p] = (sm.x_raw[2 * p] - mean) * rstd * g2.x + b2.x;
                sm.vec[2 * p + 1] = (sm.x_raw[2 * p + 1] - mean) * rstd * g2.y + b2.y;
            }
        }
        consumer_sync();
    }
    const int wt = ph.type == kPhHead ? int(kWF32) : WT;
    if (wt == kWI4) {
        for (int g = warp; g < (in >> 5); g += kConsumerWarps) {
            const float v = warp_sum(sm.vec[g * 32 + lane]);
            if (lane == 0) sm.xsum[g] = v;
        }
        consumer_sync();
    }
    GPT2_TRACE_AT(s, phase, 2);
#ifdef GPT2_TRACE
    long long waited = 0;
#endif
    // Rows: warp w owns rows w, w+8, w+16, ... of this CTA's range and takes
    // them kGroup at a time as independent chains (lanes split the columns);
    // no CTA-wide barrier until the next phase.  Row i sits in chunk i / C
    // (C = rows per stage).  A warp releases a stage (one arrival of eight)
    // once it is done with it, after waiting for its data even when it has no
    // row there, so an arrival never counts toward the stage's previous use.
    const uint32_t epoch = epoch_of(seq, phase);
    const int nrows = r1 - r0, C = ph.chunk_rows;
    const int nchunks = (nrows + C - 1) / C;
    const int cols = in >> 2;
    const float4 *x4 = reinterpret_cast<const float4 *>(sm.vec);
    const uint32_t k0 = k;
    int released = 0;       // chunks [0, released) released by this warp
    bool okw = true;
    auto release_to = [&](int q_end) {
        for (; released < q_end; ++released) {
#ifdef GPT2_TRACE
            const long long tw = clock64();
#endif
            if (okw && !wait_chunk(a, full, k0 + released)) okw = false;
#ifdef GPT2_TRACE
            waited += clock64() - tw;
#endif
            __syncwarp();
            if (lane == 0)
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty[(k0 + released) % uint32_t(a.n_stages)]))
                             : "memory");
        }
    };
    for (int i0 = warp; i0 < nrows; i0 += kConsumerWarps * kGroup) {
        const int ng = min(kGroup, (nrows - i0 + kConsumerWarps - 1) / kConsumerWarps);
        const uint8_t *stg[kGroup];
        int rl[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
            const int i = i0 + g * kConsumerWarps;
            const int q = g < ng ? i / C : 0;
            rl[g] = g < ng ? i % C : 0;
            stg[g] = ring + size_t((k0 + q) % uint32_t(a.n_stages)) * a.stage_bytes;
            if (g < ng && okw) {
#ifdef GPT2_TRACE
                const long long tw = clock64();
#endif
                if (!wait_chunk(a, full, k0 + q)) okw = false;
#ifdef GPT2_TRACE
                waited += clock64() - tw;
#endif
            }
        }
        float acc[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) acc[g] = 0.f;
        GPT2_TRACE2(i0 / 32, 0);
        if (okw) {
            for (int c = lane; c < cols; c += 32) {
                const float4 x = x4[c];
#pragma unroll
                for (int g = 0; g < kGroup; ++g) {
                    if (g < ng) {
                        if (wt == kWF32) acc[g] = col_dot<kWF32>(stg[g], rl[g], in, c, x, sm.xsum, 0, 0, acc[g]);
                        else if (wt == kWF16) acc[g] = col_dot<kWF16>(stg[g], rl[g], in, c, x, sm.xsum, 0, 0, acc[g]);
                        else acc[g] = col_dot<kWI4>(stg[g], rl[g], in, c, x, sm.xsum, ph.stage_scale_off,
                                                     ph.stage_zero_off, acc[g]);
                    }
                }
            }
        }
        GPT2_TRACE2(i0 / 32, 1);
        const float t = warp_sum4(acc, lane);
        const int g = warp_sum4_row(lane);
        GPT2_TRACE2(i0 / 32, 2);
        if ((lane & 7) == 0 && g < ng && okw) {
            const int r = r0 + i0 + g * kConsumerWarps;
            if (ph.type == kPhHead) {
                a.logits[r] = t;
                const unsigned long long key = argmax_key(t, uint32_t(r));
                best = key > best ? key : best;
            } else {
                float v = t + sm.rowval[r - r0];
                if (ph.mode == kModeLnBiasGelu) v = gelu_new(v);
                else if (ph.mode == kModeBiasRes) v = sm.x_raw[r] + v;
                ll_store(a.ll[ph.out_buf] + r, __float_as_uint(v), epoch);
            }
        }
        GPT2_TRACE2(i0 / 32, 3);
        // chunks before the one holding this warp's next row are done
        const int nxt = i0 + kConsumerWarps * kGroup;
        release_to(nxt < nrows ? nxt / C : nchunks);
        GPT2_TRACE2(i0 / 32, 4);
    }
    release_to(nchunks);
    k = k0 + uint32_t(nchunks);
    if (!okw) atomicExch(&ctl.abort, 1);   // leave at the next barrier, with every stage released
    GPT2_TRACE_AT(s, phase, 3);
#ifdef GPT2_TRACE
    if (threadIdx.x == 0 && s < 64 && phase < 64) {
        const int b = blockIdx.x == 0 ? 0 : blockIdx.x == 13 ? 1 : blockIdx.x == gridDim.x - 1 ? 2 : -1;
        if (b >= 0) g_trace[b][s][phase][4] = waited;
    }
#endif
    return true;
}


// ---- block phases: the 4 matrices of a transformer block ---------------------
//
// The CTA's whole row slice of the matrix (at most kMaxBlockRows rows) sits
// in consecutive ring stages, streamed in ahead of time.  Thread t owns the
// 4-input columns u = t, t + 256, ... of the input vector: it polls the tagged
// words of its columns and, as soon as they carry this pass's epoch,
// multiplies them into every row of the slice, so the dot products proceed
// while the rest of the vector is still arriving.  LayerNorm is folded into
// the matrix: W.LN(x) = rstd * (W.(gamma*x) - mean * c1) + c2 with
// c1 = W.gamma and c2 = W.beta precomputed from the stored weights; the mean
// and variance are combined across threads with Chan's pairwise formula in a
// fixed order while the products run.  One multi-row butterfly per warp and a
// fixed-order sum over warps finish the rows.

constexpr int kMaxUnits = 4;    // columns per thread: in <= 4 * 4 * 256 = 4096

// Sums NR per-lane values over the warp; afterwards lane l holds the total of
// row l >> (5 - log2 NR).  NR - 1 + log2(32 / NR) shuffles, fixed order.
template <int NR>
__device__ __forceinline__ float warp_sum_rows(float (&v)[kMaxBlockRows], int lane)
{
    int off = 16;
#pragma unroll
    for (int n = NR; n > 1; n >>= 1, off >>= 1) {
        const int half = n >> 1;
        const bool hi = lane & off;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = hi ? v[i] : v[i + half], keep = hi ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    return v[0];
}

// Chan's pairwise combination of (count, mean, M2).
__device__ __forceinline__ void chan_combine(float &n, float &mean, float &m2, float nb, float meanb, float m2b)
{
    const float nn = n + nb;
    if (nb == 0.f) return;
    if (n == 0.f) {
        n = nb;
        mean = meanb;
        m2 = m2b;
        return;
    }
    const float d = meanb - mean, f = nb / nn;
    mean = fmaf(d, f, mean);
    m2 = m2 + m2b + d * d * n * f;
    n = nn;
}

// Where row r of a block phase's slice sits in the ring: stage of chunk r / C,
// row r % C of that stage.
struct SliceMap {
    const uint8_t *ring;
    uint32_t k0, n_stages, stage_bytes, row_bytes, soff, zoff, C, G, zb;
    __device__ __forceinline__ const uint8_t *stage(int r) const
    {
        return ring + size_t((k0 + uint32_t(r) / C) % n_stages) * stage_bytes;
    }
};

// Dot of row r's column u (4 inputs) with z, added to acc.
template <int WT>
__device__ __forceinline__ float unit_dot(const SliceMap &m, int r, int u, const float4 &z, float acc)
{
    const uint8_t *st = m.stage(r);
    const uint32_t rr = uint32_t(r) % m.C;
    if (WT == kWF32) {
        const float4 v = reinterpret_cast<const float4 *>(st + rr * m.row_bytes)[u];
        return fmaf(v.x, z.x, fmaf(v.y, z.y, fmaf(v.z, z.z, fmaf(v.w, z.w, acc))));
    } else if (WT == kWF16) {
        const uint2 w = reinterpret_cast<const uint2 *>(st + rr * m.row_bytes)[u];
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
        return fmaf(a.x, z.x, fmaf(a.y, z.y, fmaf(b.x, z.z, fmaf(b.y, z.w, acc))));
    } else {
        // (q - zp) * s per weight, the stored definition of a dequantised weight
        const int g = u >> 3;
        const uint32_t q = reinterpret_cast<const uint16_t *>(st + rr * m.row_bytes)[u];
        const int zp = ((st + m.zoff + rr * m.zb)[g >> 1] >> ((g & 1) * 4)) & 15;
        const float sc = reinterpret_cast<const float *>(st + m.soff + rr * m.G * 4u)[g];
        const float d = fmaf(float(int(q & 15u) - zp), z.x,
                             fmaf(float(int((q >> 4) & 15u) - zp), z.y,
                                  fmaf(float(int((q >> 8) & 15u) - zp), z.z, float(int((q >> 12) & 15u) - zp) * z.w)));
        return fmaf(sc, d, acc);
    }
}

template <int WT, int NR>
__device__ __forceinline__ void block_rows(const SliceMap &m, int R, int u, const float4 &z,
                                           float (&acc)[kMaxBlockRows])
{
#pragma unroll
    for (int r = 0; r < NR; ++r)
        if (r < R) acc[r] = unit_dot<WT>(m, r, u, z, acc[r]);
}

template <int WT>
__device__ __forceinline__ bool block_phase(const PersistArgs &a, const PPhase &ph, int phase, int s, uint32_t seq,
                                            Ctl &ctl, CSmem &sm, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                            uint32_t &k, int par)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int in = ph.in, cols = in >> 2;
    const bool ln = ph.mode != kModeBiasRes;
    int r0, r1;
    cta_rows(ph, r0, r1);
    const int R = r1 - r0, C = ph.chunk_rows;
    const int nchunks = (R + C - 1) / C;
    // pass-independent loads first: this row's constants, this thread's gamma
    float rb = 0.f, rc1 = 0.f, rc2 = 0.f;
    if (tid < R) {
        rb = __ldg(ph.bias + r0 + tid);
        if (ln) {
            rc1 = __ldg(ph.c1 + r0 + tid);
            rc2 = __ldg(ph.c2 + r0 + tid);
        }
    }
    float4 g4[kMaxUnits];
#pragma unroll
    for (int j = 0; j < kMaxUnits; ++j) {
        const int u = tid + j * kConsumers;
        g4[j] = (ln && u < cols) ? __ldg(reinterpret_cast<const float4 *>(ph.ln_w) + u) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
    // No barrier here: the reduction scratch is double-buffered by the parity
    // of the block-phase count (a barrier of the block phase in between
    // separates two uses), and x_raw is rewritten only after data that this
    // CTA's own later epilogue produces has come back.
    GPT2_TRACE_AT(s, phase, 0);
    SliceMap map;
    map.ring = ring;
    map.k0 = k;
    map.n_stages = uint32_t(a.n_stages);
    map.stage_bytes = a.stage_bytes;
    map.row_bytes = WT == kWF32 ? uint32_t(in) * 4 : WT == kWF16 ? uint32_t(in) * 2 : uint32_t(in) / 2;
    map.soff = ph.stage_scale_off;
    map.zoff = ph.stage_zero_off;
    map.C = uint32_t(C);
    map.G = uint32_t(in / 32);
    map.zb = uint32_t(in / 64);
    bool ok = true;
    for (int q = 0; q < nchunks && ok; ++q) ok = wait_chunk(a, full, k + uint32_t(q));
    GPT2_TRACE_AT(s, phase, 1);

    float acc[kMaxBlockRows];
#pragma unroll
    for (int r = 0; r < kMaxBlockRows; ++r) acc[r] = 0.f;
    float sn = 0.f, smean = 0.f, sm2 = 0.f;   // this thread's LayerNorm statistics
    const uint32_t ein = epoch_of(seq, ph.in_src);
    int tok = 0, pp = 0;
    if (ph.mode == kModeEmbLnBias) {
        const int pos = a.pos0 + s;
        if (s < a.n_prompt) {
            tok = a.prompt ? __ldg(a.prompt + s) : a.tok_first;
        } else if (s == 0) {
            tok = ld_relaxed_int(&a.st->tok);
        } else {
            uint32_t b = 0;
            if (!ll_wait(a, a.ll_tok, epoch_of(seq - 1, a.n_phases - 1), b)) ok = false;
            tok = int(b);
        }
        if (tok < 0 || tok >= a.V || pos < 0 || pos >= a.P) {
            if (tid == 0) record_error(a.st, tok < 0 || tok >= a.V ? kDevErrBadToken : kDevErrBadPosition, tok);
            tok = min(max(tok, 0), a.V - 1);
        }
        pp = min(max(pos, 0), a.P - 1);
    }
    const uint64_t *src = ph.mode == kModeEmbLnBias ? nullptr : a.ll[ph.in_buf];
#pragma unroll
    for (int j = 0; j < kMaxUnits; ++j) {
        const int u = tid + j * kConsumers;
        if (u >= cols || !ok) continue;
        float4 x;
        if (ph.mode == kModeEmbLnBias) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(a.wte + size_t(tok) * in) + u);
            const float4 e = __ldg(reinterpret_cast<const float4 *>(a.wpe + size_t(pp) * in) + u);
            x = make_float4(t.x + e.x, t.y + e.y, t.z + e.z, t.w + e.w);
        } else {
            // four tagged words: wait until all carry this pass's epoch
            const uint64_t *p = src + 4 * u;
            uint64_t w0, w1, w2, w3;
            ll_load2(p, w0, w1);
            ll_load2(p + 2, w2, w3);
            unsigned long long t0 = 0;
            for (uint32_t it = 0; uint32_t(w0 >> 32) != ein || uint32_t(w1 >> 32) != ein ||
                                  uint32_t(w2 >> 32) != ein || uint32_t(w3 >> 32) != ein;
                 ++it) {
                if ((it & 63u) == 63u) {
                    if (abort_seen(a)) { ok = false; break; }
                    const unsigned long long tn = global_ns();
                    if (t0 == 0) t0 = tn;
                    else if (tn - t0 > kWaitLimitNs) { raise_abort(a, 1000 + int(blockIdx.x)); ok = false; break; }
                }
                ll_load2(p, w0, w1);
                ll_load2(p + 2, w2, w3);
            }
            if (!ok) continue;
            x = make_float4(__uint_as_float(uint32_t(w0)), __uint_as_float(uint32_t(w1)),
                            __uint_as_float(uint32_t(w2)), __uint_as_float(uint32_t(w3)));
        }
        float4 z = x;
        if (ln) {
            reinterpret_cast<float4 *>(sm.x_raw)[u] = x;      // the residual stream, for the next residual epilogue
            const float m4 = ((x.x + x.y) + (x.z + x.w)) * 0.25f;
            const float d0 = x.x - m4, d1 = x.y - m4, d2 = x.z - m4, d3 = x.w - m4;
            chan_combine(sn, smean, sm2, 4.f, m4, fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, d3 * d3))));
            z = make_float4(x.x * g4[j].x, x.y * g4[j].y, x.z * g4[j].z, x.w * g4[j].w);
        }
        if (R <= 8) block_rows<WT, 8>(map, R, u, z, acc);
        else if (R <= 16) block_rows<WT, 16>(map, R, u, z, acc);
        else block_rows<WT, 32>(map, R, u, z, acc);
    }
    if (!ok) atomicExch(&ctl.abort, 1);
    GPT2_TRACE_AT(s, phase, 2);
    // rows: per-warp multi-row sums, then a fixed-order sum over warps
    float wsum;
    int rowsh;
    if (R <= 8) { wsum = warp_sum_rows<8>(acc, lane); rowsh = 2; }
    else if (R <= 16) { wsum = warp_sum_rows<16>(acc, lane); rowsh = 1; }
    else { wsum = warp_sum_rows<32>(acc, lane); rowsh = 0; }
    if ((lane & ((1 << rowsh) - 1)) == 0) ctl.rowred[par][warp][lane >> rowsh] = wsum;
    if (ln) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float nb = __shfl_xor_sync(0xffffffffu, sn, off);
            const float mb = __shfl_xor_sync(0xffffffffu, smean, off);
            const float qb = __shfl_xor_sync(0xffffffffu, sm2, off);
            // the lower lane of each pair keeps (a, b) order so every lane ends with the same bits
            if (lane & off) { float tn = nb, tm = mb, tq = qb; chan_combine(tn, tm, tq, sn, smean, sm2); sn = tn; smean = tm; sm2 = tq; }
            else chan_combine(sn, smean, sm2, nb, mb, qb);
        }
        if (lane == 0) {
            ctl.stn[par][warp] = sn;
            ctl.stmean[par][warp] = smean;
            ctl.stm2[par][warp] = sm2;
        }
    }
    consumer_sync();   // every warp is done with the stages and has written its sums
    if (lane == 0)
        for (int q = 0; q < nchunks; ++q)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty[(k + uint32_t(q)) % uint32_t(a.n_stages)]))
                         : "memory");
    k += uint32_t(nchunks);
    if (tid < R && ok) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) t += ctl.rowred[par][w][tid];
        float y;
        if (ln) {
            float n = 0.f, mean = 0.f, m2 = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w)
                chan_combine(n, mean, m2, ctl.stn[par][w], ctl.stmean[par][w], ctl.stm2[par][w]);
            const float rstd = 1.0f / sqrtf(m2 / float(in) + a.eps);
            y = fmaf(rstd, t - mean * rc1, rc2) + rb;
        } else {
            y = t + rb;
        }
        const int r = r0 + tid;
        if (ph.mode == kModeLnBiasGelu) y = gelu_new(y);
        else if (ph.mode == kModeBiasRes) y = sm.x_raw[r] + y;
        ll_store(a.ll[ph.out_buf] + r, __float_as_uint(y), epoch_of(seq, phase));
    }
    GPT2_TRACE_AT(s, phase, 3);
    return true;
}

template <int D>
__device__ __forceinline__ bool attn_phase(const PersistArgs &a, const PPhase &ph, int phase, int s, uint32_t seq,
                                           Ctl &ctl, CSmem &sm)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x;
    if (h >= a.H) return true;
    constexpr int DPL = D / 32;
    const int E = a.H * D;
    const int pos = min(max(a.pos0 + s, 0), a.P - 1);
    float *kh = a.kcache + (size_t(ph.layer) * a.H + h) * a.P * D;
    float *vh = a.vcache + (size_t(ph.layer) * a.H + h) * a.P * D;
    consumer_sync();   // previous phase done with the scratch (and with the K/V window)
    // The cached rows 0..pos-1 do not depend on this pass: copy the first
    // kv_cap of them into shared memory (K then V) while q, k, v of this pass
    // are still being produced; rows past the window are pulled toward L2.
    const int n_pre = min(pos, sm.kv_cap);
    float *kw = sm.kv, *vw = sm.kv + size_t(sm.kv_cap) * D;
    if (tid == 0) {
        if (n_pre > 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the window's last reads came first
            const uint32_t bytes = uint32_t(n_pre) * D * 4u;
            mbar_arrive_expect_tx(sm.kv_bar, 2u * bytes);
            bulk_g2s(kw, kh, bytes, sm.kv_bar);
            bulk_g2s(vw, vh, bytes, sm.kv_bar);
        }
        if (pos > n_pre) {
            const uint32_t bytes = uint32_t(pos - n_pre) * D * 4u;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kh + size_t(n_pre) * D), "r"(bytes) : "memory");
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vh + size_t(n_pre) * D), "r"(bytes) : "memory");
        }
    }
    GPT2_TRACE_AT(s, phase, 0);
    const uint32_t ein = epoch_of(seq, ph.in_src);
    const uint64_t *qkv = a.ll[ph.in_buf];
    bool ok = true;
    // q, k, v of this head: three runs of D words, one 16-byte load per thread
    if (tid < 3 * D / 2) {
        const int part = (2 * tid) / D, d = (2 * tid) % D;
        const uint64_t *p = qkv + part * E + h * D + d;
        uint64_t w0, w1;
        ll_load2(p, w0, w1);
        unsigned long long t0 = 0;
        for (uint32_t it = 0; uint32_t(w0 >> 32) != ein || uint32_t(w1 >> 32) != ein; ++it) {
            if ((it & 63u) == 63u) {
                if (abort_seen(a)) { ok = false; break; }
                const unsigned long long t = global_ns();
                if (t0 == 0) t0 = t;
                else if (t - t0 > kWaitLimitNs) { raise_abort(a, 1000 + int(blockIdx.x)); ok = false; break; }
            }
            ll_load2(p, w0, w1);
        }
        if (ok) {
            float *dst = part == 0 ? sm.qs + d : (part == 1 ? kh : vh) + size_t(pos) * D + d;
            dst[0] = __uint_as_float(uint32_t(w0));
            dst[1] = __uint_as_float(uint32_t(w1));
            if (part > 0 && pos < sm.kv_cap) {      // this position's row of the window
                float *wdst = (part == 1 ? kw : vw) + size_t(pos) * D + d;
                wdst[0] = dst[0];
                wdst[1] = dst[1];
            }
        }
    }
    if (n_pre > 0) {
        const uint32_t par = sm.kv_uses & 1u;
        unsigned long long t0 = 0;
        uint32_t it = 0;
        while (!mbar_try_wait(sm.kv_bar, par)) {
            if ((++it & 255u) == 0) {
                if (abort_seen(a)) { ok = false; break; }
                const unsigned long long t = global_ns();
                if (t0 == 0) t0 = t;
                else if (t - t0 > kWaitLimitNs) { raise_abort(a, 4000 + int(blockIdx.x)); ok = false; break; }
            }
        }
        ++sm.kv_uses;
    }
    if (!ok) atomicExch(&ctl.abort, 1);
    consumer_sync();
    GPT2_TRACE_AT(s, phase, 1);

    const int n = pos + 1;
    const int per = (n + kConsumerWarps - 1) / kConsumerWarps;
    const int j0 = warp * per, j1 = min(n, j0 + per);
    float m = -INFINITY, l = 0.f;
    float o[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] = 0.f;
    const float4 *q4 = reinterpret_cast<const float4 *>(sm.qs);
    for (int base = j0; base < j1; base += 32) {
        const int j = base + lane;
        const bool valid = j < j1;
        float sc = -INFINITY;
        if (valid) {
            const float4 *kr = reinterpret_cast<const float4 *>((j < sm.kv_cap ? kw : kh) + size_t(j) * D);
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int i = 0; i < D / 4; i += 2) {
                const float4 k0 = kr[i], k1 = kr[i + 1], qa = q4[i], qb = q4[i + 1];
                d0 = fmaf(qa.x, k0.x, d0);
                d0 = fmaf(qa.y, k0.y, d0);
                d0 = fmaf(qa.z, k0.z, d0);
                d0 = fmaf(qa.w, k0.w, d0);
                d1 = fmaf(qb.x, k1.x, d1);
                d1 = fmaf(qb.y, k1.y, d1);
                d1 = fmaf(qb.z, k1.z, d1);
                d1 = fmaf(qb.w, k1.w, d1);
            }
            sc = (d0 + d1) * a.scale;
        }
        const float mn = fmaxf(m, warp_max(sc));
        const float corr = expf(m - mn);
        const float p = valid ? expf(sc - mn) : 0.f;
        l = fmaf(l, corr, warp_sum(p));
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[c] *= corr;
        const int cnt = min(32, j1 - base);
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            if (i < cnt) {
                const float pi = __shfl_sync(0xffffffffu, p, i);
                const float *vr = (base + i < sm.kv_cap ? vw : vh) + size_t(base + i) * D;
#pragma unroll
                for (int c = 0; c < DPL; ++c) o[c] = fmaf(pi, vr[lane + 32 * c], o[c]);
            }
        }
        m = mn;
    }
    if (lane == 0) {
        sm.wm[warp] = m;
        sm.wl[warp] = l;
    }
#pragma unroll
    for (int c = 0; c < DPL; ++c) sm.wo[warp * D + lane + 32 * c] = o[c];
    consumer_sync();
    GPT2_TRACE_AT(s, phase, 2);
    const uint32_t eout = epoch_of(seq, phase);
    for (int t = tid; t < D; t += kConsumers) {
        float M = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w)
            if (sm.wl[w] > 0.f) M = fmaxf(M, sm.wm[w]);
        float L = 0.f, O = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) {
            if (sm.wl[w] > 0.f) {
                const float e = expf(sm.wm[w] - M);
                L = fmaf(sm.wl[w], e, L);
                O = fmaf(sm.wo[w * D + t], e, O);
            }
        }
        ll_store(a.ll[ph.out_buf] + h * D + t, __float_as_uint(O / L), eout);
    }
    GPT2_TRACE_AT(s, phase, 3);
    return true;
}

// Head epilogue: CTA key -> partials; the last CTA to arrive reduces, publishes
// the token and updates the state.
__device__ __forceinline__ void head_finish(const PersistArgs &a, int s, uint32_t seq, Ctl &ctl,
                                            unsigned long long best)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    best = warp_max_u64(best);
    if (lane == 0) ctl.keys[warp] = best;
    consumer_sync();
    if (tid == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < kConsumerWarps; ++w) b = ctl.keys[w] > b ? ctl.keys[w] : b;
        a.partials[blockIdx.x] = b;
        __threadfence();
        const unsigned int t = atomicAdd(a.counter, 1u);
        ctl.last = (t == gridDim.x - 1) ? 1 : 0;
    }
    consumer_sync();
    if (ctl.last && warp == 0) {
        __threadfence();
        unsigned long long b = 0ull;
        for (int i = lane; i < int(gridDim.x); i += 32) {
            const unsigned long long v = __ldcg(a.partials + i);
            b = v > b ? v : b;
        }
        b = warp_max_u64(b);
        if (lane == 0) {
            const int32_t tok = argmax_key_index(b);
            *a.counter = 0u;
            DeviceState *st = a.st;
            st->next_tok = tok;
            if (s >= a.n_prompt - 1) {
                const int32_t n = st->n_out;
                if (a.out_ids && n >= 0 && n < a.out_cap) a.out_ids[n] = tok;
                st->n_out = n + 1;
            }
            if (s == a.n_steps - 1) {
                st->tok = tok;
                st->pos = a.pos0 + a.n_steps;
                st->seq = int32_t(seq + 1);
            }
            __threadfence();
            ll_store(a.ll_tok, uint32_t(tok), epoch_of(seq, a.n_phases - 1));
        }
    }
}

template <int WT, int D>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(const PersistArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Ctl ctl;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxRing;
    // the phase table lives in shared memory: its fields are re-read after
    // every memory-clobbering barrier or tagged store, and a shared read costs
    // ~30 cycles where a global one (the L1 is small next to the ring) costs
    // an L2 round trip
    PPhase *sph = reinterpret_cast<PPhase *>(smem + 2 * kMaxRing * 8);
    float *f = reinterpret_cast<float *>(smem + 2 * kMaxRing * 8 + kMaxPhases * sizeof(PPhase));
    CSmem sm;
    sm.x_raw = f;
    f += a.E;
    sm.vec = f;
    f += 4 * a.E;
    sm.xsum = f;
    f += (4 * a.E) / 32;
    sm.rowval = f;
    f += a.max_rows;
    sm.qs = f;
    f += D;
    sm.wm = f;
    f += kConsumerWarps;
    sm.wl = f;
    f += kConsumerWarps;
    sm.wo = f;
    f += kConsumerWarps * D;
    // K/V window: kKvWindowBytes, 16-byte aligned (everything before it is a
    // multiple of 4 floats), then its barrier
    sm.kv = f;
    sm.kv_cap = int(kKvWindowBytes / (2u * D * 4u));
    sm.kv_bar = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(f) + kKvWindowBytes);
    sm.kv_uses = 0;
    uint8_t *ring = smem + a.ring_offset;
    const int tid = threadIdx.x, warp = tid >> 5;
    {
        const int words = a.n_phases * int(sizeof(PPhase) / 4);
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.phases);
        uint32_t *dst = reinterpret_cast<uint32_t *>(sph);
        for (int i = tid; i < words; i += blockDim.x) dst[i] = src[i];
    }
    if (tid == 0) {
        for (int i = 0; i < a.n_stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        mbar_init(sm.kv_bar, 1);
        mbar_init_fence();
        ctl.abort = 0;
        ctl.last = 0;
    }
    __syncthreads();
    if (warp == kProducerWarp) {
        if ((tid & 31) == 0) producer<WT>(a, sph, ring, full, empty);
        return;
    }
    const uint32_t seq0 = uint32_t(ld_relaxed_int(&a.st->seq));
    // Every consumer thread runs every phase and every barrier of every
    // pass; after a timeout or abort the waits return at once and the work is
    // skipped, so the threads of a CTA can never end up at different barriers.
    uint32_t k = 0;
    int nblock = 0;
    for (int s = 0; s < a.n_steps; ++s) {
        const uint32_t seq = seq0 + uint32_t(s);
        unsigned long long best = 0ull;
        for (int i = 0; i < a.n_phases; ++i) {
            const PPhase &ph = sph[i];
            if (ph.type == kPhAttn) attn_phase<D>(a, ph, i, s, seq, ctl, sm);
            else if (ph.type == kPhGemv && a.block_mode == 0)
                block_phase<WT>(a, ph, i, s, seq, ctl, sm, ring, full, empty, k, (nblock++) & 1);
            else gemv_phase<WT>(a, ph, i, s, seq, ctl, sm, ring, full, empty, k, best);
            if (ph.type == kPhHead) head_finish(a, s, seq, ctl, best);
        }
    }
}

template <int WT, int D>
static cudaError_t launch_t(const PersistArgs &a, int grid, size_t smem, cudaStream_t s)
{
    void *args[] = {const_cast<PersistArgs *>(&a)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(k_decode_persistent<WT, D>), dim3(grid),
                                       dim3(kPThreads), args, smem, s);
}

cudaError_t launch_persistent(int wtype, const PersistArgs &a, int grid, size_t smem, cudaStream_t s)
{
#define GPT2_P_CASE(WT)                                          \
    switch (a.D) {                                               \
    case 32: return launch_t<WT, 32>(a, grid, smem, s);          \
    case 64: return launch_t<WT, 64>(a, grid, smem, s);          \
    case 128: return launch_t<WT, 128>(a, grid, smem, s);        \
    default: return cudaErrorInvalidValue;                       \
    }
    switch (wtype) {
    case kWF32: GPT2_P_CASE(kWF32)
    case kWF16: GPT2_P_CASE(kWF16)
    case kWI4: GPT2_P_CASE(kWI4)
    default: return cudaErrorInvalidValue;
    }
#undef GPT2_P_CASE
}

size_t persistent_fixed_smem(int E, int D, int max_rows)
{
    const size_t floats = size_t(E) + 4 * size_t(E) + (4 * size_t(E)) / 32 + size_t(max_rows) + D +
                          2 * kConsumerWarps + size_t(kConsumerWarps) * D;
    return align_up(uint32_t(2 * kMaxRing * 8 + kMaxPhases * sizeof(PPhase) + floats * 4 + kKvWindowBytes + 16),
                    128u);
}

int persistent_threads() { return kPThreads; }

// One warp per row: c1 = W.gamma, c2 = W.beta (fixed-order sums).
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

#ifdef GPT2_TRACE
extern "C" int gpt2_debug_trace(long long *host_out)
{
    return cudaMemcpyFromSymbol(host_out, g_trace, sizeof(g_trace)) == cudaSuccess ? 0 : -6;
}
extern "C" int gpt2_debug_trace2(long long *host_out)
{
    return cudaMemcpyFromSymbol(host_out, g_trace2, sizeof(g_trace2)) == cudaSuccess ? 0 : -6;
}
#endif

// Raises the kernel's dynamic shared-memory limit to `limit` (the same value
// for every model, so models of different sizes can coexist; must precede
// the launches) and reports how many CTAs of `smem` bytes fit on one SM.
template <int WT, int D>
static cudaError_t occ_t(size_t smem, size_t limit, int *blocks)
{
    cudaError_t e = cudaFuncSetAttribute(k_decode_persistent<WT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(limit));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k_decode_persistent<WT, D>, kPThreads, smem);
}

cudaError_t persistent_blocks_per_sm(int wtype, int D, size_t smem, size_t limit, int *blocks)
{
#define GPT2_O_CASE(WT)                                  \
    switch (D) {                                         \
    case 32: return occ_t<WT, 32>(smem, limit, blocks);         \
    case 64: return occ_t<WT, 64>(smem, limit, blocks);         \
    case 128: return occ_t<WT, 128>(smem, limit, blocks);       \
    default: return cudaErrorInvalidValue;               \
    }
    switch (wtype) {
    case kWF32: GPT2_O_CASE(kWF32)
    case kWF16: GPT2_O_CASE(kWF16)
    case kWI4: GPT2_O_CASE(kWI4)
    default: return cudaErrorInvalidValue;
    }
#undef GPT2_O_CASE
}

}  // namespace gpt2
