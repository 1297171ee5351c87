// Cluster decode kernel: the decode pass with two GPU-wide exchanges per
// transformer block.
//
// A pass needs the whole output vector of one step on every SM before the
// next step can start (LayerNorm needs all of x, a linear needs all of its
// input).  Measured on GB300, one such GPU-wide exchange costs ~1.4-3 us, so
// a pass of 61 of them cannot be fast.  Here one block needs two:
//
//   head clusters (one per attention head, 4 CTAs):
//     wait for x (GPU-wide) -> LN1 -> this head's q, k, v rows of the QKV
//     matrix (a quarter per CTA) -> exchanged inside the cluster through
//     distributed shared memory -> attention, positions split over the 4 CTAs,
//     partial softmax states exchanged the same way -> the head's slice of
//     the output projection (split-K by head: columns hD..hD+D, a quarter of
//     the rows per CTA) -> added into x_new
//   fc clusters (the other CTAs):
//     wait for x_new (GPU-wide) -> LN2 -> fr rows of the fc matrix, gelu_new ->
//     the matching fr columns of the MLP projection (split-K), reduced over
//     the cluster -> added into the next x
//   every CTA: wait for the last x -> LN_f -> its rows of the tied head ->
//     argmax (or a temperature draw) -> the next token (a tagged word read by
//     the next pass).
//
// GPU-wide sums are fixed-point atomic additions that carry their own count
// (see kFixScale below): integer addition does not depend on the order of the
// atomics, so every run gives the same bits, and a reader polls the words
// until their counts are complete.  Sums are double-buffered by pass parity;
// each CTA zeroes its share of the other parity after the first wait of a
// pass (by then every CTA has finished the previous pass).
//
// Weights stream through a ring of shared-memory stages (one producer thread,
// cp.async.bulk, mbarriers); a CTA's slice of a layer fits the ring, so it is
// resident before the layer's input arrives.  Every wait is bounded by 2 s of
// %globaltimer; on timeout the kernel records GPT2_ERR_TIMEOUT, raises the
// abort word and runs its remaining steps without waiting; all CTAs of a
// cluster meet at a final cluster barrier, so no CTA exits while a peer may
// still write its shared memory.
#include "cluster.h"
#include "gemv_dev.cuh"

#include <algorithm>

namespace gpt2 {

#ifdef GPT2_CTRACE
// Debug builds only: %globaltimer, SM clock and thread 0's accumulated
// ring-stage wait (clock cycles) of every CTA at the phase boundaries of two
// passes.
constexpr int kTrCtas = 160, kTrPasses = 2, kTrSlots = 208, kTrPass0 = 20;
__device__ unsigned long long g_ctrace[kTrCtas][kTrPasses][kTrSlots][6];
__device__ __forceinline__ void ctrace(int s, int slot, unsigned long long waited, const unsigned long long *sub)
{
    if (threadIdx.x == 0 && blockIdx.x < kTrCtas && s >= kTrPass0 && s < kTrPass0 + kTrPasses && slot < kTrSlots) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        g_ctrace[blockIdx.x][s - kTrPass0][slot][0] = t;
        g_ctrace[blockIdx.x][s - kTrPass0][slot][1] = clock64();
        g_ctrace[blockIdx.x][s - kTrPass0][slot][2] = waited;
        for (int i = 0; i < 3; ++i) g_ctrace[blockIdx.x][s - kTrPass0][slot][3 + i] = sub[i];
    }
}
#define CTRACE(s, slot) ctrace(s, slot, *c.twait, c.tsub)
// stamps inside a dot-product phase, at slots c.tslot + i of pass c.tpass
#define CSUB(i) ctrace(c.tpass, c.tslot + (i), *c.twait, c.tsub)
#define TSET(s, slot) (c.tpass = (s), c.tslot = (slot))
#else
#define CTRACE(s, slot) ((void)0)
#define CSUB(i) ((void)0)
#define TSET(s, slot) ((void)0)
#endif

namespace {

constexpr int kCWarps = 8;
constexpr int kCThreads = kCWarps * 32;
constexpr int kCAll = kCThreads + 32;      // + producer warp
constexpr int kCRing = kClusterRing;
// Residual sums: each contribution is one 64-bit atomic addition of
//   (round(v * 2^24) + 2^40) + 2^56
// so a word holds the biased fixed-point sum in its low 56 bits and the
// number of contributions above.  A reader polls its words until the count
// is complete: the data is its own arrival flag (one L2 round trip, no
// counter, no release fence), and integer addition makes the sum independent
// of the order of the atomics.  |v| <= kFixLimit < 2^16 keeps each term in
// [0, 2^41), so the low field holds 2^15 terms; the count field (bits 56..63)
// holds at most 255 contributions, which bounds the contributors of one sum
// (the host checks it).  A value outside the limit (or NaN) is clamped and
// recorded as a range error, never silently summed.
constexpr float kFixScale = 16777216.0f;              // 2^24
constexpr float kFixLimit = 65000.0f;
constexpr unsigned long long kFixBias = 1ull << 40;
constexpr int kCountShift = 56;
constexpr uint32_t kKvWin = 8192;          // K/V rows of this CTA's positions held in shared memory
// Attention: up to this many positions per CTA, one lane per head dimension
// (pairs of positions per warp); more, one lane per position (32 per tile).
constexpr int kLanePerDimMax = 48;
constexpr uint32_t kBarBytes = 512;        // mbarriers at the start of shared memory

// Shared-memory layout before the ring (byte offsets): barriers, x, LN(x),
// this head's q | k | v, the cluster's attention partials, the attention
// output, the MLP hidden slice, a scratch vector, the layer parameters, the
// K/V window and the layer table.
struct CLayout {
    uint32_t x, qkv, part, attn, hloc, outv, red, pr, kvw, layers, end;
};
__host__ __device__ __forceinline__ CLayout cluster_layout(int E, int D, int fr, int L, int R)
{
    auto r16 = [](uint32_t v) { return (v + 15u) & ~15u; };
    CLayout o;
    o.x = kBarBytes;
    o.qkv = o.x + r16(uint32_t(E) * 4u);
    o.part = o.qkv + r16(3u * D * 4u);
    o.attn = o.part + r16(uint32_t(kClusterSize) * (D + 4) * 4u);
    o.hloc = o.attn + r16(uint32_t(D) * 4u);
    o.outv = o.hloc + r16(uint32_t(fr) * 4u);
    o.red = o.outv + r16((uint32_t(E) + 2u * kCWarps + uint32_t(kCWarps) * D) * 4u);
    o.pr = o.red + r16(uint32_t(E) * 4u);
    o.kvw = o.pr + r16((2u * E + 2u * uint32_t(R)) * 4u);
    o.layers = o.kvw + kKvWin;
    o.end = o.layers + r16(uint32_t(sizeof(CLayer)) * uint32_t(L));
    return o;
}

// ---- primitives -------------------------------------------------------------
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory"); }

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, const float4 &v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
                 "r"(__float_as_uint(v.w)), "r"(bar)
                 : "memory");
}

// Store to a CTA of the cluster that completes `bytes` on that CTA's mbarrier
// (address and barrier both mapped into the destination CTA).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
                 "r"(__float_as_uint(v)), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void cluster_barrier_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ int ld_relaxed_i32(const int *p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_i64(long long *p, long long v)
{
    asm volatile("st.relaxed.gpu.global.s64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_add_i64(long long *p, long long v)
{
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long to_word(float v)
{
    v = fminf(fmaxf(v, -kFixLimit), kFixLimit);   // (fmaxf maps NaN to -kFixLimit)
    return (unsigned long long)(__float2ll_rn(v * kFixScale) + (long long)kFixBias) + (1ull << kCountShift);
}
__device__ __forceinline__ int word_count(unsigned long long w) { return int(w >> kCountShift); }
__device__ __forceinline__ float word_value(unsigned long long w)
{
    const long long n = (long long)(w >> kCountShift);
    const long long f = (long long)(w & ((1ull << kCountShift) - 1)) - n * (long long)kFixBias;
    return float(__ll2double_rn(f) * (1.0 / 16777216.0));
}

struct Sh {
    unsigned long long keys[kCWarps];
};

// Shared-memory views of a consumer thread.
struct CS {
    uint64_t *full, *empty, *kv_bar, *prm_bar;
    // the barriers of the cluster exchanges come in pairs, used alternately
    // (exchange n on barrier n & 1): a CTA of the cluster can run one exchange
    // ahead of another, and its stores then complete on the other barrier of
    // the pair, never on the phase this CTA is still waiting for
    uint64_t *qkv_bar, *att_bar, *red_bar, *x_bar;
    float *x, *qkv, *part, *attn, *hloc, *outv, *red, *kvw;
    float *pr;                 // this layer's LayerNorm parameters and bias slices
    const CLayer *layers;      // the layer table, copied to shared memory
    uint8_t *ring;
    uint32_t uses_qkv, uses_att, uses_kv, uses_prm, uses_red, uses_x;   // barrier phases consumed so far
#ifdef GPT2_CTRACE
    unsigned long long *twait, *tsub;
    int tpass, tslot;
#endif
};

struct Waiter {
    unsigned long long t0 = 0;
    uint32_t it = 0;
};

__device__ __forceinline__ bool aborted(const ClusterArgs &a) { return ld_relaxed_i32(&a.st->abort) != 0; }

__device__ __forceinline__ void raise_abort(const ClusterArgs &a, int info)
{
    record_error(a.st, kDevErrTimeout, info);
    atomicMax(&a.st->abort, 1);   // (never lowers the level 2 of keep_waiting_landing)
}

// One step of a bounded spin: false once the spin must end (abort or timeout).
// A limit of 0 lets no wait spin: the first one that does not succeed at
// once gives up (the test of the abort path).  Used by the waits for data
// that may never come once the pass is abandoned: ring stages, GPU-wide sums,
// the previous pass's token, free ring slots.
__device__ __forceinline__ bool keep_waiting(const ClusterArgs &a, Waiter &w, int info)
{
    if (a.wait_ns == 0) {
        raise_abort(a, info);
        return false;
    }
    if ((++w.it & 127u) != 0) return true;
    if (aborted(a)) return false;
    const unsigned long long t = global_ns();
    if (w.t0 == 0) w.t0 = t;
    else if (t - w.t0 > a.wait_ns) {
        raise_abort(a, info);
        return false;
    }
    return true;
}

// The same for waits on writes into this CTA's shared memory that have been
// issued and will land whatever happens (bulk copies of parameters and K/V
// rows, st.async stores from the cluster's CTAs, which send every exchange
// even on the abort path): they never give up early, so no write into shared
// memory is still in flight when the CTA leaves and no barrier is re-armed
// with a phase pending; only the fixed limit ends them.
// If one of these ever runs out (a fault, not an abandoned pass), the abort
// word goes to 2 and every such wait then ends at once, so the kernel still
// returns within about one limit.
__device__ __forceinline__ bool keep_waiting_landing(const ClusterArgs &a, Waiter &w, int info)
{
    if ((++w.it & 127u) != 0) return true;
    if (ld_relaxed_i32(&a.st->abort) >= 2) return false;
    const unsigned long long t = global_ns();
    if (w.t0 == 0) w.t0 = t;
    else if (t - w.t0 > kWaitLimitNs) {
        record_error(a.st, kDevErrTimeout, info);
        atomicMax(&a.st->abort, 2);
        return false;
    }
    return true;
}

__device__ __forceinline__ bool wait_stage(const ClusterArgs &a, const CS &c, uint32_t kk)
{
    const uint32_t st = kk & (kCRing - 1), par = (kk / kCRing) & 1u;
    if (mbar_test_wait(&c.full[st], par)) return true;
#ifdef GPT2_CTRACE
    const long long t0 = clock64();
#endif
    Waiter w;
    bool good = true;
    while (!mbar_try_wait(&c.full[st], par))
        if (!keep_waiting(a, w, 3000 + int(blockIdx.x))) {
            good = false;
            break;
        }
#ifdef GPT2_CTRACE
    if ((threadIdx.x & 31) == 0) atomicAdd(c.twait, (unsigned long long)(clock64() - t0));
#endif
    return good;
}

// Bounded wait on a barrier of this CTA that completes by transaction bytes
// (bulk copies, or stores from CTAs of the cluster): always waited out (see
// keep_waiting_landing).
__device__ __forceinline__ bool wait_phase(const ClusterArgs &a, uint64_t *bar, uint32_t par, int info)
{
    if (mbar_test_wait(bar, par)) return true;
    Waiter w;
    while (!try_wait_cluster(bar, par))
        if (!keep_waiting_landing(a, w, info)) return false;
    return true;
}
// One barrier, one phase per use (this CTA's bulk copies).
__device__ __forceinline__ bool wait_tx_bar(const ClusterArgs &a, uint64_t *bar, uint32_t &uses, int info)
{
    const uint32_t par = uses & 1u;
    ++uses;
    return wait_phase(a, bar, par, info);
}
// A pair of barriers used alternately (cluster exchanges): use n waits for
// phase (n / 2) & 1 of barrier n & 1.
__device__ __forceinline__ uint64_t *pair_bar(uint64_t *bars, uint32_t uses) { return bars + (uses & 1u); }
__device__ __forceinline__ bool wait_pair(const ClusterArgs &a, uint64_t *bars, uint32_t &uses, int info)
{
    const uint32_t n = uses++;
    return wait_phase(a, bars + (n & 1u), (n >> 1) & 1u, info);
}

// ---- roles and row segments ---------------------------------------------------
struct Role {
    bool head;      // a head-cluster CTA (else an fc CTA)
    int h, r;       // head and rank (head CTAs)
    int f;          // fc CTA index (fc CTAs)
    int g;          // CTA index in the grid (LM head)
};

// Geometry of one kind of segment (the same in every layer): `rows` rows of
// rb bytes (+ srb scale bytes, + zrb zero-point bytes for int4), streamed in
// chunks of `chunk` rows per ring stage; a stage holds the chunk's rows, then
// its scales at soff, then its zero points at zoff.
struct Geo {
    uint32_t rb, srb, zrb;
    int32_t rows, chunk, nch;
    uint32_t soff, zoff;
    float inv_chunk;            // row i lies in chunk floor((i + 0.5) * inv_chunk)
};
// A segment: a geometry and where its rows start in this layer.
struct Seg {
    const uint8_t *main, *sc, *zp;
};

__host__ __device__ __forceinline__ uint32_t a16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ __forceinline__ uint32_t seg_stage_bytes(uint32_t c, uint32_t rb, uint32_t srb, uint32_t zrb)
{
    return a16(c * rb) + a16(c * srb) + c * zrb;
}

// Chunk of a row index without an integer division: for i < 2^20 and
// chunks below 2^11, (i + 0.5) / chunk is at least 2^-12 away from an
// integer, far more than the float rounding of the product.
__device__ __forceinline__ int chunk_of(const Geo &g, int i)
{
    return __float2int_rz((float(i) + 0.5f) * g.inv_chunk);
}

// Largest chunk (a multiple of gran, or all rows) whose sections fit a stage.
__device__ __forceinline__ Geo make_geo(uint32_t rb, uint32_t srb, uint32_t zrb, int rows, int gran, uint32_t stage)
{
    Geo g;
    g.rb = rb;
    g.srb = srb;
    g.zrb = zrb;
    g.rows = rows;
    int c = int(stage / (rb + srb + zrb)) / gran * gran;
    while (c > gran && seg_stage_bytes(uint32_t(c), rb, srb, zrb) > stage) c -= gran;
    if (c < gran) c = gran;
    if (c > rows) c = rows > 0 ? rows : 1;
    g.chunk = c;
    g.nch = rows > 0 ? (rows + c - 1) / c : 0;
    g.soff = a16(uint32_t(c) * rb);
    g.zoff = g.soff + a16(uint32_t(c) * srb);
    g.inv_chunk = 1.0f / float(c);
    return g;
}

__device__ __forceinline__ uint32_t wt_row_bytes(int wt, int n)
{
    return wt == kWF32 ? uint32_t(n) * 4 : wt == kWF16 ? uint32_t(n) * 2 : uint32_t(n) / 2;
}

// Canonical rows of an [out][in] matrix (int4: codes [out][in/2], scales
// [out][in/32], zero points [out][in/64] two per byte).
__device__ __forceinline__ Geo long_geo(int wt, int in, int rows, uint32_t stage)
{
    const bool i4 = wt == kWI4;
    return make_geo(wt_row_bytes(wt, in), i4 ? uint32_t(in / 32) * 4 : 0, i4 ? uint32_t(in / 64) : 0, rows,
                    i4 ? 8 : 1, stage);
}
__device__ __forceinline__ Seg long_seg(const Geo &g, const void *W, const float *sc, const uint8_t *zp, int row0)
{
    Seg s;
    s.main = static_cast<const uint8_t *>(W) + size_t(row0) * g.rb;
    s.sc = sc ? reinterpret_cast<const uint8_t *>(sc) + size_t(row0) * g.srb : nullptr;
    s.zp = zp ? zp + size_t(row0) * g.zrb : nullptr;
    return s;
}

// Tile rows of `cols` columns (int4: codes [rows][cols/2], scales
// [rows][cols/32], one zero-point byte per group).
__device__ __forceinline__ Geo tile_geo(int wt, int rows, int cols, uint32_t stage)
{
    const bool i4 = wt == kWI4;
    return make_geo(wt_row_bytes(wt, cols), i4 ? uint32_t(cols / 32) * 4 : 0, i4 ? uint32_t(cols / 32) : 0, rows,
                    i4 ? 16 : 1, stage);
}
__device__ __forceinline__ Seg tile_seg(const Geo &g, const void *W, const float *sc, const uint8_t *zp, int t)
{
    return long_seg(g, W, sc, zp, t * g.rows);
}

// The geometries of a CTA's segments: head CTAs stream their gathered q, k, v
// rows (3 D/4 rows), then their tile of the output projection; fc CTAs their
// fc rows, then their tile of the MLP projection; every CTA its LM-head rows.
struct Geos {
    Geo a, b, head;
    int head_row0;
};

__device__ __forceinline__ Geos make_geos(const ClusterArgs &a, const Role &ro)
{
    Geos G;
    if (ro.head) {
        G.a = long_geo(a.wtype, a.E, 3 * (a.D / 4), a.stage_bytes);
        G.b = tile_geo(a.wtype, a.E / kClusterSize, a.D, a.stage_bytes);
    } else {
        G.a = long_geo(a.wtype, a.E, a.fr, a.stage_bytes);
        G.b = tile_geo(a.wtype, a.E, a.fr, a.stage_bytes);
    }
    // an int4 head streams whole padded shares (whole chunks of 8 rows: its
    // 12-byte zero-point rows need multiples of 4 rows per copy); rows >= V
    // are read but never stored
    const int r0 = a.head_wt == kWI4 ? ro.g * a.head_rpc : min(a.V, ro.g * a.head_rpc);
    const int r1 = a.head_wt == kWI4 ? r0 + a.head_rpc : min(a.V, r0 + a.head_rpc);
    G.head = long_geo(a.head_wt, a.E, r1 - r0, a.stage_bytes);
    G.head_row0 = r0;
    return G;
}

__device__ __forceinline__ Seg seg_a(const Role &ro, const Geos &G, const CLayer &L)
{
    return ro.head ? tile_seg(G.a, L.Wqkv, L.qkv_s, L.qkv_z, ro.h * kClusterSize + ro.r)
                   : tile_seg(G.a, L.Wfc, L.fc_s, L.fc_z, ro.f);
}
__device__ __forceinline__ Seg seg_b(const Role &ro, const Geos &G, const CLayer &L)
{
    return ro.head ? tile_seg(G.b, L.Wo_t, L.o_s, L.o_z, ro.h * kClusterSize + ro.r)
                   : tile_seg(G.b, L.Wp_t, L.p_s, L.p_z, ro.f);
}
__device__ __forceinline__ Seg seg_head(const ClusterArgs &a, const Geos &G)
{
    return long_seg(G.head, a.head_w, a.head_s, a.head_z, G.head_row0);
}

// ---- producer --------------------------------------------------------------------
__device__ __forceinline__ void stream_seg(const ClusterArgs &a, const Geo &g, const Seg &sg, uint8_t *ring,
                                           uint64_t *full, uint64_t *empty, uint32_t &k, bool &ok, uint64_t pol)
{
    const int C = g.chunk;
    for (int rs = 0; rs < g.rows && ok; rs += C) {
        const uint64_t p = pol;
        const int n = min(C, g.rows - rs);
        const uint32_t st = k & (kCRing - 1);
        if (k >= uint32_t(kCRing)) {
            const uint32_t par = ((k / kCRing) - 1u) & 1u;
            Waiter w;
            while (!mbar_try_wait(&empty[st], par)) {
                if (!keep_waiting(a, w, 2000 + int(blockIdx.x))) { ok = false; break; }
                __nanosleep(32);   // the ring is full: leave the issue slots to the consumer warps
            }
            if (!ok) break;
            // the stage's previous copy has landed (consumers that gave up on
            // it may have released it early): never re-arm a pending phase
            Waiter w2;
            while (!mbar_try_wait(&full[st], par))
                if (!keep_waiting_landing(a, w2, 2100 + int(blockIdx.x))) {
                    ok = false;
                    break;
                }
            if (!ok) break;
        }
        uint8_t *dst = ring + size_t(st) * a.stage_bytes;
        const uint32_t b0 = uint32_t(n) * g.rb, b1 = uint32_t(n) * g.srb, b2 = uint32_t(n) * g.zrb;
        mbar_arrive_expect_tx(&full[st], b0 + b1 + b2);
        bulk_g2s_hint(dst, sg.main + size_t(rs) * g.rb, b0, &full[st], p);
        if (b1) bulk_g2s_hint(dst + g.soff, sg.sc + size_t(rs) * g.srb, b1, &full[st], p);
        if (b2) bulk_g2s_hint(dst + g.zoff, sg.zp + size_t(rs) * g.zrb, b2, &full[st], p);
        ++k;
    }
}

__device__ void producer(const ClusterArgs &a, const CLayer *layers, const Role &ro, const Geos &G, uint8_t *ring,
                         uint64_t *full, uint64_t *empty)
{
    uint32_t k = 0;
    bool ok = true;
    // L2 policies: the LM head and fp32 / fp16 block matrices stream through
    // (evict first); int4 block matrices (54 MB for GPT-2 small) fit L2 and
    // are kept there across passes (evict last)
    const uint64_t pol = l2_evict_first_policy();
    const uint64_t pol_blk = a.wtype == kWI4 ? l2_evict_last_policy() : pol;
    for (int s = 0; s < a.n_steps && ok; ++s) {
        for (int l = 0; l < a.L && ok; ++l) {
            stream_seg(a, G.a, seg_a(ro, G, layers[l]), ring, full, empty, k, ok, pol_blk);
            if (ok) stream_seg(a, G.b, seg_b(ro, G, layers[l]), ring, full, empty, k, ok, pol_blk);
        }
        if (ok) stream_seg(a, G.head, seg_head(a, G), ring, full, empty, k, ok, pol);
    }
    // the copies still in flight land before the CTA leaves
    const uint32_t first = k > uint32_t(kCRing) ? k - uint32_t(kCRing) : 0u;
    for (uint32_t j = first; j < k; ++j) {
        Waiter w;
        while (!mbar_try_wait(&full[j & (kCRing - 1)], (j / kCRing) & 1u))
            if ((++w.it & 127u) == 0) {
                const unsigned long long t = global_ns();
                if (w.t0 == 0) w.t0 = t;
                else if (t - w.t0 > kWaitLimitNs) break;
            }
    }
}

// ---- consumer math -------------------------------------------------------------
// Inputs per column unit of a canonical row: 4 fp32 (16 bytes), 8 fp16 (16
// bytes) or 8 int4 codes (one 32-bit word; four words share a group's scale
// and zero point).
template <int WT>
struct UnitOf {
    static constexpr int kIn = WT == kWF32 ? 4 : 8;
    static constexpr int kF4 = kIn / 4;                    // float4 of inputs per unit
    static constexpr int kPL = 1024 / kIn / 32;            // units per lane for n_embd <= 1024
};

// 2^23 + (byte b of w), as a float: byte b of w must be below 16.
__device__ __forceinline__ float byte_f23(uint32_t w, int b)
{
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + uint32_t(b)));
}

// Shared-memory loads by 32-bit shared address (the ring and the vectors are
// addressed in the shared window explicitly, never through generic pointers).
__device__ __forceinline__ float4 lds_f4(uint32_t a)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds_u4(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f(uint32_t a)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Rows of a stage by shared address: row rr's values at m + rr * rb, its
// scales at s + rr * srb, its zero points at z + rr * zrb.
struct RowAddr {
    uint32_t m, s, z;
};
__device__ __forceinline__ RowAddr row_addr(uint32_t stage, const Geo &g, int rr)
{
    RowAddr r;
    r.m = stage + uint32_t(rr) * g.rb;
    r.s = stage + g.soff + uint32_t(rr) * g.srb;
    r.z = stage + g.zoff + uint32_t(rr) * g.zrb;
    return r;
}

// Packed pairs of fp32 values (low word first) and the paired fp32 operations
// (fma/sub .f32x2: two IEEE operations per instruction).
using F2 = unsigned long long;
__device__ __forceinline__ F2 pack2(float a, float b)
{
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float sum2(F2 r)
{
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
    return a + b;
}
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c)
{
    F2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ F2 sub2(F2 a, F2 b)
{
    F2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ void lds_f2x2(uint32_t a, F2 &lo, F2 &hi)
{
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(lo), "=l"(hi) : "r"(a));
}
__device__ __forceinline__ F2 half2_f2(uint32_t h)
{
    const float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return pack2(p.x, p.y);
}

// Unit c of a canonical row dotted with its inputs, in pairs: xu[0..2 kF4)
// hold the unit's inputs two by two; acc is a pair of partial sums.  int4:
// the 8 codes q of word c, (q - z) taken exactly as (2^23 + q) - (2^23 + z),
// the pairs' sums times the group's scale.
template <int WT>
__device__ __forceinline__ F2 canon_unit(const RowAddr &ra, int c, const F2 *xu, F2 acc)
{
    if (WT == kWF32) {
        F2 w0, w1;
        lds_f2x2(ra.m + 16u * uint32_t(c), w0, w1);
        return fma2(w1, xu[1], fma2(w0, xu[0], acc));
    } else if (WT == kWF16) {
        const uint4 u = lds_u4(ra.m + 16u * uint32_t(c));
        acc = fma2(half2_f2(u.x), xu[0], acc);
        acc = fma2(half2_f2(u.y), xu[1], acc);
        acc = fma2(half2_f2(u.z), xu[2], acc);
        return fma2(half2_f2(u.w), xu[3], acc);
    } else {
        // word c: inputs 8c..8c+7 of group c / 4; byte b of the word holds
        // inputs 2b (low nibble) and 2b + 1
        const uint32_t q = lds_u32(ra.m + 4u * uint32_t(c));
        const int grp = c >> 2;
        const float s = lds_f(ra.s + 4u * uint32_t(grp));
        const uint32_t z = (lds_u8(ra.z + uint32_t(grp >> 1)) >> ((grp & 1) * 4)) & 15u;
        const float zf = __uint_as_float(0x4B000000u | z);   // 2^23 + z, exactly
        const F2 zz = pack2(zf, zf);
        const uint32_t lo = q & 0x0F0F0F0Fu, hi = (q >> 4) & 0x0F0F0F0Fu;
        F2 d = 0ull;
#pragma unroll
        for (int b = 0; b < 4; ++b) d = fma2(sub2(pack2(byte_f23(lo, b), byte_f23(hi, b)), zz), xu[b], d);
        return fma2(pack2(s, s), d, acc);
    }
}

__device__ __forceinline__ float4 mul4(const float4 &a, const float4 &b)
{
    return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}
__device__ __forceinline__ float4 sub4(const float4 &a, float k)
{
    return make_float4(a.x - k, a.y - k, a.z - k, a.w - k);
}

// Shifted sum and sum of squares of 4 values (LayerNorm statistics).
__device__ __forceinline__ void stat4(const float4 &v, float k, float &s, float &q)
{
    const float a = v.x - k, b = v.y - k, c = v.z - k, d = v.w - k;
    s += (a + b) + (c + d);
    q = fmaf(a, a, fmaf(b, b, fmaf(c, c, fmaf(d, d, q))));
}

// Sums 8 per-lane values over the warp in 9 shuffles (each step halves the
// values a lane keeps); lane l ends with the total of value
// 4 * bit4(l) + 2 * bit3(l) + bit2(l).  The order is fixed, so every run gives
// the same bits.
__device__ __forceinline__ float warp_sum8(float (&v)[8], int lane)
{
    {
        const bool hi = lane & 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float send = hi ? v[i] : v[i + 4], keep = hi ? v[i + 4] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    {
        const bool hi = lane & 8;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float send = hi ? v[i] : v[i + 2], keep = hi ? v[i + 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    {
        const bool hi = lane & 4;
        const float send = hi ? v[0] : v[1], keep = hi ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    return v[0];
}
__device__ __forceinline__ int warp_sum8_row(int lane)
{
    return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

// The same for 4 values in 6 shuffles: lane l ends with the total of value
// 2 * bit4(l) + bit3(l).
__device__ __forceinline__ float warp_sum4(float (&v)[4], int lane)
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

// Row sums of RG (4, or up to 8) rows held across a warp: the value of row
// group_row<RG>(lane), complete in the lanes where group_writer<RG>(lane).
template <int RG>
__device__ __forceinline__ float warp_sum_rows(const float (&acc)[RG], int lane)
{
    if constexpr (RG == 4) {
        float v[4] = {acc[0], acc[1], acc[2], acc[3]};
        return warp_sum4(v, lane);
    } else {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = j < RG ? acc[j] : 0.f;
        return warp_sum8(v, lane);
    }
}
template <int RG>
__device__ __forceinline__ int group_row(int lane)
{
    return RG == 4 ? ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1) : warp_sum8_row(lane);
}
template <int RG>
__device__ __forceinline__ bool group_writer(int lane)
{
    return (lane & (RG == 4 ? 7 : 3)) == 0;
}

// Stages are consumed in windows of at most the ring's size.  Within a window
// every thread waits (on the stages' full barriers) only for the stages that
// hold the rows it reads; at the window's end one CTA barrier, then one lane
// per stage releases it (empty barriers count one arrival).  Every stage
// before a window is released before the window is waited for, so the
// producer can always fill it.  Layer segments, whose stages are resident
// ahead of time, take one window of up to the whole ring; the LM head, which
// streams, takes windows of half the ring so the producer fills one while the
// other is read.
constexpr int kStreamWindow = kCRing / 2;

__device__ __forceinline__ void window_release(const CS &c, uint32_t k, int q0, int q1)
{
    csync();
    const int tid = threadIdx.x;
    if (tid < q1 - q0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&c.empty[(k + uint32_t(q0 + tid)) & (kCRing - 1)]))
                     : "memory");
}

__device__ __forceinline__ uint32_t stage_addr(const ClusterArgs &a, const CS &c, uint32_t kk)
{
    return smem_addr(c.ring) + (kk & (kCRing - 1)) * a.stage_bytes;
}

// Temperature sampling ("Let's make GPT-2 in assembly", Step 7: divide the
// scores by a temperature, softmax, draw at random): the Gumbel-max form, the
// token with the highest logit / T - log(-log u), u = the uniform number of
// counter pos * V + id from a counter-based SplitMix64 generator (Steele, Lea
// and Flood, 2014): seed + (k + 1) * 0x9E3779B97F4A7C15 through its output
// mixer; u = (top 23 bits + 0.5) * 2^-23, which lies strictly inside (0, 1)
// (2m + 1 < 2^24 is exact in fp32).  The argmax key is built from that score;
// the stored logit stays the plain one.
__device__ __forceinline__ float sample_score(float logit, float temperature, unsigned long long seed,
                                              unsigned long long k)
{
    unsigned long long z = seed + (k + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    const float u = (float(uint32_t(z >> 41)) + 0.5f) * 1.1920928955078125e-7f;
    return logit / temperature - logf(-logf(u));
}

// Row groups of one warp in one window: rows [w0, w1), RG at a time (a short
// last group repeats its first row in the empty slots, whose sums are not
// stored: no per-row branches in the loop), lanes over the column units; each
// lane's inputs (x * gamma) are in registers, xr[m] for unit lane + 32 m.
template <int WT, bool LN, int RG, bool GELU>
__device__ __forceinline__ void canon_groups(const ClusterArgs &a, const CS &c, const Geo &g, uint32_t k, int w0,
                                             int w1, int units, const F2 (&xr)[UnitOf<WT>::kPL * UnitOf<WT>::kF4 * 2],
                                             bool &have_stats, float ssum, float ssq, int in,
                                             float &dmean, float &rstd, const float *c1, const float *cb, float *out,
                                             int logit_row0, unsigned long long &best, long long sample_k0)
{
    constexpr int kF4 = UnitOf<WT>::kF4;
    const int lane = threadIdx.x & 31, C = g.chunk;
    for (int g0 = w0; g0 < w1; g0 += RG) {
        const int ng = min(RG, w1 - g0);
        RowAddr ra[RG];
#pragma unroll
        for (int j = 0; j < RG; ++j) {
            const int i = j < ng ? g0 + j : g0;
            const int q = chunk_of(g, i);
            ra[j] = row_addr(stage_addr(a, c, k + uint32_t(q)), g, i - q * C);
        }
        F2 acc2[RG];
#pragma unroll
        for (int j = 0; j < RG; ++j) acc2[j] = 0ull;
#pragma unroll
        for (int m = 0; m < UnitOf<WT>::kPL; ++m) {
            const int u = lane + 32 * m;
            if (u < units) {
#pragma unroll
                for (int j = 0; j < RG; ++j) acc2[j] = canon_unit<WT>(ra[j], u, &xr[m * kF4 * 2], acc2[j]);
            }
        }
        float acc[RG];
#pragma unroll
        for (int j = 0; j < RG; ++j) acc[j] = sum2(acc2[j]);
        if (LN && !have_stats) {
            // the statistics' butterfly runs here, after the first group's loads
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            }
            const float inv = 1.0f / float(in);
            dmean = ssum * inv;   // mean - shift
            rstd = rsqrtf(fmaxf(fmaf(ssq, inv, -dmean * dmean), 0.f) + a.eps);
            have_stats = true;
        }
        float t = warp_sum_rows<RG>(acc, lane);
        const int jr = group_row<RG>(lane);
        if (group_writer<RG>(lane) && jr < ng) {
            const int i = g0 + jr;
            if (LN) t = rstd * fmaf(-dmean, c1[i], t) + cb[i];
            if (logit_row0 >= 0) {
                if (logit_row0 + i < a.V) {   // (rows >= V: padding of an int4 head)
                    a.logits[logit_row0 + i] = t;
                    const float score = sample_k0 >= 0 ? sample_score(t, a.temperature, a.seed,
                                                                      (unsigned long long)(sample_k0 + logit_row0 + i))
                                                       : t;
                    const unsigned long long key = argmax_key(score, uint32_t(logit_row0 + i));
                    best = key > best ? key : best;
                }
            } else {
                out[i] = GELU ? gelu_new(t) : t;
            }
        }
    }
}

// Dot products of the canonical rows of a segment (length in) with x.  Each
// lane first loads the inputs of its column units (x * gamma, LN) into
// registers and, for LN, every warp takes the statistics of x (shifted by
// x[0]) from them with the same fixed-order butterfly, so all warps get the
// same bits.  In each window, warp w takes a contiguous block of the window's
// rows, in groups of 6 (4 when the block has at most 4 rows), and waits only
// for the stages that hold them.  Results go to out[i], or, for the LM head
// (logit_row0 >= 0), to the logits and this thread's argmax key.
//
// LN: the LayerNorm before the rows is folded into them (see CLayer): each
// result is rstd * (W.(gamma*(x - s)) - (mean - s) * c1[i]) + cb[i], with the
// shift s = x[0].  Centring on s keeps the two terms of the difference small
// when the residual stream has a large common offset (|mean| >> std):
// |mean - s| <= sqrt(n) * std for any x, so the cancellation is bounded.
// The rows of a window that warp `warp` takes: [w0, w1).
__device__ __forceinline__ void warp_rows(const Geo &g, int q0, int q1, int &w0, int &w1, int &per)
{
    const int warp = threadIdx.x >> 5;
    const int r0 = q0 * g.chunk, r1 = min(g.rows, q1 * g.chunk);
    per = (r1 - r0 + kCWarps - 1) / kCWarps;
    w0 = r0 + warp * per;
    w1 = min(r1, w0 + per);
}

// Waits for the stages that hold this warp's rows of a segment's first window
// (called before the segment's input arrives, so the barrier tests overlap
// that wait; canon_rows is then told not to repeat them).
__device__ __forceinline__ void prewait_rows(const ClusterArgs &a, const CS &c, const Geo &g, uint32_t k, int win,
                                             bool &ok)
{
    int w0, w1, per;
    warp_rows(g, 0, min(g.nch, win), w0, w1, per);
    if (w0 < w1)
        for (int q = chunk_of(g, w0), qb = chunk_of(g, w1 - 1); q <= qb; ++q)
            if (ok && !wait_stage(a, c, k + uint32_t(q))) ok = false;
}

template <int WT, bool LN, bool GELU = false>
__device__ __forceinline__ void canon_rows(const ClusterArgs &a, CS &c, const Geo &g, uint32_t &k, int win, int in,
                                          const float *xin, const float *gamma, const float *c1, const float *cb,
                                          float *out, int logit_row0, unsigned long long &best, bool &ok,
                                          bool prewaited = false, long long sample_k0 = -1)
{
    constexpr int kF4 = UnitOf<WT>::kF4;
    const int lane = threadIdx.x & 31;
    const int nch = g.nch;
    const int units = in / UnitOf<WT>::kIn;
    const uint32_t xa = smem_addr(xin), ga = smem_addr(gamma);
    F2 xr[UnitOf<WT>::kPL * kF4 * 2];
    float dmean = 0.f, rstd = 0.f;
    const float shift = LN ? xin[0] : 0.f;
    float ssum = 0.f, ssq = 0.f;   // this lane's share of the LayerNorm statistics
    {
        float s1 = 0.f, q1s = 0.f;  // two chains
#pragma unroll
        for (int m = 0; m < UnitOf<WT>::kPL; ++m) {
            const int u = lane + 32 * m;
#pragma unroll
            for (int f = 0; f < kF4; ++f) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (u < units) {
                    const uint32_t off = 16u * uint32_t(u * kF4 + f);
                    v = lds_f4(xa + off);
                    if (LN) {
                        if ((m * kF4 + f) & 1) stat4(v, shift, s1, q1s);
                        else stat4(v, shift, ssum, ssq);
                        v = mul4(sub4(v, shift), lds_f4(ga + off));
                    }
                }
                xr[(m * kF4 + f) * 2] = pack2(v.x, v.y);
                xr[(m * kF4 + f) * 2 + 1] = pack2(v.z, v.w);
            }
        }
        ssum += s1;
        ssq += q1s;
    }
    bool have_stats = false;
    CSUB(0);
    for (int q0 = 0; q0 < nch; q0 += win) {
        const int q1 = min(nch, q0 + win);
        int w0, w1, per;
        warp_rows(g, q0, q1, w0, w1, per);
        if (w0 < w1 && !(prewaited && q0 == 0)) {
            const int qa = chunk_of(g, w0), qb = chunk_of(g, w1 - 1);
            for (int q = qa; q <= qb; ++q)
                if (ok && !wait_stage(a, c, k + uint32_t(q))) ok = false;
        }
        CSUB(1);
        // the row groups' shuffles need the whole warp: a lane whose wait gave
        // up (the pass is being abandoned) takes its warp out of the work
        const bool wok = __all_sync(0xffffffffu, ok);
        if (wok && w0 < w1) {
            if (per <= 4)
                canon_groups<WT, LN, 4, GELU>(a, c, g, k, w0, w1, units, xr, have_stats, ssum, ssq, in, dmean, rstd,
                                              c1, cb, out, logit_row0, best, sample_k0);
            else
                canon_groups<WT, LN, 6, GELU>(a, c, g, k, w0, w1, units, xr, have_stats, ssum, ssq, in, dmean, rstd,
                                              c1, cb, out, logit_row0, best, sample_k0);
        }
        CSUB(2);
        window_release(c, k, q0, q1);   // its barrier also publishes out[]
    }
    k += uint32_t(nch);
}

// Unit u of a tile row (stored at unit us) dotted with its inputs, read
// from the input vector at shared address v.
template <int WT>
__device__ __forceinline__ float tile_unit(const RowAddr &ra, uint32_t us, int u, uint32_t v)
{
    if (WT == kWF32) {
        const float4 w = lds_f4(ra.m + 16u * us);
        const float4 x = lds_f4(v + 16u * uint32_t(u));
        return fmaf(w.w, x.w, fmaf(w.z, x.z, w.y * x.y)) + w.x * x.x;
    } else if (WT == kWF16) {
        const uint4 w = lds_u4(ra.m + 16u * us);
        const float4 v0 = lds_f4(v + 32u * uint32_t(u)), v1 = lds_f4(v + 32u * uint32_t(u) + 16u);
        const float2 p0 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
        const float2 p1 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
        const float2 p2 = __half22float2(*reinterpret_cast<const __half2 *>(&w.z));
        const float2 p3 = __half22float2(*reinterpret_cast<const __half2 *>(&w.w));
        const float e0 = fmaf(p0.y, v0.y, p0.x * v0.x), e1 = fmaf(p1.y, v0.w, p1.x * v0.z);
        const float e2 = fmaf(p2.y, v1.y, p2.x * v1.x), e3 = fmaf(p3.y, v1.w, p3.x * v1.z);
        return (e0 + e1) + (e2 + e3);
    } else {
        const uint4 w = lds_u4(ra.m + 16u * us);
        const float s = lds_f(ra.s + 4u * uint32_t(u));
        const float zf = 8388608.0f + float(lds_u8(ra.z + uint32_t(u)));
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            const uint32_t lo = words[wi] & 0x0F0F0F0Fu, hi = (words[wi] >> 4) & 0x0F0F0F0Fu;
            const float4 v0 = lds_f4(v + 128u * uint32_t(u) + 32u * uint32_t(wi));
            const float4 v1 = lds_f4(v + 128u * uint32_t(u) + 32u * uint32_t(wi) + 16u);
            d0 = fmaf(byte_f23(lo, 0) - zf, v0.x, d0);
            d1 = fmaf(byte_f23(hi, 0) - zf, v0.y, d1);
            d0 = fmaf(byte_f23(lo, 1) - zf, v0.z, d0);
            d1 = fmaf(byte_f23(hi, 1) - zf, v0.w, d1);
            d0 = fmaf(byte_f23(lo, 2) - zf, v1.x, d0);
            d1 = fmaf(byte_f23(hi, 2) - zf, v1.y, d1);
            d0 = fmaf(byte_f23(lo, 3) - zf, v1.z, d0);
            d1 = fmaf(byte_f23(hi, 3) - zf, v1.w, d1);
        }
        return s * (d0 + d1);
    }
}

// Tile rows run with the unit loop unrolled at their usual widths: 64
// columns (the head's slice of the output projection) and 32 (an fc CTA's
// slice of the MLP projection in GPT-2 small); other widths take the loop.
template <int WT>
constexpr int kTileUnroll = WT == kWF32 ? 16 : WT == kWF16 ? 8 : 2;
template <int WT>
constexpr int kFcTileUnits = WT == kWF32 ? 8 : WT == kWF16 ? 4 : 1;

// Dot products of the tile rows of a segment (cols columns) with vin: one
// thread per row, which waits for its row's stage; 16-byte units of row r are
// stored at u ^ (r & m), so the threads of a quarter-warp read different
// banks.  out[row] for every row.  Rows of exactly UX units run with the unit
// loop unrolled (every load of a row in flight at once); with XREG (fp32,
// several rows per thread) the UX float4 of inputs are loaded into registers
// once.  The sums are taken in the same order on every path (each unit's
// fused products, then even units, odd units, and the two).
template <int WT, int UX, bool XREG>
__device__ __forceinline__ void tile_rows(const ClusterArgs &a, CS &c, const Geo &g, uint32_t &k, int win, int cols,
                                          const float *vin, float *out, bool &ok)
{
    const int tid = threadIdx.x;
    const int per_unit = WT == kWF32 ? 4 : WT == kWF16 ? 8 : 32;
    const int U = cols / per_unit;
    const int m = (U & (U - 1)) == 0 ? min(U, 8) - 1 : 0;
    const int C = g.chunk, nch = g.nch;
    const uint32_t v4 = smem_addr(vin);
    constexpr bool kReg = XREG && WT == kWF32;
    float4 xv[kReg ? UX : 1];
    if (kReg && U == UX) {
#pragma unroll
        for (int u = 0; u < (kReg ? UX : 1); ++u) xv[u] = lds_f4(v4 + 16u * uint32_t(u));
    }
    for (int q0 = 0; q0 < nch; q0 += win) {
        const int q1 = min(nch, q0 + win);
        const int r1 = min(g.rows, q1 * C);
        CSUB(0);
        if (ok)
            for (int row = q0 * C + tid; row < r1; row += kCThreads) {
                const int q = chunk_of(g, row);
                if (!wait_stage(a, c, k + uint32_t(q))) {
                    ok = false;
                    break;
                }
                const RowAddr ra = row_addr(stage_addr(a, c, k + uint32_t(q)), g, row - q * C);
                const int sw = row & m;
                float acc0 = 0.f, acc1 = 0.f;
                if (U == UX) {
#pragma unroll
                    for (int u = 0; u < UX; ++u) {
                        float part;
                        if constexpr (kReg) {
                            const float4 w = lds_f4(ra.m + 16u * uint32_t(u ^ sw));
                            const float4 x = xv[u];
                            part = fmaf(w.w, x.w, fmaf(w.z, x.z, w.y * x.y)) + w.x * x.x;
                        } else {
                            part = tile_unit<WT>(ra, uint32_t(u ^ sw), u, v4);
                        }
                        if (u & 1) acc1 += part;
                        else acc0 += part;
                    }
                } else {
#pragma unroll 2
                    for (int u = 0; u < U; ++u) {
                        const float part = tile_unit<WT>(ra, uint32_t(u ^ sw), u, v4);
                        if (u & 1) acc1 += part;
                        else acc0 += part;
                    }
                }
                out[row] = acc0 + acc1;
            }
        CSUB(2);
        window_release(c, k, q0, q1);   // its barrier also completes out[]
    }
    k += uint32_t(nch);
}

constexpr int kMaxPerThread = 8;   // n_embd <= 8 * kCThreads

__device__ __forceinline__ unsigned long long ld_word(const long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Reads a residual sum into c.x once every word holds `count` contributions.
// The CTAs of a cluster share the work: rank r polls words [r E/4, (r+1) E/4)
// (each thread its own words), then stores their values into c.x of all four
// CTAs; every thread then waits for the whole vector on x_bar.  The words carry
// the data themselves, so nothing after the poll reads memory that the
// contributors wrote; `fence` (the first wait of a pass, which the zeroing of
// the other parity's sums follows) orders this CTA's later stores after the
// contributors' earlier reads.
__device__ __forceinline__ void read_sum(const ClusterArgs &a, CS &c, int count, const long long *src, bool &ok,
                                         bool fence = false)
{
    const int tid = threadIdx.x, rq = a.E / kClusterSize;
    const int r = int(blockIdx.x) % kClusterSize;
    if (tid == 0) mbar_arrive_expect_tx(pair_bar(c.x_bar, c.uses_x), uint32_t(a.E) * 4u);
    constexpr int kW = kMaxPerThread / kClusterSize;   // words per thread
    unsigned long long v[kW];
#pragma unroll
    for (int j = 0; j < kW; ++j) {
        const int t = tid + j * kCThreads;
        v[j] = t < rq ? ld_word(src + size_t(r * rq + t) * kClusterAccStride) : 0ull;
    }
    Waiter w;
    for (;;) {
        bool done = true;
#pragma unroll
        for (int j = 0; j < kW; ++j) {
            const int t = tid + j * kCThreads;
            if (t < rq && word_count(v[j]) < count) {
                done = false;
                v[j] = ld_word(src + size_t(r * rq + t) * kClusterAccStride);
            }
        }
        if (done || !ok) break;
        if (!keep_waiting(a, w, 5000 + int(blockIdx.x))) {
            ok = false;
            break;
        }
    }
    if (fence) __threadfence();
    const uint32_t xbar = smem_addr(pair_bar(c.x_bar, c.uses_x));
#pragma unroll
    for (int j = 0; j < kW; ++j) {
        const int t = tid + j * kCThreads;
        if (t < rq) {
            const float val = word_value(v[j]);
            const uint32_t dsm = smem_addr(c.x + r * rq + t);
#pragma unroll
            for (int dst = 0; dst < kClusterSize; ++dst)
                st_async_f32(mapa(dsm, uint32_t(dst)), val, mapa(xbar, uint32_t(dst)));
        }
    }
    if (!wait_pair(a, c.x_bar, c.uses_x, 5500 + int(blockIdx.x))) ok = false;
}

// Adds values[i] (+ extra[base + i] + extra2[i] if extra is given) into
// sum[base + i], i < n, one contribution per word.  The closing barrier keeps
// the parameter area (extra2) unchanged until every thread has read it.
__device__ __forceinline__ void add_sum(const ClusterArgs &a, long long *sum, int base, const float *values,
                                        const float *extra, const float *extra2, int n)
{
    const int tid = threadIdx.x;
    for (int i = tid; i < n; i += kCThreads) {
        float v = values[i];
        if (extra) v += extra[base + i] + extra2[i];
        if (!(fabsf(v) <= kFixLimit)) record_error(a.st, kDevErrRange, base + i);
        red_add_i64(sum + size_t(base + i) * kClusterAccStride, (long long)to_word(v));
    }
    csync();
}

// ---- attention of one head, positions split over the cluster ----------------------
template <int D>
__device__ void attention(const ClusterArgs &a, CS &c, int l, int h, int r, int pos, bool &ok)
{
    constexpr int DPL = D / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *kh = a.kcache + (size_t(l) * a.H + h) * a.P * D;
    float *vh = a.vcache + (size_t(l) * a.H + h) * a.P * D;
    const int n = pos + 1;
    const int j0 = (r * n) / kClusterSize, j1 = ((r + 1) * n) / kClusterSize;
    const int jc = min(j1, pos);                       // cached rows of this CTA: [j0, jc)
    const int win = int(kKvWin / (2u * D * 4u));
    const int n_pre = max(0, min(jc - j0, win));
    float *kw = c.kvw, *vw = c.kvw + size_t(win) * D;
    if (r == 0 && tid < D) {                           // append this token's k, v to the cache
        kh[size_t(pos) * D + tid] = c.qkv[D + tid];
        vh[size_t(pos) * D + tid] = c.qkv[2 * D + tid];
    }
    if (n_pre > 0) {
        const uint32_t par = c.uses_kv & 1u;
        ++c.uses_kv;
        Waiter w;   // the bulk copies of this CTA's K/V rows always land: waited out
        while (!mbar_try_wait(c.kv_bar, par))
            if (!keep_waiting_landing(a, w, 4000 + int(blockIdx.x))) {
                ok = false;
                break;
            }
    }
    // this CTA's positions, spread over all warps.  Few positions (short
    // contexts): warp w takes positions j0 + w, j0 + w + 8, ..., two at a time,
    // each lane holding DPL consecutive dimensions, the score a butterfly over
    // the warp.  Many positions: warp w takes a contiguous block, 32 positions
    // at a time with one lane per position (online softmax per tile).  Either
    // way each warp keeps its own state (max, sum, unnormalised output),
    // merged over the warps in a fixed order below.
    const int cnt = max(0, j1 - j0);
    const bool lpd = cnt <= kLanePerDimMax;
    float m = -INFINITY, lsum = 0.f, o[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = 0.f;
    auto krow = [&](int j) -> const float * {
        return j == pos ? c.qkv + D : (j - j0 < n_pre ? kw + size_t(j - j0) * D : kh + size_t(j) * D);
    };
    auto vrow = [&](int j) -> const float * {
        return j == pos ? c.qkv + 2 * D : (j - j0 < n_pre ? vw + size_t(j - j0) * D : vh + size_t(j) * D);
    };
    const bool wok = __all_sync(0xffffffffu, ok);   // the loops' shuffles need the whole warp
    if (lpd) {
        float qv[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) qv[i] = c.qkv[lane * DPL + i];
        for (int ja = j0 + warp; ja < j1 && wok; ja += 2 * kCWarps) {
            const int jb = ja + kCWarps;
            const bool hb = jb < j1;
            const float *ka = krow(ja), *kb = krow(hb ? jb : ja);
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int i = 0; i < DPL; ++i) {
                sa = fmaf(qv[i], ka[lane * DPL + i], sa);
                sb = fmaf(qv[i], kb[lane * DPL + i], sb);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sa += __shfl_xor_sync(0xffffffffu, sa, off);
                sb += __shfl_xor_sync(0xffffffffu, sb, off);
            }
            sa *= a.scale;
            sb = hb ? sb * a.scale : -INFINITY;
            const float mn = fmaxf(m, fmaxf(sa, sb));
            const float corr = expf(m - mn);          // 0 on the first positions (m = -inf)
            const float pa = expf(sa - mn), pb = hb ? expf(sb - mn) : 0.f;
            lsum = fmaf(lsum, corr, pa + pb);
            const float *va = vrow(ja), *vb = vrow(hb ? jb : ja);
#pragma unroll
            for (int i = 0; i < DPL; ++i)
                o[i] = fmaf(pb, vb[lane * DPL + i], fmaf(pa, va[lane * DPL + i], o[i] * corr));
            m = mn;
        }
    } else {
        const int per = (cnt + kCWarps - 1) / kCWarps;
        const int w0 = j0 + warp * per, w1 = min(j1, w0 + per);
        const float4 *q4 = reinterpret_cast<const float4 *>(c.qkv);
        for (int base = w0; base < w1 && wok; base += 32) {
            const int j = base + lane;
            const bool valid = j < w1;
            float sc = -INFINITY;
            if (valid) {
                // lane j starts at unit j: the rows of a quarter-warp, 4 D
                // bytes apart, then fall in different shared-memory banks
                const float4 *kr = reinterpret_cast<const float4 *>(krow(j));
                float d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int i = 0; i < D / 4; i += 2) {
                    const int u0 = (i + lane) & (D / 4 - 1), u1 = (i + 1 + lane) & (D / 4 - 1);
                    const float4 k0 = kr[u0], k1 = kr[u1], qa = q4[u0], qb = q4[u1];
                    d0 = fmaf(qa.x, k0.x, fmaf(qa.y, k0.y, fmaf(qa.z, k0.z, fmaf(qa.w, k0.w, d0))));
                    d1 = fmaf(qb.x, k1.x, fmaf(qb.y, k1.y, fmaf(qb.z, k1.z, fmaf(qb.w, k1.w, d1))));
                }
                sc = (d0 + d1) * a.scale;
            }
            const float mn = fmaxf(m, warp_max(sc));
            const float corr = expf(m - mn);
            const float p = valid ? expf(sc - mn) : 0.f;
            lsum = fmaf(lsum, corr, warp_sum(p));
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[i] *= corr;
            // sum of p_j v_j, 8 positions at a time: their value rows are
            // loaded before any is used, so the loads overlap; lane holds
            // dimensions lane + 32 i here
            const int cntt = min(32, w1 - base);
            for (int i0 = 0; i0 < cntt; i0 += 8) {
                float pv[8], vv[8][DPL];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = min(i0 + u, cntt - 1);
                    pv[u] = __shfl_sync(0xffffffffu, p, i);
                    const float *vr = vrow(base + i);
#pragma unroll
                    for (int dd = 0; dd < DPL; ++dd) vv[u][dd] = vr[lane + 32 * dd];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i0 + u < cntt) {
#pragma unroll
                        for (int dd = 0; dd < DPL; ++dd) o[dd] = fmaf(pv[u], vv[u][dd], o[dd]);
                    }
            }
            m = mn;
        }
    }
    // merge the warps through shared scratch (outv), then send this CTA's
    // (max, sum, unnormalised output) to every CTA of the cluster; the stores
    // complete on each receiver's att_bar
    const uint32_t slot = smem_addr(c.part + size_t(r) * (D + 4));
    const uint32_t abar = smem_addr(pair_bar(c.att_bar, c.uses_att));
    {
        float *wm = c.outv, *wl = c.outv + kCWarps, *wo = c.outv + 2 * kCWarps;
        if (lane == 0) {
            wm[warp] = m;
            wl[warp] = lsum;
        }
#pragma unroll
        for (int i = 0; i < DPL; ++i) wo[warp * D + (lpd ? lane * DPL + i : lane + 32 * i)] = o[i];
        csync();
        for (int t = tid; t < D + 2; t += kCThreads) {
            float M = -INFINITY;
            for (int w = 0; w < kCWarps; ++w)
                if (wl[w] > 0.f) M = fmaxf(M, wm[w]);
            float L = 0.f, O = 0.f;
            for (int w = 0; w < kCWarps; ++w) {
                if (wl[w] > 0.f) {
                    const float e = expf(wm[w] - M);
                    L = fmaf(wl[w], e, L);
                    if (t >= 2) O = fmaf(wo[w * D + t - 2], e, O);
                }
            }
            const float v = t == 0 ? M : (t == 1 ? L : O);
            const uint32_t off = t < 2 ? uint32_t(t) * 4u : uint32_t(t + 2) * 4u;
#pragma unroll
            for (int dst = 0; dst < kClusterSize; ++dst)
                st_async_f32(mapa(slot + off, uint32_t(dst)), v, mapa(abar, uint32_t(dst)));
        }
    }
    if (!wait_pair(a, c.att_bar, c.uses_att, 6000 + int(blockIdx.x))) ok = false;
    // combine the 4 ranks in rank order (every CTA gets the same bits)
    for (int t = tid; t < D; t += kCThreads) {
        float M = -INFINITY;
        for (int q = 0; q < kClusterSize; ++q) {
            const float *pq = c.part + size_t(q) * (D + 4);
            if (pq[1] > 0.f) M = fmaxf(M, pq[0]);
        }
        float L = 0.f, O = 0.f;
        for (int q = 0; q < kClusterSize; ++q) {
            const float *pq = c.part + size_t(q) * (D + 4);
            if (pq[1] > 0.f) {
                const float e = expf(pq[0] - M);
                L = fmaf(pq[1], e, L);
                O = fmaf(pq[4 + t], e, O);
            }
        }
        c.attn[t] = O / L;
    }
}

// Issue the bulk copies of this CTA's cached K/V rows of a head (before q, k,
// v of the pass exist).
template <int D>
__device__ __forceinline__ void prefetch_kv(const ClusterArgs &a, CS &c, int l, int h, int r, int pos)
{
    if (threadIdx.x != 0) return;
    const int n = pos + 1;
    const int j0 = (r * n) / kClusterSize, j1 = ((r + 1) * n) / kClusterSize;
    const int jc = min(j1, pos);
    const int win = int(kKvWin / (2u * D * 4u));
    const int n_pre = max(0, min(jc - j0, win));
    if (n_pre <= 0) return;
    const float *kh = a.kcache + ((size_t(l) * a.H + h) * a.P + j0) * D;
    const float *vh = a.vcache + ((size_t(l) * a.H + h) * a.P + j0) * D;
    const uint32_t bytes = uint32_t(n_pre) * D * 4u;
    asm volatile("fence.proxy.async;" ::: "memory");   // cache rows written by generic stores; window last read by them
    mbar_arrive_expect_tx(c.kv_bar, 2u * bytes);
    bulk_g2s(c.kvw, kh, bytes, c.kv_bar);
    bulk_g2s(c.kvw + size_t(win) * D, vh, bytes, c.kv_bar);
}

// Zeroes this CTA's share of the other parity's sums.  Called after the
// pass's first GPU-wide wait: by then every CTA has finished the previous
// pass, the last reader of those sums.
__device__ __forceinline__ void zero_other_parity(const ClusterArgs &a, int par)
{
    const size_t words = size_t(a.L) * a.E;
    const size_t per = (words + gridDim.x - 1) / gridDim.x;
    const size_t w0 = size_t(blockIdx.x) * per, w1 = min(words, w0 + per);
    long long *zn = a.acc_new + size_t(1 - par) * words * kClusterAccStride;
    long long *zx = a.acc_next + size_t(1 - par) * words * kClusterAccStride;
    for (size_t i = w0 + threadIdx.x; i < w1; i += kCThreads) {
        st_relaxed_i64(zn + i * kClusterAccStride, 0);
        st_relaxed_i64(zx + i * kClusterAccStride, 0);
    }
}

// The LM head's hand-off: each CTA publishes its best (value, ~id) key with
// the pass's epoch (its sequence number mod 2^15) in bits 17..31, in place
// of the top bits of ~id (ids < 2^17), so the word is its own arrival flag;
// the head CTAs of the next pass (and CTA 0 after the last pass) poll all the
// keys, each thread one CTA's word, until every word carries the epoch, and
// take the maximum.  Keys of one epoch compare as untagged keys do.
constexpr unsigned long long kKeyEpochMask = 0x7FFFull << 17;

__device__ __forceinline__ unsigned long long tag_key(unsigned long long key, uint32_t seq)
{
    return (key & ~kKeyEpochMask) | ((unsigned long long)(seq & 0x7FFFu) << 17);
}
__device__ __forceinline__ int32_t tagged_key_index(unsigned long long key)
{
    return int32_t(0x1FFFFu - uint32_t(key & 0x1FFFFull));
}

__device__ __forceinline__ void publish_key(const ClusterArgs &a, Sh &sh, uint32_t seq, unsigned long long best)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    best = warp_max_u64(best);
    if (lane == 0) sh.keys[warp] = best;
    csync();
    if (tid == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < kCWarps; ++w) b = sh.keys[w] > b ? sh.keys[w] : b;
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a.partials + blockIdx.x), "l"(tag_key(b, seq))
                     : "memory");
    }
    // sh.keys is written again only after every CTA has published this pass's key
}

// The token chosen by pass `seq`: polls every CTA's key (all threads of the
// CTA call it), returns the id of the largest.  Ends with a fence: what the
// CTAs did before publishing is ordered before what follows.
__device__ __forceinline__ int32_t collect_token(const ClusterArgs &a, Sh &sh, uint32_t seq, bool &ok)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned long long want = (unsigned long long)(seq & 0x7FFFu) << 17;
    unsigned long long v = 0ull;
    if (tid < int(gridDim.x)) {
        v = ld_word(reinterpret_cast<const long long *>(a.partials + tid));
        Waiter w;
        while (ok && (v & kKeyEpochMask) != want) {
            if (!keep_waiting(a, w, 7000 + int(blockIdx.x))) ok = false;
            v = ld_word(reinterpret_cast<const long long *>(a.partials + tid));
        }
    }
    v = warp_max_u64(v);
    if (lane == 0) sh.keys[warp] = v;
    csync();
    unsigned long long b = 0ull;
    for (int w = 0; w < kCWarps; ++w) b = sh.keys[w] > b ? sh.keys[w] : b;
    __threadfence();
    csync();   // every thread has read sh.keys
    return tagged_key_index(b);
}

// CTA 0, thread 0: the state after pass s chose `tok`.
__device__ __forceinline__ void record_token(const ClusterArgs &a, int s, uint32_t seq, int32_t tok)
{
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
}

// How the fc CTAs' MLP-projection partials reach the residual sum: summed
// over the cluster first (distributed shared memory, then one contribution
// per fc cluster and word), or, with int4 weights (measured faster there),
// each fc CTA adding its whole partial vector (one contribution per fc CTA).
__device__ __forceinline__ bool mlp_direct(const ClusterArgs &a) { return a.wtype == kWI4; }
__device__ __forceinline__ int mlp_contributions(const ClusterArgs &a)
{
    return mlp_direct(a) ? a.nfc : a.nfc / kClusterSize;
}

// Bulk copies of what a CTA needs besides weights in one layer
// (L != nullptr) or in the LM head (L == nullptr) into the parameter area
// c.pr: gamma [E], the fold vectors c1 and cb of its rows [pr_rows each], and
// the bias slice of its residual sum [E].  Issued by thread 0 before the wait
// for the layer's input, so the copies overlap that wait; the area's previous
// contents were last read before the barrier that precedes this call.
__device__ __forceinline__ void issue_params(const ClusterArgs &a, CS &c, const Role &ro, const Geos &G,
                                             const CLayer *L)
{
    if (threadIdx.x != 0) return;
    const int E = a.E, R = a.pr_rows;
    float *pg = c.pr, *p1 = c.pr + E, *pc = c.pr + E + R, *pb = c.pr + E + 2 * R;
    const uint32_t ev = uint32_t(E) * 4u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (!L) {
        const uint32_t rv = uint32_t(a.head_rpc) * 4u;   // padded vectors: whole slots exist
        const size_t r0 = size_t(ro.g) * a.head_rpc;
        mbar_arrive_expect_tx(c.prm_bar, ev + 2u * rv);
        bulk_g2s(pg, a.lnf_w, ev, c.prm_bar);
        bulk_g2s(p1, a.h_c1 + r0, rv, c.prm_bar);
        bulk_g2s(pc, a.h_cb + r0, rv, c.prm_bar);
    } else if (ro.head) {
        const uint32_t rv = uint32_t(G.a.rows) * 4u, qv = ev / kClusterSize;
        const size_t r0 = size_t(ro.h * kClusterSize + ro.r) * G.a.rows;
        mbar_arrive_expect_tx(c.prm_bar, ev + 2u * rv + (ro.h == 0 ? qv : 0u));
        bulk_g2s(pg, L->ln1_w, ev, c.prm_bar);
        bulk_g2s(p1, L->q_c1 + r0, rv, c.prm_bar);
        bulk_g2s(pc, L->q_cb + r0, rv, c.prm_bar);
        if (ro.h == 0) bulk_g2s(pb, L->proj_b + size_t(ro.r) * (E / kClusterSize), qv, c.prm_bar);
    } else {
        const uint32_t rv = uint32_t(a.fr) * 4u, qv = ev / kClusterSize;
        const size_t r0 = size_t(ro.f) * a.fr;
        // x and the bias are added once: by fc cluster 0, a slice per rank
        // (or, adding partials directly, by fc CTA 0, all of them)
        const bool direct = mlp_direct(a);
        const bool first = direct ? ro.f == 0 : ro.f < kClusterSize;
        const uint32_t bv = direct ? ev : qv;
        mbar_arrive_expect_tx(c.prm_bar, ev + 2u * rv + (first ? bv : 0u));
        bulk_g2s(pg, L->ln2_w, ev, c.prm_bar);
        bulk_g2s(p1, L->f_c1 + r0, rv, c.prm_bar);
        bulk_g2s(pc, L->f_cb + r0, rv, c.prm_bar);
        if (first)
            bulk_g2s(pb, L->mlp_proj_b + (direct ? size_t(0) : size_t(ro.r) * (E / kClusterSize)), bv, c.prm_bar);
    }
}

template <int WT, int D>
__device__ void consumer(const ClusterArgs &a, CS &c, Sh &sh, const Role &ro, const Geos &G)
{
    const int tid = threadIdx.x;
    const uint32_t seq0 = uint32_t(ld_relaxed_i32(&a.st->seq));
    const int E = a.E, q4 = D / 4, rq = E / kClusterSize, R = a.pr_rows;
    const float *p1 = c.pr + E, *pc = c.pr + E + R, *pb = c.pr + E + 2 * R;
    uint32_t k = 0;
    bool ok = true;
    for (int s = 0; s < a.n_steps; ++s) {
        const uint32_t seq = seq0 + uint32_t(s);
        const int par = int(seq & 1u);
        const int pos = min(max(a.pos0 + s, 0), a.P - 1);
        unsigned long long best = 0ull;
        for (int l = 0; l < a.L; ++l) {
            const CLayer &L = c.layers[l];
            long long *an = a.acc_new + (size_t(par) * a.L + l) * E * kClusterAccStride;
            CTRACE(s, l * 16 + 0);
            issue_params(a, c, ro, G, &L);
            if (ro.head) {
                if (tid == 0) {   // this layer's phases of the two cluster exchanges
                    mbar_arrive_expect_tx(pair_bar(c.qkv_bar, c.uses_qkv), 3u * D * 4u);
                    mbar_arrive_expect_tx(pair_bar(c.att_bar, c.uses_att), uint32_t(kClusterSize) * (D + 2) * 4u);
                }
                prefetch_kv<D>(a, c, l, ro.h, ro.r, pos);
                prewait_rows(a, c, G.a, k, kCRing, ok);   // this layer's QKV rows, while x is on its way
                // x entering the block
                if (l == 0) {
                    // every pass after the first waits for the previous one (its
                    // token, tagged with its sequence number), prompt passes too:
                    // the GPU-wide order of passes is what makes reusing the
                    // sums, the exchange slots and the cache rows safe
                    int tok = 0;
                    if (s > 0) {
                        tok = collect_token(a, sh, seq - 1, ok);
                        if (blockIdx.x == 0 && tid == 0) record_token(a, s - 1, seq - 1, tok);
                    }
                    if (s < a.n_prompt) tok = a.prompt ? __ldg(a.prompt + s) : a.tok_first;
                    else if (s == 0) tok = ld_relaxed_i32(&a.st->tok);
                    if (tok < 0 || tok >= a.V || a.pos0 + s >= a.P) {
                        if (tid == 0) record_error(a.st, tok < 0 || tok >= a.V ? kDevErrBadToken : kDevErrBadPosition, tok);
                        tok = min(max(tok, 0), a.V - 1);
                    }
                    for (int i = tid; i < E; i += kCThreads)
                        c.x[i] = __ldg(a.wte + size_t(tok) * E + i) + __ldg(a.wpe + size_t(pos) * E + i);
                    zero_other_parity(a, par);
                    csync();
                } else {
                    read_sum(a, c, mlp_contributions(a),
                             a.acc_next + (size_t(par) * a.L + (l - 1)) * E * kClusterAccStride, ok);
                }
                CTRACE(s, l * 16 + 1);
                if (!wait_tx_bar(a, c.prm_bar, c.uses_prm, 9000 + int(blockIdx.x))) ok = false;
                CTRACE(s, l * 16 + 2);
                // this CTA's q, k, v rows (LayerNorm folded, bias included) ->
                // every CTA of the cluster
                TSET(s, l * 16 + 8);
                canon_rows<WT, true>(a, c, G.a, k, kCRing, E, c.x, c.pr, p1, pc, c.outv, -1, best, ok, true);
                CTRACE(s, l * 16 + 3);   // (the window's closing barrier published c.outv)
                {
                    const uint32_t qbar = smem_addr(pair_bar(c.qkv_bar, c.uses_qkv));
                    for (int t = tid; t < 3 * q4; t += kCThreads) {
                        const int part = t / q4, d = ro.r * q4 + t % q4;
                        const float v = c.outv[t];
                        const uint32_t dsm = smem_addr(c.qkv + part * D + d);
#pragma unroll
                        for (int dst = 0; dst < kClusterSize; ++dst)
                            st_async_f32(mapa(dsm, uint32_t(dst)), v, mapa(qbar, uint32_t(dst)));
                    }
                }
                if (!wait_pair(a, c.qkv_bar, c.uses_qkv, 8000 + int(blockIdx.x))) ok = false;
                CTRACE(s, l * 16 + 4);
                attention<D>(a, c, l, ro.h, ro.r, pos, ok);
                csync();   // publishes c.attn; the attention scratch in c.outv is free again
                CTRACE(s, l * 16 + 5);
                // the head's slice of the output projection, rows rank*E/4.. (+ x + bias once, by head 0)
                TSET(s, l * 16 + 11);
                tile_rows<WT, kTileUnroll<WT>, false>(a, c, G.b, k, kCRing, D, c.attn, c.outv, ok);
                CTRACE(s, l * 16 + 6);
                add_sum(a, an, ro.r * rq, c.outv, ro.h == 0 ? c.x : nullptr, pb, rq);
                CTRACE(s, l * 16 + 7);
            } else {
                if (tid == 0 && WT != kWI4)   // this layer's partial slices (see mlp_direct)
                    mbar_arrive_expect_tx(pair_bar(c.red_bar, c.uses_red), uint32_t(E) * 4u);
                prewait_rows(a, c, G.a, k, kCRing, ok);   // this layer's fc rows, while x_new is on its way
                read_sum(a, c, a.H, an, ok, l == 0);
                if (l == 0) zero_other_parity(a, par);
                CTRACE(s, l * 16 + 1);
                if (!wait_tx_bar(a, c.prm_bar, c.uses_prm, 9000 + int(blockIdx.x))) ok = false;
                CTRACE(s, l * 16 + 2);
                TSET(s, l * 16 + 8);
                // fc rows with gelu_new applied as they are written (the
                // window's closing barrier publishes c.hloc)
                canon_rows<WT, true, true>(a, c, G.a, k, kCRing, E, c.x, c.pr, p1, pc, c.hloc, -1, best, ok, true);
                CTRACE(s, l * 16 + 3);
                CTRACE(s, l * 16 + 4);
                TSET(s, l * 16 + 11);
                tile_rows<WT, kFcTileUnits<WT>, false>(a, c, G.b, k, kCRing, a.fr, c.hloc, c.outv, ok);
                CTRACE(s, l * 16 + 5);
                if constexpr (WT == kWI4) {   // (mlp_direct)
                    add_sum(a, a.acc_next + (size_t(par) * a.L + l) * E * kClusterAccStride, 0, c.outv,
                            ro.f == 0 ? c.x : nullptr, pb, E);
                } else {
                    // the cluster's four partial vectors meet first: rank r sums
                    // slice r of all four (in rank order) and adds that once
                    {
                        const int q = rq / 4;   // float4 per slice
                        const uint32_t rbar = smem_addr(pair_bar(c.red_bar, c.uses_red));
                        const float4 *o4 = reinterpret_cast<const float4 *>(c.outv);
                        for (int t = tid; t < kClusterSize * q; t += kCThreads) {
                            const int dst = t / q, u = t % q;
                            const uint32_t slot = smem_addr(c.red + ro.r * rq + u * 4);
                            st_async_f32x4(mapa(slot, uint32_t(dst)), o4[dst * q + u], mapa(rbar, uint32_t(dst)));
                        }
                        if (!wait_pair(a, c.red_bar, c.uses_red, 9500 + int(blockIdx.x))) ok = false;
                        for (int i = tid; i < rq; i += kCThreads)
                            c.outv[i] = ((c.red[i] + c.red[rq + i]) + c.red[2 * rq + i]) + c.red[3 * rq + i];
                        csync();
                    }
                    add_sum(a, a.acc_next + (size_t(par) * a.L + l) * E * kClusterAccStride, ro.r * rq, c.outv,
                            ro.f < kClusterSize ? c.x : nullptr, pb, rq);
                }
                CTRACE(s, l * 16 + 6);
            }
        }
        // LM head (every CTA)
        CTRACE(s, 200);
        issue_params(a, c, ro, G, nullptr);
        read_sum(a, c, mlp_contributions(a), a.acc_next + (size_t(par) * a.L + (a.L - 1)) * E * kClusterAccStride,
                 ok);
        CTRACE(s, 201);
        if (!wait_tx_bar(a, c.prm_bar, c.uses_prm, 9000 + int(blockIdx.x))) ok = false;
        TSET(s, 204);
        {
            const long long sk = a.temperature > 0.f ? (long long)pos * (long long)a.V : -1ll;
            if (a.head_wt == kWF16)
                canon_rows<kWF16, true>(a, c, G.head, k, kStreamWindow, E, c.x, c.pr, p1, pc, nullptr, G.head_row0,
                                        best, ok, false, sk);
            else if (a.head_wt == kWI4)
                canon_rows<kWI4, true>(a, c, G.head, k, kStreamWindow, E, c.x, c.pr, p1, pc, nullptr, G.head_row0,
                                       best, ok, false, sk);
            else
                canon_rows<kWF32, true>(a, c, G.head, k, kStreamWindow, E, c.x, c.pr, p1, pc, nullptr, G.head_row0,
                                        best, ok, false, sk);
        }
        CTRACE(s, 202);
        publish_key(a, sh, seq, best);
        if (s == a.n_steps - 1 && blockIdx.x == 0) {   // the last pass's token: CTA 0 records it
            const int32_t tok = collect_token(a, sh, seq, ok);
            if (tid == 0) record_token(a, s, seq, tok);
        }
        CTRACE(s, 203);
    }
}

template <int WT, int D>
__global__ void __cluster_dims__(kClusterSize, 1, 1) __launch_bounds__(kCAll, 1) k_decode_cluster(const ClusterArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ Sh sh;
#ifdef GPT2_CTRACE
    __shared__ unsigned long long twait, tsub[3];
#endif
    // The kernel addresses its cluster peers' shared memory by rank: run only
    // in the launch shape it was written for (the same answer in every CTA,
    // so either all CTAs return here or none does).
    {
        uint32_t nct, crank;
        asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(nct));
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
        if (nct != uint32_t(kClusterSize) || blockDim.x != uint32_t(kCAll) ||
            gridDim.x != uint32_t(kClusterSize * a.H + a.nfc) || gridDim.y != 1u || gridDim.z != 1u) {
            if (threadIdx.x == 0) record_error(a.st, kDevErrLaunchShape, int(nct));
            return;
        }
        if (crank != blockIdx.x % uint32_t(kClusterSize) && threadIdx.x == 0)
            record_error(a.st, kDevErrLaunchShape, int(blockIdx.x));
    }
    const CLayout lo = cluster_layout(a.E, D, a.fr, a.L, a.pr_rows);
    CS c;
    c.full = reinterpret_cast<uint64_t *>(smem);
    c.empty = c.full + kCRing;
    c.qkv_bar = c.empty + kCRing;   // pairs: qkv, att, red, x; then kv, prm
    c.att_bar = c.qkv_bar + 2;
    c.red_bar = c.qkv_bar + 4;
    c.x_bar = c.qkv_bar + 6;
    c.kv_bar = c.qkv_bar + 8;
    c.prm_bar = c.qkv_bar + 9;
    c.red = reinterpret_cast<float *>(smem + lo.red);
    c.x = reinterpret_cast<float *>(smem + lo.x);
    c.qkv = reinterpret_cast<float *>(smem + lo.qkv);
    c.part = reinterpret_cast<float *>(smem + lo.part);
    c.attn = reinterpret_cast<float *>(smem + lo.attn);
    c.hloc = reinterpret_cast<float *>(smem + lo.hloc);
    c.outv = reinterpret_cast<float *>(smem + lo.outv);
    c.pr = reinterpret_cast<float *>(smem + lo.pr);
    c.kvw = reinterpret_cast<float *>(smem + lo.kvw);
    CLayer *tab = reinterpret_cast<CLayer *>(smem + lo.layers);
    c.layers = tab;
    c.ring = smem + a.ring_offset;
    c.uses_qkv = c.uses_att = c.uses_kv = c.uses_prm = c.uses_red = c.uses_x = 0;
#ifdef GPT2_CTRACE
    c.twait = &twait;
    c.tsub = tsub;
#endif
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the layer table, word by word
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a.layers);
        uint32_t *dst = reinterpret_cast<uint32_t *>(tab);
        const int words = int(sizeof(CLayer) / 4) * a.L;
        for (int i = tid; i < words; i += kCAll) dst[i] = __ldg(src + i);
    }
    if (tid == 0) {
        for (int i = 0; i < kCRing; ++i) {
            mbar_init(&c.full[i], 1);
            mbar_init(&c.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(c.qkv_bar + i, 1);   // + the bytes of the 4 ranks' stores
            mbar_init(c.att_bar + i, 1);
            mbar_init(c.red_bar + i, 1);   // + the bytes of the cluster's four partial slices
            mbar_init(c.x_bar + i, 1);     // + the bytes of x, a quarter from each CTA of the cluster
        }
        mbar_init(c.kv_bar, 1);
        mbar_init(c.prm_bar, 1);
        mbar_init_fence();
#ifdef GPT2_CTRACE
        twait = 0;
        tsub[0] = tsub[1] = tsub[2] = 0;
#endif
    }
    __syncthreads();
    cluster_barrier_all();   // every CTA's barriers exist before a peer stores to them
    Role ro;
    const int cl = int(blockIdx.x) / kClusterSize;
    ro.r = int(blockIdx.x) % kClusterSize;
    ro.head = cl < a.H;
    ro.h = ro.head ? cl : -1;
    ro.f = ro.head ? -1 : (cl - a.H) * kClusterSize + ro.r;
    ro.g = int(blockIdx.x);
    const Geos G = make_geos(a, ro);
    if (warp == kCWarps) {
        if (lane == 0) producer(a, c.layers, ro, G, c.ring, c.full, c.empty);
        __syncwarp();
    } else {
        consumer<WT, D>(a, c, sh, ro, G);
    }
    __syncthreads();
    cluster_barrier_all();   // no CTA leaves while a peer may still write its shared memory
}

template <int WT, int D>
cudaError_t launch_t(const ClusterArgs &a, int n_clusters, size_t smem, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_clusters * kClusterSize);
    cfg.blockDim = dim3(kCAll);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // the cluster shape is compiled into the kernel (__cluster_dims__), so no
    // launch path can run it without its peers
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_decode_cluster<WT, D>, a);
}

template <int WT, int D>
cudaError_t occ_t(size_t smem, size_t limit, int *clusters)
{
    cudaError_t e = cudaFuncSetAttribute(k_decode_cluster<WT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(limit));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterSize * 8);
    cfg.blockDim = dim3(kCAll);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kClusterSize;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, k_decode_cluster<WT, D>, &cfg);
}

// Re-tiling of a stored [out][in] matrix (see CLayer): tile t, row i holds
// canonical row (t % rdiv) * rows + i, columns (t / rdiv) * cols + [0, cols),
// as 16-byte units stored at u ^ (i & m).  The values are the stored ones,
// moved, never recomputed (int4: the same codes, scales and zero points).
__global__ void __launch_bounds__(256) k_tile(int wt, const uint8_t *W, const float *sc, const uint8_t *zp, int in,
                                              int T, int rdiv, int rows, int cols, uint8_t *dW, float *dsc,
                                              uint8_t *dzp)
{
    const int per_unit = wt == kWF32 ? 4 : wt == kWF16 ? 8 : 32;
    const int U = cols / per_unit;
    const int m = (U & (U - 1)) == 0 ? min(U, 8) - 1 : 0;
    const long long total = (long long)T * rows * U;
    const uint32_t rb_in = wt == kWF32 ? uint32_t(in) * 4 : wt == kWF16 ? uint32_t(in) * 2 : uint32_t(in) / 2;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int u = int(idx % U);
        const long long ti = idx / U;
        const int i = int(ti % rows), t = int(ti / rows);
        const long long R = (long long)(t % rdiv) * rows + i;
        const int col0 = (t / rdiv) * cols;
        const uint4 v = *reinterpret_cast<const uint4 *>(W + R * rb_in + size_t(col0 / per_unit + u) * 16);
        *reinterpret_cast<uint4 *>(dW + (size_t(ti) * U + (u ^ (i & m))) * 16) = v;
        if (wt == kWI4) {
            const int g = col0 / 32 + u;
            dsc[size_t(ti) * U + u] = sc[R * (in / 32) + g];
            dzp[size_t(ti) * U + u] = uint8_t((zp[R * (in / 64) + g / 2] >> ((g & 1) * 4)) & 15);
        }
    }
}

// Gathers the q, k, v rows of each (head, rank) into one contiguous block of
// 3 D/4 rows: destination row j = ((h * 4 + r) * 3 + part) * D/4 + d holds
// canonical row part * E + h * D + r * D/4 + d.  Rows keep the canonical
// format (int4: codes, scales and packed zero points, moved unchanged).
__global__ void __launch_bounds__(128) k_gather_qkv(int wt, const uint8_t *W, const float *sc, const uint8_t *zp,
                                                    int E, int D, uint8_t *dW, float *dsc, uint8_t *dzp)
{
    const int j = blockIdx.x, q4 = D / 4;
    const int i = j % (3 * q4), t = j / (3 * q4);
    const int h = t / kClusterSize, r = t % kClusterSize, part = i / q4, d = i % q4;
    const size_t src = size_t(part) * E + size_t(h) * D + size_t(r) * q4 + d;
    const uint32_t rb = wt == kWF32 ? uint32_t(E) * 4 : wt == kWF16 ? uint32_t(E) * 2 : uint32_t(E) / 2;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(W + src * rb);
    uint4 *d4 = reinterpret_cast<uint4 *>(dW + size_t(j) * rb);
    for (uint32_t u = threadIdx.x; u < rb / 16; u += blockDim.x) d4[u] = s4[u];
    if (wt == kWI4) {
        for (int g = threadIdx.x; g < E / 32; g += blockDim.x) dsc[size_t(j) * (E / 32) + g] = sc[src * (E / 32) + g];
        for (int b = threadIdx.x; b < E / 64; b += blockDim.x) dzp[size_t(j) * (E / 64) + b] = zp[src * (E / 64) + b];
    }
}

}  // namespace

size_t cluster_fixed_smem(int E, int D, int fr, int L, int pr_rows)
{
    return (size_t(cluster_layout(E, D, fr, L, pr_rows).end) + 127) / 128 * 128;
}

cudaError_t launch_cluster(int wtype, const ClusterArgs &a, int n_clusters, size_t smem, cudaStream_t s)
{
#define GPT2_C_CASE(WT)                                              \
    switch (a.D) {                                                   \
    case 32: return launch_t<WT, 32>(a, n_clusters, smem, s);        \
    case 64: return launch_t<WT, 64>(a, n_clusters, smem, s);        \
    case 128: return launch_t<WT, 128>(a, n_clusters, smem, s);      \
    default: return cudaErrorInvalidValue;                           \
    }
    switch (wtype) {
    case kWF32: GPT2_C_CASE(kWF32)
    case kWF16: GPT2_C_CASE(kWF16)
    case kWI4: GPT2_C_CASE(kWI4)
    default: return cudaErrorInvalidValue;
    }
#undef GPT2_C_CASE
}

cudaError_t cluster_max_active(int wtype, int D, size_t smem, size_t limit, int *clusters)
{
#define GPT2_CO_CASE(WT)                                             \
    switch (D) {                                                     \
    case 32: return occ_t<WT, 32>(smem, limit, clusters);            \
    case 64: return occ_t<WT, 64>(smem, limit, clusters);            \
    case 128: return occ_t<WT, 128>(smem, limit, clusters);          \
    default: return cudaErrorInvalidValue;                           \
    }
    switch (wtype) {
    case kWF32: GPT2_CO_CASE(kWF32)
    case kWF16: GPT2_CO_CASE(kWF16)
    case kWI4: GPT2_CO_CASE(kWI4)
    default: return cudaErrorInvalidValue;
    }
#undef GPT2_CO_CASE
}

cudaError_t cluster_tile(int wtype, const void *W, const float *scales, const uint8_t *zeros, int in, int T,
                         int rdiv, int rows, int cols, void *dW, float *dscales, uint8_t *dzeros, cudaStream_t s)
{
    const int per_unit = wtype == kWF32 ? 4 : wtype == kWF16 ? 8 : 32;
    if (cols % per_unit || in % per_unit || T < 1 || rows < 1) return cudaErrorInvalidValue;
    const long long total = (long long)T * rows * (cols / per_unit);
    const int grid = int(std::min<long long>((total + 255) / 256, 4096));
    k_tile<<<grid, 256, 0, s>>>(wtype, static_cast<const uint8_t *>(W), scales, zeros, in, T, rdiv, rows, cols,
                                static_cast<uint8_t *>(dW), dscales, dzeros);
    return cudaGetLastError();
}

// Largest chunk of rows of `rb`/`srb`/`zrb` bytes each (gran rows at least)
// that a stage holds; 0 if not even gran rows fit.
uint32_t cluster_stage_need(int gran, uint32_t rb, uint32_t srb, uint32_t zrb)
{
    return seg_stage_bytes(uint32_t(gran), rb, srb, zrb);
}

#ifdef GPT2_CTRACE
// Debug builds only: copies the stamps to host memory (`bytes` must be the
// trace's exact size).
extern "C" int gpt2_debug_ctrace(void *stamps, size_t bytes)
{
    if (!stamps || bytes != sizeof g_ctrace) return 2;
    if (cudaMemcpyFromSymbol(stamps, g_ctrace, sizeof g_ctrace) != cudaSuccess) return 1;
    return 0;
}
#endif

cudaError_t cluster_gather_qkv(int wtype, const void *W, const float *scales, const uint8_t *zeros, int E, int D,
                               void *dW, float *dscales, uint8_t *dzeros, cudaStream_t s)
{
    if (E % 64 || D % 4 || E % D) return cudaErrorInvalidValue;
    k_gather_qkv<<<3 * E, 128, 0, s>>>(wtype, static_cast<const uint8_t *>(W), scales, zeros, E, D,
                                       static_cast<uint8_t *>(dW), dscales, dzeros);
    return cudaGetLastError();
}

}  // namespace gpt2
