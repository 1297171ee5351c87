// C ABI of libgpt2.so (include/gpt2.h): model lifecycle, the captured decode
// pass, greedy decoding, inspection and stand-alone operations.
#include "../../include/gpt2.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "batch.h"
#include "cluster.h"
#include "common.cuh"
#include "kernels.h"

using namespace gpt2;

namespace {

struct QMat {
    void *w = nullptr;
    float *scales = nullptr;
    uint8_t *zeros = nullptr;
    int in = 0, out = 0;
    size_t main_bytes = 0, scale_bytes = 0, zero_bytes = 0;
};

struct LayerDev {
    float *ln1_w, *ln1_b, *attn_b, *proj_b, *ln2_w, *ln2_b, *fc_b, *mlp_proj_b;
    QMat mat[4];   // GPT2_MAT_ATTN, _PROJ, _FC, _MLP_PROJ
};

}  // namespace

struct gpt2_model {
    gpt2_config cfg{};
    int wdtype = 0;
    cudaStream_t stream = nullptr;
    int device = 0;
    int num_sms = 0;
    // device memory
    uint8_t *arena = nullptr;        // weights
    size_t arena_bytes = 0;
    uint8_t *work = nullptr;         // cache, activations, state
    size_t work_bytes = 0;
    float *wte = nullptr, *wpe = nullptr, *lnf_w = nullptr, *lnf_b = nullptr;
    std::vector<LayerDev> layers;
    float *kcache = nullptr, *vcache = nullptr;   // [L][H][P][D]
    float *x = nullptr, *qkv = nullptr, *attn = nullptr, *h = nullptr, *logits = nullptr;
    DeviceState *st = nullptr;
    int32_t *out_ids = nullptr;
    int32_t out_cap = 0;
    unsigned long long *partials = nullptr;
    unsigned int *counter = nullptr;
    int max_head_ctas = 0;
    // captured pass
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int kernels_per_step = 0;
    // cluster path: one cooperative launch per call
    bool cluster = false;
    int32_t *prompt_buf = nullptr;
    // prompts on the tensor cores: the prompt's positions as the rows of one
    // batched step (cluster path, greedy)
    gpt2_batch *pre = nullptr;
    bool head_f16 = false;           // GPT2_FLAG_HEAD_F16: the LM head reads an fp16 copy of wte
    bool head_int4 = false;          // GPT2_FLAG_HEAD_INT4: ... or a grouped int4 copy
    uint8_t *cbuf = nullptr;         // tiled matrices, fp16 head, sums, keys, layer table
    uint8_t *c_state = nullptr;      // sums + tagged LM-head keys (zeroed together)
    size_t c_state_bytes = 0;
    ClusterArgs cargs{};
    int c_clusters = 0;
    size_t c_smem = 0;
    // host view of the cache
    int cached = 0;
    bool has_step = false;
    unsigned long long launches = 0;
};

namespace {

constexpr size_t kAlign = 256;
// Prompts of at least this many tokens run on the tensor cores (the
// prefill engine), shorter ones as single-token passes of the cluster kernel
// (measured on GB300, GPT-2 small fp32: one engine step takes 0.51-0.55 ms
// for up to 64 positions, a pass ~0.145 ms: the engine wins clearly from 5
// tokens; at 4 the two are within 0.07 ms).
constexpr int kTcPrefillMin = 5;
// Per-kernel graph path: shared-memory stage budget and stages in flight of
// each GEMV launch (measured on GB300: 96 KB in up to 4 stages).
constexpr size_t kGraphStageBudget = 96 * 1024;
constexpr int kGraphMaxStages = 4;
size_t aup(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

size_t main_bytes_of(int wdtype, int in, int out)
{
    const size_t n = size_t(in) * out;
    return wdtype == GPT2_F32 ? n * 4 : wdtype == GPT2_F16 ? n * 2 : n / 2;
}

int check_config(const gpt2_config *c, int wdtype)
{
    if (!c) return GPT2_ERR_INVALID_ARG;
    if (c->n_layer < 1 || c->n_embd < 32 || c->n_head < 1 || c->n_positions < 1 || c->vocab_size < 1)
        return GPT2_ERR_INVALID_ARG;
    if (c->n_embd % 32 || c->n_embd % c->n_head) return GPT2_ERR_INVALID_ARG;
    const int D = c->n_embd / c->n_head;
    if (D != 32 && D != 64 && D != 128) return GPT2_ERR_INVALID_ARG;
    if (!(c->ln_eps > 0.f) || !std::isfinite(c->ln_eps)) return GPT2_ERR_INVALID_ARG;
    if (wdtype != GPT2_F32 && wdtype != GPT2_F16 && wdtype != GPT2_INT4) return GPT2_ERR_INVALID_ARG;
    if (wdtype == GPT2_INT4 && c->n_embd % 128) return GPT2_ERR_INVALID_ARG;
    // index arithmetic inside kernels is 32-bit per matrix row / element count
    const long long E = c->n_embd;
    if ((long long)c->vocab_size * E > (1ll << 31) - 1) return GPT2_ERR_INVALID_ARG;
    if ((long long)c->n_positions * E > (1ll << 31) - 1) return GPT2_ERR_INVALID_ARG;
    if (4 * E * E > (1ll << 31) - 1) return GPT2_ERR_INVALID_ARG;
    return GPT2_OK;
}

bool is_device_ptr(const void *p)
{
    if (!p) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return GPT2_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? GPT2_ERR_OUT_OF_MEMORY : GPT2_ERR_CUDA;
}

#define TRY_CUDA(expr)                                  \
    do {                                                \
        cudaError_t _e = (expr);                        \
        if (_e != cudaSuccess) return cuda_status(_e);  \
    } while (0)

// Fills GEMV arguments common to every launch of a matrix.
GemvArgs gemv_for(const gpt2_model *m, const QMat &q, int ctas, int &grid, size_t budget, int max_stages)
{
    GemvArgs a;
    std::memset(&a, 0, sizeof a);
    a.W = q.w;
    a.scales = q.scales;
    a.zeros = q.zeros;
    a.in = q.in;
    a.out = q.out;
    a.eps = m->cfg.ln_eps;
    a.st = m->st;
    grid = gemv_plan(a, m->wdtype, ctas, budget, max_stages);
    return a;
}

// Records one decode pass on stream s (called under stream capture).
int record_pass(gpt2_model *m, cudaStream_t s)
{
    const gpt2_config &c = m->cfg;
    const int E = c.n_embd, H = c.n_head, D = E / H, P = c.n_positions;
    const size_t budget = kGraphStageBudget;
    const int max_stages = kGraphMaxStages;
    const int ctas = m->num_sms;
    int kernels = 0;
    bool first = true;
    auto pdl = [&]() {
        bool p = !first;
        first = false;
        return p;
    };
    for (int l = 0; l < c.n_layer; ++l) {
        const LayerDev &L = m->layers[l];
        int grid;
        // qkv = LN1(x) . W_attn + b_attn   (layer 0 builds x from the embeddings)
        GemvArgs a = gemv_for(m, L.mat[GPT2_MAT_ATTN], ctas, grid, budget, max_stages);
        a.xin = m->x;
        a.ln_w = L.ln1_w;
        a.ln_b = L.ln1_b;
        a.bias = L.attn_b;
        a.y = m->qkv;
        int mode = kModeLnBias;
        if (l == 0) {
            mode = kModeEmbLnBias;
            a.wte = m->wte;
            a.wpe = m->wpe;
            a.x_out = m->x;
            a.vocab = c.vocab_size;
            a.n_positions = P;
        }
        TRY_CUDA(launch_gemv(m->wdtype, mode, a, grid, s, pdl()));
        ++kernels;
        // attention over the cache
        AttnArgs t;
        t.qkv = m->qkv;
        t.k_cache = m->kcache + size_t(l) * H * P * D;
        t.v_cache = m->vcache + size_t(l) * H * P * D;
        t.out = m->attn;
        t.n_head = H;
        t.head_dim = D;
        t.n_positions = P;
        t.scale = float(1.0 / std::sqrt(double(D)));
        t.st = m->st;
        TRY_CUDA(launch_attention(t, s, pdl()));
        ++kernels;
        // x += attn . W_proj + b_proj
        a = gemv_for(m, L.mat[GPT2_MAT_PROJ], ctas, grid, budget, max_stages);
        a.xin = m->attn;
        a.bias = L.proj_b;
        a.y = m->x;
        TRY_CUDA(launch_gemv(m->wdtype, kModeBiasRes, a, grid, s, pdl()));
        ++kernels;
        // h = gelu_new(LN2(x) . W_fc + b_fc)
        a = gemv_for(m, L.mat[GPT2_MAT_FC], ctas, grid, budget, max_stages);
        a.xin = m->x;
        a.ln_w = L.ln2_w;
        a.ln_b = L.ln2_b;
        a.bias = L.fc_b;
        a.y = m->h;
        TRY_CUDA(launch_gemv(m->wdtype, kModeLnBiasGelu, a, grid, s, pdl()));
        ++kernels;
        // x += h . W_mlp_proj + b_mlp_proj
        a = gemv_for(m, L.mat[GPT2_MAT_MLP_PROJ], ctas, grid, budget, max_stages);
        a.xin = m->h;
        a.bias = L.mlp_proj_b;
        a.y = m->x;
        TRY_CUDA(launch_gemv(m->wdtype, kModeBiasRes, a, grid, s, pdl()));
        ++kernels;
    }
    // logits = wte . LN_f(x); argmax; greedy feedback into the state
    int grid;
    GemvArgs a;
    std::memset(&a, 0, sizeof a);
    a.W = m->wte;
    a.in = E;
    a.out = c.vocab_size;
    a.eps = c.ln_eps;
    a.st = m->st;
    grid = gemv_plan(a, kWF32, m->max_head_ctas, budget, max_stages);
    a.evict_first = 1;
    a.xin = m->x;
    a.ln_w = m->lnf_w;
    a.ln_b = m->lnf_b;
    a.y = m->logits;
    a.partials = m->partials;
    a.counter = m->counter;
    a.out_ids = m->out_ids;
    a.out_cap = m->out_cap;
    TRY_CUDA(launch_gemv(kWF32, kModeHead, a, grid, s, pdl()));
    ++kernels;
    m->kernels_per_step = kernels;
    return GPT2_OK;
}

int build_graph(gpt2_model *m)
{
    cudaStream_t cs;
    TRY_CUDA(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(cs);
        return cuda_status(e);
    }
    int rc = record_pass(m, cs);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (rc != GPT2_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return cuda_status(e);
    m->graph = g;
    e = cudaGraphInstantiate(&m->exec, g, 0);
    if (e != cudaSuccess) return cuda_status(e);
    return GPT2_OK;
}

void free_model(gpt2_model *m)
{
    if (!m) return;
    if (m->pre) prefill_engine_destroy(m->pre);
    if (m->exec) cudaGraphExecDestroy(m->exec);
    if (m->graph) cudaGraphDestroy(m->graph);
    if (m->arena) cudaFree(m->arena);
    if (m->work) cudaFree(m->work);
    if (m->cbuf) cudaFree(m->cbuf);
    delete m;
}

int read_state(gpt2_model *m, DeviceState *hs)
{
    TRY_CUDA(cudaStreamSynchronize(m->stream));
    TRY_CUDA(cudaMemcpy(hs, m->st, sizeof *hs, cudaMemcpyDeviceToHost));
    if (hs->err != kDevErrNone) {
        const int err = hs->err;
        // report once, then clear so the model stays usable: the error word,
        // the abort word, and every tagged activation (stale epochs)
        TRY_CUDA(cudaMemset(&m->st->err, 0, 3 * sizeof(int32_t)));
        if (m->cluster) {   // sums and counters restart with the sequence
            const int32_t one = 1;
            TRY_CUDA(cudaMemset(m->c_state, 0, m->c_state_bytes));
            TRY_CUDA(cudaMemcpy(&m->st->seq, &one, sizeof one, cudaMemcpyHostToDevice));
        }
        return err == kDevErrTimeout ? GPT2_ERR_TIMEOUT : err == kDevErrRange ? GPT2_ERR_RANGE : GPT2_ERR_DEVICE_STATE;
    }
    return GPT2_OK;
}

// One launch of the cluster kernel running n_steps passes.
int launch_cluster_call(gpt2_model *m, int n_steps, const int32_t *prompt, int n_prompt, int tok_first, int pos0)
{
    ClusterArgs c = m->cargs;
    c.n_steps = n_steps;
    c.prompt = prompt;
    c.n_prompt = n_prompt;
    c.tok_first = tok_first;
    c.pos0 = pos0;
    TRY_CUDA(launch_cluster(m->wdtype, c, m->c_clusters, m->c_smem, m->stream));
    m->launches += 1;
    return GPT2_OK;
}

// Whether a prompt of n tokens runs on the tensor cores (greedy only: a
// temperature draw of the first token is the cluster kernel's).
bool use_tc_prefill(const gpt2_model *m, int n)
{
    return m->pre && n >= kTcPrefillMin && !(m->cargs.temperature > 0.f);
}

int launch_step(gpt2_model *m, int32_t token, int32_t position)
{
    if (m->cluster) return launch_cluster_call(m, 1, nullptr, 1, token, position);
    TRY_CUDA(launch_set_state(m->st, token, position, kSetTokPos, m->out_ids, m->stream));
    TRY_CUDA(cudaGraphLaunch(m->exec, m->stream));
    m->launches += 1 + m->kernels_per_step;
    return GPT2_OK;
}

// Sets up the cluster decode kernel (cluster.cu): tiled copies of the two
// projection matrices, the fixed-point sums and their counters, and the
// launch shape.  Returns GPT2_OK, or a nonzero status if the path cannot run
// here (the caller then keeps the per-kernel graph).
int setup_cluster(gpt2_model *m, int32_t *prompt_buf)
{
    const gpt2_config &c = m->cfg;
    const int L = c.n_layer, E = c.n_embd, H = c.n_head, D = E / H, V = c.vocab_size, F = 4 * E;
    const int wt = m->wdtype;
    if (E % 64) return GPT2_ERR_INVALID_ARG;   // E/4 tile rows in chunks of 16
    if (E > 1024) return GPT2_ERR_INVALID_ARG;  // input vectors held in registers (1024 values)
    int optin = 0, coop = 0;
    TRY_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, m->device));
    TRY_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, m->device));
    if (!coop) return GPT2_ERR_UNSUPPORTED_DEVICE;
    const size_t limit = size_t(optin) - 1024;   // room for static shared memory
    const int ns = kClusterRing;
    // co-resident clusters at (nearly) the full shared-memory size
    int max_clusters = 0;
    TRY_CUDA(cluster_max_active(wt, D, limit, limit, &max_clusters));
    // fc CTAs: a multiple of the cluster size, each owning fr = F / nfc fc rows
    // (a multiple of one int4 group)
    int nfc = 0;
    for (int n = (max_clusters - H) * kClusterSize; n >= kClusterSize; n -= kClusterSize)
        if (F % n == 0 && (F / n) % 32 == 0) {
            nfc = n;
            break;
        }
    if (nfc == 0) return GPT2_ERR_INVALID_ARG;
    const int fr = F / nfc;
    const int n_clusters = H + nfc / kClusterSize, grid = n_clusters * kClusterSize;
    if (grid > 256) return GPT2_ERR_INVALID_ARG;   // each consumer thread polls one CTA's LM-head key
    // a residual-sum word counts its contributions in 8 bits (bits 56..63):
    // one per head cluster (x after attention), one per fc cluster (x after the
    // MLP), or one per fc CTA where those add their partials directly (int4)
    if (H > 255 || (wt == kWI4 ? nfc : nfc / kClusterSize) > 255) return GPT2_ERR_INVALID_ARG;
    if (V > (1 << 17)) return GPT2_ERR_INVALID_ARG;   // tagged keys keep 17 bits of the id
    // LM-head rows per CTA: a multiple of 4 (of 8 for an int4 head, whose shares are padded)
    const int head_rpc = m->head_int4 ? ((V + grid - 1) / grid + 7) / 8 * 8 : ((V + grid - 1) / grid + 3) / 4 * 4;
    if (m->head_int4 && E % 64) return GPT2_ERR_INVALID_ARG;
    const int pr_rows = (std::max(std::max(3 * (D / 4), fr), head_rpc) + 3) / 4 * 4;
    const size_t fixed = cluster_fixed_smem(E, D, fr, L, pr_rows);
    const uint32_t ring_offset = uint32_t((fixed + 127) / 128 * 128);
    if (ring_offset >= limit) return GPT2_ERR_INVALID_ARG;
    const uint32_t stage = uint32_t((limit - ring_offset) / ns) / 16u * 16u;
    // every segment's smallest chunk fits a stage
    auto rbw = [&](int w, int n) {
        return w == kWF32 ? uint32_t(n) * 4 : w == kWF16 ? uint32_t(n) * 2 : uint32_t(n) / 2;
    };
    const bool i4 = wt == kWI4;
    uint32_t need = cluster_stage_need(1, uint32_t(E) * 4, 0, 0);   // LM head rows
    need = std::max(need, cluster_stage_need(i4 ? 8 : 1, rbw(wt, E), i4 ? uint32_t(E / 32) * 4 : 0,
                                             i4 ? uint32_t(E / 64) : 0));
    for (int cols : {D, fr})
        need = std::max(need, cluster_stage_need(i4 ? 16 : 1, rbw(wt, cols), i4 ? uint32_t(cols / 32) * 4 : 0,
                                                 i4 ? uint32_t(cols / 32) : 0));
    if (need > stage) return GPT2_ERR_INVALID_ARG;
    m->c_smem = ring_offset + size_t(ns) * stage;
    int fit = 0;
    TRY_CUDA(cluster_max_active(wt, D, m->c_smem, limit, &fit));
    if (fit < n_clusters) return GPT2_ERR_INVALID_ARG;

    // ---- device buffer: tiles, then the zeroed state, then the layer table ----
    const size_t mat_o = main_bytes_of(wt, E, E), mat_p = main_bytes_of(wt, F, E);
    const size_t sc_o = i4 ? size_t(E) * (E / 32) * 4 : 0, zp_o = i4 ? size_t(E) * (E / 32) : 0;
    const size_t sc_p = i4 ? size_t(E) * (F / 32) * 4 : 0, zp_p = i4 ? size_t(E) * (F / 32) : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += aup(bytes);
        return o;
    };
    const size_t mat_q = main_bytes_of(wt, E, 3 * E);
    const size_t sc_q = i4 ? size_t(3 * E) * (E / 32) * 4 : 0, zp_q = i4 ? size_t(3 * E) * (E / 64) : 0;
    std::vector<size_t> o_wq(L), o_sq(L), o_zq(L), o_wo(L), o_so(L), o_zo(L), o_wp(L), o_sp(L), o_zp(L);
    for (int l = 0; l < L; ++l) {
        o_wq[l] = take(mat_q);
        if (i4) {
            o_sq[l] = take(sc_q);
            o_zq[l] = take(zp_q);
        }
        o_wo[l] = take(mat_o);
        o_wp[l] = take(mat_p);
        if (i4) {
            o_so[l] = take(sc_o);
            o_zo[l] = take(zp_o);
            o_sp[l] = take(sc_p);
            o_zp[l] = take(zp_p);
        }
    }
    std::vector<size_t> o_qc1(L), o_qcb(L), o_fc1(L), o_fcb(L);
    for (int l = 0; l < L; ++l) {
        o_qc1[l] = take(size_t(3 * E) * 4);
        o_qcb[l] = take(size_t(3 * E) * 4);
        o_fc1[l] = take(size_t(F) * 4);
        o_fcb[l] = take(size_t(F) * 4);
    }
    const size_t head_pad = size_t(head_rpc) * grid;
    const size_t o_hc1 = take(head_pad * 4), o_hcb = take(head_pad * 4);
    const size_t o_h16 = m->head_f16 ? take(size_t(V) * E * 2) : 0;   // the fp16 LM head [V][E]
    // the int4 LM head, padded to head_pad rows: codes [.][E/2], scales [.][E/32] f32, zero points [.][E/64]
    const size_t o_h4c = m->head_int4 ? take(head_pad * E / 2) : 0;
    const size_t o_h4s = m->head_int4 ? take(head_pad * (E / 32) * 4) : 0;
    const size_t o_h4z = m->head_int4 ? take(head_pad * (E / 64)) : 0;
    const size_t o_state = off;
    const size_t acc_bytes = size_t(2) * L * E * 8 * kClusterAccStride;
    const size_t o_accn = take(acc_bytes), o_accx = take(acc_bytes);
    const size_t o_keys = take(size_t(grid) * 8);   // per-CTA LM-head keys, tagged with their pass
    const size_t state_bytes = off - o_state;
    const size_t o_layers = take(sizeof(CLayer) * L);
    uint8_t *B = nullptr;
    TRY_CUDA(cudaMalloc(&B, off));
    m->cbuf = B;
    m->c_state = B + o_state;
    m->c_state_bytes = state_bytes;
    cudaStream_t s = m->stream;
    std::vector<CLayer> cl(L);
    for (int l = 0; l < L; ++l) {
        const LayerDev &Ld = m->layers[l];
        const QMat &qa = Ld.mat[GPT2_MAT_ATTN], &qo = Ld.mat[GPT2_MAT_PROJ], &qf = Ld.mat[GPT2_MAT_FC],
                   &qp = Ld.mat[GPT2_MAT_MLP_PROJ];
        CLayer &x = cl[l];
        x = CLayer{};
        x.Wqkv = B + o_wq[l];
        x.qkv_s = i4 ? reinterpret_cast<const float *>(B + o_sq[l]) : nullptr;
        x.qkv_z = i4 ? B + o_zq[l] : nullptr;
        x.ln1_w = Ld.ln1_w;
        x.ln1_b = Ld.ln1_b;
        x.attn_b = Ld.attn_b;
        x.Wo_t = B + o_wo[l];
        x.o_s = i4 ? reinterpret_cast<const float *>(B + o_so[l]) : nullptr;
        x.o_z = i4 ? B + o_zo[l] : nullptr;
        x.proj_b = Ld.proj_b;
        x.Wfc = qf.w;
        x.fc_s = qf.scales;
        x.fc_z = qf.zeros;
        x.ln2_w = Ld.ln2_w;
        x.ln2_b = Ld.ln2_b;
        x.fc_b = Ld.fc_b;
        x.Wp_t = B + o_wp[l];
        x.p_s = i4 ? reinterpret_cast<const float *>(B + o_sp[l]) : nullptr;
        x.p_z = i4 ? B + o_zp[l] : nullptr;
        x.mlp_proj_b = Ld.mlp_proj_b;
        TRY_CUDA(cluster_gather_qkv(wt, qa.w, qa.scales, qa.zeros, E, D, B + o_wq[l],
                                    i4 ? reinterpret_cast<float *>(B + o_sq[l]) : nullptr, i4 ? B + o_zq[l] : nullptr,
                                    s));
        TRY_CUDA(cluster_tile(wt, qo.w, qo.scales, qo.zeros, E, H * kClusterSize, kClusterSize, E / kClusterSize, D,
                              B + o_wo[l], i4 ? reinterpret_cast<float *>(B + o_so[l]) : nullptr,
                              i4 ? B + o_zo[l] : nullptr, s));
        TRY_CUDA(cluster_tile(wt, qp.w, qp.scales, qp.zeros, F, nfc, 1, E, fr, B + o_wp[l],
                              i4 ? reinterpret_cast<float *>(B + o_sp[l]) : nullptr, i4 ? B + o_zp[l] : nullptr, s));
    }
    // LayerNorm folded into the QKV, fc and LM-head rows, from the weights as
    // stored: c1 = W.gamma, cb = W.beta + bias (QKV in the gathered order)
    {
        float *tmp = nullptr, *d1 = nullptr, *d2 = nullptr;
        const size_t nmax = std::max(size_t(V), size_t(F));
        cudaError_t e = cudaMalloc(&tmp, size_t(F) * E * 4);
        if (e == cudaSuccess) e = cudaMalloc(&d1, nmax * 4);
        if (e == cudaSuccess) e = cudaMalloc(&d2, nmax * 4);
        std::vector<float> h1(nmax), h2(nmax), hb(nmax), g1(nmax, 0.f), g2(nmax, 0.f);
        auto fold = [&](const QMat &q, const float *gamma, const float *beta) -> cudaError_t {
            cudaError_t r = dequant_to_f32(wt, q.w, q.scales, q.zeros, q.in, q.out, tmp, s);
            if (r == cudaSuccess) r = ln_fold(tmp, gamma, beta, q.in, q.out, d1, d2, s);
            if (r == cudaSuccess) r = cudaMemcpyAsync(h1.data(), d1, size_t(q.out) * 4, cudaMemcpyDeviceToHost, s);
            if (r == cudaSuccess) r = cudaMemcpyAsync(h2.data(), d2, size_t(q.out) * 4, cudaMemcpyDeviceToHost, s);
            return r;
        };
        const int q4 = D / 4, Rq = 3 * q4;
        for (int l = 0; l < L && e == cudaSuccess; ++l) {
            const LayerDev &Ld = m->layers[l];
            e = fold(Ld.mat[GPT2_MAT_ATTN], Ld.ln1_w, Ld.ln1_b);
            if (e == cudaSuccess) e = cudaMemcpyAsync(hb.data(), Ld.attn_b, size_t(3 * E) * 4, cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) break;
            for (int j = 0; j < 3 * E; ++j) {
                const int t = j / Rq, i = j % Rq, h = t / kClusterSize, r = t % kClusterSize;
                const int src = (i / q4) * E + h * D + r * q4 + i % q4;
                g1[j] = h1[src];
                g2[j] = h2[src] + hb[src];
            }
            e = cudaMemcpy(B + o_qc1[l], g1.data(), size_t(3 * E) * 4, cudaMemcpyHostToDevice);
            if (e == cudaSuccess) e = cudaMemcpy(B + o_qcb[l], g2.data(), size_t(3 * E) * 4, cudaMemcpyHostToDevice);
            if (e == cudaSuccess) e = fold(Ld.mat[GPT2_MAT_FC], Ld.ln2_w, Ld.ln2_b);
            if (e == cudaSuccess) e = cudaMemcpyAsync(hb.data(), Ld.fc_b, size_t(F) * 4, cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) break;
            for (int j = 0; j < F; ++j) h2[j] += hb[j];
            e = cudaMemcpy(B + o_fc1[l], h1.data(), size_t(F) * 4, cudaMemcpyHostToDevice);
            if (e == cudaSuccess) e = cudaMemcpy(B + o_fcb[l], h2.data(), size_t(F) * 4, cudaMemcpyHostToDevice);
        }
        if (e == cudaSuccess) e = cudaMemsetAsync(B + o_hc1, 0, head_pad * 4, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(B + o_hcb, 0, head_pad * 4, s);
        if (m->head_f16) {
            // the fp16 head, and its LayerNorm fold constants from the stored (rounded) values
            float *wide = nullptr;
            if (e == cudaSuccess) e = convert_f16(m->wte, size_t(V) * E, B + o_h16, s);
            if (e == cudaSuccess) e = cudaMalloc(&wide, size_t(V) * E * 4);
            if (e == cudaSuccess) e = dequant_to_f32(kWF16, B + o_h16, nullptr, nullptr, E, V, wide, s);
            if (e == cudaSuccess) e = ln_fold(wide, m->lnf_w, m->lnf_b, E, V, reinterpret_cast<float *>(B + o_hc1),
                                              reinterpret_cast<float *>(B + o_hcb), s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (wide) cudaFree(wide);
        } else if (m->head_int4) {
            // quantise wte's rows (already [out][in]); padding rows stay zero (scale 0: value 0)
            float *wide = nullptr;
            uint8_t *hc = B + o_h4c, *hz = B + o_h4z;
            float *hs = reinterpret_cast<float *>(B + o_h4s);
            if (e == cudaSuccess) e = cudaMemsetAsync(hc, 0, head_pad * E / 2, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(hs, 0, head_pad * (E / 32) * 4, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(hz, 0, head_pad * (E / 64), s);
            if (e == cudaSuccess) e = quant_int4_rows(m->wte, E, V, hc, hs, hz, s);
            if (e == cudaSuccess) e = cudaMalloc(&wide, size_t(V) * E * 4);
            if (e == cudaSuccess) e = dequant_to_f32(kWI4, hc, hs, hz, E, V, wide, s);
            if (e == cudaSuccess) e = ln_fold(wide, m->lnf_w, m->lnf_b, E, V, reinterpret_cast<float *>(B + o_hc1),
                                              reinterpret_cast<float *>(B + o_hcb), s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (wide) cudaFree(wide);
        } else if (e == cudaSuccess) {
            e = ln_fold(m->wte, m->lnf_w, m->lnf_b, E, V, reinterpret_cast<float *>(B + o_hc1),
                        reinterpret_cast<float *>(B + o_hcb), s);
        }
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (tmp) cudaFree(tmp);
        if (d1) cudaFree(d1);
        if (d2) cudaFree(d2);
        TRY_CUDA(e);
    }
    for (int l = 0; l < L; ++l) {
        cl[l].q_c1 = reinterpret_cast<const float *>(B + o_qc1[l]);
        cl[l].q_cb = reinterpret_cast<const float *>(B + o_qcb[l]);
        cl[l].f_c1 = reinterpret_cast<const float *>(B + o_fc1[l]);
        cl[l].f_cb = reinterpret_cast<const float *>(B + o_fcb[l]);
    }
    TRY_CUDA(cudaMemsetAsync(m->c_state, 0, state_bytes, s));
    TRY_CUDA(cudaMemcpyAsync(B + o_layers, cl.data(), sizeof(CLayer) * L, cudaMemcpyHostToDevice, s));
    TRY_CUDA(cudaStreamSynchronize(s));

    ClusterArgs &a = m->cargs;
    a = ClusterArgs{};
    a.layers = reinterpret_cast<const CLayer *>(B + o_layers);
    a.L = L;
    a.E = E;
    a.H = H;
    a.D = D;
    a.F = F;
    a.P = c.n_positions;
    a.V = V;
    a.eps = c.ln_eps;
    a.scale = float(1.0 / std::sqrt(double(D)));
    a.nfc = nfc;
    a.fr = fr;
    a.head_rpc = head_rpc;
    a.pr_rows = pr_rows;
    a.head_w = m->head_f16 ? static_cast<const void *>(B + o_h16)
               : m->head_int4 ? static_cast<const void *>(B + o_h4c) : static_cast<const void *>(m->wte);
    a.head_s = m->head_int4 ? reinterpret_cast<const float *>(B + o_h4s) : nullptr;
    a.head_z = m->head_int4 ? B + o_h4z : nullptr;
    a.head_wt = m->head_f16 ? kWF16 : m->head_int4 ? kWI4 : kWF32;
    a.h_c1 = reinterpret_cast<const float *>(B + o_hc1);
    a.h_cb = reinterpret_cast<const float *>(B + o_hcb);
    a.acc_new = reinterpret_cast<long long *>(B + o_accn);
    a.acc_next = reinterpret_cast<long long *>(B + o_accx);
    a.kcache = m->kcache;
    a.vcache = m->vcache;
    a.logits = m->logits;
    a.partials = reinterpret_cast<unsigned long long *>(B + o_keys);
    a.out_ids = m->out_ids;
    a.out_cap = m->out_cap;
    a.st = m->st;
    a.wte = m->wte;
    a.wpe = m->wpe;
    a.lnf_w = m->lnf_w;
    a.lnf_b = m->lnf_b;
    a.wtype = wt;
    a.n_stages = ns;
    a.stage_bytes = stage;
    a.ring_offset = ring_offset;
    a.wait_ns = kWaitLimitNs;
    m->c_clusters = n_clusters;
    m->prompt_buf = prompt_buf;
    m->cluster = true;
    return GPT2_OK;
}

}  // namespace

extern "C" {

const char *gpt2_strerror(int status)
{
    switch (status) {
    case GPT2_OK: return "ok";
    case GPT2_ERR_INVALID_ARG: return "invalid argument";
    case GPT2_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case GPT2_ERR_TOKEN_RANGE: return "token outside [0, vocab_size)";
    case GPT2_ERR_POSITION_RANGE: return "position outside the context or past the cached length";
    case GPT2_ERR_NOT_READY: return "no decode step has run yet";
    case GPT2_ERR_CUDA: return "CUDA runtime error";
    case GPT2_ERR_TIMEOUT: return "a bounded device wait timed out";
    case GPT2_ERR_DEVICE_STATE: return "a kernel rejected its device-side inputs";
    case GPT2_ERR_OUT_OF_MEMORY: return "device out of memory";
    case GPT2_ERR_RANGE: return "an activation left the range of the fixed-point residual sums";
    default: return "unknown status";
    }
}

int gpt2_create(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype, void *stream, gpt2_model **out)
{
    return gpt2_create_ex(cfg, w, wdtype, 0, stream, out);
}

int gpt2_create_ex(const gpt2_config *cfg, const gpt2_weights *w, int32_t wdtype, int32_t flags, void *stream,
                   gpt2_model **out)
{
    if (!out) return GPT2_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = check_config(cfg, wdtype);
    if (rc != GPT2_OK) return rc;
    if (!w || !w->layers) return GPT2_ERR_INVALID_ARG;
    if (flags & ~int32_t(GPT2_FLAG_PER_KERNEL | GPT2_FLAG_HEAD_F16 | GPT2_FLAG_HEAD_INT4 | GPT2_FLAG_NO_TC_PREFILL))
        return GPT2_ERR_INVALID_ARG;
    if ((flags & GPT2_FLAG_HEAD_F16) && (flags & GPT2_FLAG_HEAD_INT4)) return GPT2_ERR_INVALID_ARG;
    int dev;
    TRY_CUDA(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    TRY_CUDA(cudaGetDeviceProperties(&prop, dev));
    if (!(prop.major == 10 && prop.minor == 3)) return GPT2_ERR_UNSUPPORTED_DEVICE;
    TRY_CUDA(gemv_init());
    // every tensor pointer must be device memory
    const float *top[4] = {w->wte, w->wpe, w->ln_f_w, w->ln_f_b};
    for (const float *p : top)
        if (!is_device_ptr(p)) return GPT2_ERR_INVALID_ARG;
    for (int l = 0; l < cfg->n_layer; ++l) {
        const gpt2_layer_weights &L = w->layers[l];
        const float *ps[12] = {L.ln1_w, L.ln1_b, L.attn_w, L.attn_b, L.proj_w, L.proj_b,
                               L.ln2_w, L.ln2_b, L.fc_w,   L.fc_b,   L.mlp_proj_w, L.mlp_proj_b};
        for (const float *p : ps)
            if (!is_device_ptr(p)) return GPT2_ERR_INVALID_ARG;
    }

    gpt2_model *m = new (std::nothrow) gpt2_model();
    if (!m) return GPT2_ERR_OUT_OF_MEMORY;
    m->cfg = *cfg;
    m->wdtype = wdtype;
    m->head_f16 = (flags & GPT2_FLAG_HEAD_F16) != 0;
    m->head_int4 = (flags & GPT2_FLAG_HEAD_INT4) != 0;
    m->stream = static_cast<cudaStream_t>(stream);
    m->device = dev;
    m->num_sms = prop.multiProcessorCount;
    m->max_head_ctas = std::min(m->num_sms, 1024);

    const int L = cfg->n_layer, E = cfg->n_embd, H = cfg->n_head, P = cfg->n_positions, V = cfg->vocab_size;
    const int F = 4 * E;
    const int D = E / H;
    // ---- weight arena layout ----
    const int mat_in[4] = {E, E, E, F};
    const int mat_out[4] = {3 * E, E, F, E};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += aup(bytes);
        return o;
    };
    const size_t o_wte = take(size_t(V) * E * 4), o_wpe = take(size_t(P) * E * 4);
    const size_t o_lnf_w = take(E * 4), o_lnf_b = take(E * 4);
    struct LOff {
        size_t ln1_w, ln1_b, attn_b, proj_b, ln2_w, ln2_b, fc_b, mlp_proj_b;
        size_t w[4], s[4], z[4];
    };
    std::vector<LOff> lo(L);
    for (int l = 0; l < L; ++l) {
        lo[l].ln1_w = take(E * 4);
        lo[l].ln1_b = take(E * 4);
        lo[l].attn_b = take(3 * E * 4);
        lo[l].proj_b = take(E * 4);
        lo[l].ln2_w = take(E * 4);
        lo[l].ln2_b = take(E * 4);
        lo[l].fc_b = take(F * 4);
        lo[l].mlp_proj_b = take(E * 4);
        for (int k = 0; k < 4; ++k) {
            lo[l].w[k] = take(main_bytes_of(wdtype, mat_in[k], mat_out[k]));
            if (wdtype == GPT2_INT4) {
                lo[l].s[k] = take(size_t(mat_out[k]) * (mat_in[k] / 32) * 4);
                lo[l].z[k] = take(size_t(mat_out[k]) * (mat_in[k] / 64));
            }
        }
    }
    m->arena_bytes = off;
    // ---- work area layout ----
    off = 0;
    const size_t kv = size_t(L) * H * P * D * 4;
    const size_t o_k = take(kv), o_v = take(kv);
    const size_t o_x = take(E * 4), o_qkv = take(3 * E * 4), o_attn = take(E * 4), o_h = take(F * 4);
    const size_t o_logits = take(size_t(V) * 4);
    const size_t o_st = take(sizeof(DeviceState));
    m->out_cap = P + 1;
    const size_t o_ids = take(size_t(m->out_cap) * 4);
    const size_t o_part = take(size_t(m->max_head_ctas) * 8);
    const size_t o_cnt = take(16);
    const size_t o_prompt = take(size_t(P) * 4);
    m->work_bytes = off;

    cudaError_t e = cudaMalloc(&m->arena, m->arena_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&m->work, m->work_bytes);
    if (e != cudaSuccess) {
        free_model(m);
        return cuda_status(e);
    }
    uint8_t *A = m->arena, *W = m->work;
    m->wte = reinterpret_cast<float *>(A + o_wte);
    m->wpe = reinterpret_cast<float *>(A + o_wpe);
    m->lnf_w = reinterpret_cast<float *>(A + o_lnf_w);
    m->lnf_b = reinterpret_cast<float *>(A + o_lnf_b);
    m->layers.resize(L);
    for (int l = 0; l < L; ++l) {
        LayerDev &d = m->layers[l];
        d.ln1_w = reinterpret_cast<float *>(A + lo[l].ln1_w);
        d.ln1_b = reinterpret_cast<float *>(A + lo[l].ln1_b);
        d.attn_b = reinterpret_cast<float *>(A + lo[l].attn_b);
        d.proj_b = reinterpret_cast<float *>(A + lo[l].proj_b);
        d.ln2_w = reinterpret_cast<float *>(A + lo[l].ln2_w);
        d.ln2_b = reinterpret_cast<float *>(A + lo[l].ln2_b);
        d.fc_b = reinterpret_cast<float *>(A + lo[l].fc_b);
        d.mlp_proj_b = reinterpret_cast<float *>(A + lo[l].mlp_proj_b);
        for (int k = 0; k < 4; ++k) {
            QMat &q = d.mat[k];
            q.in = mat_in[k];
            q.out = mat_out[k];
            q.w = A + lo[l].w[k];
            q.main_bytes = main_bytes_of(wdtype, q.in, q.out);
            if (wdtype == GPT2_INT4) {
                q.scales = reinterpret_cast<float *>(A + lo[l].s[k]);
                q.zeros = A + lo[l].z[k];
                q.scale_bytes = size_t(q.out) * (q.in / 32) * 4;
                q.zero_bytes = size_t(q.out) * (q.in / 64);
            }
        }
    }
    m->kcache = reinterpret_cast<float *>(W + o_k);
    m->vcache = reinterpret_cast<float *>(W + o_v);
    m->x = reinterpret_cast<float *>(W + o_x);
    m->qkv = reinterpret_cast<float *>(W + o_qkv);
    m->attn = reinterpret_cast<float *>(W + o_attn);
    m->h = reinterpret_cast<float *>(W + o_h);
    m->logits = reinterpret_cast<float *>(W + o_logits);
    m->st = reinterpret_cast<DeviceState *>(W + o_st);
    m->out_ids = reinterpret_cast<int32_t *>(W + o_ids);
    m->partials = reinterpret_cast<unsigned long long *>(W + o_part);
    m->counter = reinterpret_cast<unsigned int *>(W + o_cnt);

    // ---- copy and repack ----
    cudaStream_t s = m->stream;
    float *tmp = nullptr;
    auto fail = [&](cudaError_t err) {
        if (tmp) cudaFree(tmp);
        cudaStreamSynchronize(s);
        free_model(m);
        return cuda_status(err);
    };
#define CK(expr)                                  \
    do {                                          \
        cudaError_t _e2 = (expr);                 \
        if (_e2 != cudaSuccess) return fail(_e2); \
    } while (0)
    CK(cudaMemsetAsync(m->work, 0, m->work_bytes, s));
    CK(cudaMemcpyAsync(m->wte, w->wte, size_t(V) * E * 4, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(m->wpe, w->wpe, size_t(P) * E * 4, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(m->lnf_w, w->ln_f_w, E * 4, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpyAsync(m->lnf_b, w->ln_f_b, E * 4, cudaMemcpyDeviceToDevice, s));
    if (wdtype == GPT2_INT4) CK(cudaMalloc(&tmp, size_t(F) * E * 4));
    for (int l = 0; l < L; ++l) {
        const gpt2_layer_weights &src = w->layers[l];
        LayerDev &d = m->layers[l];
        CK(cudaMemcpyAsync(d.ln1_w, src.ln1_w, E * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.ln1_b, src.ln1_b, E * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.attn_b, src.attn_b, 3 * E * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.proj_b, src.proj_b, E * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.ln2_w, src.ln2_w, E * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.ln2_b, src.ln2_b, E * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.fc_b, src.fc_b, F * 4, cudaMemcpyDeviceToDevice, s));
        CK(cudaMemcpyAsync(d.mlp_proj_b, src.mlp_proj_b, E * 4, cudaMemcpyDeviceToDevice, s));
        const float *srcm[4] = {src.attn_w, src.proj_w, src.fc_w, src.mlp_proj_w};
        for (int k = 0; k < 4; ++k) {
            QMat &q = d.mat[k];
            if (wdtype == GPT2_F32) CK(repack_f32(srcm[k], q.in, q.out, static_cast<float *>(q.w), s));
            else if (wdtype == GPT2_F16) CK(repack_f16(srcm[k], q.in, q.out, q.w, s));
            else CK(repack_int4(srcm[k], q.in, q.out, tmp, static_cast<uint8_t *>(q.w), q.scales, q.zeros, s));
        }
    }
    CK(cudaStreamSynchronize(s));
    if (tmp) {
        cudaFree(tmp);
        tmp = nullptr;
    }
#undef CK
    rc = build_graph(m);
    if (rc != GPT2_OK) {
        free_model(m);
        return rc;
    }
    if (!(flags & GPT2_FLAG_PER_KERNEL)) {
        rc = setup_cluster(m, reinterpret_cast<int32_t *>(W + o_prompt));
        if (rc != GPT2_OK) {            // the per-kernel graph computes the pass instead
            cudaGetLastError();
            if (m->cbuf) cudaFree(m->cbuf);
            m->cbuf = nullptr;
            m->cluster = false;
        }
    }
    if (m->cluster && !(flags & GPT2_FLAG_NO_TC_PREFILL)) {
        // the prefill engine: the stored matrices and head as bf16 hi + lo planes
        std::vector<const float *> params(size_t(L) * 8);
        for (int l = 0; l < L; ++l) {
            const LayerDev &d = m->layers[l];
            const float *pv[8] = {d.ln1_w, d.ln1_b, d.attn_b, d.proj_b, d.ln2_w, d.ln2_b, d.fc_b, d.mlp_proj_b};
            for (int k = 0; k < 8; ++k) params[size_t(l) * 8 + k] = pv[k];
        }
        PrefillSrc ps;
        ps.wte = m->wte;
        ps.wpe = m->wpe;
        ps.lnf_w = m->lnf_w;
        ps.lnf_b = m->lnf_b;
        ps.params = params.data();
        ps.kc = m->kcache;
        ps.vc = m->vcache;
        ps.matrix = [m](int l, int k, float *dst, cudaStream_t st) {
            const QMat &q = m->layers[l].mat[k];
            return dequant_to_f32(m->wdtype, q.w, q.scales, q.zeros, q.in, q.out, dst, st);
        };
        ps.head = [m](float *dst, cudaStream_t st) {
            const ClusterArgs &a = m->cargs;
            if (a.head_wt == kWF32)
                return cudaMemcpyAsync(dst, m->wte, size_t(m->cfg.vocab_size) * m->cfg.n_embd * 4,
                                       cudaMemcpyDeviceToDevice, st);
            return dequant_to_f32(a.head_wt, a.head_w, a.head_s, a.head_z, m->cfg.n_embd, m->cfg.vocab_size, dst, st);
        };
        rc = prefill_engine_create(m->cfg, ps, m->stream, m->num_sms, &m->pre);
        if (rc != GPT2_OK) {
            free_model(m);
            return rc;
        }
    }
    if ((m->head_f16 || m->head_int4) && !m->cluster) {   // a separate head is read only by the cluster kernel
        free_model(m);
        return GPT2_ERR_INVALID_ARG;
    }
    // state: the epoch sequence starts at 1 (tagged words are zero)
    DeviceState init{};
    init.seq = 1;
    rc = cuda_status(cudaMemcpy(m->st, &init, sizeof init, cudaMemcpyHostToDevice));
    if (rc != GPT2_OK) {
        free_model(m);
        return rc;
    }
    *out = m;
    return GPT2_OK;
}

void gpt2_destroy(gpt2_model *m)
{
    if (!m) return;
    cudaStreamSynchronize(m->stream);
    free_model(m);
}

int gpt2_set_sampling(gpt2_model *m, float temperature, uint64_t seed)
{
    if (!m || !(temperature >= 0.f) || !std::isfinite(temperature)) return GPT2_ERR_INVALID_ARG;
    if (temperature > 0.f && !m->cluster) return GPT2_ERR_INVALID_ARG;   // drawn in the cluster kernel's head
    m->cargs.temperature = temperature;
    m->cargs.seed = (unsigned long long)seed;
    return GPT2_OK;
}

int gpt2_set_wait_limit(gpt2_model *m, uint64_t ns)
{
    if (!m) return GPT2_ERR_INVALID_ARG;
    if (!m->cluster) return GPT2_ERR_INVALID_ARG;   // the per-kernel graph has no cross-CTA waits
    m->cargs.wait_ns = (unsigned long long)ns;
    return GPT2_OK;
}

int gpt2_reset(gpt2_model *m)
{
    if (!m) return GPT2_ERR_INVALID_ARG;
    m->cached = 0;
    m->has_step = false;
    return GPT2_OK;
}

int gpt2_decode_step(gpt2_model *m, int32_t token, int32_t position, const float **dev_logits)
{
    if (!m) return GPT2_ERR_INVALID_ARG;
    if (token < 0 || token >= m->cfg.vocab_size) return GPT2_ERR_TOKEN_RANGE;
    if (position < 0 || position >= m->cfg.n_positions || position > m->cached) return GPT2_ERR_POSITION_RANGE;
    int rc = launch_step(m, token, position);
    if (rc != GPT2_OK) return rc;
    m->cached = position + 1;
    m->has_step = true;
    if (dev_logits) *dev_logits = m->logits;
    return GPT2_OK;
}

int gpt2_prefill(gpt2_model *m, const int32_t *host_ids, int32_t n)
{
    if (!m || !host_ids) return GPT2_ERR_INVALID_ARG;
    if (n < 1 || n > m->cfg.n_positions) return GPT2_ERR_POSITION_RANGE;
    for (int i = 0; i < n; ++i)
        if (host_ids[i] < 0 || host_ids[i] >= m->cfg.vocab_size) return GPT2_ERR_TOKEN_RANGE;
    gpt2_reset(m);
    if (use_tc_prefill(m, n)) {
        int rc = prefill_engine_run(m->pre, host_ids, n, m->st, m->out_ids, m->out_cap, m->logits, m->stream,
                                    &m->launches);
        if (rc != GPT2_OK) return rc;
        m->cached = n;
        m->has_step = true;
        return GPT2_OK;
    }
    if (m->cluster) {
        TRY_CUDA(cudaMemcpyAsync(m->prompt_buf, host_ids, size_t(n) * 4, cudaMemcpyHostToDevice, m->stream));
        int rc = launch_cluster_call(m, n, m->prompt_buf, n, 0, 0);
        if (rc != GPT2_OK) return rc;
        m->cached = n;
        m->has_step = true;
        return GPT2_OK;
    }
    for (int i = 0; i < n; ++i) {
        int rc = gpt2_decode_step(m, host_ids[i], i, nullptr);
        if (rc != GPT2_OK) return rc;
    }
    return GPT2_OK;
}

int gpt2_argmax(gpt2_model *m, int32_t *token_out)
{
    if (!m || !token_out) return GPT2_ERR_INVALID_ARG;
    if (!m->has_step) return GPT2_ERR_NOT_READY;
    DeviceState hs;
    int rc = read_state(m, &hs);
    if (rc != GPT2_OK) return rc;
    *token_out = hs.next_tok;
    return GPT2_OK;
}

int gpt2_decode_greedy(gpt2_model *m, int32_t n_steps)
{
    if (!m || n_steps < 0) return GPT2_ERR_INVALID_ARG;
    if (!m->has_step) return GPT2_ERR_NOT_READY;
    if ((long long)m->cached + n_steps > m->cfg.n_positions) return GPT2_ERR_POSITION_RANGE;
    if (n_steps == 0) return GPT2_OK;
    if (m->cluster) {
        int rc = launch_cluster_call(m, n_steps, nullptr, 0, 0, m->cached);
        if (rc != GPT2_OK) return rc;
    } else {
        for (int i = 0; i < n_steps; ++i) TRY_CUDA(cudaGraphLaunch(m->exec, m->stream));
        m->launches += (unsigned long long)n_steps * m->kernels_per_step;
    }
    m->cached += n_steps;
    return GPT2_OK;
}

int gpt2_generate(gpt2_model *m, const int32_t *host_prompt, int32_t n_prompt, int32_t n_steps,
                  int32_t *host_out)
{
    if (!m || !host_prompt || !host_out || n_steps < 0) return GPT2_ERR_INVALID_ARG;
    if (n_prompt < 1 || (long long)n_prompt + n_steps > m->cfg.n_positions) return GPT2_ERR_POSITION_RANGE;
    for (int i = 0; i < n_prompt; ++i)
        if (host_prompt[i] < 0 || host_prompt[i] >= m->cfg.vocab_size) return GPT2_ERR_TOKEN_RANGE;
    int rc;
    if (m->cluster) {
        gpt2_reset(m);
        TRY_CUDA(launch_set_state(m->st, 0, 0, kResetOut, m->out_ids, m->stream));
        m->launches += 1;
        if (use_tc_prefill(m, n_prompt)) {
            // the prompt on the tensor cores, then the greedy passes in one launch
            rc = prefill_engine_run(m->pre, host_prompt, n_prompt, m->st, m->out_ids, m->out_cap, m->logits,
                                    m->stream, &m->launches);
            if (rc == GPT2_OK && n_steps > 0) rc = launch_cluster_call(m, n_steps, nullptr, 0, 0, n_prompt);
        } else {
            TRY_CUDA(cudaMemcpyAsync(m->prompt_buf, host_prompt, size_t(n_prompt) * 4, cudaMemcpyHostToDevice,
                                     m->stream));
            rc = launch_cluster_call(m, n_prompt + n_steps, m->prompt_buf, n_prompt, 0, 0);
        }
        if (rc != GPT2_OK) return rc;
        m->cached = n_prompt + n_steps;
        m->has_step = true;
    } else {
        rc = gpt2_prefill(m, host_prompt, n_prompt);
        if (rc != GPT2_OK) return rc;
        TRY_CUDA(launch_set_state(m->st, 0, 0, kSeedOutWithNext, m->out_ids, m->stream));
        m->launches += 1;
        rc = gpt2_decode_greedy(m, n_steps);
        if (rc != GPT2_OK) return rc;
    }
    TRY_CUDA(cudaMemcpyAsync(host_out, m->out_ids, size_t(n_steps + 1) * 4, cudaMemcpyDeviceToHost, m->stream));
    DeviceState hs;
    return read_state(m, &hs);
}

int gpt2_copy_logits(gpt2_model *m, float *dst)
{
    if (!m || !dst) return GPT2_ERR_INVALID_ARG;
    if (!m->has_step) return GPT2_ERR_NOT_READY;
    TRY_CUDA(cudaMemcpyAsync(dst, m->logits, size_t(m->cfg.vocab_size) * 4, cudaMemcpyDefault, m->stream));
    DeviceState hs;
    return read_state(m, &hs);
}

int gpt2_sync(gpt2_model *m)
{
    if (!m) return GPT2_ERR_INVALID_ARG;
    DeviceState hs;
    return read_state(m, &hs);
}

int gpt2_matrix_bytes(const gpt2_model *m, int32_t which, size_t *main_bytes, size_t *scale_bytes,
                      size_t *zero_bytes)
{
    if (!m || which < 0 || which > 3) return GPT2_ERR_INVALID_ARG;
    const QMat &q = m->layers[0].mat[which];
    if (main_bytes) *main_bytes = q.main_bytes;
    if (scale_bytes) *scale_bytes = q.scale_bytes;
    if (zero_bytes) *zero_bytes = q.zero_bytes;
    return GPT2_OK;
}

int gpt2_export_matrix(gpt2_model *m, int32_t layer, int32_t which, void *dst_main, void *dst_scales,
                       void *dst_zeros)
{
    if (!m || layer < 0 || layer >= m->cfg.n_layer || which < 0 || which > 3) return GPT2_ERR_INVALID_ARG;
    const QMat &q = m->layers[layer].mat[which];
    if (dst_main) TRY_CUDA(cudaMemcpyAsync(dst_main, q.w, q.main_bytes, cudaMemcpyDefault, m->stream));
    if (dst_scales && q.scales)
        TRY_CUDA(cudaMemcpyAsync(dst_scales, q.scales, q.scale_bytes, cudaMemcpyDefault, m->stream));
    if (dst_zeros && q.zeros)
        TRY_CUDA(cudaMemcpyAsync(dst_zeros, q.zeros, q.zero_bytes, cudaMemcpyDefault, m->stream));
    TRY_CUDA(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_export_dequant(gpt2_model *m, int32_t layer, int32_t which, float *dst)
{
    if (!m || !dst || layer < 0 || layer >= m->cfg.n_layer || which < 0 || which > 3) return GPT2_ERR_INVALID_ARG;
    if (!is_device_ptr(dst)) return GPT2_ERR_INVALID_ARG;
    const QMat &q = m->layers[layer].mat[which];
    TRY_CUDA(dequant_to_f32(m->wdtype, q.w, q.scales, q.zeros, q.in, q.out, dst, m->stream));
    TRY_CUDA(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_export_kv(gpt2_model *m, int32_t layer, int32_t n_rows, float *dst_k, float *dst_v)
{
    if (!m || layer < 0 || layer >= m->cfg.n_layer) return GPT2_ERR_INVALID_ARG;
    const int H = m->cfg.n_head, D = m->cfg.n_embd / H, P = m->cfg.n_positions;
    if (n_rows < 0 || n_rows > P) return GPT2_ERR_INVALID_ARG;
    for (int h = 0; h < H; ++h) {
        const size_t src = (size_t(layer) * H + h) * P * D;
        const size_t dst = size_t(h) * n_rows * D;
        const size_t bytes = size_t(n_rows) * D * 4;
        if (dst_k) TRY_CUDA(cudaMemcpyAsync(dst_k + dst, m->kcache + src, bytes, cudaMemcpyDefault, m->stream));
        if (dst_v) TRY_CUDA(cudaMemcpyAsync(dst_v + dst, m->vcache + src, bytes, cudaMemcpyDefault, m->stream));
    }
    TRY_CUDA(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_kernels_per_step(const gpt2_model *m, int32_t *count)
{
    if (!m || !count) return GPT2_ERR_INVALID_ARG;
    *count = m->cluster ? 1 : m->kernels_per_step;
    return GPT2_OK;
}

int gpt2_launch_count(const gpt2_model *m, uint64_t *count)
{
    if (!m || !count) return GPT2_ERR_INVALID_ARG;
    *count = m->launches;
    return GPT2_OK;
}

int gpt2_path(const gpt2_model *m, int32_t *path)
{
    if (!m || !path) return GPT2_ERR_INVALID_ARG;
    *path = m->cluster ? GPT2_PATH_CLUSTER : GPT2_PATH_PER_KERNEL;
    return GPT2_OK;
}

int gpt2_op_layernorm(const float *x, const float *gamma, const float *beta, int32_t rows, int32_t n, float eps,
                      float *y, void *stream)
{
    if (!x || !gamma || !beta || !y || rows < 0 || n < 1 || n % 4 || !(eps > 0.f)) return GPT2_ERR_INVALID_ARG;
    if (rows == 0) return GPT2_OK;
    TRY_CUDA(launch_layernorm_rows(x, gamma, beta, rows, n, eps, y, static_cast<cudaStream_t>(stream)));
    return GPT2_OK;
}

// Workspace of the stand-alone head: a 16-byte arrival counter, then one
// 8-byte (value, index) key per CTA; the grid never exceeds 1024 CTAs.
static constexpr int kOpHeadMaxCtas = 1024;

size_t gpt2_op_head_argmax_workspace(int32_t vocab, int32_t n_embd)
{
    (void)vocab;
    (void)n_embd;
    return 16 + size_t(kOpHeadMaxCtas) * 8;
}

int gpt2_op_head_argmax(const float *x, const float *ln_w, const float *ln_b, float eps, const float *wte,
                        int32_t vocab, int32_t n_embd, float *logits, int32_t *dev_token, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    if (!x || !ln_w || !ln_b || !wte || !logits || !dev_token || !workspace) return GPT2_ERR_INVALID_ARG;
    if (vocab < 1 || n_embd < 4 || n_embd % 4 || !(eps > 0.f)) return GPT2_ERR_INVALID_ARG;
    if ((long long)vocab * n_embd > (1ll << 31) - 1) return GPT2_ERR_INVALID_ARG;
    if (workspace_bytes < gpt2_op_head_argmax_workspace(vocab, n_embd)) return GPT2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 || reinterpret_cast<uintptr_t>(wte) % 16)
        return GPT2_ERR_INVALID_ARG;
    int dev, sms;
    TRY_CUDA(gemv_init());
    TRY_CUDA(cudaGetDevice(&dev));
    TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemvArgs a;
    std::memset(&a, 0, sizeof a);
    a.W = wte;
    a.in = n_embd;
    a.out = vocab;
    a.eps = eps;
    const int grid = gemv_plan(a, kWF32, std::min(sms, kOpHeadMaxCtas), 96 * 1024, 4);
    a.evict_first = 1;
    a.xin = x;
    a.ln_w = ln_w;
    a.ln_b = ln_b;
    a.y = logits;
    a.counter = static_cast<unsigned int *>(workspace);
    a.partials = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(workspace) + 16);
    a.dev_token = dev_token;
    TRY_CUDA(cudaMemsetAsync(a.counter, 0, sizeof(unsigned int), s));
    TRY_CUDA(launch_gemv(kWF32, kModeHead, a, grid, s, false));
    return GPT2_OK;
}

}  // extern "C"
