// gpt2_op_head_argmax_noalloc: the stand-alone final LayerNorm + tied head +
// argmax for callers that must not allocate device memory.
//
// Who needs it: some hosts own every byte of device memory themselves — an
// inference server that hands each plugin fixed, pre-sized buffers from its
// own pool, or a runtime whose steady-state loop must never enter (and never
// block in, or fragment) the CUDA allocator.  Such a caller can pass inputs and
// outputs but cannot cudaMalloc the small workspace gpt2_op_head_argmax needs.
// This variant runs the same kernel with that workspace taken from a fixed
// array in the library's own device memory instead.
//
// The scratch array below exists once per GPU that loads the library and
// stays until the process exits.  Every call on a device uses the same array,
// so two calls whose kernels overlap on the GPU (on different streams, or from
// different threads) race on it and give wrong results; serialise them.  The
// array keeps whatever the last call left in it, so each call clears the part
// that must start at zero (the arrival counter) before its kernel runs.
#include "../../include/gpt2.h"

#include <cuda.h>

#include <cstring>
#include <mutex>

#include "kernels.h"

using namespace gpt2;

namespace {

// Scratch layout: a 16-byte arrival counter, then one 8-byte packed
// (value, index) key per CTA.  The kernel uses one CTA per 256 vocabulary
// rows (at most), so 512 keys cover a vocabulary of 131072.
constexpr int kRowsPerCta = 256;
constexpr int kMaxCtas = 512;
constexpr size_t kScratchBytes = 16 + size_t(kMaxCtas) * 8;   // 4112 bytes
static_assert(size_t(kRowsPerCta) * kMaxCtas == GPT2_NOALLOC_MAX_VOCAB, "limit in gpt2.h");

static __device__ __align__(256) unsigned char g_head_scratch[kScratchBytes];

// In host code `g_head_scratch` names a host-side stand-in, not device memory;
// the device address comes from cudaGetSymbolAddress, looked up once per
// device with that device current.  The module is loaded into the device's
// context, so the address is remembered together with that context: after
// cudaDeviceReset (or any new primary context) the array may sit elsewhere,
// and the next call looks it up again instead of using a stale address.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};
CUcontext g_ctx[kMaxDevices] = {};

using CtxGetCurrent = CUresult (*)(CUcontext *);

// The current context, through the driver entry point the runtime hands out
// (no link against the driver library).
cudaError_t current_context(CUcontext *ctx)
{
    static CtxGetCurrent fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !p) return cudaErrorNotSupported;
        fn = reinterpret_cast<CtxGetCurrent>(p);
    }
    return fn(ctx) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GPT2_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GPT2_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    // the first runtime call on a device creates its primary context, so the
    // lookup comes first and the context is read after it
    CUcontext ctx = nullptr;
    if (g_addr[dev]) {
        e = current_context(&ctx);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GPT2_ERR_CUDA;
        }
    }
    if (!g_addr[dev] || ctx != g_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_head_scratch);
        if (e == cudaSuccess) e = current_context(&ctx);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return GPT2_ERR_CUDA;
        }
        g_addr[dev] = p;
        g_ctx[dev] = ctx;
    }
    *out = g_addr[dev];
    return GPT2_OK;
}

}  // namespace

extern "C" int gpt2_op_head_argmax_noalloc(const float *x, const float *ln_w, const float *ln_b, float eps,
                                           const float *wte, int32_t vocab, int32_t n_embd, float *logits,
                                           int32_t *dev_token, void *stream)
{
    if (!x || !ln_w || !ln_b || !wte || !logits || !dev_token) return GPT2_ERR_INVALID_ARG;
    if (vocab < 1 || n_embd < 4 || n_embd % 4 || !(eps > 0.f)) return GPT2_ERR_INVALID_ARG;
    if (vocab > GPT2_NOALLOC_MAX_VOCAB) return GPT2_ERR_INVALID_ARG;   // more keys than the scratch holds
    if ((long long)vocab * n_embd > (1ll << 31) - 1) return GPT2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(wte) % 16) return GPT2_ERR_INVALID_ARG;
    void *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != GPT2_OK) return rc;
    cudaError_t e = gemv_init();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GPT2_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemvArgs a;
    std::memset(&a, 0, sizeof a);
    a.W = wte;
    a.in = n_embd;
    a.out = vocab;
    a.eps = eps;
    const int ctas = (vocab + kRowsPerCta - 1) / kRowsPerCta;
    const int grid = gemv_plan(a, kWF32, ctas, 96 * 1024, 4);   // grid <= ctas <= kMaxCtas
    if (grid > kMaxCtas) return GPT2_ERR_INVALID_ARG;
    a.evict_first = 1;
    a.xin = x;
    a.ln_w = ln_w;
    a.ln_b = ln_b;
    a.y = logits;
    a.counter = static_cast<unsigned int *>(scratch);
    a.partials = reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(scratch) + 16);
    a.dev_token = dev_token;
    e = cudaMemsetAsync(a.counter, 0, sizeof(unsigned int), s);   // left over from the last call
    if (e == cudaSuccess) e = launch_gemv(kWF32, kModeHead, a, grid, s, false);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GPT2_ERR_CUDA;
    }
    return GPT2_OK;
}
