// accept_noalloc.cu -- svf_spec_accept for callers that cannot hand the
// library any device scratch memory.
//
// Some callers have no way to allocate device memory at the point where they
// run the acceptance step: an inference runtime that hands a plugin only its
// input and output buffers, a serving loop that reserved every byte of HBM
// up front and forbids allocation afterwards, or host code that must not
// risk the implicit synchronisation an allocation can bring. This entry
// point runs the same kernels as svf_spec_accept. Vocabularies up to 262144
// need no scratch; for larger ones the streaming kernels' scratch (the
// per-row, per-chunk softmax statistics) lives in a fixed array that the
// library itself defines in device memory. Every GPU that loads the library
// holds that array until the process exits.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace svf {
namespace {

// 4 MiB: room for (4 MiB - 256) / 16 = 262128 (row, chunk) statistics
// entries of the streaming kernels. None of the five workloads needs any
// (their vocabularies are at most 151936, which the on-chip walk holds); a
// batch of 64 sequences x 31 nodes at the largest streamed vocabulary,
// 786432, needs 32000 bytes.
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
    void *ctx;   // the context the address was looked up in
    void *addr;  // device address of g_accept_scratch there
};
ScratchAddr g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// The current context (the runtime's primary context of the current device
// once it is initialised), or nullptr when the driver entry point is missing.
void *current_context() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    CUcontext c = nullptr;
    if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the array on the current device. In host code the
// array's name only stands in for the symbol, so the address is asked of the
// runtime once per device and context and kept; a new context on the device
// (after cudaDeviceReset, for instance) reloads the module, and the address
// is looked up again.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SVF_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &e = g_scratch[dev];
    void *ctx = current_context();
    if (e.addr == nullptr || ctx == nullptr || e.ctx != ctx) {
        // the lookup also initialises the device's primary context if needed
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_accept_scratch) != cudaSuccess || ptr == nullptr)
            return SVF_ERR_LAUNCH;
        e.ctx = current_context();
        e.addr = ptr;
    }
    *out = e.addr;
    return SVF_OK;
}

}  // namespace
}  // namespace svf

using namespace svf;

extern "C" int svf_spec_accept_noalloc(const float *target_logits, const float *draft_logits,
                                       const int32_t *tokens, const int32_t *parent,
                                       const float *u_accept, const float *u_bonus, int B, int N,
                                       int V, int32_t *accept_len, int32_t *path,
                                       int32_t *out_tokens, float *ratio, int32_t *status,
                                       svf_stream_t stream) {
    if (B < 0 || N < 0 || V < 0) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!target_logits || !draft_logits || !tokens || !parent || !u_accept || !u_bonus ||
        !accept_len || !path || !out_tokens || !status)
        return SVF_ERR_ARG;
    if (N < 1 || N > 1024 || V < 1 || V > 786432) return SVF_ERR_UNSUPPORTED;
    if ((V & 3) == 0 && (((uintptr_t)target_logits | (uintptr_t)draft_logits) & 15u))
        return SVF_ERR_ARG;
    if (accept_workspace_bytes(B, N, V) > kNoAllocScratchBytes) return SVF_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SVF_OK) return rc;
    cudaError_t e = launch_accept(target_logits, draft_logits, tokens, parent, u_accept, u_bonus,
                                  B, N, V, accept_len, path, out_tokens, ratio, scratch, status,
                                  reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}
