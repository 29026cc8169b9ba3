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
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace svf {
namespace {

// 4 MiB: room for (rows x chunks) statistics of up to 262,112 (B*N*chunks)
// entries, far beyond the workloads (a 64 x 31-node batch with a 128K
// vocabulary needs 32 KB).
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device. In host code the
// array's name only stands in for the symbol, so the address is asked of the
// runtime once per device and kept.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SVF_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_accept_scratch) != cudaSuccess || ptr == nullptr)
            return SVF_ERR_LAUNCH;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
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
