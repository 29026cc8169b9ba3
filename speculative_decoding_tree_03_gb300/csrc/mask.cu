// mask.cu -- ancestor bitmasks of BFS-flattened draft trees.
//
// "EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree Verification 详解, B:
// every node attends to its ancestors and itself, never to siblings or
// cousins. One CTA per sequence holds parent[] in shared memory; each thread
// takes nodes and walks their parent links to the root, setting one bit per
// node passed. The walk is O(depth) per node, and parent[i] < i bounds it.
#include "common.cuh"
#include "internal.h"

namespace svf {

constexpr int kMaxMaskWords = 16;  // N <= 1024

__global__ void __launch_bounds__(1024) tree_mask_kernel(const int32_t *__restrict__ parent,
                                                         int N, int W,
                                                         uint64_t *__restrict__ anc,
                                                         int32_t *__restrict__ depth,
                                                         int32_t *__restrict__ status) {
    extern __shared__ int32_t sp[];
    const int b = blockIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    const int32_t *par = parent + (size_t)b * N;
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const int p = par[i];
        sp[i] = p;
        bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    }
    bad = __syncthreads_or(bad);
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        uint64_t *row = anc + ((size_t)b * N + i) * W;
        uint64_t words[kMaxMaskWords];
#pragma unroll
        for (int w = 0; w < kMaxMaskWords; ++w) words[w] = 0;
        int d = 0;
        if (bad) {
            words[i >> 6] = 1ull << (i & 63);
        } else {
            d = -1;
            for (int a = i; a != -1; a = sp[a]) {
                words[a >> 6] |= 1ull << (a & 63);
                ++d;
            }
        }
        for (int w = 0; w < W; ++w) row[w] = words[w];
        if (depth) depth[(size_t)b * N + i] = d;
    }
    if (threadIdx.x == 0) status[b] = bad ? SVF_DEV_BAD_PARENT : 0;
}

cudaError_t launch_tree_mask(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                             int32_t *status, cudaStream_t stream) {
    const int W = (N + 63) / 64;
    int threads = ((N + 31) / 32) * 32;
    if (threads > 1024) threads = 1024;
    return launch_pdl(tree_mask_kernel, dim3((unsigned)B), dim3((unsigned)threads),
                      N * sizeof(int32_t), stream, 0u, parent, N, W, anc, depth, status);
}

}  // namespace svf
