// internal.h -- launchers shared between the kernel files and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <tuple>

#include "specverify.h"

namespace svf {

// Ancestor bitmasks (mask.cu).
cudaError_t launch_tree_mask(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                             int32_t *status, cudaStream_t stream);

// A bounded wait that runs out on purpose (selftest.cu).
cudaError_t launch_selftest_wait(int32_t *result, unsigned long long deadline_ns,
                                 cudaStream_t stream);

// EAGLE-2 tree construction (eagle2.cu).
constexpr int kEagle2MaxK = 16;
constexpr int kEagle2MaxPool = 2048;
constexpr int kEagle2MaxV = 1 << 20;  // draft vocabulary of svf_eagle2_expand
size_t eagle2_finalize_smem(int C);
cudaError_t launch_eagle2_init(const int32_t *root_tokens, int B, int C, int32_t *parent,
                               int32_t *depth, int32_t *token, double *value, int32_t *count,
                               cudaStream_t stream);
cudaError_t launch_eagle2_expand(const float *rows, int B, int R, int V, int k,
                                 const int32_t *frontier, int C, int32_t *parent, int32_t *depth,
                                 int32_t *token, double *value, int32_t *count, int32_t *next,
                                 int32_t *status, cudaStream_t stream);
cudaError_t launch_eagle2_finalize(int B, int C, const int32_t *parent, const int32_t *depth,
                                   const int32_t *token, const double *value,
                                   const int32_t *count, int n_nodes, int32_t *out_parent,
                                   int32_t *out_token, double *out_value, int32_t *out_cid,
                                   int32_t *n_out, cudaStream_t stream);

// The acceptance walk on bf16 logits (accept.cu; on-chip vocabularies only).
bool accept_bf16_supported(int V);
cudaError_t launch_accept_bf16(const __nv_bfloat16 *target, const __nv_bfloat16 *draft,
                               const int32_t *tokens, const int32_t *parent,
                               const float *u_accept, const float *u_bonus, int B, int N, int V,
                               int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                               float *ratio, int32_t *status, cudaStream_t stream);

// Target-only acceptance variants (accept_target.cu): greedy or one-hot q;
// the rows of vocabularies above kMaxOnChipVocab stream from memory
// (accept_target_stream.cu).
bool accept_target_supported(int V);
cudaError_t launch_accept_target(bool greedy, const float *target, const int32_t *tokens,
                                 const int32_t *parent, const float *u_accept,
                                 const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                                 int32_t *path, int32_t *out_tokens, float *ratio,
                                 int32_t *status, cudaStream_t stream);
cudaError_t launch_accept_target_bf16(bool greedy, const __nv_bfloat16 *target,
                                      const int32_t *tokens, const int32_t *parent,
                                      const float *u_accept, const float *u_bonus, int B, int N,
                                      int V, int32_t *accept_len, int32_t *path,
                                      int32_t *out_tokens, float *ratio, int32_t *status,
                                      cudaStream_t stream);
cudaError_t launch_accept_target_stream(bool greedy, const float *target, const int32_t *tokens,
                                        const int32_t *parent, const float *u_accept,
                                        const float *u_bonus, int B, int N, int V,
                                        int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                                        float *ratio, int32_t *status, cudaStream_t stream);
cudaError_t launch_accept_target_stream_bf16(bool greedy, const __nv_bfloat16 *target,
                                             const int32_t *tokens, const int32_t *parent,
                                             const float *u_accept, const float *u_bonus, int B,
                                             int N, int V, int32_t *accept_len, int32_t *path,
                                             int32_t *out_tokens, float *ratio, int32_t *status,
                                             cudaStream_t stream);

// Arguments of one KV commit call (kv_commit.cu).
struct KvCommitArgs {
    void *k_cache;
    void *v_cache;
    int num_layers;
    long long layer_stride;  // elements
    int num_pages;
    int page_size;
    const int32_t *page_table;
    int max_pages;
    const int32_t *seq_lens;
    const int32_t *path;
    const int32_t *accept_len;
    int B, N, Hkv, D, elem_size;
    int32_t *new_seq_lens;
    int32_t *freed_pages;
    int max_free;
    int32_t *n_freed;
    int32_t *status;
};
cudaError_t launch_kv_commit(const KvCommitArgs &a, cudaStream_t stream);

// Arguments of one tree-attention call, shared by both attention kernels.
struct AttnArgs {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    int num_pages, page_size;
    const int32_t *page_table;
    int max_pages;
    const int32_t *seq_lens;
    const uint64_t *anc;
    int B, N, Hq, Hkv, D, dtype;
    float sm_scale;
    void *out;
    float *lse;
    int32_t *status;
    // non-null: the ancestor masks are built from parent[] inside the
    // tensor-core kernel (anc above is then ignored) and written out as
    // svf_tree_mask_build writes them (each output nullable)
    const int32_t *parent = nullptr;
    uint64_t *anc_out = nullptr;
    int32_t *depth_out = nullptr;
    int32_t *mask_status = nullptr;
};

// CUDA-core path for fp32 (and any dtype): one warp per (sequence, node, head) (attn_simt.cu).
cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t stream);

// Tensor-core path for bf16 (attn_tc.cu).
size_t attn_tc_workspace_bytes(int B, int N, int Hq, int Hkv, int max_pages, int page_size);
int attn_tc_splits(int B, int N, int Hq, int Hkv, int max_pages, int page_size);
bool attn_tc_supported(int max_pages, int page_size);
int launch_attn_tc(const AttnArgs &a, void *workspace, size_t ws_bytes, cudaStream_t stream);
// Test hook: the deadline of the tensor-core attention kernel's waits (ns;
// 0 or less restores the default of 2 s).
void attn_tc_set_wait_ns(long long ns);
// Test hook: the chunk count (cluster size) of later calls, 1..8; 0 restores
// the host model's choice. A forced count selects the cluster kernel.
void attn_tc_force_splits(int s);
int attn_tc_forced_splits();
long long attn_tc_wait_ns();

// Persistent tensor-core path for bf16 (attn_sk.cu): one CTA per SM over an
// equal share of all units' tiles; split units merge through the workspace,
// which must be zero-filled before its first use (every call leaves it so).
bool attn_sk_supported(int Hq, int Hkv);
size_t attn_sk_workspace_bytes(int B, int N, int Hq, int Hkv);
int launch_attn_sk(const AttnArgs &a, void *workspace, size_t ws_bytes, cudaStream_t stream);
// Which bf16 kernel runs: 0 the library's choice, 1 the cluster kernel, 2 the
// persistent kernel (test hook).
void attn_set_kernel(int which);
int attn_choose_kernel(const AttnArgs &a, const void *workspace, size_t ws_bytes);

// Acceptance walk (accept.cu): rows of the visited nodes held in the registers
// of one CTA cluster up to kMaxOnChipVocab, streamed from memory beyond that
// (accept_stream.cu, with a statistics pre-pass into the workspace).
constexpr int kMaxOnChipVocab = 262144;
constexpr int kMaxStreamVocab = 786432;
bool accept_supported(int V);
bool accept_on_chip(int V);
size_t accept_workspace_bytes(int B, int N, int V);
cudaError_t launch_accept(const float *target, const float *draft, const int32_t *tokens,
                          const int32_t *parent, const float *u_accept, const float *u_bonus, int B,
                          int N, int V, int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                          float *ratio, void *workspace, int32_t *status, cudaStream_t stream);
size_t accept_stream_workspace_bytes(int B, int N, int V);
cudaError_t launch_accept_stream(const float *target, const float *draft, const int32_t *tokens,
                                 const int32_t *parent, const float *u_accept,
                                 const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                                 int32_t *path, int32_t *out_tokens, float *ratio, void *workspace,
                                 int32_t *status, cudaStream_t stream);

// Target logits from the LM head (lm_head.cu): logits[r][v] = h[r] . W[v],
// bf16 operands, fp32 accumulation on the tensor cores. Returns an svf_status.
bool lm_head_supported(int R, int H, int V);
int launch_lm_head(const void *hidden, const void *weight, int R, int H, int V, float *logits,
                   int32_t *status, cudaStream_t stream);

int num_sms();

// Clusters of `cl` CTAs of `kern` that can be resident at once on the
// current device, from the occupancy calculator (cached); 0 if unknown.
template <typename K>
inline int resident_clusters(K kern, int nt, size_t smem, int cl) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, size_t, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(reinterpret_cast<const void *>(kern), nt, smem, cl, dev);
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    bool ok = true;  // every call below succeeded
    if (cl > 8)
        ok = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
             cudaSuccess;
    if (ok && smem > 48 * 1024)
        ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
             cudaSuccess;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)cl);
        cfg.blockDim = dim3((unsigned)nt);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)cl;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            n = 0;
            ok = false;
        }
    }
    // a failed query is not the caller's error: clear it (only then)
    if (!ok) (void)cudaGetLastError();
    cache[key] = n;
    return n;
}


// Launch with programmatic stream serialization (and a cluster size when
// cluster_x > 0): the kernel may be scheduled while the previous kernel on the stream
// drains; its griddepcontrol.wait orders every global access after it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 0) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// The same with the cluster along y (cluster_y CTAs of consecutive blockIdx.y).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster_y(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, unsigned cluster_y, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_y > 0) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = cluster_y;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

}  // namespace svf
