// api.cu -- extern "C" entry points declared in include/specverify.h.
//
// Host-side argument checks, the per-call status reset, and the choice of
// kernel: fp32 inputs take the CUDA-core attention kernel, bf16 inputs the
// tensor-core kernel. All work is enqueued on the caller's stream.
#include <limits.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool tc_page_size_ok(int ps) {
    return ps == 16 || ps == 32 || ps == 64 || (ps > 0 && ps % 128 == 0);
}

}  // namespace svf

using namespace svf;

extern "C" {

int svf_version(void) { return 100; }

const char *svf_status_string(int code) {
    switch (code) {
        case SVF_OK: return "ok";
        case SVF_ERR_ARG: return "invalid argument";
        case SVF_ERR_UNSUPPORTED: return "unsupported size or dtype";
        case SVF_ERR_LAUNCH: return "CUDA launch or driver call failed";
        case SVF_ERR_WORKSPACE: return "workspace missing or too small";
        case SVF_ERR_SCRATCH_LIMIT: return "request exceeds the fixed 4 MiB scratch of the allocation-free call";
        case SVF_DEV_BAD_PARENT: return "device: parent[] is not a BFS-flattened tree";
        case SVF_DEV_BAD_TOKEN: return "device: draft token outside the vocabulary";
        case SVF_DEV_BAD_PAGE: return "device: page id outside the cache";
        case SVF_DEV_BAD_LENGTH: return "device: sequence length outside its page table";
        case SVF_DEV_TIMEOUT: return "device: an internal wait timed out";
        case SVF_DEV_BAD_PATH: return "device: accepted path is not a root path in BFS order";
        case SVF_DEV_BAD_CLUSTER: return "device: kernel ran without its thread-block cluster";
        default: return "unknown status";
    }
}

int svf_tree_mask_build(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                        int32_t *status, svf_stream_t stream) {
    if (B < 0 || N < 0) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (N < 1 || N > 1024) return SVF_ERR_UNSUPPORTED;
    if (!parent || !anc || !status) return SVF_ERR_ARG;
    cudaError_t e = launch_tree_mask(parent, B, N, anc, depth, status,
                                     reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

size_t svf_tree_verify_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int dtype,
                                           int max_pages, int page_size) {
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages <= 0 ||
        page_size <= 0)
        return 0;
    if (dtype != SVF_BF16 || D != 128) return 0;
    const size_t tc_bytes = attn_tc_workspace_bytes(B, N, Hq, Hkv, max_pages, page_size);
    const size_t sk_bytes = attn_sk_workspace_bytes(B, N, Hq, Hkv);
    return tc_bytes > sk_bytes ? tc_bytes : sk_bytes;
}

static int tree_attn_common(const void *q, const void *k_cache, const void *v_cache,
                            int num_pages, int page_size, const int32_t *page_table,
                            int max_pages, const int32_t *seq_lens, const uint64_t *anc,
                            const int32_t *parent, uint64_t *anc_out, int32_t *depth_out,
                            int32_t *mask_status, int B, int N, int Hq, int Hkv, int D, int dtype,
                            float sm_scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, int32_t *status, svf_stream_t stream) {
    if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || num_pages <= 0 || page_size <= 0 ||
        max_pages <= 0)
        return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || (!anc && !parent) || !out ||
        !status)
        return SVF_ERR_ARG;
    if (N < 1 || N > 64 || Hq % Hkv != 0) return SVF_ERR_UNSUPPORTED;
    if ((long long)num_pages * page_size > INT_MAX) return SVF_ERR_UNSUPPORTED;
    if ((long long)max_pages * page_size > INT_MAX) return SVF_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    AttnArgs a;
    a.q = q; a.k_cache = k_cache; a.v_cache = v_cache;
    a.num_pages = num_pages; a.page_size = page_size;
    a.page_table = page_table; a.max_pages = max_pages;
    a.seq_lens = seq_lens; a.anc = anc;
    a.B = B; a.N = N; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.dtype = dtype;
    a.sm_scale = sm_scale; a.out = out; a.lse = lse; a.status = status;
    if (dtype == SVF_F32) {
        if (D != 64 && D != 128) return SVF_ERR_UNSUPPORTED;
        if (parent) {
            // the CUDA-core path reads the masks from memory: build them first
            if (!anc_out || !mask_status) return SVF_ERR_ARG;
            if (launch_tree_mask(parent, B, N, anc_out, depth_out, mask_status, s) != cudaSuccess)
                return SVF_ERR_LAUNCH;
            a.anc = anc_out;
        }
        if (cudaMemsetAsync(status, 0, sizeof(int32_t) * (size_t)B, s) != cudaSuccess)
            return SVF_ERR_LAUNCH;
        return launch_attn_simt(a, s) == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
    }
    if (dtype != SVF_BF16) return SVF_ERR_UNSUPPORTED;
    if (D != 128 || !tc_page_size_ok(page_size)) return SVF_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return SVF_ERR_ARG;
    a.parent = parent;
    a.anc_out = anc_out;
    a.depth_out = depth_out;
    a.mask_status = mask_status;
    // the kernels store every sequence's status word themselves
    const int which = attn_choose_kernel(a, workspace, workspace_bytes);
    if (which < 0) return SVF_ERR_WORKSPACE;
    if (which == 2) return launch_attn_sk(a, workspace, workspace_bytes, s);
    return launch_attn_tc(a, workspace, workspace_bytes, s);
}

int svf_tree_verify_attn(const void *q, const void *k_cache, const void *v_cache, int num_pages,
                         int page_size, const int32_t *page_table, int max_pages,
                         const int32_t *seq_lens, const uint64_t *anc, int B, int N, int Hq,
                         int Hkv, int D, int dtype, float sm_scale, void *out, float *lse,
                         void *workspace, size_t workspace_bytes, int32_t *status,
                         svf_stream_t stream) {
    if (B > 0 && !anc) return SVF_ERR_ARG;
    return tree_attn_common(q, k_cache, v_cache, num_pages, page_size, page_table, max_pages,
                            seq_lens, anc, nullptr, nullptr, nullptr, nullptr, B, N, Hq, Hkv, D,
                            dtype, sm_scale, out, lse, workspace, workspace_bytes, status, stream);
}

int svf_tree_mask_attn(const int32_t *parent, uint64_t *anc, int32_t *depth,
                       int32_t *mask_status, const void *q, const void *k_cache,
                       const void *v_cache, int num_pages, int page_size,
                       const int32_t *page_table, int max_pages, const int32_t *seq_lens, int B,
                       int N, int Hq, int Hkv, int D, int dtype, float sm_scale, void *out,
                       float *lse, void *workspace, size_t workspace_bytes, int32_t *status,
                       svf_stream_t stream) {
    if (B > 0 && !parent) return SVF_ERR_ARG;
    return tree_attn_common(q, k_cache, v_cache, num_pages, page_size, page_table, max_pages,
                            seq_lens, nullptr, parent, anc, depth, mask_status, B, N, Hq, Hkv, D,
                            dtype, sm_scale, out, lse, workspace, workspace_bytes, status, stream);
}

size_t svf_spec_accept_workspace_size(int B, int N, int V) {
    if (B <= 0 || N <= 0 || V <= 0) return 0;
    return accept_workspace_bytes(B, N, V);
}

int svf_spec_accept(const float *target_logits, const float *draft_logits, const int32_t *tokens,
                    const int32_t *parent, const float *u_accept, const float *u_bonus, int B,
                    int N, int V, int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                    float *ratio, void *workspace, size_t workspace_bytes, int32_t *status,
                    svf_stream_t stream) {
    if (B < 0 || N < 0 || V < 0) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!target_logits || !draft_logits || !tokens || !parent || !u_accept || !u_bonus ||
        !accept_len || !path || !out_tokens || !status)
        return SVF_ERR_ARG;
    if (N < 1 || N > 1024 || V < 1 || !accept_supported(V)) return SVF_ERR_UNSUPPORTED;
    if ((V & 3) == 0 && (!aligned16(target_logits) || !aligned16(draft_logits)))
        return SVF_ERR_ARG;
    const size_t need = accept_workspace_bytes(B, N, V);
    if (need > 0 && (!workspace || workspace_bytes < need)) return SVF_ERR_WORKSPACE;
    cudaError_t e = launch_accept(target_logits, draft_logits, tokens, parent, u_accept, u_bonus,
                                  B, N, V, accept_len, path, out_tokens, ratio, workspace, status,
                                  reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_debug_set_attn_wait_ns(long long ns) {
    attn_tc_set_wait_ns(ns);
    return SVF_OK;
}

int svf_debug_set_attn_splits(int splits) {
    if (splits < 0 || splits > 8) return SVF_ERR_ARG;
    attn_tc_force_splits(splits);
    return SVF_OK;
}

int svf_debug_set_attn_kernel(int which) {
    if (which < 0 || which > 2) return SVF_ERR_ARG;
    attn_set_kernel(which);
    return SVF_OK;
}

int svf_lm_head(const void *hidden, const void *weight, int R, int H, int V, float *logits,
                int32_t *status, svf_stream_t stream) {
    if (R < 0 || H < 0 || V < 0) return SVF_ERR_ARG;
    if (R == 0) return SVF_OK;
    if (!hidden || !weight || !logits) return SVF_ERR_ARG;
    if (!lm_head_supported(R, H, V)) return SVF_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(weight)) return SVF_ERR_ARG;
    return launch_lm_head(hidden, weight, R, H, V, logits, status,
                          reinterpret_cast<cudaStream_t>(stream));
}

int svf_spec_accept_lmhead(const void *hidden, const void *weight, const float *draft_logits,
                           const int32_t *tokens, const int32_t *parent, const float *u_accept,
                           const float *u_bonus, int B, int N, int H, int V,
                           float *target_logits, int32_t *accept_len, int32_t *path,
                           int32_t *out_tokens, float *ratio, int32_t *lm_status,
                           int32_t *status, svf_stream_t stream) {
    if (B < 0 || N < 0 || H < 0 || V < 0) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!hidden || !weight || !draft_logits || !tokens || !parent || !u_accept || !u_bonus ||
        !target_logits || !accept_len || !path || !out_tokens || !status)
        return SVF_ERR_ARG;
    if (N < 1 || N > 1024 || V < 1 || !accept_on_chip(V) ||
        !lm_head_supported(B * N, H, V) || (long long)B * N > (1 << 24))
        return SVF_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(weight)) return SVF_ERR_ARG;
    if ((V & 3) == 0 && (!aligned16(target_logits) || !aligned16(draft_logits)))
        return SVF_ERR_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int rc = launch_lm_head(hidden, weight, B * N, H, V, target_logits, lm_status, s);
    if (rc != SVF_OK) return rc;
    cudaError_t e = launch_accept(target_logits, draft_logits, tokens, parent, u_accept, u_bonus,
                                  B, N, V, accept_len, path, out_tokens, ratio, nullptr, status,
                                  s);
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_spec_accept_bf16(const void *target_logits, const void *draft_logits,
                         const int32_t *tokens, const int32_t *parent, const float *u_accept,
                         const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                         int32_t *path, int32_t *out_tokens, float *ratio, int32_t *status,
                         svf_stream_t stream) {
    if (B < 0 || N < 0 || V < 0) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!target_logits || !draft_logits || !tokens || !parent || !u_accept || !u_bonus ||
        !accept_len || !path || !out_tokens || !status)
        return SVF_ERR_ARG;
    if (N < 1 || N > 1024 || V < 1 || !accept_bf16_supported(V)) return SVF_ERR_UNSUPPORTED;
    if ((V & 3) == 0 && (((uintptr_t)target_logits | (uintptr_t)draft_logits) & 7u) != 0)
        return SVF_ERR_ARG;
    cudaError_t e = launch_accept_bf16(reinterpret_cast<const __nv_bfloat16 *>(target_logits),
                                       reinterpret_cast<const __nv_bfloat16 *>(draft_logits),
                                       tokens, parent, u_accept, u_bonus, B, N, V, accept_len,
                                       path, out_tokens, ratio, status,
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

// Shared checks of the target-only variants; 1 for an empty batch. Rows of
// V % 4 == 0 logits are read four at a time: 16-byte (fp32) or 8-byte (bf16)
// aligned.
static int accept_variant_args(const void *target, size_t elem, const int32_t *tokens,
                               const int32_t *parent, int B, int N, int V,
                               const int32_t *accept_len, const int32_t *path,
                               const int32_t *out_tokens, const int32_t *status) {
    if (B < 0 || N < 0 || V < 0) return SVF_ERR_ARG;
    if (B == 0) return 1;
    if (!target || !tokens || !parent || !accept_len || !path || !out_tokens || !status)
        return SVF_ERR_ARG;
    if (N < 1 || N > 1024 || V < 1 || !accept_target_supported(V)) return SVF_ERR_UNSUPPORTED;
    if ((V & 3) == 0 && ((uintptr_t)target % (4 * elem)) != 0) return SVF_ERR_ARG;
    return SVF_OK;
}

int svf_spec_accept_greedy(const float *target_logits, const int32_t *tokens,
                           const int32_t *parent, int B, int N, int V, int32_t *accept_len,
                           int32_t *path, int32_t *out_tokens, int32_t *status,
                           svf_stream_t stream) {
    const int rc = accept_variant_args(target_logits, sizeof(float), tokens, parent, B, N, V,
                                       accept_len, path, out_tokens, status);
    if (rc != SVF_OK) return rc > 0 ? SVF_OK : rc;
    cudaError_t e = launch_accept_target(true, target_logits, tokens, parent, nullptr, nullptr, B,
                                         N, V, accept_len, path, out_tokens, nullptr, status,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_spec_accept_onehot(const float *target_logits, const int32_t *tokens,
                           const int32_t *parent, const float *u_accept, const float *u_bonus,
                           int B, int N, int V, int32_t *accept_len, int32_t *path,
                           int32_t *out_tokens, float *ratio, int32_t *status,
                           svf_stream_t stream) {
    const int rc = accept_variant_args(target_logits, sizeof(float), tokens, parent, B, N, V,
                                       accept_len, path, out_tokens, status);
    if (rc != SVF_OK) return rc > 0 ? SVF_OK : rc;
    if (!u_accept || !u_bonus) return SVF_ERR_ARG;
    cudaError_t e = launch_accept_target(false, target_logits, tokens, parent, u_accept, u_bonus,
                                         B, N, V, accept_len, path, out_tokens, ratio, status,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_spec_accept_greedy_bf16(const void *target_logits, const int32_t *tokens,
                                const int32_t *parent, int B, int N, int V, int32_t *accept_len,
                                int32_t *path, int32_t *out_tokens, int32_t *status,
                                svf_stream_t stream) {
    const int rc = accept_variant_args(target_logits, sizeof(__nv_bfloat16), tokens, parent, B,
                                       N, V, accept_len, path, out_tokens, status);
    if (rc != SVF_OK) return rc > 0 ? SVF_OK : rc;
    cudaError_t e = launch_accept_target_bf16(
        true, reinterpret_cast<const __nv_bfloat16 *>(target_logits), tokens, parent, nullptr,
        nullptr, B, N, V, accept_len, path, out_tokens, nullptr, status,
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_spec_accept_onehot_bf16(const void *target_logits, const int32_t *tokens,
                                const int32_t *parent, const float *u_accept,
                                const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                                int32_t *path, int32_t *out_tokens, float *ratio,
                                int32_t *status, svf_stream_t stream) {
    const int rc = accept_variant_args(target_logits, sizeof(__nv_bfloat16), tokens, parent, B,
                                       N, V, accept_len, path, out_tokens, status);
    if (rc != SVF_OK) return rc > 0 ? SVF_OK : rc;
    if (!u_accept || !u_bonus) return SVF_ERR_ARG;
    cudaError_t e = launch_accept_target_bf16(
        false, reinterpret_cast<const __nv_bfloat16 *>(target_logits), tokens, parent, u_accept,
        u_bonus, B, N, V, accept_len, path, out_tokens, ratio, status,
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_eagle2_init(const int32_t *root_tokens, int B, int capacity, int32_t *pool_parent,
                    int32_t *pool_depth, int32_t *pool_token, double *pool_value,
                    int32_t *pool_count, svf_stream_t stream) {
    if (B < 0 || capacity < 1) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!root_tokens || !pool_parent || !pool_depth || !pool_token || !pool_value || !pool_count)
        return SVF_ERR_ARG;
    if (capacity > kEagle2MaxPool) return SVF_ERR_UNSUPPORTED;
    cudaError_t e = launch_eagle2_init(root_tokens, B, capacity, pool_parent, pool_depth,
                                       pool_token, pool_value, pool_count,
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_eagle2_expand(const float *draft_rows, int B, int R, int V, int k,
                      const int32_t *frontier, int capacity, int32_t *pool_parent,
                      int32_t *pool_depth, int32_t *pool_token, double *pool_value,
                      int32_t *pool_count, int32_t *next_frontier, int32_t *status,
                      svf_stream_t stream) {
    if (B < 0 || R < 0 || V < 0 || k < 0 || capacity < 1) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!draft_rows || !frontier || !pool_parent || !pool_depth || !pool_token || !pool_value ||
        !pool_count || !next_frontier)
        return SVF_ERR_ARG;
    if (R < 1 || R > 65535 || k < 1 || k > kEagle2MaxK || k > V || V > kEagle2MaxV ||
        capacity > kEagle2MaxPool)
        return SVF_ERR_UNSUPPORTED;
    cudaError_t e = launch_eagle2_expand(draft_rows, B, R, V, k, frontier, capacity, pool_parent,
                                         pool_depth, pool_token, pool_value, pool_count,
                                         next_frontier, status,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_eagle2_finalize(int B, int capacity, const int32_t *pool_parent,
                        const int32_t *pool_depth, const int32_t *pool_token,
                        const double *pool_value, const int32_t *pool_count, int n_nodes,
                        int32_t *parent, int32_t *tokens, double *values, int32_t *cids,
                        int32_t *n_out, svf_stream_t stream) {
    if (B < 0 || capacity < 1 || n_nodes < 0) return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!pool_parent || !pool_depth || !pool_token || !pool_value || !pool_count || !parent ||
        !tokens || !values || !cids || !n_out)
        return SVF_ERR_ARG;
    if (n_nodes < 1 || n_nodes > 1024 || capacity > kEagle2MaxPool) return SVF_ERR_UNSUPPORTED;
    cudaError_t e = launch_eagle2_finalize(B, capacity, pool_parent, pool_depth, pool_token,
                                           pool_value, pool_count, n_nodes, parent, tokens,
                                           values, cids, n_out,
                                           reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_selftest_wait_timeout(int32_t *result, long long deadline_ns, svf_stream_t stream) {
    if (!result || deadline_ns < 1000 || deadline_ns > 1000000000ll) return SVF_ERR_ARG;
    cudaError_t e = launch_selftest_wait(result, (unsigned long long)deadline_ns,
                                         reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

int svf_kv_commit(void *k_cache, void *v_cache, int num_layers, long long layer_stride,
                  int num_pages, int page_size, const int32_t *page_table, int max_pages,
                  const int32_t *seq_lens, const int32_t *path, const int32_t *accept_len, int B,
                  int N, int Hkv, int D, int dtype, int32_t *new_seq_lens, int32_t *freed_pages,
                  int max_free, int32_t *n_freed, int32_t *status, svf_stream_t stream) {
    if (B < 0 || N < 0 || num_layers < 0 || Hkv <= 0 || D <= 0 || num_pages <= 0 ||
        page_size <= 0 || max_pages <= 0 || max_free < 0 || layer_stride < 0)
        return SVF_ERR_ARG;
    if (B == 0) return SVF_OK;
    if (!k_cache || !v_cache || !page_table || !seq_lens || !path || !accept_len ||
        !new_seq_lens || !status || (max_free > 0 && !freed_pages))
        return SVF_ERR_ARG;
    if (N < 1 || N > 1024 || num_layers < 1 || num_layers > 65535) return SVF_ERR_UNSUPPORTED;
    const int elem = dtype == SVF_BF16 ? 2 : dtype == SVF_F32 ? 4 : 0;
    if (elem == 0 || ((long long)Hkv * D * elem) % 16 != 0) return SVF_ERR_UNSUPPORTED;
    if ((long long)num_pages * page_size > INT_MAX || (long long)max_pages * page_size > INT_MAX)
        return SVF_ERR_UNSUPPORTED;
    const long long layer_elems = (long long)num_pages * page_size * Hkv * D;
    if (num_layers > 1 && layer_stride < layer_elems) return SVF_ERR_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || (layer_stride * elem) % 16 != 0)
        return SVF_ERR_ARG;
    KvCommitArgs a;
    a.k_cache = k_cache; a.v_cache = v_cache;
    a.num_layers = num_layers; a.layer_stride = num_layers > 1 ? layer_stride : 0;
    a.num_pages = num_pages; a.page_size = page_size;
    a.page_table = page_table; a.max_pages = max_pages;
    a.seq_lens = seq_lens; a.path = path; a.accept_len = accept_len;
    a.B = B; a.N = N; a.Hkv = Hkv; a.D = D; a.elem_size = elem;
    a.new_seq_lens = new_seq_lens; a.freed_pages = max_free > 0 ? freed_pages : nullptr;
    a.max_free = max_free; a.n_freed = n_freed; a.status = status;
    cudaError_t e = launch_kv_commit(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

}  // extern "C"
