// eagle2.cu -- EAGLE-2 dynamic draft-tree construction on the device.
//
// "EAGLE 演化史", § E.2: a node's value is the product of the draft
// confidences on its root path, a confidence being the draft softmax
// probability of the node's own token. Expansion grows the tree round by
// round: the k most valuable nodes of the last round are expanded into their
// k most probable draft tokens each. Rerank keeps the N most valuable nodes,
// a connected subtree because values shrink along every path, and the target
// verifies them flattened in BFS order. § E.3 works one expansion step; "The
// EAGLE Family" (EAGLE-2) describes the same expand-then-rerank procedure.
//
// The drafter runs between rounds, so the construction is three calls on a
// per-sequence node pool (creation id = pool index; the root is id 0):
//   eagle2_init_kernel      the root;
//   eagle2_rows_kernel      one CTA per frontier row: softmax statistics and
//                           the row's top-k tokens in one pass over V, then
//                           the k children written at fixed pool slots;
//   eagle2_select_kernel    the next frontier, the k best new children;
//   eagle2_finalize_kernel  rerank and BFS numbering, one CTA per sequence.
// The row pass is bound by HBM (R rows of V floats per sequence and round);
// the rest is a few hundred values per sequence, bound by latency.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

namespace e2 {

constexpr int kRowThreads = 1024;
constexpr int kSelThreads = 256;
constexpr int kFinThreads = 512;

// (logit, id) order of the top-k search: larger logit first, then lower id.
__device__ __forceinline__ bool before(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

}  // namespace e2

__global__ void eagle2_init_kernel(const int32_t *__restrict__ root_tokens, int B, int C,
                                   int32_t *__restrict__ parent, int32_t *__restrict__ depth,
                                   int32_t *__restrict__ token, double *__restrict__ value,
                                   int32_t *__restrict__ count) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const size_t o = (size_t)b * C;
    parent[o] = -1;
    depth[o] = 0;
    token[o] = root_tokens[b];
    value[o] = 1.0;
    count[b] = 1;
}

// One CTA per (frontier row r, sequence b). Child i of frontier node f gets
// pool slot count[b] + r k + i.
template <int KMAX>  // merge list length, KMAX >= k
__global__ void __launch_bounds__(e2::kRowThreads) eagle2_rows_kernel(
    const float *__restrict__ rows, int R, int V, int k, const int32_t *__restrict__ frontier,
    int C, int32_t *__restrict__ parent, int32_t *__restrict__ depth, int32_t *__restrict__ token,
    double *__restrict__ value, const int32_t *__restrict__ count) {
    using namespace e2;
    constexpr int NW = kRowThreads / 32;
    const int r = blockIdx.x, b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ float s_m[NW];
    __shared__ double s_z[NW];
    __shared__ int s_win[KMAX];
    __shared__ float s_winv[KMAX];
    pdl_wait();
    pdl_launch_dependents();
    const int f = frontier[(size_t)b * R + r];
    if (f < 0 || f >= min(count[b], C)) return;  // an unused frontier slot
    const float *row = rows + ((size_t)b * R + r) * (size_t)V;

    // one pass: each thread's running (max, sum e^(l - max)); each warp's
    // top-k, kept sorted (best first) in lanes 0 .. k-1 of (wv, wi). A chunk
    // of 32 elements (one per lane) is compared with the warp's k-th entry and
    // only the lanes that beat it (a ballot) are inserted, one at a time.
    float m = -INFINITY;
    float z = 0.0f;
    float wv = -INFINITY;
    int wi = INT_MAX;
    float tv = -INFINITY;  // the warp's k-th entry, identical in every lane
    int tix = INT_MAX;
    constexpr int kBatch = KMAX >= 16 ? 8 : 16;
    // the loop bound is the warp's first element, so every lane of a warp runs
    // the same iterations (the ballots and shuffles need the whole warp)
    for (int v0 = threadIdx.x; v0 - lane < V; v0 += kBatch * kRowThreads) {
        float lb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + u * kRowThreads;
            lb[u] = v < V ? __ldg(row + v) : -INFINITY;
        }
        // running (max, sum e^(l - max)): one rescale per batch
        float bm = lb[0];
#pragma unroll
        for (int u = 1; u + 1 < kBatch; u += 2) bm = fmax3(bm, lb[u], lb[u + 1]);
        if (kBatch % 2 == 0) bm = fmaxf(bm, lb[kBatch - 1]);
        if (bm > m) {
            z = (m == -INFINITY) ? 0.0f : z * ex2_approx((m - bm) * 1.4426950408889634f);
            m = bm;
        }
        if (m != -INFINITY) {  // (a thread with no element yet keeps z = 0)
            const float ml2 = m * 1.4426950408889634f;
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                z += ex2_approx(fmaf(lb[u], 1.4426950408889634f, -ml2));
        }
        // candidates for the warp's top-k
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + u * kRowThreads;
            const float l = lb[u];
            unsigned mask = __ballot_sync(0xffffffffu, v < V && before(l, v, tv, tix));
            if (!mask) continue;
            while (mask) {
                const int src = __ffs(mask) - 1;
                mask &= mask - 1;
                const float cv = __shfl_sync(0xffffffffu, l, src);
                const int ci = __shfl_sync(0xffffffffu, v, src);
                // position = entries that stay ahead of the candidate
                const int pos = __popc(__ballot_sync(0xffffffffu,
                                                     lane < k && before(wv, wi, cv, ci)));
                const float upv = __shfl_up_sync(0xffffffffu, wv, 1);
                const int upi = __shfl_up_sync(0xffffffffu, wi, 1);
                if (pos < k && lane < k) {
                    if (lane == pos) {
                        wv = cv;
                        wi = ci;
                    } else if (lane > pos) {
                        wv = upv;
                        wi = upi;
                    }
                }
            }
            tv = __shfl_sync(0xffffffffu, wv, k - 1);
            tix = __shfl_sync(0xffffffffu, wi, k - 1);
        }
    }
    // softmax statistics of the row: (max, sum) over the warp and the CTA
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float zw = (m == -INFINITY) ? 0.0f : z * ex2_approx((m - M) * 1.4426950408889634f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zw += __shfl_xor_sync(0xffffffffu, zw, o);
    __shared__ float s_lv[NW][KMAX];
    __shared__ int s_li[NW][KMAX];
    if (lane == 0) {
        s_m[warp] = M;
        s_z[warp] = (double)zw;
    }
    if (lane < k) {
        s_lv[warp][lane] = wv;
        s_li[warp][lane] = wi;
    }
    __syncthreads();
    float Mc = -INFINITY;
    for (int w = 0; w < NW; ++w) Mc = fmaxf(Mc, s_m[w]);
    static_assert(NW == 32, "one lane of warp 0 per warp");
    __shared__ double s_Z;
    if (warp == 0) {
        // the row's normaliser: one lane per warp, fp32 exponentials and an
        // fp64 sum (this part's fp64 pipe is slow, so no fp64 exp)
        double t = s_m[lane] == -INFINITY
                       ? 0.0
                       : s_z[lane] * (double)ex2_approx((s_m[lane] - Mc) * 1.4426950408889634f);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) s_Z = t;
        // the row's top-k: a k-way merge of the warps' sorted lists, lane w
        // holding warp w's list as a shift register (head = element 0)
        float hv[KMAX];
        int hx[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            hv[j] = j < k ? s_lv[lane][j] : -INFINITY;
            hx[j] = j < k ? s_li[lane][j] : INT_MAX;
        }
        for (int i = 0; i < k; ++i) {
            float bv = hv[0];
            int bi = hx[0];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (before(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (lane == 0) {
                s_win[i] = bi;
                s_winv[i] = bv;
            }
            if (hx[0] == bi) {
#pragma unroll
                for (int j = 0; j < KMAX - 1; ++j) {
                    hv[j] = hv[j + 1];
                    hx[j] = hx[j + 1];
                }
                hv[KMAX - 1] = -INFINITY;
                hx[KMAX - 1] = INT_MAX;
            }
        }
    }
    __syncthreads();

    // children: value = parent value * confidence
    const double Z = s_Z;
    if (threadIdx.x < k) {
        const int i = threadIdx.x;
        const long long slot = (long long)count[b] + (long long)r * k + i;
        if (slot < C && s_win[i] != INT_MAX) {
            const size_t o = (size_t)b * C;
            const double conf =
                (double)ex2_approx((s_winv[i] - Mc) * 1.4426950408889634f) / Z;
            parent[o + slot] = f;
            depth[o + slot] = depth[o + f] + 1;
            token[o + slot] = s_win[i];
            value[o + slot] = value[o + f] * conf;
        }
    }
}

// The next frontier: the k best of this round's new nodes by (value desc,
// id asc), -1 padded; then the pool count moves past them.
__global__ void __launch_bounds__(e2::kSelThreads) eagle2_select_kernel(
    int R, int k, const int32_t *__restrict__ frontier, int C, const double *__restrict__ value,
    int32_t *__restrict__ count, int32_t *__restrict__ next) {
    const int b = blockIdx.x;
    __shared__ int s_valid;
    pdl_wait();
    pdl_launch_dependents();
    const int first = min(count[b], C);
    if (threadIdx.x == 0) {
        int nv = 0;
        while (nv < R && frontier[(size_t)b * R + nv] >= 0 && frontier[(size_t)b * R + nv] < first)
            ++nv;
        s_valid = nv;
    }
    for (int i = threadIdx.x; i < k; i += blockDim.x) next[(size_t)b * k + i] = -1;
    __syncthreads();
    const int last = min(C, first + s_valid * k);
    // values are >= 0: their IEEE bit patterns order like the values, and
    // integer compares avoid this part's slow fp64 pipe
    const unsigned long long *pv =
        reinterpret_cast<const unsigned long long *>(value) + (size_t)b * C;
    for (int c = first + (int)threadIdx.x; c < last; c += blockDim.x) {
        const unsigned long long vc = pv[c];
        int rank = 0;
        for (int d = first; d < last; ++d) {
            const unsigned long long vd = pv[d];
            rank += (vd > vc || (vd == vc && d < c)) ? 1 : 0;
        }
        if (rank < k) next[(size_t)b * k + rank] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) count[b] = last;
}

// Rerank and BFS numbering of one sequence's pool.
__global__ void __launch_bounds__(e2::kFinThreads) eagle2_finalize_kernel(
    int C, const int32_t *__restrict__ pparent, const int32_t *__restrict__ pdepth,
    const int32_t *__restrict__ ptoken, const double *__restrict__ pvalue,
    const int32_t *__restrict__ pcount, int n_nodes, int32_t *__restrict__ out_parent,
    int32_t *__restrict__ out_token, double *__restrict__ out_value, int32_t *__restrict__ out_cid,
    int32_t *__restrict__ n_out) {
    extern __shared__ __align__(8) unsigned char dyn[];
    // [C] values as ordered integer keys (values are >= 0; 0 for non-nodes)
    unsigned long long *sv = reinterpret_cast<unsigned long long *>(dyn);
    // the 8-byte arrays first, so every array stays aligned for any C
    unsigned long long *kv = sv + C;                   // [C] key of kept node j
    int *sd = reinterpret_cast<int *>(kv + C);         // [C] depth
    int *sp = sd + C;                                  // [C] parent id
    int *sidx = sp + C;                                // [C] new index, -1 if not kept
    int *snew = sidx + C;                              // [C] new index being computed
    int *skept = snew + C;                             // [C] kept nodes by rerank rank
    int *kd = skept + C;                               // [C] depth of kept node j
    int *kpn = kd + C;                                 // [C] its parent's new index
    __shared__ int s_kept, s_maxd, s_at, s_lvl;
    const int b = blockIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    const size_t o = (size_t)b * C;
    const int cnt = min(pcount[b], C);
    if (threadIdx.x == 0) {
        s_kept = 0;
        s_maxd = 0;
        s_lvl = 0;
    }
    for (int c = threadIdx.x; c < cnt; c += blockDim.x) {
        const int pc = pparent[o + c];
        const bool ok = c == 0 || (pc >= 0 && pc < c);  // parents precede children
        sv[c] = ok ? (unsigned long long)__double_as_longlong(pvalue[o + c]) : 0ull;
        sd[c] = ok ? pdepth[o + c] : -1;
        sp[c] = ok ? pc : 0;
        sidx[c] = -1;
    }
    for (int i = threadIdx.x; i < n_nodes; i += blockDim.x) {
        out_parent[(size_t)b * n_nodes + i] = -1;
        out_token[(size_t)b * n_nodes + i] = -1;
        out_value[(size_t)b * n_nodes + i] = 0.0;
        out_cid[(size_t)b * n_nodes + i] = -1;
    }
    __syncthreads();
    // rerank: rank of every non-root node by (value desc, depth asc, id asc)
    for (int c = 1 + (int)threadIdx.x; c < cnt; c += blockDim.x) {
        const unsigned long long vc = sv[c];
        const int dc = sd[c];
        if (dc < 1) continue;  // not a node of the tree
        int rank = 0;
        for (int d = 1; d < cnt; ++d) {
            const unsigned long long vd = sv[d];
            if (sd[d] < 1) continue;
            rank += (vd > vc || (vd == vc && (sd[d] < dc || (sd[d] == dc && d < c)))) ? 1 : 0;
        }
        if (rank < n_nodes - 1) {
            sidx[c] = -2;  // kept, not yet numbered
            skept[rank] = c;
            atomicAdd(&s_kept, 1);
            atomicMax(&s_maxd, dc);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        sidx[0] = 0;
        s_at = 1;
    }
    __syncthreads();
    // BFS numbering, a level at a time: (parent's new index, value desc, id
    // asc); the ranks of a level are all computed before any is published
    // Only the kept nodes are scanned, from flat per-node copies (independent
    // loads in the inner loop): skept[j] lists them by rerank rank, kd/kv hold
    // their depth and key, kpn the parent's new index for the current level.
    const int nk = s_kept;
    for (int j = threadIdx.x; j < nk; j += blockDim.x) {
        const int c = skept[j];
        kd[j] = sd[c];
        kv[j] = sv[c];
    }
    __syncthreads();
    for (int d = 1; d <= s_maxd; ++d) {
        const int base = s_at;
        for (int j = threadIdx.x; j < nk; j += blockDim.x)
            kpn[j] = kd[j] == d ? sidx[sp[skept[j]]] : -1;
        __syncthreads();
        for (int j = threadIdx.x; j < nk; j += blockDim.x) {
            if (kd[j] != d) continue;
            const int pc = kpn[j], c = skept[j];
            const unsigned long long vc = kv[j];
            int rank = 0;
            for (int q = 0; q < nk; ++q) {
                if (kd[q] != d) continue;
                const int pe = kpn[q];
                const unsigned long long ve = kv[q];
                rank += (pe < pc || (pe == pc && (ve > vc || (ve == vc && skept[q] < c)))) ? 1 : 0;
            }
            snew[j] = base + rank;
        }
        __syncthreads();
        for (int j = threadIdx.x; j < nk; j += blockDim.x) {
            if (kd[j] == d) {
                sidx[skept[j]] = snew[j];
                atomicAdd(&s_lvl, 1);
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            s_at += s_lvl;
            s_lvl = 0;
        }
        __syncthreads();
    }
    // outputs
    for (int c = threadIdx.x; c < cnt; c += blockDim.x) {
        const int ni = sidx[c];
        if (ni < 0 || ni >= n_nodes) continue;
        const size_t q = (size_t)b * n_nodes + ni;
        out_parent[q] = c == 0 ? -1 : sidx[sp[c]];
        out_token[q] = ptoken[o + c];
        out_value[q] = pvalue[o + c];
        out_cid[q] = c;
    }
    if (threadIdx.x == 0) n_out[b] = s_at;
}

// ---------------------------------------------------------------- host side

size_t eagle2_finalize_smem(int C) {
    return (size_t)C * (2 * sizeof(unsigned long long) + 7 * sizeof(int));
}

cudaError_t launch_eagle2_init(const int32_t *root_tokens, int B, int C, int32_t *parent,
                               int32_t *depth, int32_t *token, double *value, int32_t *count,
                               cudaStream_t stream) {
    const unsigned blocks = (unsigned)((B + 127) / 128);
    return launch_pdl(eagle2_init_kernel, dim3(blocks), dim3(128), 0, stream, 0u, root_tokens, B,
                      C, parent, depth, token, value, count);
}

cudaError_t launch_eagle2_expand(const float *rows, int B, int R, int V, int k,
                                 const int32_t *frontier, int C, int32_t *parent, int32_t *depth,
                                 int32_t *token, double *value, int32_t *count, int32_t *next,
                                 cudaStream_t stream) {
    cudaError_t e;
#define SVF_E2ROWS(K_)                                                                          \
    e = launch_pdl(eagle2_rows_kernel<K_>, dim3((unsigned)R, (unsigned)B),                        \
                   dim3(e2::kRowThreads), 0, stream, 0u, rows, R, V, k, frontier, C, parent,      \
                   depth, token, value, (const int32_t *)count)
    if (k <= 1) SVF_E2ROWS(1);
    else if (k <= 2) SVF_E2ROWS(2);
    else if (k <= 4) SVF_E2ROWS(4);
    else if (k <= 8) SVF_E2ROWS(8);
    else SVF_E2ROWS(16);
#undef SVF_E2ROWS
    if (e != cudaSuccess) return e;
    return launch_pdl(eagle2_select_kernel, dim3((unsigned)B), dim3(e2::kSelThreads), 0, stream,
                      0u, R, k, frontier, C, (const double *)value, count, next);
}

cudaError_t launch_eagle2_finalize(int B, int C, const int32_t *parent, const int32_t *depth,
                                   const int32_t *token, const double *value,
                                   const int32_t *count, int n_nodes, int32_t *out_parent,
                                   int32_t *out_token, double *out_value, int32_t *out_cid,
                                   int32_t *n_out, cudaStream_t stream) {
    const size_t smem = eagle2_finalize_smem(C);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(eagle2_finalize_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(eagle2_finalize_kernel, dim3((unsigned)B), dim3(e2::kFinThreads), smem,
                      stream, 0u, C, parent, depth, token, value, count, n_nodes, out_parent,
                      out_token, out_value, out_cid, n_out);
}

}  // namespace svf
