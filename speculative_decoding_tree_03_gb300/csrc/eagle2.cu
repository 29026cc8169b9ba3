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
//   eagle2_rows_kernel      a cluster of CTAs per frontier row: softmax
//                           statistics and the row's top-k tokens in one
//                           pass over V, then the k children written at
//                           fixed pool slots;
//   eagle2_select_kernel    the next frontier, the k best new children;
//   eagle2_finalize_kernel  rerank and BFS numbering, one CTA per sequence.
// The row pass is bound by HBM (R rows of V floats per sequence and round);
// the rest is a few hundred values per sequence, bound by latency.
#include <float.h>
#include <limits.h>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace svf {

namespace e2 {

constexpr int kRowThreads = 512;
constexpr int kSelThreads = 256;
constexpr int kFinThreads = 512;
constexpr int kMaxSlices = 8;          // CTAs per row (a portable cluster)

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

// One cluster of P CTAs per (frontier row r, sequence b), each CTA over a
// contiguous slice of the row. A CTA streams its slice once through a ring of
// shared-memory stages filled by bulk copies (element loads when the rows are
// not 16-byte aligned): every thread keeps a running (max, sum e^(l - max))
// and its own best (logit, id). The k-th best of the CTA's thread bests, T,
// bounds the slice's top-k from below, and only the (at most k) threads whose
// best reaches T can hold a top-k element: they re-read their elements (from
// cache) and post those that reach T into the freed stage memory, for an
// exact rank. Rank 0 of the cluster merges the slices' statistics and top-k
// lists (sent into its shared memory) and writes the children: child i of
// frontier node f gets pool slot count[b] + r k + i. A stage wait that gives
// up marks the row's child slots with token kTimeoutToken.
namespace e2 {

constexpr int kGroups = 4;                          // float4 groups per thread per batch
constexpr int kPerBatch = 4 * kGroups;              // elements per thread per batch
constexpr int kBatchElems = kRowThreads * kPerBatch;  // one stage: 32 KB
constexpr int kStages = 3;
constexpr size_t kRowSmem = (size_t)kStages * kBatchElems * sizeof(float);
constexpr int kCandCap = (int)(kRowSmem / 8);       // (logit, id) pairs in the stages
constexpr int kMaxBatches = 48;                     // KMAX * 16 * kMaxBatches <= kCandCap
constexpr int kTimeoutToken = -2;

// element j of a thread's batch at `base`: group j / 4, lane j % 4
__device__ __forceinline__ int elem_id(int base, int j) {
    return base + ((j >> 2) * kRowThreads + (int)threadIdx.x) * 4 + (j & 3);
}

// A thread's 16 elements of the batch at `base` from global memory; -inf past
// `hi`. VEC: 16-byte loads (the row start and `hi` are multiples of 4).
template <bool VEC>
__device__ __forceinline__ void load_batch(const float *__restrict__ row, int base, int hi,
                                           float (&x)[kPerBatch]) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        const int i = elem_id(base, 4 * g);
        if (VEC) {
            float4 t = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (i < hi) t = __ldg(reinterpret_cast<const float4 *>(row + i));
            x[4 * g] = t.x;
            x[4 * g + 1] = t.y;
            x[4 * g + 2] = t.z;
            x[4 * g + 3] = t.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) x[4 * g + c] = i + c < hi ? __ldg(row + i + c) : -INFINITY;
        }
    }
}

// The same 16 elements from a stage holding the batch at `base`.
__device__ __forceinline__ void load_stage(const float *st, int base, int hi,
                                           float (&x)[kPerBatch]) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
        const int off = (g * kRowThreads + (int)threadIdx.x) * 4;
        float4 t = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (base + off < hi) t = *reinterpret_cast<const float4 *>(st + off);
        x[4 * g] = t.x;
        x[4 * g + 1] = t.y;
        x[4 * g + 2] = t.z;
        x[4 * g + 3] = t.w;
    }
}

// The k best of n <= 32 sorted lists (best first, k entries each, ids
// distinct except INT_MAX fillers), by one warp: lane q holds the head of
// list q, and each round the best head (a shuffle reduction) is taken and
// its list advances. Lane 0 writes the k entries, best first.
template <int KMAX>
__device__ __forceinline__ void merge_lists(const float (*lv)[KMAX], const int (*li)[KMAX], int n,
                                            int k, float *outv, int *outi) {
    const int lane = threadIdx.x & 31;
    int h = 0;
    float hv = lane < n ? lv[lane][0] : -INFINITY;
    int hx = lane < n ? li[lane][0] : INT_MAX;
    const int o0 = n > 16 ? 16 : n > 8 ? 8 : n > 4 ? 4 : n > 2 ? 2 : 1;
    for (int i = 0; i < k; ++i) {
        float bv = hv;
        int bi = hx;
        for (int o = o0; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (before(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            outv[i] = bv;
            outi[i] = bi;
        }
        if (hx == bi && bi != INT_MAX && lane < n) {
            ++h;
            hv = h < k ? lv[lane][h] : -INFINITY;
            hx = h < k ? li[lane][h] : INT_MAX;
        }
    }
}

}  // namespace e2

template <int KMAX, bool VEC>  // KMAX >= k; VEC: bulk copies of 16-byte aligned rows
__global__ void __launch_bounds__(e2::kRowThreads, 2) eagle2_rows_kernel(
    const float *__restrict__ rows, int R, int V, int k, int P,
    const int32_t *__restrict__ frontier, int C, int32_t *__restrict__ parent,
    int32_t *__restrict__ depth, int32_t *__restrict__ token, double *__restrict__ value,
    const int32_t *__restrict__ count) {
    using namespace e2;
    constexpr int NW = kRowThreads / 32;
    static_assert(NW <= 32 && NW * KMAX <= kRowThreads, "one lane of warp 0 per warp");
    static_assert(KMAX * kPerBatch * kMaxBatches <= kCandCap, "candidate bound");
    extern __shared__ __align__(128) unsigned char e2_dyn[];
    float *stage = reinterpret_cast<float *>(e2_dyn);              // [kStages][kBatchElems]
    float *s_cv = reinterpret_cast<float *>(e2_dyn);               // candidates, afterwards
    int *s_ci = reinterpret_cast<int *>(e2_dyn + (size_t)kCandCap * sizeof(float));
    __shared__ __align__(8) uint64_t s_full[kStages];
    __shared__ int s_abort;
    __shared__ float s_rm[kMaxSlices];            // rank 0: the slices' maxima
    __shared__ double s_rz[kMaxSlices];           //   their sums
    __shared__ int s_rbad[kMaxSlices];            //   their wait failures
    __shared__ float s_rv[kMaxSlices][KMAX];      //   their top-k lists
    __shared__ int s_ri[kMaxSlices][KMAX];
    __shared__ float s_m[NW];
    __shared__ double s_z[NW];
    __shared__ double s_Z;
    __shared__ float s_lv[NW][KMAX];              // each warp's best thread bests
    __shared__ int s_li[NW][KMAX];
    __shared__ float s_winv[KMAX];
    __shared__ int s_win[KMAX];
    __shared__ int s_nc;
    __shared__ int s_nsel;
    __shared__ int s_sel[kRowThreads];            // threads holding candidates
    const int r = blockIdx.x / P, rank = blockIdx.x % P, b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // this CTA's slice of the row, a multiple of 32 elements wide
    const int per = ((V + P - 1) / P + 31) & ~31;
    const int lo = rank * per, hi = min(V, lo + per);
    const int nb = hi > lo ? (hi - lo + kBatchElems - 1) / kBatchElems : 0;
    pdl_wait();
    pdl_launch_dependents();
    if (P > 1) cluster_arrive();  // waited on before the first remote store
    const int f = frontier[(size_t)b * R + r];
    if (f < 0 || f >= min(count[b], C)) return;  // an unused frontier slot
    const float *row = rows + ((size_t)b * R + r) * (size_t)V;
    constexpr float kLog2e = 1.4426950408889634f;
    // the parent's value and depth, read early (its slot is older than count)
    const size_t po = (size_t)b * C;
    const double vf = (rank == 0 && threadIdx.x < k) ? value[po + f] : 0.0;
    const int df = (rank == 0 && threadIdx.x < k) ? depth[po + f] : 0;

    auto issue = [&](int c) {  // batch c of the slice into stage c % kStages
        const int start = lo + c * kBatchElems;
        const uint32_t bytes = (uint32_t)min(kBatchElems, hi - start) * 4u;
        uint64_t *bar = &s_full[c % kStages];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load_smem(stage + (size_t)(c % kStages) * kBatchElems, row + start, bytes, bar);
    };
    if (VEC && threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) mbar_init(&s_full[s], 1);
        mbar_fence_init();
        for (int c = 0; c < min(kStages, nb); ++c) issue(c);
    }
    __syncthreads();

    // the one pass over the slice
    float m = -INFINITY, z = 0.0f;
    float bv = -INFINITY;
    int bi = INT_MAX;
    bool bad = false;  // a stage wait gave up (the same in every thread)
    int c = 0;
    for (; c < nb; ++c) {
        const int base = lo + c * kBatchElems;
        float x[kPerBatch];
        if (VEC) {
            if (mbar_wait(&s_full[c % kStages], (uint32_t)(c / kStages) & 1u, &s_abort))
                load_stage(stage + (size_t)(c % kStages) * kBatchElems, base, hi, x);
            else
                bad = true;
            // every thread is done with this stage: refill it
            if (__syncthreads_or(bad)) {
                bad = true;
                break;
            }
            if (threadIdx.x == 0 && c + kStages < nb) issue(c + kStages);
        } else {
            load_batch<false>(row, base, hi, x);
        }
        float bm = fmax3(x[0], x[1], x[2]);
#pragma unroll
        for (int j = 3; j + 1 < kPerBatch; j += 2) bm = fmax3(bm, x[j], x[j + 1]);
        bm = fmaxf(bm, x[kPerBatch - 1]);
        if (bm > m) {  // one rescale per batch
            z = (m == -INFINITY) ? 0.0f : z * ex2_approx((m - bm) * kLog2e);
            m = bm;
        }
        if (m != -INFINITY) {
            const float ml2 = m * kLog2e;
#pragma unroll
            for (int j = 0; j < kPerBatch; ++j) z += ex2_approx(fmaf(x[j], kLog2e, -ml2));
        }
        if (bm > bv || (bm == bv && bi == INT_MAX)) {
            // a new best for this thread: the batch's first element equal to
            // bm (ids grow with j and from batch to batch)
            int bj = -1;
#pragma unroll
            for (int j = kPerBatch - 1; j >= 0; --j)
                if (x[j] == bm && elem_id(base, j) < hi) bj = j;
            if (bj >= 0 && before(bm, elem_id(base, bj), bv, bi)) {
                bv = bm;
                bi = elem_id(base, bj);
            }
        }
    }
    if (VEC && bad && threadIdx.x == 0) {
        // let the copies still in flight land before the memory is reused
        s_abort = 0;
        for (int d = c; d < min(c + kStages, nb); ++d)
            mbar_wait_for(&s_full[d % kStages], (uint32_t)(d / kStages) & 1u, &s_abort,
                          kWaitDeadlineNs);
    }

    // softmax statistics of the slice: (max, sum) over the warp and the CTA
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float zw = (m == -INFINITY) ? 0.0f : z * ex2_approx((m - M) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zw += __shfl_xor_sync(0xffffffffu, zw, o);
    // the warp's thread bests sorted best first (a bitonic sort over lanes)
    float sv = bv;
    int si = bi;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, sv, stride);
            const int oi = __shfl_xor_sync(0xffffffffu, si, stride);
            const bool best_first = (lane & size) == 0;
            const bool low = (lane & stride) == 0;
            const bool take = (best_first == low) ? before(ov, oi, sv, si) : before(sv, si, ov, oi);
            if (take) {
                sv = ov;
                si = oi;
            }
        }
    }
    if (lane == 0) {
        s_m[warp] = M;
        s_z[warp] = (double)zw;
    }
    if (lane < k) {
        s_lv[warp][lane] = sv;
        s_li[warp][lane] = si;
    }
    if (threadIdx.x < k) {
        s_winv[threadIdx.x] = -INFINITY;
        s_win[threadIdx.x] = INT_MAX;
    }
    if (threadIdx.x == 0) s_nc = 0;
    __syncthreads();
    float Mc = -INFINITY;
    for (int w = 0; w < NW; ++w) Mc = fmaxf(Mc, s_m[w]);
    if (warp == 0) {
        // T: the k-th best of the thread bests
        merge_lists<KMAX>(s_lv, s_li, NW, k, s_winv, s_win);
        if (lane == 0) s_nsel = 0;
    } else if (warp == 1) {
        // the slice's normaliser: one lane per warp, fp32 exponentials and an
        // fp64 sum (this part's fp64 pipe is slow, so no fp64 exp)
        double t = (lane < NW && s_m[lane] != -INFINITY)
                       ? s_z[lane] * (double)ex2_approx((s_m[lane] - Mc) * kLog2e)
                       : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) s_Z = t;
    }
    __syncthreads();
    const float tv = s_winv[k - 1];
    const int ti = s_win[k - 1];
    // only the threads whose best reaches T hold candidates; a warp re-reads
    // each such thread's elements (from cache), eight loads per lane at a time
    if (!bad && !before(tv, ti, bv, bi)) s_sel[atomicAdd(&s_nsel, 1)] = (int)threadIdx.x;
    __syncthreads();
    const int nsel = s_nsel;
    const int nel = nb * kPerBatch;  // elements per thread
    for (int q = warp; q < nsel; q += NW) {
        const int t = s_sel[q];
        for (int j0 = 0; j0 < nel; j0 += 8 * 32) {
            float xv[8];
            int xi[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u * 32 + lane;  // element j: batch j / 16, slot j % 16
                const int jj = j % kPerBatch;
                xi[u] = lo + (j / kPerBatch) * kBatchElems +
                        ((jj >> 2) * kRowThreads + t) * 4 + (jj & 3);
                xv[u] = (j < nel && xi[u] < hi) ? __ldg(row + xi[u]) : -INFINITY;
                if (j >= nel) xi[u] = INT_MAX;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (xi[u] < hi && !before(tv, ti, xv[u], xi[u])) {
                    const int slot = atomicAdd(&s_nc, 1);
                    if (slot < kCandCap) {
                        s_cv[slot] = xv[u];
                        s_ci[slot] = xi[u];
                    }
                }
            }
        }
    }
    __syncthreads();
    // the slice's top-k: each candidate's rank among the candidates
    const int nc = min(s_nc, kCandCap);
    if ((int)threadIdx.x >= nc && (int)threadIdx.x < k) {
        s_winv[threadIdx.x] = -INFINITY;
        s_win[threadIdx.x] = INT_MAX;
    }
    for (int e = threadIdx.x; e < nc; e += kRowThreads) {
        const float cv = s_cv[e];
        const int ci = s_ci[e];
        int pos = 0;
        for (int d = 0; d < nc; ++d) pos += before(s_cv[d], s_ci[d], cv, ci) ? 1 : 0;
        if (pos < k) {
            s_winv[pos] = cv;
            s_win[pos] = ci;
        }
    }
    __syncthreads();

    float Mg = Mc;
    bool any_bad = bad;
    if (P > 1) {
        // every slice's (max, sum, failure, top-k) into rank 0's shared memory
        cg::cluster_group cl = cg::this_cluster();
        cluster_wait();  // every CTA of the cluster has started
        if (threadIdx.x == 0) {
            *cl.map_shared_rank(&s_rm[rank], 0) = Mc;
            *cl.map_shared_rank(&s_rz[rank], 0) = s_Z;
            *cl.map_shared_rank(&s_rbad[rank], 0) = bad ? 1 : 0;
        }
        if (threadIdx.x < k) {
            *cl.map_shared_rank(&s_rv[rank][threadIdx.x], 0) = s_winv[threadIdx.x];
            *cl.map_shared_rank(&s_ri[rank][threadIdx.x], 0) = s_win[threadIdx.x];
        }
        cluster_arrive();
        cluster_wait();
        if (rank != 0) return;  // nothing reads this CTA's memory any more
        Mg = -INFINITY;
        for (int q = 0; q < P; ++q) {
            Mg = fmaxf(Mg, s_rm[q]);
            any_bad = any_bad || s_rbad[q] != 0;
        }
        if (warp == 0) {
            merge_lists<KMAX>(s_rv, s_ri, P, k, s_winv, s_win);
        } else if (warp == 1) {
            double t = (lane < P && s_rm[lane] != -INFINITY)
                           ? s_rz[lane] * (double)ex2_approx((s_rm[lane] - Mg) * kLog2e)
                           : 0.0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            if (lane == 0) s_Z = t;
        }
        __syncthreads();
    }

    // children: value = parent value * confidence
    const double Z = s_Z;
    if (threadIdx.x < k) {
        const int i = threadIdx.x;
        const long long slot = (long long)count[b] + (long long)r * k + i;
        if (slot < C && any_bad) {
            token[po + slot] = kTimeoutToken;
        } else if (slot < C && s_win[i] != INT_MAX) {
            const double conf = (double)ex2_approx((s_winv[i] - Mg) * kLog2e) / Z;
            parent[po + slot] = f;
            depth[po + slot] = df + 1;
            token[po + slot] = s_win[i];
            value[po + slot] = vf * conf;
        }
    }
}

// The next frontier: the k best of this round's new nodes by (value desc,
// id asc), -1 padded; then the pool count moves past them. status[b] (when
// given) reports a row of this round whose stage wait gave up.
__global__ void __launch_bounds__(e2::kSelThreads) eagle2_select_kernel(
    int R, int k, const int32_t *__restrict__ frontier, int C, const double *__restrict__ value,
    const int32_t *__restrict__ token, int32_t *__restrict__ count, int32_t *__restrict__ next,
    int32_t *__restrict__ status) {
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
    int timed_out = 0;
    for (int c = first + (int)threadIdx.x; c < last; c += blockDim.x)
        timed_out |= token[(size_t)b * C + c] == e2::kTimeoutToken ? 1 : 0;
    timed_out = __syncthreads_or(timed_out);
    if (threadIdx.x == 0) {
        count[b] = last;
        if (status) status[b] = timed_out ? SVF_DEV_TIMEOUT : 0;
    }
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
    int *lcnt = sidx + C;                              // [C] kept nodes per depth
    int *skept = lcnt + C;                             // [C] kept nodes by rerank rank
    int *kd = skept + C;                               // [C] depth of kept node j
    int *kpn = kd + C;                                 // [C] its parent's new index
    __shared__ int s_kept, s_maxd;
    const int b = blockIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    const size_t o = (size_t)b * C;
    const int cnt = min(pcount[b], C);
    if (threadIdx.x == 0) {
        s_kept = 0;
        s_maxd = 0;
    }
    // a slot that is not a node gets key 0 and depth INT_MAX: it never ranks
    // ahead of a node, so the rank loops need no branch
    for (int c = threadIdx.x; c < cnt; c += blockDim.x) {
        const int pc = pparent[o + c];
        const int dc = pdepth[o + c];
        // parents precede children, so a depth is at most the node's id
        const bool ok = c == 0 || (pc >= 0 && pc < c && dc >= 1 && dc <= c);
        sv[c] = ok ? (unsigned long long)__double_as_longlong(pvalue[o + c]) : 0ull;
        sd[c] = ok ? dc : INT_MAX;
        sp[c] = ok ? pc : 0;
        sidx[c] = -1;
        lcnt[c] = 0;
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
        if (dc < 1 || dc == INT_MAX) continue;  // not a node of the tree
        int rank = 0;
#pragma unroll 8
        for (int d = 1; d < cnt; ++d) {
            const unsigned long long vd = sv[d];
            const int dd = sd[d];
            rank += (int)((vd > vc) | ((vd == vc) & ((dd < dc) | ((dd == dc) & (d < c)))));
        }
        if (rank < n_nodes - 1) {
            sidx[c] = -2;  // kept, not yet numbered
            skept[rank] = c;
            atomicAdd(&s_kept, 1);
            atomicAdd(&lcnt[dc], 1);
            atomicMax(&s_maxd, dc);
        }
    }
    if (threadIdx.x == 0) sidx[0] = 0;
    __syncthreads();
    // BFS numbering, a level at a time: (parent's new index, value desc, id
    // asc). Only the kept nodes are scanned, from flat copies: skept[j] lists
    // them by rerank rank, kd/kv hold their depth and key, kpn the parent's
    // new index for the current level (INT_MAX off the level, so that those
    // never rank ahead). A level's new indices start after all shallower
    // kept nodes (lcnt), and the level is numbered in one pass that reads no
    // index it writes.
    const int nk = s_kept;
    for (int j = threadIdx.x; j < nk; j += blockDim.x) {
        const int c = skept[j];
        kd[j] = sd[c];
        kv[j] = sv[c];
    }
    __syncthreads();
    int base = 1;
    for (int d = 1; d <= s_maxd; ++d) {
        for (int j = threadIdx.x; j < nk; j += blockDim.x)
            kpn[j] = kd[j] == d ? sidx[sp[skept[j]]] : INT_MAX;
        __syncthreads();
        for (int j = threadIdx.x; j < nk; j += blockDim.x) {
            const int pc = kpn[j];
            if (pc == INT_MAX) continue;
            const int c = skept[j];
            const unsigned long long vc = kv[j];
            int rank = 0;
#pragma unroll 4
            for (int q = 0; q < nk; ++q) {
                const int pe = kpn[q];
                const unsigned long long ve = kv[q];
                rank += (int)((pe < pc) | ((pe == pc) & ((ve > vc) | ((ve == vc) & (skept[q] < c)))));
            }
            sidx[c] = base + rank;
        }
        base += lcnt[d];
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
    if (threadIdx.x == 0) n_out[b] = 1 + nk;
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
                                 int32_t *status, cudaStream_t stream) {
    cudaError_t e;
    // CTAs per row: enough to fill the SMs (two CTAs each) when the rows are
    // few, at least one batch each, and enough to keep every thread within
    // kMaxBatches batches (the bound on the candidate list)
    const long long nrows = (long long)R * B;
    const long long slots = 2ll * num_sms();
    int P = nrows >= slots ? 1 : (int)(slots / nrows);
    const int p_elems = (V + e2::kBatchElems - 1) / e2::kBatchElems;
    if (P > p_elems) P = p_elems;
    if (P > e2::kMaxSlices) P = e2::kMaxSlices;
    if (P < 1) P = 1;
    auto slice = [V](int p) { return ((V + p - 1) / p + 31) & ~31; };
    while (P < e2::kMaxSlices && slice(P) > e2::kMaxBatches * e2::kBatchElems) ++P;
    if (slice(P) > e2::kMaxBatches * e2::kBatchElems) return cudaErrorInvalidValue;
    const bool vec = V % 4 == 0 && ((uintptr_t)rows & 15) == 0;
#define SVF_E2ROWS(K_)                                                                          \
    do {                                                                                        \
        auto kern = vec ? eagle2_rows_kernel<K_, true> : eagle2_rows_kernel<K_, false>;         \
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,             \
                                 (int)e2::kRowSmem);                                            \
        if (e != cudaSuccess) return e;                                                         \
        e = launch_pdl(kern, dim3((unsigned)(R * P), (unsigned)B), dim3(e2::kRowThreads),       \
                       e2::kRowSmem, stream, P > 1 ? (unsigned)P : 0u, rows, R, V, k, P,       \
                       frontier, C, parent, depth, token, value, (const int32_t *)count);       \
    } while (0)
    if (k <= 1) SVF_E2ROWS(1);
    else if (k <= 2) SVF_E2ROWS(2);
    else if (k <= 4) SVF_E2ROWS(4);
    else if (k <= 8) SVF_E2ROWS(8);
    else SVF_E2ROWS(16);
#undef SVF_E2ROWS
    if (e != cudaSuccess) return e;
    return launch_pdl(eagle2_select_kernel, dim3((unsigned)B), dim3(e2::kSelThreads), 0, stream,
                      0u, R, k, frontier, C, (const double *)value, (const int32_t *)token, count,
                      next, status);
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
