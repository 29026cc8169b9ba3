// accept.cu -- lossless acceptance walk over a verified draft tree.
//
// "Eagle vs DFlash" (speculative sampling): a draft token x is accepted with
// probability min(1, p(x)/q(x)); on rejection the replacement comes from
// normalize(max(0, p - q)). "EAGLE 演化史", § Tree Verification 详解, C:
// walk from the root, test the children of the current node in order, after a
// rejected child subtract q from the (residual) target distribution and test
// the next sibling; if every child is rejected sample from that residual; the
// accepted path is the longest accepted prefix; the bonus token is drawn at
// the last node.
//
// One kernel, one sequence per CTA cluster (or per CTA for small
// vocabularies). The walk only ever needs the two logits rows of the nodes it
// visits, so those are the only rows it reads: every CTA of the cluster owns
// a fixed slice of the vocabulary and holds its slice of the current node's
// target and draft rows in registers, as 128-element groups (one float4 per
// lane per group). Per visited node:
//   1. load the node's two rows (the draft row only if the node has
//      children) into registers, and ask L2 for the first child's rows;
//   2. softmax statistics: per-thread (max, sum e^(l - max)) pairs, merged
//      over the warp, the CTA and (through distributed shared memory, in rank
//      order) the cluster, so that every CTA holds identical (m, Z) values;
//   3. scale the registers to probabilities p_v and q_v;
//   4. test the children in ascending index order from scalars gathered at
//      kernel start; a rejection needs the mass of the next residual, a
//      register-only pass over the slice plus one cluster exchange.
// The residual after k rejections is kept in closed form,
// p~ = max(0, p - c q)/S with c_0 = 0, S_0 = 1, c_{k+1} = c_k + S_k and
// S_{k+1} = sum_v max(0, p_v - c_{k+1} q_v): subtracting q from
// max(0, p - c q)/S and renormalising gives exactly that form. The bonus token
// is an inverse-CDF search: rank totals, then 128-element group sums of the
// crossing slice, then the crossing inside one group, found by the warp whose
// registers hold it. Group sums are fp32; prefixes over groups, slices and
// residual masses are fp64.
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace svf {

namespace acc {
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCluster = 16;
constexpr int kLargeThreads = 512;  // threads per CTA of the clustered variants
// The wide variant for large batches: 11 warps x 16 slots per lane and row,
// the largest slices the register file holds, so a sequence needs fewer CTAs
// and more clusters are resident at once.
constexpr int kWideThreads = 352;
constexpr int kWideSlots = 16;
}  // namespace acc

// 2^(l log2 e - ml2): e^(l - m) for ml2 = m log2 e, in one FFMA and one MUFU op.
__device__ __forceinline__ float e2(float l, float ml2) {
    return ex2_approx(fmaf(l, acc::kLog2e, -ml2));
}

// Online (max, sum e^(x - max)) pair merge. Symmetric in its two operands, so
// butterfly reductions leave the same value in every lane.
__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    if (m2 > m) {
        s = fmaf(s, ex2_approx((m - m2) * acc::kLog2e), s2);
        m = m2;
    } else {
        s = fmaf(s2, ex2_approx((m2 - m) * acc::kLog2e), s);
    }
}

__device__ __forceinline__ float4 neg_inf4() {
    return make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
}

// This warp's slice of one logits row: group k covers elements
// [128 (g0 + k), 128 (g0 + k) + 128), lane l holds elements 4l .. 4l + 3 of
// it; elements past V read as -inf.
template <int E4, bool VEC>
__device__ __forceinline__ void load_slice(const float *__restrict__ row, int V, int g0, int lane,
                                           float4 (&x)[E4]) {
#pragma unroll
    for (int k = 0; k < E4; ++k) {
        const int v0 = (g0 + k) * 128 + lane * 4;
        if (VEC) {
            x[k] = v0 < V ? __ldg(reinterpret_cast<const float4 *>(row + v0)) : neg_inf4();
        } else {
            x[k].x = v0 + 0 < V ? __ldg(row + v0 + 0) : -INFINITY;
            x[k].y = v0 + 1 < V ? __ldg(row + v0 + 1) : -INFINITY;
            x[k].z = v0 + 2 < V ? __ldg(row + v0 + 2) : -INFINITY;
            x[k].w = v0 + 3 < V ? __ldg(row + v0 + 3) : -INFINITY;
        }
    }
}

// The same slice of a bf16 row (VEC: four bf16, 8 bytes, per load), widened
// exactly to fp32.
template <int E4, bool VEC>
__device__ __forceinline__ void load_slice(const __nv_bfloat16 *__restrict__ row, int V, int g0,
                                           int lane, float4 (&x)[E4]) {
#pragma unroll
    for (int k = 0; k < E4; ++k) {
        const int v0 = (g0 + k) * 128 + lane * 4;
        if (VEC) {
            if (v0 < V) {
                const uint2 u = __ldg(reinterpret_cast<const uint2 *>(row + v0));
                x[k] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                   __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
            } else {
                x[k] = neg_inf4();
            }
        } else {
            x[k].x = v0 + 0 < V ? __bfloat162float(row[v0 + 0]) : -INFINITY;
            x[k].y = v0 + 1 < V ? __bfloat162float(row[v0 + 1]) : -INFINITY;
            x[k].z = v0 + 2 < V ? __bfloat162float(row[v0 + 2]) : -INFINITY;
            x[k].w = v0 + 3 < V ? __bfloat162float(row[v0 + 3]) : -INFINITY;
        }
    }
}

__device__ __forceinline__ float ldg_logit(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldg_logit(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// Replace the logits of a thread's slice by e^(l - m_t), m_t the thread's own
// maximum; returns (m_t, sum). A thread with no element returns (-inf, 0).
template <int E4>
__device__ __forceinline__ float2 exp_in_place(float4 (&x)[E4]) {
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < E4; ++k) m = fmaxf(m, fmaxf(fmaxf(x[k].x, x[k].y), fmaxf(x[k].z, x[k].w)));
    const float ml2 = m == -INFINITY ? 0.0f : m * acc::kLog2e;
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < E4; ++k) {
        x[k].x = e2(x[k].x, ml2);
        x[k].y = e2(x[k].y, ml2);
        x[k].z = e2(x[k].z, ml2);
        x[k].w = e2(x[k].w, ml2);
        s += (x[k].x + x[k].y) + (x[k].z + x[k].w);
    }
    return make_float2(m, s);
}

template <int E4>
__device__ __forceinline__ void scale_in_place(float4 (&x)[E4], float f) {
#pragma unroll
    for (int k = 0; k < E4; ++k) {
        x[k].x *= f;
        x[k].y *= f;
        x[k].z *= f;
        x[k].w *= f;
    }
}

// The current distribution at one element: the target softmax (c = 0) or the
// residual numerator max(0, p - c q).
__device__ __forceinline__ float resid(float p, float q, float c) {
    return c == 0.0f ? p : fmaxf(0.0f, fmaf(-c, q, p));
}

// Double-float: a value hi + lo with |lo| <= ulp(hi) / 2, for residual masses
// and CDF prefixes (about 44 significant bits on the fp32 pipes; this part's
// fp64 units are far slower).
struct DF {
    float hi, lo;
};

__device__ __forceinline__ DF df_add(DF a, DF b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    float e = (a.hi - (s - bb)) + (b.hi - bb);
    e += a.lo + b.lo;
    const float hi = s + e;
    return {hi, e - (hi - s)};
}

__device__ __forceinline__ DF df_mul(DF a, float u) {
    const float p = a.hi * u;
    float e = fmaf(a.hi, u, -p);
    e = fmaf(a.lo, u, e);
    const float hi = p + e;
    return {hi, e - (hi - p)};
}

__device__ __forceinline__ bool df_gt(DF a, DF b) {
    return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ DF df_shfl_up(DF a, int d) {
    return {__shfl_up_sync(0xffffffffu, a.hi, d), __shfl_up_sync(0xffffffffu, a.lo, d)};
}

__device__ __forceinline__ DF df_shfl(DF a, int src) {
    return {__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}

// (max, sum e^(x - max)) of a warp: the maximum first, then every lane
// rescales its own sum once. Butterflies leave the same value in every lane.
__device__ __forceinline__ float2 warp_max_sum(float m, float s) {
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float t = (m == -INFINITY) ? 0.0f : s * ex2_approx((m - M) * acc::kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return make_float2(M, t);
}

// Per-CTA shared state of the walk, next to the per-node arrays.
struct WalkSmem {
    float4 recv[2][acc::kMaxCluster];  // records pushed by every rank, by exchange parity
    uint64_t bar[2];                   // completes when every rank's record has landed
    float4 red[32];                    // per-warp partial statistics
    DF run_incl[32];                   // warp 0: inclusive prefix of its lanes' group runs
    int bad;
    int abort;
    int gsel;                          // bonus search: group picked in this CTA (-1: none)
    int gmode;                         // 1 when gsel holds the crossing, else the last group
    DF gbase;                          // mass before gsel (gmode 1)
};

template <int NT, int E4, bool VEC, bool CLUSTER, typename T>
__global__ void __launch_bounds__(NT, 1) accept_walk_kernel(
    const T *__restrict__ target, const T *__restrict__ draft,
    const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
    const float *__restrict__ u_accept, const float *__restrict__ u_bonus, int N, int V, int CL,
    int32_t *__restrict__ accept_len, int32_t *__restrict__ path,
    int32_t *__restrict__ out_tokens, float *__restrict__ ratio, int32_t *__restrict__ status) {
    constexpr int NW = NT / 32;
    constexpr int NG = NW * E4;          // 128-element groups per CTA
    constexpr int PER = (NG + 31) / 32;  // groups per lane in the CTA prefix
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = CLUSTER ? (int)(blockIdx.x % (unsigned)CL) : 0;
    const long long b = CLUSTER ? (long long)(blockIdx.x / (unsigned)CL) : (long long)blockIdx.x;
    const int ncta = CLUSTER ? CL : 1;
    const size_t base = (size_t)b * N;
    const int g0 = (rank * NW + warp) * E4;  // first group of this warp's slice
    const bool lead = rank == 0;

    extern __shared__ __align__(16) unsigned char dyn[];
    float2 *slx = reinterpret_cast<float2 *>(dyn);      // [N] (target, draft) logit of c's token
    float *su = reinterpret_cast<float *>(slx + N);     // [N] u_accept
    int32_t *sp = reinterpret_cast<int32_t *>(su + N);  // [N] parent
    int32_t *stok = sp + N;                             // [N] token
    int32_t *sfirst = stok + N;                         // [N] first child, -1 for a leaf
    int32_t *snext = sfirst + N;                        // [N] next sibling, -1 for the last
    float *G = reinterpret_cast<float *>(snext + N);    // [NG] group sums of the last pass
    __shared__ WalkSmem ws;

    pdl_wait();
    pdl_launch_dependents();
    // This thread's own tree entry is read first: the set-up waits for it,
    // and loads issued after the root's rows would return behind them.
    const int i0 = threadIdx.x;
    int pp0 = -1, tk0 = 0;
    float ua0 = 0.0f;
    if (i0 < N) {
        pp0 = parent[base + i0];
        tk0 = tokens[base + i0];
        ua0 = u_accept[base + i0];
    }
    // the root's rows go out next: their latency hides behind the set-up
    float4 P[E4], Q[E4];
    load_slice<E4, VEC>(target + base * V, V, g0, lane, P);
    if (N > 1) {
        load_slice<E4, VEC>(draft + base * V, V, g0, lane, Q);
    } else {
#pragma unroll
        for (int k = 0; k < E4; ++k) Q[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // then node i0's token logits at its parent's rows (a parent's draft row
    // is read because it has a child), when both of its indexes are valid; an
    // invalid tree is reported below and nothing else is read. Node i0 keeps
    // the pair in registers until the first test, so these loads overlap the
    // set-up and the root's statistics.
    float2 lx_mine = make_float2(0.0f, 0.0f);
    if (i0 > 0 && i0 < N && pp0 >= 0 && pp0 < i0 && tk0 >= 0 && tk0 < V) {
        const size_t row = (base + pp0) * (size_t)V + tk0;
        lx_mine = make_float2(ldg_logit(target + row), ldg_logit(draft + row));
    }

    // ---- the tree: parents, tokens, uniforms; validity; child lists
    if (threadIdx.x == 0) {
        ws.bad = 0;
        ws.abort = 0;
    }
    for (int i = threadIdx.x; i < N; i += NT) sfirst[i] = INT_MAX;
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const bool mine = i == i0;
        const int pp = mine ? pp0 : parent[base + i];
        const int tk = mine ? tk0 : tokens[base + i];
        sp[i] = pp;
        stok[i] = tk;
        su[i] = mine ? ua0 : u_accept[base + i];
        const bool pok = i == 0 ? pp == -1 : (pp >= 0 && pp < i);
        if (!pok) bad |= SVF_DEV_BAD_PARENT;
        if (i > 0 && (tk < 0 || tk >= V)) bad |= SVF_DEV_BAD_TOKEN;
        if (i > 0 && pok) atomicMin(&sfirst[pp], i);
        if (lead) {
            path[base + i] = -1;
            out_tokens[base + i] = -1;
            if (ratio) ratio[base + i] = __int_as_float(0x7fc00000);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(FULL, bad, o);
    if (lane == 0 && bad) atomicOr(&ws.bad, bad);
    if (CLUSTER && threadIdx.x == 0) {
        mbar_init(&ws.bar[0], 1);
        mbar_init(&ws.bar[1], 1);
        mbar_fence_init();
    }
    __syncthreads();
    bad = ws.bad;
    if (lead && threadIdx.x == 0) {
        status[b] = bad;
        accept_len[b] = 0;
    }
    if (bad) return;  // every CTA of the cluster read the same tree and leaves here
    // peers may push records once every CTA's barriers are initialised
    if (CLUSTER) cluster_arrive();

    // siblings in ascending index order; the token logits of the nodes past
    // the first NT at their parents' rows
    for (int i = threadIdx.x; i < N; i += NT) {
        if (sfirst[i] == INT_MAX) sfirst[i] = -1;
        int nx = -1;
        if (i > 0) {
            const int pp = sp[i];
            for (int c = i + 1; c < N; ++c)
                if (sp[c] == pp) {
                    nx = c;
                    break;
                }
            if (i >= NT) {
                const size_t row = (base + pp) * (size_t)V + stok[i];
                slx[i] = make_float2(ldg_logit(target + row), ldg_logit(draft + row));
            }
        }
        snext[i] = nx;
    }
    // every thread reads the child lists from here on (a root without
    // children is marked -1 just above)
    __syncthreads();
    if (CLUSTER) cluster_wait();

    // One exchange: warp 0 pushes this CTA's record into slot `rank` of every
    // CTA of the cluster and waits (bounded) until every rank's record has
    // landed in its own slots; then the CTA's threads read them locally.
    int ph = 0, last_ph = 0;
    auto exchange = [&](float4 rec) {
        const int s = ph & 1;
        if (warp == 0) {
            if (!CLUSTER) {
                if (lane == 0) ws.recv[s][0] = rec;
            } else {
                if (lane == 0) mbar_arrive_expect_tx(&ws.bar[s], (uint32_t)ncta * 16u);
                if (lane < ncta)
                    st_async_v4(cluster_map(&ws.recv[s][rank], (uint32_t)lane), rec,
                                cluster_map(&ws.bar[s], (uint32_t)lane));
                const bool ok = __all_sync(FULL, mbar_wait_cluster(&ws.bar[s], (ph >> 1) & 1));
                if (lane == 0 && !ok) ws.abort = 1;
            }
        }
        __syncthreads();
        last_ph = ph++;
        return s;
    };
    // Sum of the ranks' masses of one exchange, as a fixed butterfly over the
    // lanes (lane r holds rank r): the same value in every thread of every CTA.
    auto rank_sum = [&](int s) -> DF {
        DF t = lane < ncta ? DF{ws.recv[s][lane].x, ws.recv[s][lane].y} : DF{0.0f, 0.0f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const DF y = {__shfl_xor_sync(FULL, t.hi, o), __shfl_xor_sync(FULL, t.lo, o)};
            t = (lane & o) ? df_add(y, t) : df_add(t, y);
        }
        return t;
    };
    // Mass of max(0, p - c q) (or of p for c = 0) over the vocabulary: group
    // sums into G, this CTA's total over lane runs of PER groups, then the
    // totals of all ranks in rank order.
    auto mass_pass = [&](float c) -> DF {
#pragma unroll
        for (int k = 0; k < E4; ++k) {
            const float w0 = resid(P[k].x, Q[k].x, c), w1 = resid(P[k].y, Q[k].y, c);
            const float w2 = resid(P[k].z, Q[k].z, c), w3 = resid(P[k].w, Q[k].w, c);
            const float gs = warp_sum(((w0 + w1) + w2) + w3);
            if (lane == 0) G[warp * E4 + k] = gs;
        }
        __syncthreads();
        float4 rec = make_float4(0.f, 0.f, 0.f, 0.f);
        if (warp == 0) {
            DF part = {0.0f, 0.0f};
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int gi = lane * PER + i;
                if (gi < NG) part = df_add(part, DF{G[gi], 0.0f});
            }
            DF incl = part;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const DF y = df_shfl_up(incl, o);
                if (lane >= o) incl = df_add(incl, y);
            }
            ws.run_incl[lane] = incl;
            const DF tot = df_shfl(incl, 31);
            rec = make_float4(tot.hi, tot.lo, 0.f, 0.f);
        }
        const int s = exchange(rec);
        return rank_sum(s);
    };

    // ---- the walk: every thread of every CTA takes the same decisions
    int cur = 0, len = 0;
    float coef = 0.0f;
    DF mass = {1.0f, 0.0f};
    bool hold = false;  // G and the last exchange hold the current distribution
    bool aborted = false;
    if (lead && threadIdx.x == 0) path[base] = 0;
    for (;;) {
        const int c1 = sfirst[cur];
        const bool kids = c1 >= 0;
        if (VEC && kids && threadIdx.x == 0) {
            // ask L2 for this CTA's slice of the first child's rows
            const int s0 = rank * NG * 128;
            if (s0 < V) {
                const uint32_t bytes = (uint32_t)min(NG * 128, V - s0) * (uint32_t)sizeof(T);
                prefetch_l2_bulk(target + (base + c1) * V + s0, bytes);
                if (sfirst[c1] >= 0) prefetch_l2_bulk(draft + (base + c1) * V + s0, bytes);
            }
        }
        // softmax statistics of the node's rows, identical in every CTA
        const float2 tp = exp_in_place<E4>(P);
        const float2 tq = kids ? exp_in_place<E4>(Q) : make_float2(-INFINITY, 0.0f);
        const float2 wp = warp_max_sum(tp.x, tp.y);
        const float2 wq = warp_max_sum(tq.x, tq.y);
        if (lane == 0) ws.red[warp] = make_float4(wp.x, wp.y, wq.x, wq.y);
        __syncthreads();
        float4 rec = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        if (warp == 0) {
            const float4 t = lane < NW ? ws.red[lane] : rec;
            const float2 cp = warp_max_sum(t.x, t.y);
            const float2 cq = warp_max_sum(t.z, t.w);
            rec = make_float4(cp.x, cp.y, cq.x, cq.y);
        }
        const int s = exchange(rec);
        if (ws.abort) {
            aborted = true;
            break;
        }
        // lane r of every warp takes rank r's record; the same butterflies
        // run in every CTA, so every CTA gets the same (m, Z)
        const float4 rr = lane < ncta ? ws.recv[s][lane] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        const float2 gp = warp_max_sum(rr.x, rr.y);
        const float2 gq = warp_max_sum(rr.z, rr.w);
        const float mp = gp.x, zp = gp.y, mq = gq.x, zq = gq.y;
        if (cur == 0) {
            if (threadIdx.x > 0 && (int)threadIdx.x < N) slx[threadIdx.x] = lx_mine;  // i < NT above
            __syncthreads();
        }
        // registers -> probabilities: e^(l - m_t) * e^(m_t - m) / Z
        const float apl2 = mp * acc::kLog2e, inv_zp = 1.0f / zp;
        scale_in_place<E4>(P, tp.x == -INFINITY ? 0.0f : e2(tp.x, apl2) * inv_zp);
        float aql2 = 0.0f, inv_zq = 1.0f;
        if (kids) {
            aql2 = mq * acc::kLog2e;
            inv_zq = 1.0f / zq;
            scale_in_place<E4>(Q, tq.x == -INFINITY ? 0.0f : e2(tq.x, aql2) * inv_zq);
        }

        // the children, in ascending index order
        int next = -1;
        for (int c = c1; c >= 0; c = snext[c]) {
            const float2 lx = slx[c];
            const float px = e2(lx.x, apl2) * inv_zp;
            const float qx = e2(lx.y, aql2) * inv_zq;
            const float r = fmaxf(0.0f, fmaf(-coef, qx, px));
            const bool accepted = su[c] * qx * mass.hi < r;
            if (lead && threadIdx.x == 0 && ratio) ratio[base + c] = r / (mass.hi * qx);
            if (accepted) {
                next = c;
                break;
            }
            // rejected: the residual max(0, p - (coef + mass) q) and its mass
            const float cn = df_add(DF{coef, 0.0f}, mass).hi;
            const DF S = mass_pass(cn);
            if (ws.abort) {
                aborted = true;
                break;
            }
            if (S.hi > 0.0f) {
                coef = cn;
                mass = S;
                hold = true;
            } else {
                hold = false;  // no mass: the distribution stays as it was
            }
        }
        if (aborted || next < 0) break;
        ++len;
        if (lead && threadIdx.x == 0) {
            path[base + len] = next;
            out_tokens[base + len - 1] = stok[next];
        }
        cur = next;
        coef = 0.0f;
        mass = DF{1.0f, 0.0f};
        hold = false;
        load_slice<E4, VEC>(target + (base + cur) * V, V, g0, lane, P);
        if (sfirst[cur] >= 0) load_slice<E4, VEC>(draft + (base + cur) * V, V, g0, lane, Q);
    }

    // ---- bonus token at the last node, from its target softmax or its residual
    DF total = mass;
    if (!aborted && !hold) {
        total = mass_pass(coef);
        aborted = ws.abort != 0;
    }
    if (aborted) {
        // a peer stopped answering: report it. Every wait above is bounded, so
        // every CTA of the cluster reaches the closing barrier.
        if (lead && threadIdx.x == 0) {
            accept_len[b] = len;
            atomicOr(&status[b], SVF_DEV_TIMEOUT);
        }
        if (CLUSTER) {
            cluster_arrive();
            cluster_wait();
        }
        return;
    }
    const int lp = last_ph & 1;
    const DF thr = df_mul(total, u_bonus[b]);
    // the rank whose slice holds the crossing, else (rounding) the last one with mass
    int owner = -1, last_pos = -1;
    DF owner_before = {0.0f, 0.0f};
    {
        const DF v = lane < ncta ? DF{ws.recv[lp][lane].x, ws.recv[lp][lane].y} : DF{0.0f, 0.0f};
        DF incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const DF y = df_shfl_up(incl, o);
            if (lane >= o) incl = df_add(y, incl);
        }
        DF excl = df_shfl_up(incl, 1);
        if (lane == 0) excl = DF{0.0f, 0.0f};
        const unsigned hit = __ballot_sync(FULL, lane < ncta && df_gt(incl, thr));
        const unsigned pos = __ballot_sync(FULL, lane < ncta && v.hi > 0.0f);
        if (hit) {
            owner = __ffs(hit) - 1;
            owner_before = df_shfl(excl, owner);
        }
        if (pos) last_pos = 31 - __clz(pos);
    }
    if (CLUSTER) cluster_arrive();  // no more traffic between the CTAs
    const bool crossing = owner >= 0;
    if (!crossing) owner = last_pos;
    if (owner == rank) {
        if (warp == 0) {
            // the group of the crossing: the first lane run whose prefix passes
            // thr, then that run group by group
            int gsel = -1, mode = 0;
            DF gb = {0.0f, 0.0f};
            if (crossing) {
                const DF incl = ws.run_incl[lane];
                DF excl = df_shfl_up(incl, 1);
                if (lane == 0) excl = DF{0.0f, 0.0f};
                const unsigned hit = __ballot_sync(FULL, df_gt(df_add(owner_before, incl), thr));
                if (hit) {
                    const int l0 = __ffs(hit) - 1;
                    if (lane == l0) {
                        DF run = df_add(owner_before, excl);
                        for (int i = l0 * PER; i < min(NG, (l0 + 1) * PER); ++i) {
                            const DF nx = df_add(run, DF{G[i], 0.0f});
                            if (df_gt(nx, thr)) {
                                gsel = i;
                                break;
                            }
                            run = nx;
                        }
                        gb = run;
                    }
                    gsel = __shfl_sync(FULL, gsel, l0);
                    gb = df_shfl(gb, l0);
                    mode = gsel >= 0 ? 1 : 0;
                }
            }
            if (gsel < 0) {
                // no crossing (rounding): the last group with mass
                int lastg = -1;
                for (int i = min(NG, (lane + 1) * PER) - 1; i >= lane * PER; --i)
                    if (G[i] > 0.0f) {
                        lastg = i;
                        break;
                    }
                const unsigned has = __ballot_sync(FULL, lastg >= 0);
                if (has) gsel = __shfl_sync(FULL, lastg, 31 - __clz(has));
                gb = DF{0.0f, 0.0f};
                mode = 0;
            }
            if (lane == 0) {
                ws.gsel = gsel;
                ws.gbase = gb;
                ws.gmode = mode;
            }
        }
        __syncthreads();
        const int gsel = ws.gsel;
        if (gsel < 0) {
            if (threadIdx.x == 0) out_tokens[base + len] = -1;
        } else if (warp == gsel / E4) {
            const int ks = gsel - warp * E4;
            float4 pp = P[0], qq = Q[0];
#pragma unroll
            for (int k = 1; k < E4; ++k)
                if (k == ks) {
                    pp = P[k];
                    qq = Q[k];
                }
            const bool by_crossing = ws.gmode != 0;
            const float w[4] = {resid(pp.x, qq.x, coef), resid(pp.y, qq.y, coef),
                                resid(pp.z, qq.z, coef), resid(pp.w, qq.w, coef)};
            float a[4];
            a[0] = w[0];
            a[1] = a[0] + w[1];
            a[2] = a[1] + w[2];
            a[3] = a[2] + w[3];
            float incl = a[3];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += y;
            }
            const DF lbase = df_add(ws.gbase, DF{incl - a[3], 0.0f});
            int hit = -1, lastw = -1;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (by_crossing && hit < 0 && df_gt(df_add(lbase, DF{a[e], 0.0f}), thr)) hit = e;
                if (w[e] > 0.0f) lastw = e;
            }
            const unsigned bh = __ballot_sync(FULL, hit >= 0);
            const unsigned bl = __ballot_sync(FULL, lastw >= 0);
            const int v0 = (rank * NG + gsel) * 128;
            int pick = -1;
            if (bh) {
                const int src = __ffs(bh) - 1;
                pick = v0 + src * 4 + __shfl_sync(FULL, hit, src);
            } else if (bl) {
                const int src = 31 - __clz(bl);
                pick = v0 + src * 4 + __shfl_sync(FULL, lastw, src);
            }
            if (lane == 0) out_tokens[base + len] = pick;
        }
    }
    if (lead && threadIdx.x == 0) accept_len[b] = len;
    if (CLUSTER) cluster_wait();
}

// ---------------------------------------------------------------- host side

namespace {

struct WalkCfg {
    int nt, e4, cl;
};

constexpr int kLargeCap = acc::kLargeThreads / 32 * 128;  // elements per CTA per float4 slot
static_assert(kLargeCap * 8 * acc::kMaxCluster == kMaxOnChipVocab,
              "the largest on-chip configuration holds exactly kMaxOnChipVocab elements");

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Threads, float4 slots per lane and CTAs per sequence for a vocabulary of V.
bool walk_config(int B, int V, WalkCfg *cfg) {
    if (V <= 128) *cfg = {32, 1, 1};
    else if (V <= 512) *cfg = {32, 4, 1};
    else if (V <= 1024) *cfg = {128, 2, 1};
    else if (V <= 4096) *cfg = {128, 8, 1};
    else {
        int e4 = 1;
        while (e4 < 8 && ceil_div(V, (long long)kLargeCap * e4) > acc::kMaxCluster) e4 *= 2;
        int cl = ceil_div(V, (long long)kLargeCap * e4);
        if (cl > acc::kMaxCluster) return false;
        // many sequences: fewer, fuller CTAs per sequence
        while (e4 < 8 && (long long)B * cl > num_sms()) {
            e4 *= 2;
            cl = ceil_div(V, (long long)kLargeCap * e4);
        }
        *cfg = {acc::kLargeThreads, e4, cl};
    }
    return true;
}

size_t walk_smem(int N, const WalkCfg &c) {
    return (size_t)N * (sizeof(float2) + sizeof(float) + 4 * sizeof(int32_t)) +
           (size_t)(c.nt / 32) * c.e4 * sizeof(float) + 16;
}

template <int NT, int E4, bool VEC, bool CLUSTER, typename T>
cudaError_t launch_walk(const WalkCfg &c, const T *target, const T *draft,
                        const int32_t *tokens, const int32_t *parent, const float *u_accept,
                        const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                        int32_t *path, int32_t *out_tokens, float *ratio, int32_t *status,
                        cudaStream_t stream) {
    auto kern = accept_walk_kernel<NT, E4, VEC, CLUSTER, T>;
    const size_t smem = walk_smem(N, c);
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (CLUSTER && c.cl > 8) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const unsigned blocks = (unsigned)((long long)B * (CLUSTER ? c.cl : 1));
    return launch_pdl(kern, dim3(blocks), dim3(NT), smem, stream, CLUSTER ? (unsigned)c.cl : 0u,
                      target, draft, tokens, parent, u_accept, u_bonus, N, V, CLUSTER ? c.cl : 1,
                      accept_len, path, out_tokens, ratio, status);
}

template <bool VEC, typename T>
cudaError_t dispatch_walk(const WalkCfg &c, const T *target, const T *draft,
                          const int32_t *tokens, const int32_t *parent, const float *u_accept,
                          const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                          int32_t *path, int32_t *out_tokens, float *ratio, int32_t *status,
                          cudaStream_t stream) {
#define SVF_WALK(NT_, E4_, CL_)                                                                  \
    return launch_walk<NT_, E4_, VEC, CL_, T>(c, target, draft, tokens, parent, u_accept,       \
                                              u_bonus,                                         \
                                           B, N, V, accept_len, path, out_tokens, ratio, status, \
                                           stream)
    if constexpr (sizeof(T) == 4) {
        // More sequences than one wave of the widest 512-thread slices: take
        // the wide variant when its smaller clusters need fewer waves (fp32
        // rows; on bf16 rows it measured slower: 78.6 against 71-74 us on
        // the 70B batch).
        if (c.nt == acc::kLargeThreads && c.e4 == 8 && (long long)B * c.cl > num_sms()) {
            constexpr int cap = acc::kWideThreads / 32 * 128 * acc::kWideSlots;
            WalkCfg w{acc::kWideThreads, acc::kWideSlots, ceil_div(V, (long long)cap)};
            const int r8 = resident_clusters(
                accept_walk_kernel<acc::kLargeThreads, 8, VEC, true, T>, acc::kLargeThreads,
                walk_smem(N, c), c.cl);
            const int rw = resident_clusters(
                accept_walk_kernel<acc::kWideThreads, acc::kWideSlots, VEC, true, T>,
                acc::kWideThreads, walk_smem(N, w), w.cl);
            if (r8 > 0 && rw > 0 && w.cl <= acc::kMaxCluster &&
                ceil_div(B, rw) < ceil_div(B, r8))
                return launch_walk<acc::kWideThreads, acc::kWideSlots, VEC, true, T>(
                    w, target, draft, tokens, parent, u_accept, u_bonus, B, N, V, accept_len,
                    path, out_tokens, ratio, status, stream);
        }
    }
    if (c.nt == 32) {
        if (c.e4 == 1) SVF_WALK(32, 1, false);
        SVF_WALK(32, 4, false);
    }
    if (c.nt == 128) {
        if (c.e4 == 2) SVF_WALK(128, 2, false);
        SVF_WALK(128, 8, false);
    }
    switch (c.e4) {
        case 1: SVF_WALK(acc::kLargeThreads, 1, true);
        case 2: SVF_WALK(acc::kLargeThreads, 2, true);
        case 4: SVF_WALK(acc::kLargeThreads, 4, true);
        default: SVF_WALK(acc::kLargeThreads, 8, true);
    }
#undef SVF_WALK
}

}  // namespace

bool accept_supported(int V) { return V >= 1 && V <= kMaxStreamVocab; }

bool accept_on_chip(int V) {
    WalkCfg c;
    return walk_config(1, V, &c);
}

size_t accept_workspace_bytes(int B, int N, int V) {
    return accept_on_chip(V) ? 0 : accept_stream_workspace_bytes(B, N, V);
}

cudaError_t launch_accept(const float *target, const float *draft, const int32_t *tokens,
                          const int32_t *parent, const float *u_accept, const float *u_bonus, int B,
                          int N, int V, int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                          float *ratio, void *workspace, int32_t *status, cudaStream_t stream) {
    WalkCfg c;
    if (!walk_config(B, V, &c))
        return launch_accept_stream(target, draft, tokens, parent, u_accept, u_bonus, B, N, V,
                                    accept_len, path, out_tokens, ratio, workspace, status,
                                    stream);
    return (V & 3) == 0 ? dispatch_walk<true, float>(c, target, draft, tokens, parent, u_accept,
                                                     u_bonus, B, N, V, accept_len, path,
                                                     out_tokens, ratio, status, stream)
                        : dispatch_walk<false, float>(c, target, draft, tokens, parent, u_accept,
                                                      u_bonus, B, N, V, accept_len, path,
                                                      out_tokens, ratio, status, stream);
}

bool accept_bf16_supported(int V) { return V >= 1 && accept_on_chip(V); }

cudaError_t launch_accept_bf16(const __nv_bfloat16 *target, const __nv_bfloat16 *draft,
                               const int32_t *tokens, const int32_t *parent,
                               const float *u_accept, const float *u_bonus, int B, int N, int V,
                               int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                               float *ratio, int32_t *status, cudaStream_t stream) {
    WalkCfg c;
    if (!walk_config(B, V, &c)) return cudaErrorInvalidValue;
    return (V & 3) == 0
               ? dispatch_walk<true, __nv_bfloat16>(c, target, draft, tokens, parent, u_accept,
                                                    u_bonus, B, N, V, accept_len, path,
                                                    out_tokens, ratio, status, stream)
               : dispatch_walk<false, __nv_bfloat16>(c, target, draft, tokens, parent, u_accept,
                                                     u_bonus, B, N, V, accept_len, path,
                                                     out_tokens, ratio, status, stream);
}

}  // namespace svf
