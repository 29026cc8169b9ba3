// accept_stream.cu -- the acceptance walk for vocabularies too large to hold on chip.
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
// accept.cu holds the rows of the visited node in the registers of one CTA
// cluster; past that capacity the rows stream from memory on every pass, and
// this file does that. Two kernels:
//   accept_rowstats  streams every logits row the walk may touch once: the
//                    target row of every node, the draft row of every node
//                    with children. Per (row, chunk): max m and
//                    Z = sum 2^((l - m) log2 e).
//   accept_walk      one cluster of CTAs (or one warp for small
//                    vocabularies) per sequence; each CTA owns a slice of the
//                    vocabulary. A prologue gathers every child's p_parent(x),
//                    q_parent(x) and uniform into shared memory, so every
//                    decision is taken (identically, by every thread) from
//                    shared memory. A rejection needs the mass of the new
//                    residual, one pass over the parent's two rows; the CTAs
//                    of the cluster add their slices and exchange the totals
//                    through distributed shared memory. The residual after k
//                    rejections is kept in closed form, p~ = max(0, p - c q)/S
//                    with c_0 = 0, S_0 = 1, c_{k+1} = c_k + S_k and
//                    S_{k+1} = sum_v max(0, p_v - c_{k+1} q_v): subtracting q
//                    from max(0, p - c q)/S and renormalising gives exactly
//                    that form. The bonus token is an inverse-CDF search: the
//                    cluster's slice totals, then 128-element group sums of
//                    the crossing slice, then the crossing inside one group.
// Element probabilities are 2^(l log2 e - m log2 e) / Z: one FFMA and one
// ex2.approx per element. Group sums are fp32; prefixes over groups, slices
// and residual masses are fp64.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace svf {

namespace accs {
constexpr int kSmallV = 2048;      // at or below: one warp per row / per sequence
constexpr int kCluster = 8;        // CTAs per sequence above that
constexpr int kWalkThreads = 512;  // threads per walk CTA above that
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace acc

// 2^(l log2 e - ml2) with ml2 = m log2 e: e^(l - m) in one FFMA and one MUFU op.
__device__ __forceinline__ float se2(float l, float ml2) {
    return ex2_approx(fmaf(l, accs::kLog2e, -ml2));
}

// Online (max, sum 2^((x - max) log2 e)) pair merge.
__device__ __forceinline__ void sms_merge(float &m, float &s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    if (m2 > m) {
        s = fmaf(s, ex2_approx((m - m2) * accs::kLog2e), s2);
        m = m2;
    } else {
        s = fmaf(s2, ex2_approx((m2 - m) * accs::kLog2e), s);
    }
}

__device__ __forceinline__ void sms_add4(float &m, float &s, float4 x) {
    const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (mx > m) {
        s = (m == -INFINITY) ? 0.0f : s * ex2_approx((m - mx) * accs::kLog2e);
        m = mx;
    }
    const float ml2 = m * accs::kLog2e;
    s += (se2(x.x, ml2) + se2(x.y, ml2)) + (se2(x.z, ml2) + se2(x.w, ml2));
}

__device__ __forceinline__ void sms_add(float &m, float &s, float x) {
    sms_add4(m, s, make_float4(x, -INFINITY, -INFINITY, -INFINITY));
}

// Does node j of sequence b have a child?  (parent[] in global memory)
__device__ __forceinline__ bool stream_has_child(const int32_t *par, int N, int j, int lane,
                                               int width) {
    int hit = 0;
    for (int c = j + 1 + lane; c < N; c += width) hit |= (par[c] == j);
    return hit != 0;
}

// Row statistics. One warp per row (small V) or one block per chunk of a row
// (large V; a row splits into `nchunks` chunks of `chunk` elements so that
// small batches still fill the GPU). part[kind][row][chunk] = (m, Z) over
// that chunk; kind 0 = target, 1 = draft (rows of leaves are skipped).
template <bool WARP_PER_ROW>
__global__ void __launch_bounds__(256) accept_rowstats_kernel(const float *__restrict__ target,
                                                              const float *__restrict__ draft,
                                                              const int32_t *__restrict__ parent,
                                                              int B, int N, int V, int nchunks,
                                                              int chunk,
                                                              float2 *__restrict__ part) {
    const int kind = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long rows = (long long)B * N;
    long long r;
    int tid, width, c = 0, beg = 0, end = V;
    if (WARP_PER_ROW) {
        r = (long long)blockIdx.x * 8 + warp;
        tid = lane;
        width = 32;
        if (r >= rows) return;
    } else {
        r = blockIdx.x / nchunks;
        c = blockIdx.x % nchunks;
        beg = c * chunk;
        end = min(V, beg + chunk);
        tid = threadIdx.x;
        width = blockDim.x;
    }
    const int b = (int)(r / N), j = (int)(r % N);
    if (kind == 1) {
        bool hc;
        if (WARP_PER_ROW) {
            hc = __any_sync(0xffffffffu, stream_has_child(parent + (size_t)b * N, N, j, lane, 32));
        } else {
            hc = __syncthreads_or(stream_has_child(parent + (size_t)b * N, N, j, tid, width));
        }
        if (!hc) return;
    }
    const float *row = (kind == 0 ? target : draft) + (size_t)r * V;
    float m = -INFINITY, s = 0.0f;
    if ((V & 3) == 0) {
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        const int e4 = end >> 2;
        int i = (beg >> 2) + tid;
        for (; i + 3 * width < e4; i += 4 * width) {
            const float4 a0 = __ldg(row4 + i);
            const float4 a1 = __ldg(row4 + i + width);
            const float4 a2 = __ldg(row4 + i + 2 * width);
            const float4 a3 = __ldg(row4 + i + 3 * width);
            sms_add4(m, s, a0);
            sms_add4(m, s, a1);
            sms_add4(m, s, a2);
            sms_add4(m, s, a3);
        }
        for (; i < e4; i += width) sms_add4(m, s, __ldg(row4 + i));
    } else {
        for (int i = beg + tid; i < end; i += width) sms_add(m, s, __ldg(row + i));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        sms_merge(m, s, m2, s2);
    }
    float2 *dst = part + ((size_t)kind * rows + r) * nchunks + c;
    if (WARP_PER_ROW) {
        if (lane == 0) *dst = make_float2(m, s);
        return;
    }
    __shared__ float sm[32], ss[32];
    if (lane == 0) {
        sm[warp] = m;
        ss[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        m = lane < nw ? sm[lane] : -INFINITY;
        s = lane < nw ? ss[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            sms_merge(m, s, m2, s2);
        }
        if (lane == 0) *dst = make_float2(m, s);
    }
}

// The residual (or target) distribution at one node, in closed form:
// w_v = max(0, p_v - c q_v), p = softmax(target row), q = softmax(draft row).
struct StreamResidual {
    const float *t;
    const float *d;
    float tl2, zt, dl2, zd;  // m log2 e and Z of each row
    float c;                 // 0: plain target softmax (draft row not read)
    __device__ __forceinline__ float w(float tv, float dv) const {
        const float p = se2(tv, tl2) / zt;
        if (c == 0.0f) return p;
        return fmaxf(0.0f, fmaf(-c, se2(dv, dl2) / zd, p));
    }
};

// Four consecutive elements starting at v0 (zeros past V).
template <bool VEC4>
__device__ __forceinline__ void sload4(const StreamResidual &R, int v0, int V, float *w) {
    if (VEC4) {
        if (v0 < V) {
            const float4 tv = __ldg(reinterpret_cast<const float4 *>(R.t + v0));
            float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (R.c != 0.0f) dv = __ldg(reinterpret_cast<const float4 *>(R.d + v0));
            w[0] = R.w(tv.x, dv.x);
            w[1] = R.w(tv.y, dv.y);
            w[2] = R.w(tv.z, dv.z);
            w[3] = R.w(tv.w, dv.w);
        } else {
            w[0] = w[1] = w[2] = w[3] = 0.0f;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int v = v0 + e;
            w[e] = v < V ? R.w(__ldg(R.t + v), R.c != 0.0f ? __ldg(R.d + v) : 0.0f) : 0.0f;
        }
    }
}

// Group sums over this CTA's slice of groups [g0, g1): G[g - g0] = sum of w
// over elements [128 g, 128 g + 128) in fp32 (lanes add four elements, the
// warp a butterfly). A warp keeps four groups' loads in flight. Returns the
// slice total, added in fp64 in group order (same on every thread).
template <int NT, bool VEC4>
__device__ double stream_slice_sums(const StreamResidual &R, int V, int g0, int g1, float *G, double *sh_d) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ng = g1 - g0;
    __syncthreads();  // earlier readers of G are done
    for (int k0 = warp * 4; k0 < ng; k0 += (NT / 32) * 4) {
        float w[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) sload4<VEC4>(R, (g0 + k0 + k) * 128 + lane * 4, V, w[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float gs = warp_sum(((w[k][0] + w[k][1]) + w[k][2]) + w[k][3]);
            if (lane == 0 && k0 + k < ng) G[k0 + k] = gs;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // lane l adds a contiguous run of groups; the runs are then added in order
        const int per = (ng + 31) / 32;
        double part = 0.0;
        for (int k = 0; k < per; ++k) {
            const int gi = lane * per + k;
            if (gi < ng) part += (double)G[gi];
        }
        double incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) sh_d[0] = incl;
    }
    __syncthreads();
    const double tot = sh_d[0];
    __syncthreads();
    return tot;
}

// Per-sequence shared state of the walk (one copy per CTA).
struct StreamWalkShared {
    double slot[2];  // this CTA's slice total, exchanged (double-buffered by pass parity)
    double scratch;
    int bad;
};

// Sum of the slice totals of the CTAs of this sequence, in rank order. Every
// CTA computes the same fp64 value; *before_me gets the sum over lower ranks
// and per_rank[] every rank's total.
template <int CL>
__device__ double stream_cluster_total(StreamWalkShared &ws, double mine, int pass, double *before_me,
                                double *per_rank) {
    if (CL == 1) {
        *before_me = 0.0;
        per_rank[0] = mine;
        return mine;
    }
    cg::cluster_group cluster = cg::this_cluster();
    const int slot = pass & 1;
    if (threadIdx.x == 0) ws.slot[slot] = mine;
    cluster.sync();
    double total = 0.0, before = 0.0;
    const unsigned me = cluster.block_rank();
    double v[CL];
#pragma unroll
    for (int r = 0; r < CL; ++r) v[r] = *cluster.map_shared_rank(&ws.slot[slot], r);
#pragma unroll
    for (int r = 0; r < CL; ++r) {
        per_rank[r] = v[r];
        if ((unsigned)r < me) before += v[r];
        total += v[r];
    }
    *before_me = before;
    return total;
}

template <int NT, int CL, bool VEC4>
__global__ void __launch_bounds__(NT) accept_stream_walk_kernel(
    const float *__restrict__ target, const float *__restrict__ draft,
    const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
    const float *__restrict__ u_accept, const float *__restrict__ u_bonus, int N, int V,
    const float2 *__restrict__ part, int nchunks, long long rows,
    int32_t *__restrict__ accept_len, int32_t *__restrict__ path,
    int32_t *__restrict__ out_tokens, float *__restrict__ ratio, int32_t *__restrict__ status) {
    extern __shared__ double dyn[];
    const int ngroups = (V + 127) >> 7;
    const int gper = (ngroups + CL - 1) / CL;
    const int rank = CL > 1 ? (int)blockIdx.x % CL : 0;
    const int b = CL > 1 ? (int)blockIdx.y : (int)blockIdx.x;
    const int g0 = min(ngroups, rank * gper), g1 = min(ngroups, g0 + gper);
    float2 *st_t = reinterpret_cast<float2 *>(dyn);          // [N] target (m log2 e, Z)
    float2 *st_d = st_t + N;                                  // [N] draft
    float2 *pq = st_d + N;                                    // [N] p_par(x_c), q_par(x_c)
    float *su = reinterpret_cast<float *>(pq + N);            // [N] u_accept
    int32_t *sp = reinterpret_cast<int32_t *>(su + N);        // [N] parent
    int32_t *stok = sp + N;                                   // [N] tokens
    int32_t *sch = stok + N;                                  // [N] has a child
    float *G = reinterpret_cast<float *>(sch + N);            // [gper] group sums of the slice
    __shared__ StreamWalkShared ws;
    __shared__ double per_rank[accs::kCluster];
    const bool lead = rank == 0;

    const size_t base = (size_t)b * N;
    if (threadIdx.x == 0) ws.bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) sch[i] = 0;
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const int pp = parent[base + i];
        const int tk = tokens[base + i];
        sp[i] = pp;
        stok[i] = tk;
        if (i == 0 ? pp != -1 : (pp < 0 || pp >= i)) bad |= SVF_DEV_BAD_PARENT;
        if (i > 0 && (tk < 0 || tk >= V)) bad |= SVF_DEV_BAD_TOKEN;
        if (lead) {
            path[base + i] = -1;
            out_tokens[base + i] = -1;
            if (ratio) ratio[base + i] = __int_as_float(0x7fc00000);
        }
    }
    for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicOr(&ws.bad, bad);
    __syncthreads();
    bad = ws.bad;
    if (lead && threadIdx.x == 0) {
        status[b] = bad;
        accept_len[b] = 0;
    }
    if (bad) {
        if (CL > 1) cg::this_cluster().sync();
        return;
    }

    // prologue: row statistics of every node, and every child's gathered
    // probabilities under its parent's target and draft softmax
    for (int i = 1 + threadIdx.x; i < N; i += NT) sch[sp[i]] = 1;
    __syncthreads();
    {
        // one warp per row: lanes load chunks in parallel, a butterfly merges
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int j = warp; j < N; j += NT / 32) {
            float mt = -INFINITY, zt = 0.0f, md = -INFINITY, zd = 0.0f;
            const bool internal = sch[j] != 0;
            for (int c = lane; c < nchunks; c += 32) {
                const float2 a = part[(base + j) * nchunks + c];
                sms_merge(mt, zt, a.x, a.y);
                if (internal) {
                    const float2 d = part[(rows + base + j) * nchunks + c];
                    sms_merge(md, zd, d.x, d.y);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, mt, o);
                const float z2 = __shfl_xor_sync(0xffffffffu, zt, o);
                sms_merge(mt, zt, m2, z2);
                const float m3 = __shfl_xor_sync(0xffffffffu, md, o);
                const float z3 = __shfl_xor_sync(0xffffffffu, zd, o);
                sms_merge(md, zd, m3, z3);
            }
            if (lane == 0) {
                st_t[j] = make_float2(mt * accs::kLog2e, zt);
                st_d[j] = internal ? make_float2(md * accs::kLog2e, zd) : make_float2(0.0f, 1.0f);
            }
        }
    }
    __syncthreads();
    for (int c = 1 + threadIdx.x; c < N; c += NT) {
        const int j = sp[c], x = stok[c];
        const float tv = target[(base + j) * V + x];
        const float dv = draft[(base + j) * V + x];
        pq[c] = make_float2(se2(tv, st_t[j].x) / st_t[j].y, se2(dv, st_d[j].x) / st_d[j].y);
        su[c] = u_accept[base + c];
    }
    __syncthreads();

    // walk: every thread of every CTA takes the same decisions
    int cur = 0, len = 0, pass = 0;
    double coef = 0.0, mass = 1.0;
    bool groups_hold_residual = false;
    double slice_before = 0.0;
    if (lead && threadIdx.x == 0) path[base] = 0;
    for (;;) {
        bool moved = false;
        for (int c = cur + 1; c < N; ++c) {
            if (sp[c] != cur) continue;
            const double px = (double)pq[c].x, qx = (double)pq[c].y;
            double r = px - coef * qx;
            r = r > 0.0 ? r : 0.0;
            const bool accepted = (double)su[c] * qx * mass < r;
            if (lead && threadIdx.x == 0 && ratio) ratio[base + c] = (float)(r / (mass * qx));
            if (accepted) {
                ++len;
                if (lead && threadIdx.x == 0) {
                    path[base + len] = c;
                    out_tokens[base + len - 1] = stok[c];
                }
                cur = c;
                coef = 0.0;
                mass = 1.0;
                groups_hold_residual = false;
                moved = true;
                break;
            }
            // rejected: mass of max(0, p - (coef + mass) q) over the vocabulary
            StreamResidual R;
            R.t = target + (base + cur) * V;
            R.d = draft + (base + cur) * V;
            R.tl2 = st_t[cur].x; R.zt = st_t[cur].y; R.dl2 = st_d[cur].x; R.zd = st_d[cur].y;
            R.c = (float)(coef + mass);
            const double mine = stream_slice_sums<NT, VEC4>(R, V, g0, g1, G, &ws.scratch);
            double before;
            const double S = stream_cluster_total<CL>(ws, mine, pass++, &before, per_rank);
            if (S > 0.0) {
                coef = (double)R.c;
                mass = S;
                groups_hold_residual = true;
                slice_before = before;
            } else {
                groups_hold_residual = false;
            }
        }
        if (!moved) break;
    }

    // bonus token at the last node, from its target softmax or its residual
    StreamResidual R;
    R.t = target + (base + cur) * V;
    R.tl2 = st_t[cur].x;
    R.zt = st_t[cur].y;
    R.c = (float)coef;
    R.d = coef != 0.0 ? draft + (base + cur) * V : R.t;
    R.dl2 = coef != 0.0 ? st_d[cur].x : 0.0f;
    R.zd = coef != 0.0 ? st_d[cur].y : 1.0f;
    double total;
    if (groups_hold_residual) {
        total = mass;
    } else {
        const double mine = stream_slice_sums<NT, VEC4>(R, V, g0, g1, G, &ws.scratch);
        total = stream_cluster_total<CL>(ws, mine, pass++, &slice_before, per_rank);
    }
    const double thr = (double)u_bonus[b] * total;
    // the CTA whose slice holds the crossing, else (rounding) the last one with mass
    int owner = -1, last_pos = -1;
    {
        double acc_before = 0.0;
        for (int r2 = 0; r2 < CL; ++r2) {
            const double v = per_rank[r2];
            if (owner < 0 && acc_before + v > thr) owner = r2;
            if (v > 0.0) last_pos = r2;
            acc_before += v;
        }
    }
    const bool crossing = owner >= 0;
    if (!crossing) owner = last_pos;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (owner == rank && warp == 0) {
        const int ng = g1 - g0;
        // group of the crossing: running fp64 sum over the slice's groups
        int gsel = -1;
        double gb = slice_before;
        if (lane == 0) {
            if (crossing) {
                for (int k = 0; k < ng; ++k) {
                    if (gb + (double)G[k] > thr) {
                        gsel = k;
                        break;
                    }
                    gb += (double)G[k];
                }
            }
            if (gsel < 0) {  // no crossing found: last group with mass
                for (int k = ng - 1; k >= 0; --k)
                    if (G[k] > 0.0f) {
                        gsel = k;
                        break;
                    }
                gb = 0.0;
            }
        }
        gsel = __shfl_sync(0xffffffffu, gsel, 0);
        gb = __shfl_sync(0xffffffffu, gb, 0);
        int pick = -1;
        if (gsel >= 0) {
            float w[4];
            sload4<VEC4>(R, (g0 + gsel) * 128 + lane * 4, V, w);
            float a[4];
            a[0] = w[0];
            a[1] = a[0] + w[1];
            a[2] = a[1] + w[2];
            a[3] = a[2] + w[3];
            float incl = a[3];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const double lbase = gb + (double)(incl - a[3]);
            int hit = -1, lastw = -1;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (crossing && hit < 0 && lbase + (double)a[e] > thr) hit = e;
                if (w[e] > 0.0f) lastw = e;
            }
            const unsigned bh = __ballot_sync(0xffffffffu, hit >= 0);
            const unsigned bl = __ballot_sync(0xffffffffu, lastw >= 0);
            if (bh) {
                const int src = __ffs(bh) - 1;
                pick = (g0 + gsel) * 128 + src * 4 + __shfl_sync(0xffffffffu, hit, src);
            } else if (bl) {
                const int src = 31 - __clz(bl);
                pick = (g0 + gsel) * 128 + src * 4 + __shfl_sync(0xffffffffu, lastw, src);
            }
        }
        if (lane == 0) out_tokens[base + len] = pick;
    }
    if (lead && threadIdx.x == 0) accept_len[b] = len;
    if (CL > 1) cg::this_cluster().sync();  // peers may still read this CTA's slots
}

static int stream_stat_chunks(long long rows, int V, int *chunk) {
    if (V <= accs::kSmallV) {
        *chunk = V;
        return 1;
    }
    const long long want = 4LL * num_sms();
    long long n = (want + 2 * rows - 1) / (2 * rows);
    const long long maxn = (V + 4095) / 4096;
    if (n > maxn) n = maxn;
    if (n < 1) n = 1;
    if (n > 64) n = 64;
    int ch = (int)((V + n - 1) / n);
    ch = (ch + 1023) / 1024 * 1024;
    *chunk = ch;
    return (V + ch - 1) / ch;
}

size_t accept_stream_workspace_bytes(int B, int N, int V) {
    int chunk;
    const int n = stream_stat_chunks((long long)B * N, V, &chunk);
    return (size_t)2 * B * N * n * sizeof(float2) + 256;
}

template <int NT, int CL, bool VEC4>
static cudaError_t launch_stream_walk(const float *target, const float *draft, const int32_t *tokens,
                               const int32_t *parent, const float *u_accept,
                               const float *u_bonus, int B, int N, int V, const float2 *part,
                               int nchunks, int32_t *accept_len, int32_t *path,
                               int32_t *out_tokens, float *ratio, int32_t *status,
                               cudaStream_t stream) {
    const int ngroups = (V + 127) >> 7;
    const int gper = (ngroups + CL - 1) / CL;
    const size_t smem = (size_t)N * (3 * sizeof(float2) + sizeof(float) + 3 * sizeof(int32_t)) +
                        (size_t)gper * sizeof(float) + 16;
    auto kern = accept_stream_walk_kernel<NT, CL, VEC4>;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const long long rows = (long long)B * N;
    if (CL == 1) {
        kern<<<B, NT, smem, stream>>>(target, draft, tokens, parent, u_accept, u_bonus, N, V, part,
                                      nchunks, rows, accept_len, path, out_tokens, ratio, status);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, B, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, target, draft, tokens, parent, u_accept, u_bonus, N, V,
                              part, nchunks, rows, accept_len, path, out_tokens, ratio, status);
}

cudaError_t launch_accept_stream(const float *target, const float *draft, const int32_t *tokens,
                          const int32_t *parent, const float *u_accept, const float *u_bonus, int B,
                          int N, int V, int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                          float *ratio, void *workspace, int32_t *status, cudaStream_t stream) {
    float2 *part = reinterpret_cast<float2 *>(
        (reinterpret_cast<uintptr_t>(workspace) + 255) & ~static_cast<uintptr_t>(255));
    const long long rows = (long long)B * N;
    int chunk;
    const int nchunks = stream_stat_chunks(rows, V, &chunk);
    if (V <= accs::kSmallV) {
        dim3 grid((unsigned)((rows + 7) / 8), 2);
        accept_rowstats_kernel<true><<<grid, 256, 0, stream>>>(target, draft, parent, B, N, V, 1,
                                                               V, part);
    } else {
        dim3 grid((unsigned)(rows * nchunks), 2);
        accept_rowstats_kernel<false><<<grid, 256, 0, stream>>>(target, draft, parent, B, N, V,
                                                                nchunks, chunk, part);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const bool vec4 = (V & 3) == 0;
    if (V <= accs::kSmallV) {
        return vec4 ? launch_stream_walk<32, 1, true>(target, draft, tokens, parent, u_accept, u_bonus, B,
                                              N, V, part, nchunks, accept_len, path, out_tokens,
                                              ratio, status, stream)
                    : launch_stream_walk<32, 1, false>(target, draft, tokens, parent, u_accept, u_bonus,
                                               B, N, V, part, nchunks, accept_len, path,
                                               out_tokens, ratio, status, stream);
    }
    constexpr int NT = accs::kWalkThreads, CL = accs::kCluster;
    return vec4 ? launch_stream_walk<NT, CL, true>(target, draft, tokens, parent, u_accept, u_bonus, B, N,
                                           V, part, nchunks, accept_len, path, out_tokens, ratio,
                                           status, stream)
                : launch_stream_walk<NT, CL, false>(target, draft, tokens, parent, u_accept, u_bonus, B,
                                            N, V, part, nchunks, accept_len, path, out_tokens,
                                            ratio, status, stream);
}

}  // namespace svf
