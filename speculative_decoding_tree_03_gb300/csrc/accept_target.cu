// accept_target.cu -- acceptance variants that read only target rows.
//
// Greedy (temperature 0). "Eagle vs DFlash", § A fair evaluation protocol:
// greedy speculative decoding must reproduce a target-only run. At
// temperature 0 the target emits the argmax of its row, so the walk accepts
// the first child (ascending index) whose token is the argmax of the current
// node's target row and stops when no child carries it; the bonus token is
// that argmax. Equal maxima resolve to the lowest token id.
//
// One-hot candidates. The speculative sampling rule ("Eagle vs DFlash":
// accept x with probability min(1, p(x)/q(x)), on rejection continue from
// normalize(max(0, p - q))) with q = one-hot(candidate) for every child: the
// form that stays lossless when siblings are a deterministic top-k rather
// than draws from q. A child with token x is accepted iff u < p~(x); a
// rejection removes x's mass from p~. After rejecting the distinct tokens R
// at one node, p~ = p restricted to the other tokens, divided by 1 - p(R), so
// every test is a scalar: p~(x) = p(x) / (1 - p(R)) for x not in R, 0 for x
// in R. The bonus token is the inverse CDF of p~ at u_bonus.
//
// Logits are fp32 or bf16 (widened exactly to fp32 on load); the arithmetic
// is the same for both.
//
// Layout as in accept.cu: one CTA cluster per sequence (one CTA for small
// vocabularies), each CTA owning a fixed slice of the vocabulary and holding
// its slice of the current node's target row in registers as 128-element
// groups (lane l holds elements 4l .. 4l + 3 of each group). Per visited node
// the CTAs merge per-thread (max, argmax) or (max, sum e^(l - max)) records
// over the warp, the CTA and, through distributed shared memory in rank
// order, the cluster, so that every CTA reaches the same decision.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

namespace tgt {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCluster = 16;
constexpr int kClusterThreads = 512;
constexpr int kWideSlots = 16;  // slots per lane for large batches (one row in registers)
constexpr int kSmallThreads = 128;

// Elements past V read as -inf.
template <int E4, bool VEC>
__device__ __forceinline__ void load_row(const float *__restrict__ row, int V, int g0, int lane,
                                         float4 (&x)[E4]) {
#pragma unroll
    for (int k = 0; k < E4; ++k) {
        const long long e0 = 128ll * (g0 + k) + 4 * lane;
        if (VEC && e0 + 3 < V) {
            x[k] = __ldg(reinterpret_cast<const float4 *>(row + e0));
        } else {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = (e0 + i < V) ? __ldg(row + e0 + i) : -INFINITY;
            x[k] = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
}

// The same groups of a bf16 row (VEC: four bf16, 8 bytes, per load), widened
// exactly to fp32.
template <int E4, bool VEC>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *__restrict__ row, int V, int g0,
                                         int lane, float4 (&x)[E4]) {
#pragma unroll
    for (int k = 0; k < E4; ++k) {
        const long long e0 = 128ll * (g0 + k) + 4 * lane;
        if (VEC && e0 + 3 < V) {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(row + e0));
            x[k] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                               __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
        } else {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = (e0 + i < V) ? __bfloat162float(row[e0 + i]) : -INFINITY;
            x[k] = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
}

__device__ __forceinline__ float logit_at(const float *p) { return __ldg(p); }
__device__ __forceinline__ float logit_at(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// (value, index) maximum with ties to the lower index.
__device__ __forceinline__ void amax_merge(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

__device__ __forceinline__ void warp_amax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax_merge(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
}

// (max, sum e^(x - max)) merge.
__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    if (m2 > m) {
        s = s * ex2_approx((m - m2) * kLog2e) + s2;
        m = m2;
    } else {
        s += s2 * ex2_approx((m2 - m) * kLog2e);
    }
}

__device__ __forceinline__ void warp_ms(float &m, float &s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ms_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
}

__device__ __forceinline__ float4 pack_double(double d, float z = 0.0f, float w = 0.0f) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(d);
    return make_float4(__uint_as_float((uint32_t)u), __uint_as_float((uint32_t)(u >> 32)), z, w);
}

__device__ __forceinline__ double unpack_double(const float4 &r) {
    return __longlong_as_double((long long)(((unsigned long long)__float_as_uint(r.y) << 32) |
                                            __float_as_uint(r.x)));
}

struct TargetSmem {
    float4 recv[2][kMaxCluster];  // records of every rank, by exchange parity
    uint64_t bar[2];
    float4 red[32];               // per-warp partials
    double wsum[32];              // per-warp masses (bonus search)
    int bad;
    int abort;
    int pick;                     // bonus: element found in this CTA, -1 if none
    double dtmp[2];               // bonus: threshold, mass before the crossing warp
    int isel[3];                  // bonus: crossing rank, found flag, crossing warp
};

__device__ __forceinline__ void set_comp(float4 &v, int i, float x) {
    if (i == 0) v.x = x;
    else if (i == 1) v.y = x;
    else if (i == 2) v.z = x;
    else v.w = x;
}

}  // namespace tgt

template <int NT, int E4, bool VEC, bool CLUSTER, bool GREEDY, typename T>
__global__ void __launch_bounds__(NT, 1) accept_target_kernel(
    const T *__restrict__ target, const int32_t *__restrict__ tokens,
    const int32_t *__restrict__ parent, const float *__restrict__ u_accept,
    const float *__restrict__ u_bonus, int N, int V, int CL, int32_t *__restrict__ accept_len,
    int32_t *__restrict__ path, int32_t *__restrict__ out_tokens, float *__restrict__ ratio,
    int32_t *__restrict__ status) {
    using namespace tgt;
    constexpr int NW = NT / 32;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = CLUSTER ? (int)(blockIdx.x % (unsigned)CL) : 0;
    const long long b = CLUSTER ? (long long)(blockIdx.x / (unsigned)CL) : (long long)blockIdx.x;
    const int ncta = CLUSTER ? CL : 1;
    const size_t base = (size_t)b * N;
    const int g0 = (rank * NW + warp) * E4;
    const bool lead = rank == 0;

    extern __shared__ __align__(16) unsigned char dyn[];
    float *slx = reinterpret_cast<float *>(dyn);        // [N] target logit of c's token at its parent
    float *su = slx + N;                                // [N] u_accept
    int32_t *sp = reinterpret_cast<int32_t *>(su + N);  // [N] parent
    int32_t *stok = sp + N;                             // [N] token
    int32_t *sfirst = stok + N;                         // [N] first child, -1 for a leaf
    int32_t *snext = sfirst + N;                        // [N] next sibling, -1 for the last
    __shared__ TargetSmem ws;

    pdl_wait();
    pdl_launch_dependents();
    // This thread's own tree entry is read first: the set-up waits for it,
    // and loads issued after the root's row would return behind them.
    const int i0 = threadIdx.x;
    int pp0 = -1, tk0 = 0;
    float ua0 = 0.0f;
    if (i0 < N) {
        pp0 = parent[base + i0];
        tk0 = tokens[base + i0];
        if (!GREEDY) ua0 = u_accept[base + i0];
    }
    float4 P[E4];
    load_row<E4, VEC>(target + base * V, V, g0, lane, P);
    // one-hot: node i0's token logit at its parent's row, when both of its
    // indexes are valid (an invalid tree is reported below)
    float lx0 = 0.0f;
    if (!GREEDY && i0 > 0 && i0 < N && pp0 >= 0 && pp0 < i0 && tk0 >= 0 && tk0 < V)
        lx0 = logit_at(target + (base + pp0) * (size_t)V + tk0);

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
        su[i] = GREEDY ? 0.0f : (mine ? ua0 : u_accept[base + i]);
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
    if (lead && threadIdx.x == 0) path[base] = 0;
    if (CLUSTER) cluster_arrive();
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
            if (!GREEDY)
                slx[i] = i == i0 ? lx0 : logit_at(target + (base + pp) * (size_t)V + stok[i]);
        }
        snext[i] = nx;
    }
    if (CLUSTER) cluster_wait();

    // One exchange: every thread has finished with the previous records; warp
    // 0 pushes this CTA's record into slot `rank` of every CTA of the cluster
    // and waits (bounded) until every rank's record has landed here.
    int ph = 0;
    auto exchange = [&](float4 rec) -> int {
        const int s = ph & 1;
        __syncthreads();
        if (warp == 0) {
            if (!CLUSTER) {
                if (lane == 0) ws.recv[s][0] = rec;
            } else {
                if (lane == 0) mbar_arrive_expect_tx(&ws.bar[s], (uint32_t)ncta * 16u);
                if (lane < ncta)
                    st_async_v4(cluster_map(&ws.recv[s][rank], (uint32_t)lane), rec,
                                cluster_map(&ws.bar[s], (uint32_t)lane));
                const bool okw = __all_sync(FULL, mbar_wait_cluster(&ws.bar[s], (ph >> 1) & 1));
                if (lane == 0 && !okw) ws.abort = 1;
            }
        }
        __syncthreads();
        ++ph;
        return s;
    };

    int cur = 0, len = 0, bonus = -1;
    bool ok = true;
    for (;;) {
        if (GREEDY) {
            // ---- argmax of the node's target row, ties to the lowest id
            float bv = -INFINITY;
            int bi = INT_MAX;
#pragma unroll
            for (int k = 0; k < E4; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float v = comp(P[k], e);
                    if (v > bv) {
                        bv = v;
                        bi = 128 * (g0 + k) + 4 * lane + e;
                    }
                }
            warp_amax(bv, bi);
            if (lane == 0) ws.red[warp] = make_float4(bv, __int_as_float(bi), 0.0f, 0.0f);
            __syncthreads();
            float4 rec = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (warp == 0) {
                float v = lane < NW ? ws.red[lane].x : -INFINITY;
                int i = lane < NW ? __float_as_int(ws.red[lane].y) : INT_MAX;
                warp_amax(v, i);
                rec = make_float4(v, __int_as_float(i), 0.0f, 0.0f);
            }
            const int s = exchange(rec);
            if (ws.abort) {
                ok = false;
                break;
            }
            float v = -INFINITY;
            int a = INT_MAX;
            for (int r = 0; r < ncta; ++r)
                amax_merge(v, a, ws.recv[s][r].x, __float_as_int(ws.recv[s][r].y));
            int nxt = -1;
            for (int c = sfirst[cur]; c != -1; c = snext[c])
                if (stok[c] == a) {
                    nxt = c;
                    break;
                }
            if (nxt < 0) {
                bonus = a;
                break;
            }
            ++len;
            if (lead && threadIdx.x == 0) {
                path[base + len] = nxt;
                out_tokens[base + len - 1] = a;
            }
            cur = nxt;
            load_row<E4, VEC>(target + (base + cur) * V, V, g0, lane, P);
            continue;
        }

        // ---- one-hot candidates: softmax statistics of the node's row
        float mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < E4; ++k)
            mt = fmaxf(fmaxf(fmaxf(mt, P[k].x), fmaxf(P[k].y, P[k].z)), P[k].w);
        float st = 0.0f;
        if (mt != -INFINITY) {
            const float ml2 = mt * kLog2e;
#pragma unroll
            for (int k = 0; k < E4; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) st += ex2_approx(fmaf(comp(P[k], e), kLog2e, -ml2));
        }
        warp_ms(mt, st);
        if (lane == 0) ws.red[warp] = make_float4(mt, st, 0.0f, 0.0f);
        __syncthreads();
        float4 rec = make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
        if (warp == 0) {
            float m = -INFINITY, z = 0.0f;
            for (int w = 0; w < NW; ++w) ms_merge(m, z, ws.red[w].x, ws.red[w].y);
            rec = make_float4(m, z, 0.0f, 0.0f);
        }
        const int s = exchange(rec);
        if (ws.abort) {
            ok = false;
            break;
        }
        float M = -INFINITY, Z = 0.0f;
        for (int r = 0; r < ncta; ++r) ms_merge(M, Z, ws.recv[s][r].x, ws.recv[s][r].y);
        // ---- the children in order: scalar tests against p~ = p / (1 - p(R)),
        // decided by one thread (fp32 exponentials, fp64 mass and division;
        // this part's fp64 pipe is slow, so no fp64 exp)
        if (threadIdx.x == 0) {
            double rej_mass = 0.0;
            int pick = -1;
            for (int c = sfirst[cur]; c != -1; c = snext[c]) {
                const int x = stok[c];
                bool dup = false;  // an earlier (rejected) sibling with the same token
                for (int c2 = sfirst[cur]; c2 != c; c2 = snext[c2]) dup |= stok[c2] == x;
                const double px = (double)ex2_approx((slx[c] - M) * kLog2e) / (double)Z;
                const double pt = dup ? 0.0 : px / (1.0 - rej_mass);
                if (lead && ratio) ratio[base + c] = (float)pt;
                if ((double)su[c] < pt) {
                    pick = c;
                    break;
                }
                if (!dup) rej_mass += px;
            }
            ws.pick = pick;
        }
        __syncthreads();
        const int nxt = ws.pick;
        if (nxt >= 0) {
            ++len;
            if (lead && threadIdx.x == 0) {
                path[base + len] = nxt;
                out_tokens[base + len - 1] = stok[nxt];
            }
            cur = nxt;
            load_row<E4, VEC>(target + (base + cur) * V, V, g0, lane, P);
            continue;
        }
        // ---- bonus: inverse CDF of p~ (the node's softmax without the
        // rejected children's tokens) at u_bonus, as masses e^(l - M)
        const float ml2 = M * kLog2e;
        float gs[E4];
        float tt = 0.0f;
#pragma unroll
        for (int k = 0; k < E4; ++k) {
            float acc = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int idx = 128 * (g0 + k) + 4 * lane + e;
                float ev = ex2_approx(fmaf(comp(P[k], e), kLog2e, -ml2));
                for (int c = sfirst[cur]; c != -1; c = snext[c])
                    if (stok[c] == idx) ev = 0.0f;
                set_comp(P[k], e, ev);
                acc += ev;
            }
            gs[k] = acc;
            tt += acc;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tt += __shfl_xor_sync(FULL, tt, o);
        if (lane == 0) ws.wsum[warp] = (double)tt;
        __syncthreads();
        // fp64 bookkeeping by one thread (this part's fp64 rate is low)
        if (threadIdx.x == 0) {
            double cta_tot = 0.0;
            for (int w = 0; w < NW; ++w) cta_tot += ws.wsum[w];
            ws.dtmp[0] = cta_tot;
        }
        __syncthreads();
        const int s2 = exchange(pack_double(ws.dtmp[0]));
        if (ws.abort) {
            ok = false;
            break;
        }
        if (threadIdx.x == 0) {
            double all = 0.0;
            for (int r = 0; r < ncta; ++r) all += unpack_double(ws.recv[s2][r]);
            const double thr0 = (double)u_bonus[b] * all;
            // crossing rank (else the last rank with mass), and the mass before it
            int rs0 = -1, rlast = -1;
            double before0 = 0.0, run = 0.0, before_last = 0.0;
            for (int r = 0; r < ncta; ++r) {
                const double m = unpack_double(ws.recv[s2][r]);
                if (m > 0.0) {
                    rlast = r;
                    before_last = run;
                }
                if (rs0 < 0 && run + m > thr0 && m > 0.0) {
                    rs0 = r;
                    before0 = run;
                }
                run += m;
            }
            const bool crossing0 = rs0 >= 0;
            if (!crossing0) {
                rs0 = rlast;
                before0 = before_last;
            }
            // this CTA's crossing warp (else its last warp with mass)
            int wsel0 = -1, wlast = -1;
            double wb0 = before0, wrun = before0, wb_last = before0;
            if (rank == rs0) {
                for (int w = 0; w < NW; ++w) {
                    const double m = ws.wsum[w];
                    if (m > 0.0) {
                        wlast = w;
                        wb_last = wrun;
                    }
                    if (crossing0 && wsel0 < 0 && wrun + m > thr0 && m > 0.0) {
                        wsel0 = w;
                        wb0 = wrun;
                    }
                    wrun += m;
                }
                if (wsel0 < 0) {
                    wsel0 = wlast;
                    wb0 = wb_last;
                }
            }
            ws.dtmp[0] = thr0;
            ws.dtmp[1] = wb0;
            ws.isel[0] = rs0;
            ws.isel[1] = crossing0 ? 1 : 0;
            ws.isel[2] = wsel0;
            ws.pick = -1;
        }
        __syncthreads();
        const double thr = ws.dtmp[0];
        const int rs = ws.isel[0];
        const bool crossing = ws.isel[1] != 0;
        if (rank == rs) {
            // the crossing warp, then group, lane and element
            const int wsel = ws.isel[2];
            const double wb = ws.dtmp[1];
            if (warp == wsel) {
                bool found = false;
                double grun = wb;
                int kl = -1;
                double kl_base = wb;
#pragma unroll
                for (int k = 0; k < E4; ++k) {
                    float gf = gs[k];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) gf += __shfl_xor_sync(FULL, gf, o);
                    const double g = (double)gf;
                    if (!found && g > 0.0) {
                        kl = k;
                        kl_base = grun;
                        if (crossing && grun + g > thr) found = true;
                    }
                    if (!found) grun += g;
                }
                // within group kl: inclusive scan of the lanes' sums
                int kk = kl < 0 ? 0 : kl;
                float mine = 0.0f;
#pragma unroll
                for (int k = 0; k < E4; ++k)
                    if (k == kk) mine = gs[k];
                double inc = (double)mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double t = __shfl_up_sync(FULL, inc, o);
                    if (lane >= o) inc += t;
                }
                const double lane_base = kl_base + inc - (double)mine;
                const unsigned cross = __ballot_sync(FULL, found && mine > 0.0f &&
                                                                kl_base + inc > thr);
                const unsigned pos = __ballot_sync(FULL, mine > 0.0f);
                int lsel = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : -1);
                if (kl >= 0 && lsel >= 0 && lane == lsel) {
                    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < E4; ++k)
                        if (k == kk) q4 = P[k];
                    double c2 = lane_base;
                    int pick = -1, plast = -1;
                    for (int e = 0; e < 4; ++e) {
                        const float ev = comp(q4, e);
                        if (ev > 0.0f) plast = e;
                        c2 += (double)ev;
                        if (cross && pick < 0 && ev > 0.0f && c2 > thr) pick = e;
                    }
                    if (pick < 0) pick = plast;
                    if (pick >= 0) ws.pick = 128 * (g0 + kk) + 4 * lane + pick;
                }
            }
        }
        __syncthreads();
        const int s3 = exchange(make_float4(__int_as_float(ws.pick), 0.0f, 0.0f, 0.0f));
        if (ws.abort) {
            ok = false;
            break;
        }
        for (int r = 0; r < ncta; ++r) bonus = max(bonus, __float_as_int(ws.recv[s3][r].x));
        break;
    }
    if (lead && threadIdx.x == 0) {
        out_tokens[base + len] = ok ? bonus : -1;
        accept_len[b] = len;
        if (!ok) status[b] |= SVF_DEV_TIMEOUT;
    }
    if (CLUSTER) {
        cluster_arrive();
        cluster_wait();
    }
}

// ---------------------------------------------------------------- host side

namespace {

struct TargetCfg {
    int nt, e4, cl;
};

int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

bool target_config(int B, int V, TargetCfg *c) {
    if (V <= 4 * tgt::kSmallThreads * 8) {
        int e4 = 1;
        while (e4 < 8 && (long long)tgt::kSmallThreads * 4 * e4 < V) e4 *= 2;
        *c = {tgt::kSmallThreads, e4, 1};
        return true;
    }
    const long long cap = (long long)tgt::kClusterThreads * 4;  // elements per CTA per slot
    int e4 = 1;
    while (e4 < 8 && cdiv(V, cap * e4) > tgt::kMaxCluster) e4 *= 2;
    int cl = cdiv(V, cap * e4);
    if (cl > tgt::kMaxCluster) return false;
    while (e4 < 8 && (long long)B * cl > num_sms()) {
        e4 *= 2;
        cl = cdiv(V, cap * e4);
    }
    *c = {tgt::kClusterThreads, e4, cl};
    return true;
}

template <int NT, int E4, bool VEC, bool CLUSTER, bool GREEDY, typename T>
cudaError_t launch_target(const TargetCfg &c, const T *target, const int32_t *tokens,
                          const int32_t *parent, const float *u_accept, const float *u_bonus,
                          int B, int N, int V, int32_t *accept_len, int32_t *path,
                          int32_t *out_tokens, float *ratio, int32_t *status,
                          cudaStream_t stream) {
    auto kern = accept_target_kernel<NT, E4, VEC, CLUSTER, GREEDY, T>;
    const size_t smem = (size_t)N * 6 * sizeof(int32_t);
    if (CLUSTER && c.cl > 8) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const unsigned blocks = (unsigned)((long long)B * (CLUSTER ? c.cl : 1));
    return launch_pdl(kern, dim3(blocks), dim3(NT), smem, stream, CLUSTER ? (unsigned)c.cl : 0u,
                      target, tokens, parent, u_accept, u_bonus, N, V, CLUSTER ? c.cl : 1,
                      accept_len, path, out_tokens, ratio, status);
}

template <bool VEC, bool GREEDY, typename T>
cudaError_t dispatch_target(const TargetCfg &c, const T *target, const int32_t *tokens,
                            const int32_t *parent, const float *u_accept, const float *u_bonus,
                            int B, int N, int V, int32_t *accept_len, int32_t *path,
                            int32_t *out_tokens, float *ratio, int32_t *status,
                            cudaStream_t stream) {
#define SVF_TGT(NT_, E4_, CL_)                                                                   \
    return launch_target<NT_, E4_, VEC, CL_, GREEDY, T>(c, target, tokens, parent, u_accept,    \
                                                     u_bonus, B, N, V, accept_len, path,        \
                                                     out_tokens, ratio, status, stream)
    if (c.nt == tgt::kClusterThreads && c.e4 == 8 && (long long)B * c.cl > num_sms()) {
        // More sequences than one wave of 8-slot clusters: 16 slots per lane
        // halve the cluster, taken when that needs fewer waves.
        TargetCfg w{tgt::kClusterThreads, tgt::kWideSlots,
                    cdiv(V, (long long)tgt::kClusterThreads * 4 * tgt::kWideSlots)};
        const size_t smem = (size_t)N * 6 * sizeof(int32_t);
        const int r8 = resident_clusters(
            accept_target_kernel<tgt::kClusterThreads, 8, VEC, true, GREEDY, T>,
            tgt::kClusterThreads, smem, c.cl);
        const int rw = resident_clusters(
            accept_target_kernel<tgt::kClusterThreads, tgt::kWideSlots, VEC, true, GREEDY, T>,
            tgt::kClusterThreads, smem, w.cl);
        if (r8 > 0 && rw > 0 && cdiv(B, rw) < cdiv(B, r8))
            return launch_target<tgt::kClusterThreads, tgt::kWideSlots, VEC, true, GREEDY, T>(
                w, target, tokens, parent, u_accept, u_bonus, B, N, V, accept_len, path,
                out_tokens, ratio, status, stream);
    }
    if (c.nt == tgt::kSmallThreads) {
        switch (c.e4) {
            case 1: SVF_TGT(tgt::kSmallThreads, 1, false);
            case 2: SVF_TGT(tgt::kSmallThreads, 2, false);
            case 4: SVF_TGT(tgt::kSmallThreads, 4, false);
            default: SVF_TGT(tgt::kSmallThreads, 8, false);
        }
    }
    switch (c.e4) {
        case 1: SVF_TGT(tgt::kClusterThreads, 1, true);
        case 2: SVF_TGT(tgt::kClusterThreads, 2, true);
        case 4: SVF_TGT(tgt::kClusterThreads, 4, true);
        default: SVF_TGT(tgt::kClusterThreads, 8, true);
    }
#undef SVF_TGT
}

}  // namespace

// On chip up to kMaxOnChipVocab; the streaming kernels of
// accept_target_stream.cu above that, up to kMaxStreamVocab.
bool accept_target_supported(int V) { return V >= 1 && V <= kMaxStreamVocab; }

static bool accept_target_on_chip(int V) {
    TargetCfg c;
    return V >= 1 && target_config(1, V, &c);
}

template <typename T>
cudaError_t launch_target_walk(bool greedy, const T *target, const int32_t *tokens,
                               const int32_t *parent, const float *u_accept,
                               const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                               int32_t *path, int32_t *out_tokens, float *ratio,
                               int32_t *status, cudaStream_t stream) {
    TargetCfg c;
    if (!target_config(B, V, &c)) return cudaErrorInvalidValue;
    const bool vec = (V & 3) == 0;
    if (greedy)
        return vec ? dispatch_target<true, true>(c, target, tokens, parent, u_accept, u_bonus, B,
                                                 N, V, accept_len, path, out_tokens, ratio,
                                                 status, stream)
                   : dispatch_target<false, true>(c, target, tokens, parent, u_accept, u_bonus,
                                                  B, N, V, accept_len, path, out_tokens, ratio,
                                                  status, stream);
    return vec ? dispatch_target<true, false>(c, target, tokens, parent, u_accept, u_bonus, B, N,
                                              V, accept_len, path, out_tokens, ratio, status,
                                              stream)
               : dispatch_target<false, false>(c, target, tokens, parent, u_accept, u_bonus, B,
                                               N, V, accept_len, path, out_tokens, ratio, status,
                                               stream);
}

cudaError_t launch_accept_target(bool greedy, const float *target, const int32_t *tokens,
                                 const int32_t *parent, const float *u_accept,
                                 const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                                 int32_t *path, int32_t *out_tokens, float *ratio,
                                 int32_t *status, cudaStream_t stream) {
    if (!accept_target_on_chip(V))
        return launch_accept_target_stream(greedy, target, tokens, parent, u_accept, u_bonus, B,
                                           N, V, accept_len, path, out_tokens, ratio, status,
                                           stream);
    return launch_target_walk(greedy, target, tokens, parent, u_accept, u_bonus, B, N, V,
                              accept_len, path, out_tokens, ratio, status, stream);
}

cudaError_t launch_accept_target_bf16(bool greedy, const __nv_bfloat16 *target,
                                      const int32_t *tokens, const int32_t *parent,
                                      const float *u_accept, const float *u_bonus, int B, int N,
                                      int V, int32_t *accept_len, int32_t *path,
                                      int32_t *out_tokens, float *ratio, int32_t *status,
                                      cudaStream_t stream) {
    if (!accept_target_on_chip(V))
        return launch_accept_target_stream_bf16(greedy, target, tokens, parent, u_accept,
                                                u_bonus, B, N, V, accept_len, path, out_tokens,
                                                ratio, status, stream);
    return launch_target_walk(greedy, target, tokens, parent, u_accept, u_bonus, B, N, V,
                              accept_len, path, out_tokens, ratio, status, stream);
}

}  // namespace svf
