// accept_target_stream.cu -- greedy and one-hot acceptance for vocabularies
// too large to hold on chip (262144 < V <= 786432).
//
// The rules are those of accept_target.cu ("Eagle vs DFlash": at temperature
// 0 the target emits the argmax of its row; with q = one-hot(candidate) a
// child with token x is accepted iff u < p~(x), a rejection removes x's mass
// from p~, and the bonus token is the inverse CDF of p~). There a cluster
// holds the current node's target row in registers; here each CTA of the
// cluster streams its slice of the row from memory on every pass instead:
//   greedy   one pass per visited node: (max, argmax) with ties to the lower
//            id, merged over the warp, the CTA and the cluster in rank order;
//   one-hot  one pass per visited node: (max, sum e^(l - max)); the tests
//            are scalars from the children's gathered logits; when every
//            child is rejected (or at a leaf) one more pass gives the masses
//            of p~ per warp slice, and the crossing warp re-reads its groups
//            to find the group, lane and element of the inverse CDF.
// Each warp owns a contiguous run of 128-element groups of its CTA's slice,
// so the inverse-CDF search goes rank -> warp -> group -> lane -> element in
// vocabulary order. Group sums are fp32, masses across groups, warps and
// ranks fp64, as in the on-chip kernel. No workspace.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

namespace tgs {
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kCluster = 8;     // CTAs per sequence (portable cluster size)
constexpr int kThreads = 512;
constexpr int kMaxKids = 64;    // children of one node whose tokens a bonus pass excludes

// Four consecutive elements from e0 (-inf past V); VEC: one 16-byte (fp32)
// or 8-byte (bf16) load.
template <bool VEC>
__device__ __forceinline__ float4 load4(const float *__restrict__ row, long long e0, int V) {
    if (VEC && e0 + 3 < V) return __ldg(reinterpret_cast<const float4 *>(row + e0));
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (e0 + i < V) ? __ldg(row + e0 + i) : -INFINITY;
    return make_float4(v[0], v[1], v[2], v[3]);
}
template <bool VEC>
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *__restrict__ row, long long e0, int V) {
    if (VEC && e0 + 3 < V) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(row + e0));
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (e0 + i < V) ? __bfloat162float(row[e0 + i]) : -INFINITY;
    return make_float4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ float logit_at(const float *p) { return __ldg(p); }
__device__ __forceinline__ float logit_at(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

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

// (max, sum e^(x - max)) merge
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

__device__ __forceinline__ float4 pack_double(double d) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(d);
    return make_float4(__uint_as_float((uint32_t)u), __uint_as_float((uint32_t)(u >> 32)), 0.f, 0.f);
}

__device__ __forceinline__ double unpack_double(const float4 &r) {
    return __longlong_as_double((long long)(((unsigned long long)__float_as_uint(r.y) << 32) |
                                            __float_as_uint(r.x)));
}

struct StreamTargetSmem {
    float4 recv[2][kCluster];  // records of every rank, by exchange parity
    uint64_t bar[2];
    float4 red[32];            // per-warp partials
    double wsum[32];           // per-warp masses (bonus search)
    int kid_tok[kMaxKids];     // tokens of the current node's children (bonus exclusion)
    int nkids;
    int bad;
    int abort;
    int pick;
    double dtmp[2];
    int isel[3];
};
}  // namespace tgs

template <int NT, bool VEC, bool CLUSTER, bool GREEDY, typename T>
__global__ void __launch_bounds__(NT, 1) accept_target_stream_kernel(
    const T *__restrict__ target, const int32_t *__restrict__ tokens,
    const int32_t *__restrict__ parent, const float *__restrict__ u_accept,
    const float *__restrict__ u_bonus, int N, int V, int CL, int32_t *__restrict__ accept_len,
    int32_t *__restrict__ path, int32_t *__restrict__ out_tokens, float *__restrict__ ratio,
    int32_t *__restrict__ status) {
    using namespace tgs;
    constexpr int NW = NT / 32;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = CLUSTER ? (int)(blockIdx.x % (unsigned)CL) : 0;
    const long long b = CLUSTER ? (long long)(blockIdx.x / (unsigned)CL) : (long long)blockIdx.x;
    const int ncta = CLUSTER ? CL : 1;
    const size_t base = (size_t)b * N;
    const bool lead = rank == 0;
    // this warp's groups [wg0, wg1): contiguous runs in vocabulary order
    const int ngroups = (V + 127) >> 7;
    const int gper = (ngroups + ncta - 1) / ncta;
    const int cg0 = min(ngroups, rank * gper), cg1 = min(ngroups, cg0 + gper);
    const int wper = (cg1 - cg0 + NW - 1) / NW;
    const int wg0 = min(cg1, cg0 + warp * wper), wg1 = min(cg1, wg0 + wper);

    extern __shared__ __align__(16) unsigned char dyn[];
    float *slx = reinterpret_cast<float *>(dyn);        // [N] target logit of c's token at its parent
    float *su = slx + N;                                // [N] u_accept
    int32_t *sp = reinterpret_cast<int32_t *>(su + N);  // [N] parent
    int32_t *stok = sp + N;                             // [N] token
    int32_t *sfirst = stok + N;                         // [N] first child, -1 for a leaf
    int32_t *snext = sfirst + N;                        // [N] next sibling, -1 for the last
    __shared__ StreamTargetSmem ws;

    pdl_wait();
    pdl_launch_dependents();

    // ---- the tree: parents, tokens, uniforms; validity; child lists
    if (threadIdx.x == 0) {
        ws.bad = 0;
        ws.abort = 0;
    }
    for (int i = threadIdx.x; i < N; i += NT) sfirst[i] = INT_MAX;
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const int pp = parent[base + i];
        const int tk = tokens[base + i];
        sp[i] = pp;
        stok[i] = tk;
        su[i] = GREEDY ? 0.0f : u_accept[base + i];
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
            if (!GREEDY) slx[i] = logit_at(target + (base + pp) * (size_t)V + stok[i]);
        }
        snext[i] = nx;
    }
    if (CLUSTER) cluster_wait();

    // One exchange: warp 0 pushes this CTA's record into slot `rank` of
    // every CTA of the cluster and waits (bounded) until every rank's record
    // has landed here.
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
        const T *row = target + (base + cur) * (size_t)V;
        if (GREEDY) {
            // ---- argmax of the node's target row, ties to the lowest id
            float bv = -INFINITY;
            int bi = INT_MAX;
            for (int g = wg0; g < wg1; ++g) {
                const long long e0 = 128ll * g + 4 * lane;
                const float4 x = load4<VEC>(row, e0, V);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float v = comp(x, e);
                    if (v > bv) {
                        bv = v;
                        bi = (int)e0 + e;
                    }
                }
            }
            warp_amax(bv, bi);
            if (lane == 0) ws.red[warp] = make_float4(bv, __int_as_float(bi), 0.0f, 0.0f);
            __syncthreads();
            float4 rec = make_float4(-INFINITY, __int_as_float(INT_MAX), 0.0f, 0.0f);
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
            continue;
        }

        // ---- one-hot candidates: softmax statistics of the node's row
        float mt = -INFINITY, st = 0.0f;
        for (int g = wg0; g < wg1; ++g) {
            const float4 x = load4<VEC>(row, 128ll * g + 4 * lane, V);
            const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
            if (mx == -INFINITY) continue;
            if (mx > mt) {
                st = (mt == -INFINITY) ? 0.0f : st * ex2_approx((mt - mx) * kLog2e);
                mt = mx;
            }
            const float ml2 = mt * kLog2e;
#pragma unroll
            for (int e = 0; e < 4; ++e) st += ex2_approx(fmaf(comp(x, e), kLog2e, -ml2));
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
        // decided by one thread (fp32 exponentials, fp64 mass and division)
        if (threadIdx.x == 0) {
            double rej_mass = 0.0;
            int pick = -1, nk = 0;
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
                if (!dup) {
                    rej_mass += px;
                    if (nk < kMaxKids) ws.kid_tok[nk] = x;
                    ++nk;
                }
            }
            ws.pick = pick;
            ws.nkids = nk;
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
            continue;
        }
        // ---- bonus: inverse CDF of p~ (the node's softmax without the
        // rejected children's tokens) at u_bonus, as masses e^(l - M)
        const int nk = ws.nkids;
        const float ml2 = M * kLog2e;
        // element mass: e^(l - M), 0 for a rejected token
        auto mass_of = [&](const float4 &x, long long e0, int e) -> float {
            const int idx = (int)e0 + e;
            float ev = ex2_approx(fmaf(comp(x, e), kLog2e, -ml2));
            if (nk <= kMaxKids) {
                for (int k = 0; k < nk; ++k)
                    if (ws.kid_tok[k] == idx) ev = 0.0f;
            } else {
                for (int c = sfirst[cur]; c != -1; c = snext[c])
                    if (stok[c] == idx) ev = 0.0f;
            }
            return ev;
        };
        float tt = 0.0f;
        for (int g = wg0; g < wg1; ++g) {
            const long long e0 = 128ll * g + 4 * lane;
            const float4 x = load4<VEC>(row, e0, V);
            float acc = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc += mass_of(x, e0, e);
            tt += acc;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tt += __shfl_xor_sync(FULL, tt, o);
        if (lane == 0) ws.wsum[warp] = (double)tt;
        __syncthreads();
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
        if (rank == rs && warp == ws.isel[2]) {
            // the crossing warp re-reads its groups: the crossing group (else
            // its last group with mass), then lane and element
            const double wb = ws.dtmp[1];
            bool found = false;
            double grun = wb, kl_base = wb;
            int kl = -1;
            for (int g = wg0; g < wg1 && !found; ++g) {
                const long long e0 = 128ll * g + 4 * lane;
                const float4 x = load4<VEC>(row, e0, V);
                float gf = 0.0f;
#pragma unroll
                for (int e = 0; e < 4; ++e) gf += mass_of(x, e0, e);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) gf += __shfl_xor_sync(FULL, gf, o);
                const double gd = (double)gf;
                if (gd > 0.0) {
                    kl = g;
                    kl_base = grun;
                    if (crossing && grun + gd > thr) found = true;
                }
                if (!found) grun += gd;
            }
            if (kl >= 0) {
                // within group kl: inclusive scan of the lanes' sums
                const long long e0 = 128ll * kl + 4 * lane;
                const float4 x = load4<VEC>(row, e0, V);
                float ev[4];
                float mine = 0.0f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    ev[e] = mass_of(x, e0, e);
                    mine += ev[e];
                }
                double inc = (double)mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double t = __shfl_up_sync(FULL, inc, o);
                    if (lane >= o) inc += t;
                }
                const double lane_base = kl_base + inc - (double)mine;
                const unsigned cross =
                    __ballot_sync(FULL, found && mine > 0.0f && kl_base + inc > thr);
                const unsigned pos = __ballot_sync(FULL, mine > 0.0f);
                const int lsel = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : -1);
                if (lsel >= 0 && lane == lsel) {
                    double c2 = lane_base;
                    int pick = -1, plast = -1;
                    for (int e = 0; e < 4; ++e) {
                        if (ev[e] > 0.0f) plast = e;
                        c2 += (double)ev[e];
                        if (cross && pick < 0 && ev[e] > 0.0f && c2 > thr) pick = e;
                    }
                    if (pick < 0) pick = plast;
                    if (pick >= 0) ws.pick = (int)e0 + pick;
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

size_t stream_target_smem(int N) {
    return (size_t)N * (2 * sizeof(float) + 4 * sizeof(int32_t)) + 16;
}

template <bool VEC, bool GREEDY, typename T>
cudaError_t launch_stream_target(const T *target, const int32_t *tokens, const int32_t *parent,
                                 const float *u_accept, const float *u_bonus, int B, int N, int V,
                                 int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                                 float *ratio, int32_t *status, cudaStream_t stream) {
    auto kern = accept_target_stream_kernel<tgs::kThreads, VEC, true, GREEDY, T>;
    const size_t smem = stream_target_smem(N);
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int cl = tgs::kCluster;
    return launch_pdl(kern, dim3((unsigned)((long long)B * cl)), dim3(tgs::kThreads), smem,
                      stream, (unsigned)cl, target, tokens, parent, u_accept, u_bonus, N, V, cl,
                      accept_len, path, out_tokens, ratio, status);
}

template <typename T>
cudaError_t dispatch_stream_target(bool greedy, const T *target, const int32_t *tokens,
                                   const int32_t *parent, const float *u_accept,
                                   const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                                   int32_t *path, int32_t *out_tokens, float *ratio,
                                   int32_t *status, cudaStream_t stream) {
    const bool vec = (V & 3) == 0;
#define SVF_TS(VEC_, G_)                                                                         \
    return launch_stream_target<VEC_, G_, T>(target, tokens, parent, u_accept, u_bonus, B, N, V, \
                                             accept_len, path, out_tokens, ratio, status, stream)
    if (greedy) {
        if (vec) SVF_TS(true, true);
        SVF_TS(false, true);
    }
    if (vec) SVF_TS(true, false);
    SVF_TS(false, false);
#undef SVF_TS
}

}  // namespace

cudaError_t launch_accept_target_stream(bool greedy, const float *target, const int32_t *tokens,
                                        const int32_t *parent, const float *u_accept,
                                        const float *u_bonus, int B, int N, int V,
                                        int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                                        float *ratio, int32_t *status, cudaStream_t stream) {
    return dispatch_stream_target<float>(greedy, target, tokens, parent, u_accept, u_bonus, B, N,
                                         V, accept_len, path, out_tokens, ratio, status, stream);
}

cudaError_t launch_accept_target_stream_bf16(bool greedy, const __nv_bfloat16 *target,
                                             const int32_t *tokens, const int32_t *parent,
                                             const float *u_accept, const float *u_bonus, int B,
                                             int N, int V, int32_t *accept_len, int32_t *path,
                                             int32_t *out_tokens, float *ratio, int32_t *status,
                                             cudaStream_t stream) {
    return dispatch_stream_target<__nv_bfloat16>(greedy, target, tokens, parent, u_accept,
                                                 u_bonus, B, N, V, accept_len, path, out_tokens,
                                                 ratio, status, stream);
}

}  // namespace svf
