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
// Two kernels:
//   accept_rowstats  streams every logits row the walk may touch once: the
//                    target row of every node, the draft row of every node
//                    with children. Per row: max m and Z = sum exp(l - m).
//   accept_walk      one CTA (or one warp for small vocabularies) per
//                    sequence. Tests use gathered logits only. A rejection
//                    needs the mass of the new residual, one reduction over
//                    the parent's two rows. The residual after k rejections
//                    is kept in closed form, p~ = max(0, p - c q) / S with
//                    c_0 = 0, S_0 = 1 and c_{k+1} = c_k + S_k,
//                    S_{k+1} = sum_v max(0, p_v - c_{k+1} q_v): subtracting q
//                    from max(0, p - c q) / S and renormalising gives exactly
//                    that form. The bonus token is an inverse-CDF search:
//                    128-element group sums, their prefix in fp64, then the
//                    crossing inside one group.
// Element probabilities are exp(l - m) / Z in fp32 with the accurate expf;
// the rounding error of l - m is carried as a first-order correction.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

namespace acc {
constexpr int kMaxGroups = 6144;  // V <= 786432 in groups of 128
constexpr int kSmallV = 2048;     // at or below: one warp per row / per sequence
}  // namespace acc

// exp(a - b) with the rounding error of the fp32 difference folded back in
// (two-sum of a and -b; first-order correction e * err). Infinite inputs fall
// back to the plain expf.
__device__ __forceinline__ float exp_diff(float a, float b) {
    const float s = a - b;
    const float e = expf(s);
    const float bp = s - a;
    const float ap = s - bp;
    const float err = (a - ap) + (-b - bp);
    return isfinite(err) ? fmaf(e, err, e) : e;
}

// Online (max, sum e^{x - max}) pair merge.
__device__ __forceinline__ void ms_merge(float &m, float &s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    if (m2 > m) {
        s = s * exp_diff(m, m2) + s2;
        m = m2;
    } else {
        s = s + s2 * exp_diff(m2, m);
    }
}

__device__ __forceinline__ void ms_add(float &m, float &s, float x) {
    if (x > m) {
        s = (m == -INFINITY) ? 0.0f : s * exp_diff(m, x);
        m = x;
    }
    s += exp_diff(x, m);
}

__device__ __forceinline__ void ms_add4(float &m, float &s, float4 x) {
    const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
    if (mx > m) {
        s = (m == -INFINITY) ? 0.0f : s * exp_diff(m, mx);
        m = mx;
    }
    s += (exp_diff(x.x, m) + exp_diff(x.y, m)) + (exp_diff(x.z, m) + exp_diff(x.w, m));
}

// Does node j of sequence b have a child?  (parent[] in global memory)
__device__ __forceinline__ bool has_child_lane(const int32_t *par, int N, int j, int lane,
                                               int width) {
    int hit = 0;
    for (int c = j + 1 + lane; c < N; c += width) hit |= (par[c] == j);
    return hit != 0;
}

// One warp per row (small V) or one block per row (large V).
// stats[kind][row] = (m, Z), kind 0 = target, 1 = draft; rows = b * N + j.
template <bool WARP_PER_ROW>
__global__ void __launch_bounds__(256) accept_rowstats_kernel(const float *__restrict__ target,
                                                              const float *__restrict__ draft,
                                                              const int32_t *__restrict__ parent,
                                                              int B, int N, int V,
                                                              float2 *__restrict__ stats) {
    const int kind = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long rows = (long long)B * N;
    long long r;
    int tid, width;
    if (WARP_PER_ROW) {
        r = (long long)blockIdx.x * 8 + warp;
        tid = lane;
        width = 32;
        if (r >= rows) return;
    } else {
        r = blockIdx.x;
        tid = threadIdx.x;
        width = blockDim.x;
    }
    const int b = (int)(r / N), j = (int)(r % N);
    if (kind == 1) {
        bool hc;
        if (WARP_PER_ROW) {
            hc = __any_sync(0xffffffffu, has_child_lane(parent + (size_t)b * N, N, j, lane, 32));
        } else {
            hc = __syncthreads_or(has_child_lane(parent + (size_t)b * N, N, j, tid, width));
        }
        if (!hc) return;
    }
    const float *row = (kind == 0 ? target : draft) + (size_t)r * V;
    float m = -INFINITY, s = 0.0f;
    if ((V & 3) == 0) {
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        const int V4 = V >> 2;
        int i = tid;
        for (; i + 3 * width < V4; i += 4 * width) {
            const float4 a0 = __ldg(row4 + i);
            const float4 a1 = __ldg(row4 + i + width);
            const float4 a2 = __ldg(row4 + i + 2 * width);
            const float4 a3 = __ldg(row4 + i + 3 * width);
            ms_add4(m, s, a0);
            ms_add4(m, s, a1);
            ms_add4(m, s, a2);
            ms_add4(m, s, a3);
        }
        for (; i < V4; i += width) ms_add4(m, s, __ldg(row4 + i));
    } else {
        for (int i = tid; i < V; i += width) ms_add(m, s, __ldg(row + i));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_merge(m, s, m2, s2);
    }
    if (WARP_PER_ROW) {
        if (lane == 0) stats[(size_t)kind * rows + r] = make_float2(m, s);
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
            ms_merge(m, s, m2, s2);
        }
        if (lane == 0) stats[(size_t)kind * rows + r] = make_float2(m, s);
    }
}

// The residual (or target) distribution at one node, in closed form:
// w_v = max(0, p_v - c q_v) with p = softmax(target row), q = softmax(draft row).
struct Residual {
    const float *t;
    const float *d;
    float mt, zt, md, zd;
    float c;  // 0: plain target softmax (draft row not read)
    __device__ __forceinline__ float w(float tv, float dv) const {
        const float p = exp_diff(tv, mt) / zt;
        if (c == 0.0f) return p;
        const float q = exp_diff(dv, md) / zd;
        return fmaxf(0.0f, p - c * q);
    }
};

// Four consecutive elements starting at v0 (zeros past V).
template <bool VEC4>
__device__ __forceinline__ void load4(const Residual &R, int v0, int V, float *w) {
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

// Block-wide exclusive prefix sum of one double per thread; *total gets the sum.
template <int NT>
__device__ __forceinline__ double block_excl_scan(double x, double *total, double *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (NT == 32) {
        *total = __shfl_sync(0xffffffffu, incl, 31);
        return incl - x;
    }
    __syncthreads();
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        double w = lane < NT / 32 ? scratch[lane] : 0.0;
        double wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < NT / 32) scratch[lane] = wi - w;
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    const double res = scratch[warp] + incl - x;
    *total = scratch[32];
    __syncthreads();
    return res;
}

// Group sums G[g] = sum of w over elements [128 g, 128 g + 128), each lane
// adding its four elements in fp32, the 32 lane sums in fp64. Returns the
// total (same on every thread).
template <int NT, bool VEC4>
__device__ double group_sums(const Residual &R, int V, double *G, double *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ngroups = (V + 127) >> 7;
    __syncthreads();  // earlier readers of G are done
    for (int g = warp; g < ngroups; g += NT / 32) {
        float w[4];
        load4<VEC4>(R, g * 128 + lane * 4, V, w);
        const float ls = ((w[0] + w[1]) + w[2]) + w[3];
        const double gs = warp_sum_d((double)ls);
        if (lane == 0) G[g] = gs;
    }
    __syncthreads();
    const int seg = (ngroups + NT - 1) / NT;
    double mine = 0.0;
    for (int k = 0; k < seg; ++k) {
        const int g = threadIdx.x * seg + k;
        if (g < ngroups) mine += G[g];
    }
    double total;
    block_excl_scan<NT>(mine, &total, scratch);
    return total;
}

// Inverse CDF: the smallest v with sum_{u <= v} w_u > thr = u * sum(w);
// else the last v with w_v > 0. The prefix is exact in the order it is
// formed: group sums G (fp64 of fp32 lane sums), their running sum in fp64,
// and inside the chosen group each lane's fp32 running sum on top of the fp64
// prefix of the lanes before it.
template <int NT, bool VEC4>
__device__ int inverse_cdf(const Residual &R, int V, float u, double *G, double *scratch,
                           int *sh, double *sbase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ngroups = (V + 127) >> 7;
    const int seg = (ngroups + NT - 1) / NT;
    group_sums<NT, VEC4>(R, V, G, scratch);
    double mine = 0.0;
    for (int k = 0; k < seg; ++k) {
        const int g = threadIdx.x * seg + k;
        if (g < ngroups) mine += G[g];
    }
    double total;
    double base = block_excl_scan<NT>(mine, &total, scratch);
    const double thr = (double)u * total;
    if (threadIdx.x == 0) {
        sh[0] = 0x7fffffff;
        sh[1] = -1;
    }
    __syncthreads();
    int found = -1;
    for (int k = 0; k < seg; ++k) {
        const int g = threadIdx.x * seg + k;
        if (g >= ngroups) break;
        if (base + G[g] > thr) {
            found = g;
            atomicMin(&sh[0], g);
            break;
        }
        base += G[g];
    }
    __syncthreads();
    int gsel = sh[0];
    if (found >= 0 && found == gsel) *sbase = base;
    if (gsel == 0x7fffffff) {
        // no crossing (rounding): the last group with positive mass
        if (threadIdx.x == 0) {
            int g = ngroups - 1;
            while (g >= 0 && !(G[g] > 0.0)) --g;
            sh[0] = g;
            *sbase = 0.0;
        }
    }
    __syncthreads();
    const bool crossing = gsel != 0x7fffffff;
    gsel = sh[0];
    if (warp == 0 && gsel >= 0) {
        float w[4];
        load4<VEC4>(R, gsel * 128 + lane * 4, V, w);
        float a[4];
        a[0] = w[0];
        a[1] = a[0] + w[1];
        a[2] = a[1] + w[2];
        a[3] = a[2] + w[3];
        double incl = (double)a[3];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const double lbase = *sbase + incl - (double)a[3];
        int hit = -1, last = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (crossing && hit < 0 && lbase + (double)a[e] > thr) hit = e;
            if (w[e] > 0.0f) last = e;
        }
        const unsigned bh = __ballot_sync(0xffffffffu, hit >= 0);
        const unsigned bl = __ballot_sync(0xffffffffu, last >= 0);
        int pick = -1;
        if (bh) {
            const int src = __ffs(bh) - 1;
            pick = gsel * 128 + src * 4 + __shfl_sync(0xffffffffu, hit, src);
        } else if (bl) {
            const int src = 31 - __clz(bl);
            pick = gsel * 128 + src * 4 + __shfl_sync(0xffffffffu, last, src);
        }
        if (lane == 0) sh[1] = pick;
    }
    __syncthreads();
    const int res = sh[1];
    __syncthreads();
    return res;
}

template <int NT, bool VEC4>
__global__ void __launch_bounds__(NT) accept_walk_kernel(
    const float *__restrict__ target, const float *__restrict__ draft,
    const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
    const float *__restrict__ u_accept, const float *__restrict__ u_bonus, int N, int V,
    const float2 *__restrict__ stats, long long rows, int32_t *__restrict__ accept_len,
    int32_t *__restrict__ path, int32_t *__restrict__ out_tokens, float *__restrict__ ratio,
    int32_t *__restrict__ status) {
    extern __shared__ double dyn[];
    double *G = dyn;                                       // [ngroups]
    int32_t *sp = reinterpret_cast<int32_t *>(G + ((V + 127) >> 7));  // parent [N]
    int32_t *stok = sp + N;                                // tokens [N]
    __shared__ double scratch[34];
    __shared__ int sh[4];
    __shared__ int s_acc;
    __shared__ double s_base;

    const int b = blockIdx.x;
    const size_t base = (size_t)b * N;
    if (threadIdx.x == 0) sh[3] = 0;
    __syncthreads();
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += NT) {
        const int pp = parent[base + i];
        const int tk = tokens[base + i];
        sp[i] = pp;
        stok[i] = tk;
        if (i == 0 ? pp != -1 : (pp < 0 || pp >= i)) bad |= SVF_DEV_BAD_PARENT;
        if (i > 0 && (tk < 0 || tk >= V)) bad |= SVF_DEV_BAD_TOKEN;
        path[base + i] = -1;
        out_tokens[base + i] = -1;
        if (ratio) ratio[base + i] = __int_as_float(0x7fc00000);
    }
    // OR-reduce the error bits over the block
    for (int o = 16; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicOr(&sh[3], bad);
    __syncthreads();
    bad = sh[3];
    if (threadIdx.x == 0) {
        status[b] = bad;
        accept_len[b] = 0;
    }
    if (bad) return;

    int cur = 0, len = 0;
    double coef = 0.0, mass = 1.0;
    if (threadIdx.x == 0) path[base] = 0;
    for (;;) {
        const float2 st = stats[base + cur];
        bool moved = false;
        for (int c = cur + 1; c < N; ++c) {
            if (sp[c] != cur) continue;
            const float2 sd = stats[rows + base + cur];
            const int x = stok[c];
            if (threadIdx.x == 0) {
                const float px = exp_diff(target[(base + cur) * V + x], st.x) / st.y;
                const float qx = exp_diff(draft[(base + cur) * V + x], sd.x) / sd.y;
                double r = (double)px - coef * (double)qx;
                r = r > 0.0 ? r : 0.0;
                const double lhs = (double)u_accept[base + c] * (double)qx * mass;
                s_acc = lhs < r;
                if (ratio) ratio[base + c] = (float)(r / (mass * (double)qx));
            }
            __syncthreads();
            const int accepted = s_acc;
            __syncthreads();
            if (accepted) {
                ++len;
                if (threadIdx.x == 0) {
                    path[base + len] = c;
                    out_tokens[base + len - 1] = x;
                }
                cur = c;
                coef = 0.0;
                mass = 1.0;
                moved = true;
                break;
            }
            // rejected: mass of max(0, p - (coef + mass) q)
            Residual R;
            R.t = target + (base + cur) * V;
            R.d = draft + (base + cur) * V;
            R.mt = st.x; R.zt = st.y; R.md = sd.x; R.zd = sd.y;
            const double nc = coef + mass;
            R.c = (float)nc;
            const double S = group_sums<NT, VEC4>(R, V, G, scratch);
            if (S > 0.0) {
                coef = (double)R.c;
                mass = S;
            }
            __syncthreads();
        }
        if (!moved) break;
    }
    // bonus token at the last node, from its target softmax or its residual
    Residual R;
    const float2 st = stats[base + cur];
    R.t = target + (base + cur) * V;
    R.mt = st.x;
    R.zt = st.y;
    R.c = (float)coef;
    if (coef != 0.0) {
        const float2 sd = stats[rows + base + cur];
        R.d = draft + (base + cur) * V;
        R.md = sd.x;
        R.zd = sd.y;
    } else {
        R.d = R.t;
        R.md = 0.0f;
        R.zd = 1.0f;
    }
    const int bonus = inverse_cdf<NT, VEC4>(R, V, u_bonus[b], G, scratch, sh, &s_base);
    if (threadIdx.x == 0) {
        out_tokens[base + len] = bonus;
        accept_len[b] = len;
    }
}

size_t accept_workspace_bytes(int B, int N, int V) {
    (void)V;
    return (size_t)2 * B * N * sizeof(float2) + 256;
}

template <int NT, bool VEC4>
static cudaError_t launch_walk(const float *target, const float *draft, const int32_t *tokens,
                               const int32_t *parent, const float *u_accept,
                               const float *u_bonus, int B, int N, int V, const float2 *stats,
                               int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                               float *ratio, int32_t *status, cudaStream_t stream) {
    const size_t smem = (size_t)((V + 127) >> 7) * sizeof(double) + (size_t)2 * N * sizeof(int32_t);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(accept_walk_kernel<NT, VEC4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    accept_walk_kernel<NT, VEC4><<<B, NT, smem, stream>>>(
        target, draft, tokens, parent, u_accept, u_bonus, N, V, stats, (long long)B * N,
        accept_len, path, out_tokens, ratio, status);
    return cudaGetLastError();
}

cudaError_t launch_accept(const float *target, const float *draft, const int32_t *tokens,
                          const int32_t *parent, const float *u_accept, const float *u_bonus, int B,
                          int N, int V, int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                          float *ratio, void *workspace, int32_t *status, cudaStream_t stream) {
    float2 *stats = reinterpret_cast<float2 *>(
        (reinterpret_cast<uintptr_t>(workspace) + 255) & ~static_cast<uintptr_t>(255));
    const long long rows = (long long)B * N;
    if (V <= acc::kSmallV) {
        dim3 grid((unsigned)((rows + 7) / 8), 2);
        accept_rowstats_kernel<true><<<grid, 256, 0, stream>>>(target, draft, parent, B, N, V, stats);
    } else {
        dim3 grid((unsigned)rows, 2);
        accept_rowstats_kernel<false><<<grid, 256, 0, stream>>>(target, draft, parent, B, N, V, stats);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const bool vec4 = (V & 3) == 0;
    if (V <= acc::kSmallV) {
        return vec4 ? launch_walk<32, true>(target, draft, tokens, parent, u_accept, u_bonus, B, N,
                                           V, stats, accept_len, path, out_tokens, ratio, status,
                                           stream)
                    : launch_walk<32, false>(target, draft, tokens, parent, u_accept, u_bonus, B,
                                            N, V, stats, accept_len, path, out_tokens, ratio,
                                            status, stream);
    }
    return vec4 ? launch_walk<1024, true>(target, draft, tokens, parent, u_accept, u_bonus, B, N,
                                         V, stats, accept_len, path, out_tokens, ratio, status,
                                         stream)
                : launch_walk<1024, false>(target, draft, tokens, parent, u_accept, u_bonus, B, N,
                                          V, stats, accept_len, path, out_tokens, ratio, status,
                                          stream);
}

}  // namespace svf
