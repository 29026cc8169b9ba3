// attn_simt.cu -- tree attention on CUDA cores (fp32 inputs; also accepts bf16).
//
// "EAGLE 演化史", § Tree Verification 详解, A-B: node i of sequence b attends
// to the cached prefix t < L_b and to tree positions L_b + j for j an ancestor
// of i or i itself. One 4-warp CTA owns one (sequence, node, query head);
// each warp takes every fourth block of 32 tokens: each lane scores one token
// of the block, and an online softmax (running max, running sum, rescaled
// accumulator; the lanes split head_dim for the output) folds the visible
// tokens in. The warps' states merge at the end. fp32 arithmetic throughout
// with the accurate expf.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Eight consecutive elements of a K or V row, widened to fp32. VEC: the row
// is 16-byte aligned (two float4 loads, or one load of eight bf16).
template <bool VEC>
__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    if (VEC) {
        const float4 u = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 v = __ldg(reinterpret_cast<const float4 *>(p + 4));
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
        x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __ldg(p + i);
    }
}
template <bool VEC>
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8]) {
    if (VEC) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __bfloat162float(p[i]);
    }
}

template <typename Elt, int E, bool VEC>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a, float scale) {
    constexpr int D = 32 * E;
    constexpr int NWARP = 4;  // warps per row, each over every fourth block
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const long long rowid = blockIdx.x;  // (b, i, h)
    const int h = (int)(rowid % a.Hq);
    const int i = (int)((rowid / a.Hq) % a.N);
    const int b = (int)(rowid / ((long long)a.N * a.Hq));
    const int G = a.Hq / a.Hkv;
    const int g = h / G;
    const int L = a.seq_lens[b];
    const long long Tlen = (long long)L + a.N;
    const int ps = a.page_size;
    const int32_t *pt = a.page_table + (size_t)b * a.max_pages;

    // every warp checks the whole page range, so every warp takes the same
    // branch below
    int err = 0;
    if (L < 0 || Tlen > (long long)a.max_pages * ps) {
        err = SVF_DEV_BAD_LENGTH;
    } else {
        const int npages = (int)((Tlen + ps - 1) / ps);
        for (int p = lane; p < npages; p += 32) {
            const int id = pt[p];
            if (id < 0 || id >= a.num_pages) err = SVF_DEV_BAD_PAGE;
        }
        err = __reduce_or_sync(0xffffffffu, err);
    }
    const size_t row = ((size_t)b * a.N + i) * a.Hq + h;
    Elt *outp = reinterpret_cast<Elt *>(a.out) + row * D;
    if (err) {
        if (w == 0) {
#pragma unroll
            for (int e = 0; e < E; ++e) outp[lane * E + e] = from_f<Elt>(0.0f);
            if (lane == 0) {
                if (a.lse) a.lse[row] = 0.0f;
                atomicOr(&a.status[b], err);
            }
        }
        return;
    }

    const Elt *qp = reinterpret_cast<const Elt *>(a.q) + row * D;
    // the q row in shared memory: every lane reads all of it per token
    __shared__ float sq[32 * E];
    for (int d = threadIdx.x; d < D; d += blockDim.x) sq[d] = to_f(qp[d]);
    __syncthreads();
    const uint64_t anc = a.anc[(size_t)b * a.N + i];
    const Elt *kc = reinterpret_cast<const Elt *>(a.k_cache);
    const Elt *vc = reinterpret_cast<const Elt *>(a.v_cache);
    // Blocks of 32 tokens, block k to warp k % 4: lane j scores token t0 + j
    // over the whole head (the whole q row is read by every lane), the block's
    // maximum rescales the warp's running output once, and the output lanes
    // (which split head_dim) then fold the block's V rows in, whose loads are
    // independent of one another. The four warps' states merge at the end.
    float mx = -INFINITY, l = 0.0f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.0f;
    for (long long t0 = 32ll * w; t0 < Tlen; t0 += 32 * NWARP) {
        const long long t = t0 + lane;
        bool vis = t < Tlen;
        if (vis && t >= L) vis = (anc >> (int)(t - L)) & 1ull;
        size_t off_t = 0;
        float s = -INFINITY;
        if (vis) {
            off_t = (((size_t)pt[t / ps] * ps + (size_t)(t % ps)) * a.Hkv + g) * D;
            // the K row in pieces of 64 elements, each piece's loads issued
            // together
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int d0 = 0; d0 < D; d0 += 64) {
                float kx[8][8];
#pragma unroll
                for (int c = 0; c < 8; ++c) load8<VEC>(kc + off_t + d0 + 8 * c, kx[c]);
#pragma unroll
                for (int c = 0; c < 8; ++c)
#pragma unroll
                    for (int q = 0; q < 8; q += 2) {
                        s0 = fmaf(sq[d0 + 8 * c + q], kx[c][q], s0);
                        s1 = fmaf(sq[d0 + 8 * c + q + 1], kx[c][q + 1], s1);
                    }
            }
            s = (s0 + s1) * scale;
        }
        const float bm = warp_max(s);
        if (bm == -INFINITY) continue;  // nothing visible in this block
        const float mn = fmaxf(mx, bm);
        const float corr = expf(mx - mn);  // 0 on the first visible block
        const float p = vis ? expf(s - mn) : 0.0f;
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= corr;
        mx = mn;
        // VB V rows per batch: the (predicated) loads go out together; a
        // token with p = 0 is not read (its slot may hold anything)
        constexpr int VB = E <= 2 ? 16 : 8;
        for (int j0 = 0; j0 < 32; j0 += VB) {
            float pj[VB], vv[VB][E];
#pragma unroll
            for (int u = 0; u < VB; ++u) {
                pj[u] = __shfl_sync(0xffffffffu, p, j0 + u);
                const size_t oj = __shfl_sync(0xffffffffu, off_t, j0 + u);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    vv[u][e] = pj[u] != 0.0f ? to_f(vc[oj + lane * E + e]) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < VB; ++u)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(pj[u], vv[u][e], acc[e]);
        }
    }
    // merge the warps' (max, sum, output): each scaled by e^(max_w - M)
    __shared__ float s_mx[NWARP], s_l[NWARP], s_acc[NWARP][32 * E];
    if (lane == 0) {
        s_mx[w] = mx;
        s_l[w] = l;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) s_acc[w][lane * E + e] = acc[e];
    __syncthreads();
    if (w != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int v = 0; v < NWARP; ++v) M = fmaxf(M, s_mx[v]);
    float f[NWARP], lt = 0.0f;
#pragma unroll
    for (int v = 0; v < NWARP; ++v) {
        f[v] = s_mx[v] == -INFINITY ? 0.0f : expf(s_mx[v] - M);
        lt = fmaf(s_l[v], f[v], lt);
    }
    const float inv = 1.0f / lt;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        float o = 0.0f;
#pragma unroll
        for (int v = 0; v < NWARP; ++v) o = fmaf(s_acc[v][lane * E + e], f[v], o);
        outp[lane * E + e] = from_f<Elt>(o * inv);
    }
    if (lane == 0 && a.lse) a.lse[row] = M + logf(lt);
}

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t stream) {
    const long long blocks = (long long)a.B * a.N * a.Hq;  // one 4-warp CTA per row
    const int threads = 128;
    const float scale = a.sm_scale > 0.0f ? a.sm_scale : 1.0f / sqrtf((float)a.D);
    // K rows start at multiples of D elements: vector loads when the caches
    // are 16-byte aligned
    const bool vec = ((reinterpret_cast<uintptr_t>(a.k_cache) |
                       reinterpret_cast<uintptr_t>(a.v_cache)) & 15u) == 0;
#define SVF_SIMT(T_, E_)                                                                       \
    do {                                                                                       \
        if (vec)                                                                               \
            attn_simt_kernel<T_, E_, true><<<(unsigned)blocks, threads, 0, stream>>>(a, scale); \
        else                                                                                   \
            attn_simt_kernel<T_, E_, false><<<(unsigned)blocks, threads, 0, stream>>>(a, scale);\
    } while (0)
    if (a.dtype == SVF_F32) {
        if (a.D == 64) SVF_SIMT(float, 2);
        else SVF_SIMT(float, 4);
    } else {
        if (a.D == 64) SVF_SIMT(__nv_bfloat16, 2);
        else SVF_SIMT(__nv_bfloat16, 4);
    }
#undef SVF_SIMT
    return cudaGetLastError();
}

}  // namespace svf
