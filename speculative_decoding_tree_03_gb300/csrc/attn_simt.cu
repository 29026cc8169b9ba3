// attn_simt.cu -- tree attention on CUDA cores (fp32 inputs; also accepts bf16).
//
// "EAGLE 演化史", § Tree Verification 详解, A-B: node i of sequence b attends
// to the cached prefix t < L_b and to tree positions L_b + j for j an ancestor
// of i or i itself. One warp owns one (sequence, node, query head): the lanes
// split head_dim, a shuffle reduction gives each score, and an online softmax
// (running max, running sum, rescaled accumulator) folds the visible tokens in
// order. fp32 arithmetic throughout with the accurate expf.
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

template <typename Elt, int E>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a, float scale) {
    constexpr int D = 32 * E;
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long total = (long long)a.B * a.N * a.Hq;
    if (warp >= total) return;
    const int h = (int)(warp % a.Hq);
    const int i = (int)((warp / a.Hq) % a.N);
    const int b = (int)(warp / ((long long)a.N * a.Hq));
    const int G = a.Hq / a.Hkv;
    const int g = h / G;
    const int L = a.seq_lens[b];
    const long long Tlen = (long long)L + a.N;
    const int ps = a.page_size;
    const int32_t *pt = a.page_table + (size_t)b * a.max_pages;

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
#pragma unroll
        for (int e = 0; e < E; ++e) outp[lane * E + e] = from_f<Elt>(0.0f);
        if (lane == 0) {
            if (a.lse) a.lse[row] = 0.0f;
            atomicOr(&a.status[b], err);
        }
        return;
    }

    float q[E];
    const Elt *qp = reinterpret_cast<const Elt *>(a.q) + row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) q[e] = to_f(qp[e]);
    const uint64_t anc = a.anc[(size_t)b * a.N + i];

    float mx = -INFINITY, l = 0.0f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.0f;
    const Elt *kc = reinterpret_cast<const Elt *>(a.k_cache);
    const Elt *vc = reinterpret_cast<const Elt *>(a.v_cache);
    for (long long t = 0; t < Tlen; ++t) {
        if (t >= L) {
            const int j = (int)(t - L);
            if (!((anc >> j) & 1ull)) continue;
        }
        const int page = pt[t / ps];
        const int slot = (int)(t % ps);
        const size_t off = (((size_t)page * ps + slot) * a.Hkv + g) * D + lane * E;
        float s = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) s = fmaf(q[e], to_f(kc[off + e]), s);
        s = warp_sum(s) * scale;
        const float mn = fmaxf(mx, s);
        const float corr = expf(mx - mn);
        const float p = expf(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(p, to_f(vc[off + e]), acc[e] * corr);
        mx = mn;
    }
    const float inv = 1.0f / l;
#pragma unroll
    for (int e = 0; e < E; ++e) outp[lane * E + e] = from_f<Elt>(acc[e] * inv);
    if (lane == 0 && a.lse) a.lse[row] = mx + logf(l);
}

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t stream) {
    const long long warps = (long long)a.B * a.N * a.Hq;
    const int threads = 128;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    const float scale = a.sm_scale > 0.0f ? a.sm_scale : 1.0f / sqrtf((float)a.D);
    if (a.dtype == SVF_F32) {
        if (a.D == 64)
            attn_simt_kernel<float, 2><<<(unsigned)blocks, threads, 0, stream>>>(a, scale);
        else
            attn_simt_kernel<float, 4><<<(unsigned)blocks, threads, 0, stream>>>(a, scale);
    } else {
        if (a.D == 64)
            attn_simt_kernel<__nv_bfloat16, 2><<<(unsigned)blocks, threads, 0, stream>>>(a, scale);
        else
            attn_simt_kernel<__nv_bfloat16, 4><<<(unsigned)blocks, threads, 0, stream>>>(a, scale);
    }
    return cudaGetLastError();
}

}  // namespace svf
