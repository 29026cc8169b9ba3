// lm_head.cu -- target logits of every tree node from its hidden state, on the
// 5th-generation tensor cores, and the acceptance walk fed by them.
//
// "The EAGLE Family", § Why predict features instead of tokens?: the target
// distribution at a node is softmax(W_LM h), h the node's last hidden state.
// "EAGLE 演化史", § Tree Verification 详解, D.2: the verify pass's bandwidth
// cost sits in the LM head and the softmax over N·|V|. One call computes
//     logits[r][v] = sum_k h[r][k] W[v][k]      (bf16 operands, fp32 sums)
// for every node r of the batch (R = B·N rows) and vocabulary entry v, reading
// the weight once, and svf_spec_accept_lmhead hands those rows to the walk.
//
// A persistent GEMM: one CTA per SM (or a cluster of C CTAs sharing one tile
// of hidden states), tiles of 128 vocabulary rows x BN hidden rows, K in
// blocks of 64. The weight tile is the MMA's A operand (M = 128, K-major),
// the hidden-state tile its B operand (N = BN <= 256, K-major), both staged
// by TMA with 128-byte swizzle in a ring of stages; the accumulator lives in
// tensor memory, two buffers of BN columns, so the epilogue of one tile runs
// while the next one accumulates. Roles:
//   warp 0      producer: TMA of the weight tile and of this CTA's slice of
//               the hidden tile (multicast to the cluster when C > 1);
//   warp 1      MMA issuer (one thread): 4 MMAs per stage, then a commit that
//               frees the stage in every CTA of the cluster;
//   warps 2-5   epilogue: tensor memory -> registers -> fp32 logits, one
//               vocabulary row per thread, so a warp's stores of one hidden
//               row are 128 contiguous bytes.
// Tile order: the hidden tiles of one group of vocabulary rows are taken by
// consecutive clusters, so a weight tile is read from HBM once and reused
// from L2.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace svf {

namespace lmh {
constexpr int BM = 128;                 // vocabulary rows per tile (MMA M)
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle row
constexpr int A_BYTES = BM * BK * 2;    // 16 KB of weight per stage
constexpr int MAX_STAGES = 16;
constexpr int THREADS = 192;
constexpr int SMEM_BUDGET = 200 * 1024;  // stage ring
constexpr int MAX_BN = 256;
}  // namespace lmh

struct LmhParams {
    int R, H, V;
    int BN;        // hidden rows per tile: a multiple of 32, at most 256
    int C;         // CTAs of a cluster sharing one hidden tile
    int n_tiles;   // ceil(R / BN)
    int m_groups;  // ceil(ceil(V / 128) / C)
    int groups;    // m_groups * n_tiles
    int kblocks;   // H / 64
    int stages;
    uint32_t idesc;
    uint32_t tmem_cols;
    unsigned long long wait_ns;
    float *logits;   // [R, V]
    int32_t *status; // nullable: SVF_DEV_TIMEOUT when a wait gave up
};

__device__ __forceinline__ bool lmh_warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              unsigned long long ns) {
    const bool ok = mbar_wait_for(bar, parity, abort, ns);
    return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(lmh::THREADS, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmh,
                   LmhParams p) {
    using namespace lmh;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const int b_bytes = p.BN * 128;
    uint8_t *sA = smem;
    uint8_t *sB = smem + S * A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + S * b_bytes);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *acc_full = empty + MAX_STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!cluster_shape_is((uint32_t)p.C, 1u, 1u)) {
        // not the cluster the multicasts address: the whole cluster leaves
        // at once, touching no peer
        pdl_wait();
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, SVF_DEV_BAD_CLUSTER);
        return;
    }
    const uint32_t rank = p.C > 1 ? cluster_ctarank() : 0u;
    const uint16_t mask = (uint16_t)((1u << p.C) - 1u);
    const int cluster_id = blockIdx.x / p.C;
    const int num_clusters = gridDim.x / p.C;
    const int my_groups =
        cluster_id < p.groups ? (p.groups - 1 - cluster_id) / num_clusters + 1 : 0;
    const int slice_rows = p.BN / p.C;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], (uint32_t)p.C);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmw);
        tma_prefetch_desc(&tmh);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // every CTA's barriers exist before any peer multicasts into it
    if (p.C > 1) {
        cluster_arrive();
        cluster_wait();
    }
    pdl_wait();
    pdl_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;  // producer: k-blocks loaded

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Each cluster starts its k loop at its own offset (spread evenly over
        // H) and wraps around: clusters that start together then read
        // different columns of their weight rows instead of the same 128-byte
        // column of every row. The sum over k is the same set of terms.
        const int rot = (int)((long long)cluster_id * p.kblocks / num_clusters) % p.kblocks;
        bool ok = true;
        for (int i = 0; i < my_groups && ok; ++i) {
            const int g = cluster_id + i * num_clusters;
            const int mg = g / p.n_tiles, nt = g % p.n_tiles;
            const int m0 = (mg * p.C + (int)rank) * BM;
            const int n0 = nt * p.BN;
            for (int kb = 0; kb < p.kblocks; ++kb) {
                const int s = issued % S, use = issued / S;
                const int kc = (kb + rot < p.kblocks ? kb + rot : kb + rot - p.kblocks) * BK;
                if (use > 0 &&
                    !(ok = lmh_warp_wait(&empty[s], (uint32_t)((use - 1) & 1), abort_flag,
                                         p.wait_ns)))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(A_BYTES + b_bytes));
                    tma_load_2d(sA + s * A_BYTES, &tmw, kc, m0, &full[s]);
                    if (p.C == 1)
                        tma_load_2d(sB + s * b_bytes, &tmh, kc, n0, &full[s]);
                    else
                        tma_load_2d_multicast(sB + s * b_bytes + (int)rank * slice_rows * 128,
                                              &tmh, kc, n0 + (int)rank * slice_rows,
                                              &full[s], mask);
                }
                __syncwarp();
                ++issued;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        bool ok = true;
        int it = 0;
        for (int i = 0; i < my_groups && ok; ++i) {
            const int ab = i & 1, ause = i >> 1;
            if (ause > 0 && !(ok = lmh_warp_wait(&acc_empty[ab], (uint32_t)((ause - 1) & 1),
                                                 abort_flag, p.wait_ns)))
                break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(ab * p.BN);
            for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
                const int s = it % S, use = it / S;
                if (!(ok = lmh_warp_wait(&full[s], (uint32_t)(use & 1), abort_flag, p.wait_ns)))
                    break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a = smem_u32(sA + s * A_BYTES);
                    const uint32_t b = smem_u32(sB + s * b_bytes);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_ss(d, smem_desc_sw128(a + k * 32, 16, 1024),
                                smem_desc_sw128(b + k * 32, 16, 1024), p.idesc,
                                (kb > 0 || k > 0) ? 1u : 0u);
                    if (p.C == 1)
                        umma_commit(&empty[s]);
                    else
                        umma_commit_multicast(&empty[s], mask);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&acc_full[ab]);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        bool ok = true;
        for (int i = 0; i < my_groups && ok; ++i) {
            const int g = cluster_id + i * num_clusters;
            const int mg = g / p.n_tiles, nt = g % p.n_tiles;
            const int m0 = (mg * p.C + (int)rank) * BM;
            const int n0 = nt * p.BN;
            const int ab = i & 1, ause = i >> 1;
            if (!(ok = lmh_warp_wait(&acc_full[ab], (uint32_t)(ause & 1), abort_flag, p.wait_ns)))
                break;
            tc_fence_after();
            const int v = m0 + q * 32 + lane;
            const bool v_ok = v < p.V;
            float *col = p.logits + v;
            for (int c = 0; c < p.BN; c += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + (uint32_t)(ab * p.BN + c), r);
                tmem_wait_ld();
                const int rows_left = p.R - (n0 + c);
                if (v_ok) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < rows_left)
                            col[(size_t)(n0 + c + j) * p.V] = __uint_as_float(r[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
        }
    }

    // ---- leave only when nothing is in flight towards this CTA: every load
    // it issued has landed in every CTA of its cluster, and every commit of
    // every cluster CTA that frees one of this CTA's stages has arrived
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        volatile int never = 0;
        const int last = issued;
        for (int s = 0; s < S && s < last; ++s) {
            const int use = (last - 1 - s) / S;
            mbar_wait_for(&full[s], (uint32_t)(use & 1), &never, kWaitDeadlineNs);
            mbar_wait_for(&empty[s], (uint32_t)(use & 1), &never, kWaitDeadlineNs);
        }
    }
    __syncthreads();
    if (p.C > 1) {
        cluster_arrive();
        cluster_wait();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
    if (threadIdx.x == 0 && *abort_flag && p.status) atomicOr(p.status, SVF_DEV_TIMEOUT);
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 lmh_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [rows, H] bf16, row-major; boxes of 64 columns x box_rows rows, 128-byte swizzle.
static bool make_rows_map(CUtensorMap *map, const void *base, int rows, int H, int box_rows) {
    auto enc = lmh_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static size_t lmh_smem_bytes(int BN, int stages) {
    return 1024 + (size_t)stages * (lmh::A_BYTES + BN * 128) +
           (2 * lmh::MAX_STAGES + 4) * 8 + 16;
}

bool lm_head_supported(int R, int H, int V) {
    return R >= 1 && V >= 1 && H >= 64 && H % 64 == 0 && H <= (1 << 16) && R <= (1 << 24) &&
           V <= (1 << 24);
}

// The tile shape and cluster size for R hidden rows and V vocabulary rows.
static void lmh_config(int R, int V, int *BN, int *C, int *n_tiles) {
    const int nt = (R + lmh::MAX_BN - 1) / lmh::MAX_BN;
    int bn = (R + nt - 1) / nt;
    bn = (bn + 31) / 32 * 32;
    *BN = bn;
    *n_tiles = nt;
    // Many hidden rows make the GEMM compute-bound and the hidden tile is
    // re-read for every weight tile: four CTAs then share it by multicast.
    // Few rows leave it memory-bound on the weight, which each CTA streams.
    const int m_tiles = (V + lmh::BM - 1) / lmh::BM;
    *C = (R >= 512 && bn % (8 * 4) == 0 && m_tiles >= 16) ? 4 : 1;
}

int launch_lm_head(const void *hidden, const void *weight, int R, int H, int V, float *logits,
                   int32_t *status, cudaStream_t stream) {
    if (!lm_head_supported(R, H, V)) return SVF_ERR_UNSUPPORTED;
    int BN, C, n_tiles;
    lmh_config(R, V, &BN, &C, &n_tiles);
    const int stage_bytes = lmh::A_BYTES + BN * 128;
    int stages = lmh::SMEM_BUDGET / stage_bytes;
    if (stages > lmh::MAX_STAGES) stages = lmh::MAX_STAGES;
    CUtensorMap tmw, tmh;
    if (!make_rows_map(&tmw, weight, V, H, lmh::BM) ||
        !make_rows_map(&tmh, hidden, R, H, BN / C))
        return SVF_ERR_LAUNCH;
    LmhParams p;
    p.R = R;
    p.H = H;
    p.V = V;
    p.BN = BN;
    p.C = C;
    p.n_tiles = n_tiles;
    const int m_tiles = (V + lmh::BM - 1) / lmh::BM;
    p.m_groups = (m_tiles + C - 1) / C;
    p.groups = p.m_groups * n_tiles;
    p.kblocks = H / lmh::BK;
    p.stages = stages;
    p.idesc = idesc_bf16_f32(128, BN, false, false);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * BN)) cols <<= 1;
    p.tmem_cols = cols;
    p.wait_ns = kWaitDeadlineNs;
    p.logits = logits;
    p.status = status;
    const size_t smem = lmh_smem_bytes(BN, stages);
    if (cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return SVF_ERR_LAUNCH;
    // persistent: as many CTAs (clusters) as can be resident at once
    int clusters = num_sms() / C;
    if (C > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(C * clusters));
        cfg.blockDim = dim3(lmh::THREADS);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)C;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, lm_head_kernel, &cfg) == cudaSuccess &&
            active > 0 && active < clusters)
            clusters = active;
    }
    if (clusters > p.groups) clusters = p.groups;
    if (clusters < 1) clusters = 1;
    if (launch_pdl(lm_head_kernel, dim3((unsigned)(clusters * C)), dim3(lmh::THREADS), smem,
                   stream, C > 1 ? (unsigned)C : 0u, tmw, tmh, p) != cudaSuccess)
        return SVF_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? SVF_OK : SVF_ERR_LAUNCH;
}

}  // namespace svf
