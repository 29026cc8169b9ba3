// attn_tc_common.cuh -- what the two tensor-core tree-attention kernels share:
// the tile geometry, the warp roles' sizes, the visibility of a tile's columns
// and the TMA descriptors of the K/V cache and of q.
//
// attn_tc.cu runs one CTA per (sequence, KV head, row block, KV chunk) and
// merges the chunks of a unit inside a thread-block cluster; attn_sk.cu runs
// one persistent CTA per SM over an equal share of all units' tiles and
// merges the pieces of a unit split between CTAs through a workspace.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"

namespace svf {

namespace tc {
constexpr int BN = 64;                      // KV tokens per tile
constexpr int HD = 128;                     // head_dim
constexpr int HALF_BYTES = 128 * HD * 2;    // 32 KB of Q per 128-row half
constexpr int Q_COL_BYTES = 128 * 128;      // one 64-dim block of 128 Q rows
constexpr int TILE_BYTES = BN * HD * 2;     // 16 KB per K or V tile
constexpr int KV_COL_BYTES = BN * 128;      // one 64-dim block of a 64-token tile
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int MAX_BOX_ROWS = 64;            // TMA box height (tokens)
// S buffers per row half: 2 x 2 x 64 columns of S plus 2 x 128 of O fill the
// 512 TMEM columns with two halves; one half has room for four.
__host__ __device__ constexpr int sbuffers_for(int NH) { return NH == 1 ? 4 : 2; }
// Warps: a K and a V producer, a QK issuer and a PV issuer per half, four
// softmax warps per half. One thread issuing tcgen05.mma (or TMA copies)
// sustains about one instruction per 100 cycles; several issuing warps
// overlap, so each stream gets its own warp.
__host__ __device__ constexpr int first_softmax_warp(int NH) { return 2 + 2 * NH; }
__host__ __device__ constexpr int threads_for(int NH) { return 32 * (2 + 6 * NH); }
}  // namespace tc

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          unsigned long long ns) {
    const bool ok = mbar_wait_for(bar, parity, abort, ns);
    return __all_sync(0xffffffffu, ok);
}

// Visibility of the 32 columns t = L + off + i (i = 0..31) for a row whose
// ancestor set is `anc`: prefix columns (t < L) are visible, tree column
// L + j is visible iff bit j of anc is set; columns past the tree have no bit.
__device__ __forceinline__ uint32_t visible_bits(long long off, uint64_t anc) {
    if (off <= -32) return 0xffffffffu;
    if (off >= 64) return 0u;
    if (off < 0) {
        const int sh = (int)(-off);
        return ((1u << sh) - 1u) | (uint32_t)(anc << sh);
    }
    return (uint32_t)(anc >> (int)off);
}

// ---------------------------------------------------------------- host side

static inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// K or V cache [num_pages * page_size tokens][Hkv][128] as a 3-D map; boxes
// of 64 dims x 1 head x one page (at most 64 tokens), 128-byte swizzle.
static inline bool make_kv_map(CUtensorMap *map, const void *base, int num_pages, int page_size,
                               int Hkv) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int box_rows = page_size < tc::MAX_BOX_ROWS ? page_size : tc::MAX_BOX_ROWS;
    cuuint64_t dims[3] = {(cuuint64_t)tc::HD, (cuuint64_t)Hkv,
                          (cuuint64_t)num_pages * (cuuint64_t)page_size};
    cuuint64_t strides[2] = {(cuuint64_t)tc::HD * 2, (cuuint64_t)Hkv * tc::HD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// q [B][N][Hq][128] as a 4-D map; a box is 64 dims x G heads x 128/G nodes of
// one sequence: 128 query rows (node, grouped head) of one KV head.
static inline bool make_q_map(CUtensorMap *map, const void *q, int B, int N, int Hq, int G) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)tc::HD, (cuuint64_t)Hq, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)tc::HD * 2, (cuuint64_t)Hq * tc::HD * 2,
                             (cuuint64_t)N * Hq * tc::HD * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Rows per CTA: one half of up to 128 rows, or two halves of up to 256. Two
// halves per CTA beat two one-half CTAs per KV head (which read every K/V
// tile twice, from L2 or by multicast) on this part.
static inline int row_halves(int M) { return M > 128 ? 2 : 1; }

}  // namespace svf
