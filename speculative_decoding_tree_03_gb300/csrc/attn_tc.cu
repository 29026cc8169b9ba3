// attn_tc.cu -- tree attention on the 5th-generation tensor cores (bf16, head_dim 128).
//
// "EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree Verification 详解, A-B:
// one target pass verifies the whole tree; node i sees the cached prefix and
// tree positions L_b + j for j an ancestor of i (or i). The pages size the
// cost as O(N·P) reads of the prefix plus a sparse O(N·avg_depth) tree part
// (D.2), so the kernel is a KV-streaming decode kernel: every query row of one
// (sequence, KV head) -- N nodes x G grouped heads -- shares each K/V tile.
//
// One CTA = (KV split, KV head [x row block], sequence). Roles:
//   warp 0      TMA producer: K and V tiles of 128 tokens, page by page
//               (128-byte swizzle), into a 2-stage ring.
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma:
//                 S_h  = Q_h K^T  (A, B from shared memory, M=128, N=128)
//                 O_h += P_h V    (A = P from tensor memory, B = V MN-major)
//   warps 2..   softmax: one thread per query row (= TMEM lane). Reads S
//               from TMEM, applies the ancestor mask on the tile(s) that
//               reach the tree, keeps a lazily-updated running max (O is
//               rescaled only when the max grows by more than 2^8), writes
//               P as bf16 into the S columns, and finally reads O.
// With more than 128 rows (N*G > 128) the rows form two halves with their own
// S/O accumulators; the halves interleave on the tensor pipe.
//
// Splits of the KV range write normalised partial outputs and their
// log-sum-exp to the workspace; attn_combine_kernel merges them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace svf {

namespace tc {
constexpr int BN = 128;                  // KV tokens per tile
constexpr int HD = 128;                  // head_dim
// Ring depths for K and V tiles (32 KB each). One 128-row half (32 KB of Q)
// fits 3 + 3 stages; two halves (64 KB of Q) fit 5 stages. There K frees as
// soon as the QK^T that reads it completes, early enough for 2 stages, while
// V waits for its PV, the last use of a tile, and gets the third stage.
__host__ __device__ constexpr int kstages_for(int NH) { return NH == 1 ? 3 : 2; }
__host__ __device__ constexpr int vstages_for(int NH) { return 3; }
constexpr int CRING = 16;  // page coordinates kept for tiles ahead of the V ring
constexpr int HALF_BYTES = 128 * HD * 2;  // 32 KB: 128 rows x 128 bf16
constexpr int ATOM_COL_BYTES = 128 * 128;  // one 64-element column block of a 128-row tile
constexpr int TILE_BYTES = BN * HD * 2;   // 32 KB per K or V tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int PREFETCH = 3;               // tiles pulled into L2 ahead of the smem ring
constexpr int MAX_BOX_ROWS = 32;          // TMA box height (tokens) for large pages
}  // namespace tc

struct TcParams {
    const __nv_bfloat16 *q;
    const int32_t *page_table;
    const int32_t *seq_lens;
    const uint64_t *anc;
    int B, N, Hq, Hkv, G, M;
    int num_pages, page_size, max_pages;
    int splits, row_blocks;
    int q_tma;        // 1: Q arrives by TMA (G a power of two <= 128)
    float scale_log2;
    __nv_bfloat16 *out;
    float *lse;
    float *part_o;    // [splits, B, N, Hq, HD]
    float *part_lse;  // [splits, B, N, Hq]
    int32_t *status;
};

template <int NH>
struct TcSmem {
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + NH * tc::HALF_BYTES;
    static constexpr int kKS = tc::kstages_for(NH);
    static constexpr int kVS = tc::vstages_for(NH);
    static constexpr int kV = kK + kKS * tc::TILE_BYTES;
    static constexpr int kBar = kV + kVS * tc::TILE_BYTES;
    static constexpr int kNumBars = 2 * kKS + 2 * kVS + 3 * 2 + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 64;
    static constexpr int kDynamic = kBytes + 1024;  // slack to align the base to 1 KB
};

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, abort);
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

template <int NH>
__global__ void __launch_bounds__(64 + 128 * NH, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmq, TcParams p) {
    using S = TcSmem<NH>;
    using namespace tc;
    constexpr int KS = S::kKS;
    constexpr int VS = S::kVS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + S::kQ;
    uint8_t *sK = smem + S::kK;
    uint8_t *sV = smem + S::kV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint64_t *k_full = bars;
    uint64_t *k_empty = k_full + KS;
    uint64_t *v_full = k_empty + KS;
    uint64_t *v_empty = v_full + VS;
    // S slots: the two row halves (NH = 2), or two buffers of one half (NH = 1)
    uint64_t *s_full = v_empty + VS;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = p_full + 2;
    uint64_t *q_full = o_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *err_flag = reinterpret_cast<int *>(smem + S::kMisc + 8);

    // tensor memory: S slot k at columns [128 k, 128 k + 128), O of half h at
    // [256 + 128 h, ...); P is written over the first 64 columns of its S slot
    constexpr uint32_t kTmemCols = 512;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y / p.row_blocks;
    const int rb = blockIdx.y % p.row_blocks;
    const int b = blockIdx.z;

    const int L = p.seq_lens[b];
    const long long T = (long long)L + p.N;
    const bool len_ok = L >= 0 && T <= (long long)p.max_pages * p.page_size;
    const int ntiles = len_ok ? (int)((T + BN - 1) / BN) : 0;
    const int chunk = (ntiles + p.splits - 1) / p.splits;
    const int j0 = split * chunk;
    const int j1 = min(j0 + chunk, ntiles);

    // Page-table lookup of one tile, one box per lane of the producer warp:
    // the starting slot of box `lane` (a slot past the cache, zero-filled by
    // TMA, for boxes past the sequence or with a page id outside the cache).
    // Every index fits in 32 bits (num_pages * page_size <= INT_MAX).
    const int ps = p.page_size;
    const int box_rows = ps < MAX_BOX_ROWS ? ps : MAX_BOX_ROWS;
    const int boxes = BN / box_rows;
    const int oob = p.num_pages * ps;
    const int Ti = (int)T;
    const int32_t *__restrict__ pt = p.page_table + (size_t)b * p.max_pages;
    auto lane_coord = [&](int j, int &bad) -> int {
        if (lane >= boxes || j >= j1) return oob;
        const int t0 = j * BN + lane * box_rows;
        if (t0 >= Ti) return oob;
        const int page = t0 / ps;
        const int id = __ldg(pt + page);
        if (id < 0 || id >= p.num_pages) {
            bad = 1;
            return oob;
        }
        return id * ps + (t0 - page * ps);
    };
    // Lane 0 issues the K (or V) boxes of one tile into one stage; lane x's
    // coordinate is broadcast by shuffle (all lanes of warp 0 take part).
    auto issue_boxes = [&](const CUtensorMap *map, uint8_t *dst, uint64_t *bar, int my_coord) {
        int cs[BN / 16];
        for (int x = 0; x < boxes; ++x) cs[x] = __shfl_sync(0xffffffffu, my_coord, x);
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, TILE_BYTES);
            for (int x = 0; x < boxes; ++x)
                for (int dh = 0; dh < 2; ++dh)
                    tma_load_3d(dst + dh * ATOM_COL_BYTES + x * box_rows * 128, map, dh * 64, g,
                                cs[x], bar);
        }
    };
    auto prefetch_coord = [&](int c) {
        if (lane < boxes && c != oob) {
            for (int dh = 0; dh < 2; ++dh) {
                tma_prefetch_l2_3d(&tmk, dh * 64, g, c);
                tma_prefetch_l2_3d(&tmv, dh * 64, g, c);
            }
        }
    };
    // page coordinates of upcoming tiles, kept in a ring indexed by tile
    int ring[CRING];
    int bad_pages = 0;
    int filled = j0;  // tiles [j0, filled) have their coordinates in the ring
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k <= PREFETCH; ++k) ring[(j0 + k) % CRING] = lane_coord(j0 + k, bad_pages);
        filled = j0 + PREFETCH + 1;
        const int bad0 = __reduce_or_sync(0xffffffffu, bad_pages);
        if (lane == 0) {
            *err_flag = bad0;
            for (int s2 = 0; s2 < KS; ++s2) {
                mbar_init(&k_full[s2], 1);
                mbar_init(&k_empty[s2], 1);
            }
            for (int s2 = 0; s2 < VS; ++s2) {
                mbar_init(&v_full[s2], 1);
                mbar_init(&v_empty[s2], 1);
            }
            for (int k = 0; k < 2; ++k) {
                mbar_init(&s_full[k], 1);
                mbar_init(&p_full[k], 128);
                mbar_init(&o_done[k], 1);
            }
            mbar_init(q_full, 1);
            *abort_flag = 0;
            mbar_fence_init();
            if (!len_ok) atomicOr(&p.status[b], SVF_DEV_BAD_LENGTH);
            if (j0 < j1 && p.q_tma) {
                // rows (node, head) of this block: box = 64 dims x G heads x 128/G nodes
                mbar_arrive_expect_tx(q_full, NH * HALF_BYTES);
                const int nodes = 128 / p.G;
                for (int hh = 0; hh < NH; ++hh)
                    for (int dh = 0; dh < 2; ++dh)
                        tma_load_4d(sQ + hh * HALF_BYTES + dh * ATOM_COL_BYTES, &tmq, dh * 64,
                                    g * p.G, (rb * NH + hh) * nodes, b, q_full);
            }
        }
        __syncwarp();
        if (j0 < j1) {
            const int c0 = ring[j0 % CRING];
            issue_boxes(&tmk, sK, &k_full[0], c0);
            issue_boxes(&tmv, sV, &v_full[0], c0);
#pragma unroll
            for (int k = 1; k <= PREFETCH; ++k) prefetch_coord(ring[(j0 + k) % CRING]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (!p.q_tma && threadIdx.x >= 64) {
        // Q rows -> shared memory by the softmax threads (K-major, 128-byte
        // swizzle: 16-byte chunk c of row r lands at chunk c ^ (r % 8)).
        const int tid = threadIdx.x - 64;
        constexpr int kIters = 16;
        uint4 v[kIters];
#pragma unroll
        for (int k = 0; k < kIters; ++k) {
            const int idx = tid + k * 128 * NH;
            const int row = idx >> 4, c = idx & 15;
            const int R = rb * 128 * NH + row;
            v[k] = make_uint4(0, 0, 0, 0);
            if (R < p.M) {
                const int node = R / p.G, hq = g * p.G + R % p.G;
                v[k] = *reinterpret_cast<const uint4 *>(
                    p.q + (((size_t)b * p.N + node) * p.Hq + hq) * HD + c * 8);
            }
        }
#pragma unroll
        for (int k = 0; k < kIters; ++k) {
            const int idx = tid + k * 128 * NH;
            const int row = idx >> 4, c = idx & 15;
            const int hh = row >> 7, r = row & 127, dh = c >> 3, c8 = c & 7;
            *reinterpret_cast<uint4 *>(sQ + hh * HALF_BYTES + dh * ATOM_COL_BYTES + r * 128 +
                                       ((c8 ^ (r & 7)) << 4)) = v[k];
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (j0 < j1 && warp == 0) {
        // ------------------------------------------------------------ producer
        // K and V of every tile, each into its own ring as soon as a stage is
        // free (polling both, K first), the page coordinates PREFETCH tiles
        // ahead of the next K tile, and those tiles pulled into L2.
        int kj = j0 + 1, vj = j0 + 1;  // next tiles to issue
        int bad = bad_pages;
        // one page-table load in flight: its coordinate is stored (and its
        // boxes prefetched) at the next K issue, when the load has landed
        int pending_tile = -1, pending = oob;
        unsigned long long t_last = globaltimer_ns();
        while ((kj < j1 || vj < j1) && !*abort_flag) {
            bool progressed = false;
            if (kj < j1) {
                const int it = kj - j0, st = it % KS, use = it / KS;
                bool free_ = use == 0 || mbar_test_wait(&k_empty[st], (use - 1) & 1);
                free_ = __shfl_sync(0xffffffffu, free_, 0);
                if (free_) {
                    issue_boxes(&tmk, sK + st * TILE_BYTES, &k_full[st], ring[kj % CRING]);
                    ++kj;
                    if (pending_tile >= 0) {
                        ring[pending_tile % CRING] = pending;
                        prefetch_coord(pending);
                    }
                    pending_tile = filled;
                    pending = lane_coord(filled, bad);
                    ++filled;
                    progressed = true;
                }
            }
            if (vj < kj && vj < j1) {
                const int it = vj - j0, st = it % VS, use = it / VS;
                bool free_ = use == 0 || mbar_test_wait(&v_empty[st], (use - 1) & 1);
                free_ = __shfl_sync(0xffffffffu, free_, 0);
                if (free_) {
                    issue_boxes(&tmv, sV + st * TILE_BYTES, &v_full[st], ring[vj % CRING]);
                    ++vj;
                    progressed = true;
                }
            }
            if (progressed) {
                t_last = globaltimer_ns();
            } else {
                __nanosleep(64);
                if (globaltimer_ns() - t_last > kWaitDeadlineNs) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
            }
        }
        bad = __reduce_or_sync(0xffffffffu, bad);
        if (lane == 0) {
            if (bad || *err_flag) {
                *err_flag = 1;
                atomicOr(&p.status[b], SVF_DEV_BAD_PAGE);
            }
            // Never leave with copies in flight: wait (bounded, ignoring the
            // abort flag) for the last use of every stage that was loaded.
            volatile int never = 0;
            const int nk = kj - j0, nv = vj - j0;
            for (int st = 0; st < KS && st < nk; ++st)
                mbar_wait(&k_full[st], ((nk - 1 - st) / KS) & 1, &never);
            for (int st = 0; st < VS && st < nv; ++st)
                mbar_wait(&v_full[st], ((nv - 1 - st) / VS) & 1, &never);
            if (p.q_tma) mbar_wait(q_full, 0, &never);
        }
    } else if (j0 < j1 && warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD, false, true);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            // S_slot = Q_h K^T
            auto issue_qk = [&](int stage, int h, int slot) {
                const uint32_t d = tmem + slot * 128;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * ATOM_COL_BYTES + (kk & 3) * 32;
                    umma_ss(d, smem_desc_sw128(aQ + h * HALF_BYTES + off, 16, 1024),
                            smem_desc_sw128(aK + stage * TILE_BYTES + off, 16, 1024), idesc_qk,
                            kk > 0);
                }
                umma_commit(&s_full[slot]);
            };
            // O_h += P_slot V
            auto issue_pv = [&](int stage, int h, int slot, bool first) {
                const uint32_t d = tmem + 256 + h * 128;
                const uint32_t a = tmem + slot * 128;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_ts(d, a + kk * 8,
                            smem_desc_sw128(aV + stage * TILE_BYTES + kk * 2048, ATOM_COL_BYTES,
                                            1024),
                            idesc_pv, (!first || kk > 0) ? 1u : 0u);
                umma_commit(&o_done[slot]);
            };
            auto kst = [&](int it) { return it % KS; };
            auto kph = [&](int it) { return (uint32_t)((it / KS) & 1); };
            auto vst = [&](int it) { return it % VS; };
            auto vph = [&](int it) { return (uint32_t)((it / VS) & 1); };
            bool ok = !p.q_tma || mbar_wait(q_full, 0, abort_flag);
            if (NH == 2) {
                // Ping-pong: PV(h0, j), QK(h0, j+1), PV(h1, j), QK(h1, j+1), so
                // one half's softmax overlaps the other half's MMAs. A slot's S
                // (and the P written over it) is reused only after its PV is done.
                ok = ok && mbar_wait(&k_full[kst(0)], kph(0), abort_flag);
                if (ok) {
                    tc_fence_after();
                    issue_qk(kst(0), 0, 0);
                    issue_qk(kst(0), 1, 1);
                    umma_commit(&k_empty[kst(0)]);
                }
                for (int j = j0; ok && j < j1; ++j) {
                    const int it = j - j0;
                    const bool more = j + 1 < j1;
                    if (!(ok = mbar_wait(&v_full[vst(it)], vph(it), abort_flag))) break;
                    for (int h = 0; h < 2 && ok; ++h) {
                        if (!(ok = mbar_wait(&p_full[h], it & 1, abort_flag))) break;
                        tc_fence_after();
                        issue_pv(vst(it), h, h, it == 0);
                        if (h == 1) umma_commit(&v_empty[vst(it)]);
                        if (more) {
                            if (h == 0 &&
                                !(ok = mbar_wait(&k_full[kst(it + 1)], kph(it + 1), abort_flag)))
                                break;
                            if (!(ok = mbar_wait(&o_done[h], it & 1, abort_flag))) break;
                            tc_fence_after();
                            issue_qk(kst(it + 1), h, h);
                            if (h == 1) umma_commit(&k_empty[kst(it + 1)]);
                        }
                    }
                }
            } else {
                // One half, S double-buffered: QK(j + 2) goes into the slot PV(j)
                // has just finished reading, while the softmax works on tile j + 1.
                for (int k = 0; k < 2 && ok && j0 + k < j1; ++k) {
                    if (!(ok = mbar_wait(&k_full[kst(k)], kph(k), abort_flag))) break;
                    tc_fence_after();
                    issue_qk(kst(k), 0, k);
                    umma_commit(&k_empty[kst(k)]);
                }
                for (int j = j0; ok && j < j1; ++j) {
                    const int it = j - j0, slot = it & 1;
                    const uint32_t sph = (uint32_t)((it >> 1) & 1);
                    if (!(ok = mbar_wait(&v_full[vst(it)], vph(it), abort_flag))) break;
                    if (!(ok = mbar_wait(&p_full[slot], sph, abort_flag))) break;
                    tc_fence_after();
                    issue_pv(vst(it), 0, slot, it == 0);
                    umma_commit(&v_empty[vst(it)]);
                    if (j + 2 < j1) {
                        if (!(ok = mbar_wait(&k_full[kst(it + 2)], kph(it + 2), abort_flag)))
                            break;
                        if (!(ok = mbar_wait(&o_done[slot], sph, abort_flag))) break;
                        tc_fence_after();
                        issue_qk(kst(it + 2), 0, slot);
                        umma_commit(&k_empty[kst(it + 2)]);
                    }
                }
            }
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ softmax
        const int h = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int R = rb * 128 * NH + h * 128 + r;
        const bool row_valid = R < p.M;
        const int node = row_valid ? R / p.G : 0;
        const int hq = g * p.G + (row_valid ? R % p.G : 0);
        const uint64_t anc = row_valid ? p.anc[(size_t)b * p.N + node] : 0ull;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + 256 + h * 128;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = j0; j < j1; ++j) {
            const int it = j - j0, s = it % VS, use = it / VS;
            // S slot of this tile and the parity of its barriers
            const int slot = NH == 2 ? h : (it & 1);
            const uint32_t sph = NH == 2 ? (uint32_t)(it & 1) : (uint32_t)((it >> 1) & 1);
            const uint32_t tS = tmem + lane_off + slot * 128;
            if (!(ok = warp_wait(&s_full[slot], sph, abort_flag))) break;
            tc_fence_after();
            const long long tbase = (long long)j * BN;
            const bool masked_tile = tbase + BN > L;  // this tile reaches the tree
            // pass 1: row max of the visible scores, two 64-column halves
            float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll 1
            for (int c64 = 0; c64 < 2; ++c64) {
                uint32_t v[64];
                tmem_ld32(tS + c64 * 64, v);
                tmem_ld32(tS + c64 * 64 + 32, v + 32);
                tmem_wait_ld();
                if (masked_tile) {
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const uint32_t vis = visible_bits(tbase + 64 * c64 + 32 * c2 - L, anc);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            v[32 * c2 + c] = ((vis >> c) & 1u) ? v[32 * c2 + c] : 0xff800000u;
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    m0 = fmaxf(m0, __uint_as_float(v[c]));
                    m1 = fmaxf(m1, __uint_as_float(v[c + 1]));
                    m2 = fmaxf(m2, __uint_as_float(v[c + 2]));
                    m3 = fmaxf(m3, __uint_as_float(v[c + 3]));
                }
            }
            const float mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sl2;
            // lazy rescale: move the reference max only when it grows by > 2^8
            const bool need = mx > m_ref + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ex2_approx(m_ref - mx) : 1.0f;
                if (need) {
                    l *= alpha;
                    m_ref = mx;
                }
                if (it > 0) {
                    if (NH == 1) {
                        // O is being accumulated by PV(j - 1) on the other slot
                        const int pit = it - 1;
                        if (!(ok = warp_wait(&o_done[pit & 1], (uint32_t)((pit >> 1) & 1),
                                             abort_flag)))
                            break;
                        tc_fence_after();
                    }
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t o[32];
                        tmem_ld32(tO + c4 * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(tO + c4 * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            // pass 2: P = 2^(s*scale - m_ref) as bf16 pairs; the 32 packed
            // columns of half c64 go over S columns [32 c64, 32 c64 + 32),
            // which pass 2 has already read
            const float mneg = m_ref == -INFINITY ? 0.0f : -m_ref;
            float r0 = 0.0f, r1 = 0.0f;
#pragma unroll 1
            for (int c64 = 0; c64 < 2; ++c64) {
                uint32_t v[64];
                tmem_ld32(tS + c64 * 64, v);
                tmem_ld32(tS + c64 * 64 + 32, v + 32);
                tmem_wait_ld();
                if (masked_tile) {
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const uint32_t vis = visible_bits(tbase + 64 * c64 + 32 * c2 - L, anc);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            v[32 * c2 + c] = ((vis >> c) & 1u) ? v[32 * c2 + c] : 0xff800000u;
                    }
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(v[2 * c]), sl2, mneg));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(v[2 * c + 1]), sl2, mneg));
                    r0 += p0;
                    r1 += p1;
                    v[c] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tS + c64 * 32, v);
            }
            tmem_wait_st();
            l += r0 + r1;
            // V rows past the sequence end may hold anything: zero them before PV.
            if (h == 0 && tbase + BN > T) {
                if (!(ok = warp_wait(&v_full[s], use & 1, abort_flag))) break;
                if (tbase + r >= T) {
                    uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int dh = 0; dh < 2; ++dh)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4 *>(sV + s * TILE_BYTES + dh * ATOM_COL_BYTES +
                                                       r * 128 + c * 16) = z;
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&p_full[slot]);
        }
        // epilogue
        if (ok && j0 < j1) {
            const int lit = j1 - j0 - 1;  // the last PV of this half
            ok = NH == 2 ? warp_wait(&o_done[h], (uint32_t)(lit & 1), abort_flag)
                         : warp_wait(&o_done[lit & 1], (uint32_t)((lit >> 1) & 1), abort_flag);
        }
        tc_fence_after();
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const float lse_v =
            l > 0.0f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        const size_t row = ((size_t)b * p.N + node) * p.Hq + hq;
#pragma unroll 1
        for (int c64 = 0; c64 < 2; ++c64) {
            uint32_t o[64];
            if (j0 < j1 && ok) {
                tmem_ld32(tO + c64 * 64, o);
                tmem_ld32(tO + c64 * 64 + 32, o + 32);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) o[c] = 0;
            }
            if (row_valid) {
                if (p.splits == 1) {
                    uint4 *op = reinterpret_cast<uint4 *>(p.out + row * HD + c64 * 64);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
                        op[k] = w;
                    }
                } else {
                    float4 *op = reinterpret_cast<float4 *>(
                        p.part_o + ((size_t)split * p.B * p.N * p.Hq + row) * HD + c64 * 64);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        op[k] = make_float4(__uint_as_float(o[4 * k + 0]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                            __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
                }
            }
        }
        if (row_valid) {
            if (p.splits == 1) {
                if (p.lse) p.lse[row] = (j0 < j1) ? lse_v : 0.0f;
            } else {
                p.part_lse[(size_t)split * p.B * p.N * p.Hq + row] = (j0 < j1) ? lse_v : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&p.status[b], SVF_DEV_TIMEOUT);
    // With a single split this CTA wrote final outputs: a sequence with a bad
    // page gets zeros (every CTA of the sequence saw the same page table).
    if (p.splits == 1 && *err_flag && warp >= 2) {
        const int h = (warp - 2) >> 2;
        const int R = rb * 128 * NH + h * 128 + (warp & 3) * 32 + lane;
        if (R < p.M) {
            const size_t row = ((size_t)b * p.N + R / p.G) * p.Hq + g * p.G + R % p.G;
            uint4 z = make_uint4(0, 0, 0, 0);
            for (int k = 0; k < HD / 8; ++k)
                *reinterpret_cast<uint4 *>(p.out + row * HD + 8 * k) = z;
            if (p.lse) p.lse[row] = 0.0f;
        }
    }
}

// Merge split partials: lse = log sum_s e^{lse_s}, out = sum_s e^{lse_s - lse} o_s.
// One warp per (sequence, node, head) row; lane s holds split s's lse (and
// s + 32's), and the partial rows are loaded eight splits at a time so their
// latencies overlap. A sequence with any status bit set gets zeros.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float *__restrict__ part_o,
                                                           const float *__restrict__ part_lse,
                                                           int splits, long long rows, int per_b,
                                                           const int32_t *__restrict__ status,
                                                           __nv_bfloat16 *__restrict__ out,
                                                           float *__restrict__ lse) {
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int b = (int)(row / per_b);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse_out = 0.0f;
    if (status[b] == 0) {
        const float l0 = lane < splits ? part_lse[(size_t)lane * rows + row] : -INFINITY;
        const float l1 = lane + 32 < splits ? part_lse[(size_t)(lane + 32) * rows + row] : -INFINITY;
        const float mx = warp_max(fmaxf(l0, l1));
        if (mx != -INFINITY) {
            const float w0 = l0 == -INFINITY ? 0.0f : expf(l0 - mx);
            const float w1 = l1 == -INFINITY ? 0.0f : expf(l1 - mx);
            const float wsum = warp_sum(w0 + w1);
            for (int s0 = 0; s0 < splits; s0 += 8) {
                float4 o[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    o[k] = s0 + k < splits
                               ? *reinterpret_cast<const float4 *>(
                                     part_o + ((size_t)(s0 + k) * rows + row) * 128 + lane * 4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int sidx = s0 + k;
                    const float wa = __shfl_sync(0xffffffffu, w0, sidx & 31);
                    const float wb = __shfl_sync(0xffffffffu, w1, sidx & 31);
                    const float w = sidx < 32 ? wa : wb;
                    acc.x = fmaf(w, o[k].x, acc.x);
                    acc.y = fmaf(w, o[k].y, acc.y);
                    acc.z = fmaf(w, o[k].z, acc.z);
                    acc.w = fmaf(w, o[k].w, acc.w);
                }
            }
            const float inv = 1.0f / wsum;
            acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
            lse_out = mx + logf(wsum);
        }
    }
    uint2 w;
    w.x = pack_bf16x2(acc.x, acc.y);
    w.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2 *>(out + (size_t)row * 128 + lane * 4) = w;
    if (lse && lane == 0) lse[row] = lse_out;
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

static bool make_kv_map(CUtensorMap *map, const void *base, int num_pages, int page_size, int Hkv) {
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

static bool make_q_map(CUtensorMap *map, const void *q, int B, int N, int Hq, int G) {
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

static int row_halves(int M) { return M > 128 ? 2 : 1; }

int attn_tc_splits(int B, int N, int Hq, int Hkv, int max_pages, int page_size) {
    const int G = Hq / Hkv;
    const int M = N * G;
    const int NH = row_halves(M);
    const int row_blocks = (M + 128 * NH - 1) / (128 * NH);
    const long long units = (long long)B * Hkv * row_blocks;
    const long long kv_max = (long long)max_pages * page_size;
    const int tiles = (int)((kv_max + tc::BN - 1) / tc::BN);
    const int C = num_sms();
    // partial output write + read per split and unit, in units of one KV tile
    const double part_tiles = (double)(128 * NH) * (tc::HD + 1) * 4 * 2 / (2.0 * tc::TILE_BYTES);
    double best = 1e300;
    int best_s = 1;
    const int smax = tiles < 64 ? tiles : 64;
    for (int s = 1; s <= smax; ++s) {
        const long long waves = (units * s + C - 1) / C;
        const int per_cta = (tiles + s - 1) / s;
        const double t_chain = (double)waves * (per_cta + 1.0) + (s > 1 ? 0.5 : 0.0);
        const double t_bytes = (double)units * (tiles + (s > 1 ? s * part_tiles : 0.0)) / C;
        const double t = t_chain > t_bytes ? t_chain : t_bytes;
        if (t < best - 1e-9) {
            best = t;
            best_s = s;
        }
    }
    return best_s;
}

size_t attn_tc_workspace_bytes(int B, int N, int Hq, int Hkv, int max_pages, int page_size) {
    const int s = attn_tc_splits(B, N, Hq, Hkv, max_pages, page_size);
    if (s <= 1) return 0;
    const size_t rows = (size_t)B * N * Hq;
    return (size_t)s * rows * (tc::HD + 1) * sizeof(float) + 256;
}

int launch_attn_tc(const AttnArgs &a, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    const int G = a.Hq / a.Hkv;
    const int M = a.N * G;
    const int NH = row_halves(M);
    const int row_blocks = (M + 128 * NH - 1) / (128 * NH);
    const int splits = attn_tc_splits(a.B, a.N, a.Hq, a.Hkv, a.max_pages, a.page_size);
    const size_t need = attn_tc_workspace_bytes(a.B, a.N, a.Hq, a.Hkv, a.max_pages, a.page_size);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return SVF_ERR_WORKSPACE;

    CUtensorMap tmk, tmv, tmq;
    if (!make_kv_map(&tmk, a.k_cache, a.num_pages, a.page_size, a.Hkv) ||
        !make_kv_map(&tmv, a.v_cache, a.num_pages, a.page_size, a.Hkv))
        return SVF_ERR_LAUNCH;
    // Q by TMA when a box of 128 rows is G heads x 128/G nodes
    const bool q_tma = G <= 128 && (G & (G - 1)) == 0;
    if (q_tma) {
        if (!make_q_map(&tmq, a.q, a.B, a.N, a.Hq, G)) return SVF_ERR_LAUNCH;
    } else {
        memset(&tmq, 0, sizeof(tmq));
    }

    TcParams p;
    p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    p.page_table = a.page_table;
    p.seq_lens = a.seq_lens;
    p.anc = a.anc;
    p.B = a.B; p.N = a.N; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.M = M;
    p.num_pages = a.num_pages; p.page_size = a.page_size; p.max_pages = a.max_pages;
    p.splits = splits;
    p.row_blocks = row_blocks;
    p.q_tma = q_tma ? 1 : 0;
    const float scale = a.sm_scale > 0.0f ? a.sm_scale : 1.0f / sqrtf((float)a.D);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    const size_t rows = (size_t)a.B * a.N * a.Hq;
    if (splits > 1) {
        uintptr_t base = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~(uintptr_t)255;
        p.part_o = reinterpret_cast<float *>(base);
        p.part_lse = p.part_o + (size_t)splits * rows * tc::HD;
    } else {
        p.part_o = nullptr;
        p.part_lse = nullptr;
    }
    p.status = a.status;

    dim3 grid(splits, a.Hkv * row_blocks, a.B);
    if (NH == 1) {
        const int smem = TcSmem<1>::kDynamic;
        cudaFuncSetAttribute(attn_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        attn_tc_kernel<1><<<grid, 64 + 128, smem, stream>>>(tmk, tmv, tmq, p);
    } else {
        const int smem = TcSmem<2>::kDynamic;
        cudaFuncSetAttribute(attn_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        attn_tc_kernel<2><<<grid, 64 + 256, smem, stream>>>(tmk, tmv, tmq, p);
    }
    if (cudaGetLastError() != cudaSuccess) return SVF_ERR_LAUNCH;
    if (splits > 1) {
        const long long threads = (long long)rows * 32;
        const int blocks = (int)((threads + 255) / 256);
        attn_combine_kernel<<<blocks, 256, 0, stream>>>(
            p.part_o, p.part_lse, splits, (long long)rows, a.N * a.Hq, a.status, p.out, a.lse);
        if (cudaGetLastError() != cudaSuccess) return SVF_ERR_LAUNCH;
    }
    return SVF_OK;
}

}  // namespace svf
