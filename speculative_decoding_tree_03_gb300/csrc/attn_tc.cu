// attn_tc.cu -- tree attention on the 5th-generation tensor cores (bf16, head_dim 128).
//
// "EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree Verification 详解, A-B:
// one target pass verifies the whole tree; node i sees the cached prefix and
// tree positions L_b + j for j an ancestor of i (or i). The pages size the
// cost as O(N·P) reads of the prefix plus a sparse O(N·avg_depth) tree part
// (D.2), so the kernel is a KV-streaming decode kernel: every query row of one
// (sequence, KV head) -- N nodes x G grouped heads -- shares each K/V tile.
//
// One CTA = (KV head [x row block], KV chunk, sequence); up to 128 rows form
// one half (NH = 1), up to 256 rows two halves (NH = 2). Roles:
//   warps 0, 1    producers of K (warp 0) and V (warp 1): tiles of 64
//                 tokens, one TMA box per page (64 tokens at most) and
//                 64-dim half, 128-byte swizzle, issued by several lanes at
//                 once into two rings. Every box's coordinate is computed
//                 once, at kernel start, into shared memory. The V producer
//                 also zeroes V rows past the sequence end in the last tile.
//   warp 2 + h    QK issuer of half h: S_h,b = Q_h K^T (A, B from shared
//                 memory, M=128, N=64) into S buffer b = tile mod SB, once
//                 the PV that read that buffer is done. Warp 2 also owns the
//                 tensor-memory allocation.
//   warp 2+NH+h   PV issuer of half h: O_h += P_h,b V (A = P from tensor
//                 memory, B = V MN-major) once the softmax wrote P.
//                 A thread issuing tcgen05.mma sustains about one MMA per 100
//                 cycles; separate issuing warps overlap, so every chain gets
//                 its own.
//   4 warps per h softmax: one thread per query row (= TMEM lane). Reads the
//                 64 S columns of a tile, applies the ancestor mask on the
//                 tiles that reach the tree, keeps a lazily-updated running
//                 max (O is rescaled only when the max grows by more than
//                 2^8), writes P as bf16 over the first 32 S columns, and
//                 finally reads O.
//
// Chunks of the KV range: the S CTAs of one (sequence, KV head, row block)
// form a thread-block cluster; each takes an equal share of that sequence's
// own tiles (from seq_lens, not from the page-table capacity). At the end
// they merge through distributed shared memory: every CTA writes its rows'
// log-sum-exp and normalised partial O rows into its own shared memory, one
// cluster barrier publishes them, and each CTA merges a share of the rows
// from the whole cluster (remote loads issued together) and writes the
// final bf16 output. Nothing goes through global memory and no second
// kernel runs.
#include <string.h>

#include <atomic>

#include "attn_tc_common.cuh"
#include "internal.h"

namespace svf {

namespace tc {
constexpr int CMAX_TILES = 256;             // tiles of one CTA (coordinates in smem)
constexpr int MAX_BOXES = CMAX_TILES * (BN / 16);
// K/V ring depths: two halves of Q (64 KB) leave room for 9 stages of 16 KB,
// one half for 11. A V stage is held two tiles longer than a K stage (its PV
// comes after the next tile's QK), so V gets the extra stage.
__host__ __device__ constexpr int kstages_for(int NH) { return NH == 1 ? 5 : 4; }
__host__ __device__ constexpr int vstages_for(int NH) { return NH == 1 ? 6 : 5; }
constexpr int kFixedTiles = 3;              // prologue + epilogue cost, in tiles
constexpr float kMergeTiles = 1.5f;         // the in-cluster merge, in tiles
constexpr int kMaxSplits = 8;               // cluster size (portable limit)
constexpr int kMinChunkTiles = 4;           // smallest chunk worth a cluster
}  // namespace tc

struct TcParams {
    const __nv_bfloat16 *q;
    const int32_t *page_table;
    const int32_t *seq_lens;
    const uint64_t *anc;
    int B, N, Hq, Hkv, G, M;
    int num_pages, page_size, max_pages;
    int splits, row_blocks;  // splits: CTAs per cluster, one chunk each
    int q_tma;        // 1: Q arrives by TMA (G a power of two <= 128)
    float scale_log2;
    unsigned long long wait_ns;  // deadline of every wait but the final drains
    __nv_bfloat16 *out;
    float *lse;
    int32_t *status;
    const int32_t *parent;  // non-null: build the ancestor masks here (N <= 64)
    uint64_t *anc_out;      // with parent: the masks written out (nullable)
    int32_t *depth_out;     // nullable
    int32_t *mask_status;   // nullable
};

template <int NH>
struct TcSmem {
    static constexpr int kKS = tc::kstages_for(NH);
    static constexpr int kVS = tc::vstages_for(NH);
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + NH * tc::HALF_BYTES;
    static constexpr int kV = kK + kKS * tc::TILE_BYTES;
    static constexpr int kCrd = kV + kVS * tc::TILE_BYTES;
    static constexpr int kBar = kCrd + tc::MAX_BOXES * 4;
    static constexpr int kNumBars = 2 * kKS + 2 * kVS + 4 * NH * tc::sbuffers_for(NH) + 2 + 2 * NH;
    static constexpr int kMisc = kBar + kNumBars * 8;
    // merge: per-row log2-sum-exp of this CTA, merged value, contributing CTAs
    static constexpr int kLse = kMisc + 64;
    static constexpr int kFin = kLse + 128 * NH * 4;
    static constexpr int kMask = kFin + 128 * NH * 4;
    // ancestor masks and parent[] of the sequence when built here (N <= 64)
    static constexpr int kAnc = kMask + 128 * NH * 4;
    static constexpr int kBytes = kAnc + 64 * 8 + 64 * 4;
    // weighted O rows of the merge reuse the K/V rings (free by then)
    static_assert(kCrd - kK >= 128 * NH * tc::HD * 4, "merge rows fit in the rings");
    static constexpr int kDynamic = kBytes + 1024;  // slack to align the base to 1 KB
    static_assert(kDynamic <= 227 * 1024, "shared memory budget");
};

template <int NH>
__global__ void __launch_bounds__(tc::threads_for(NH), 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmq, TcParams p) {
    using S = TcSmem<NH>;
    using namespace tc;
    constexpr int KS = S::kKS;
    constexpr int VS = S::kVS;
    constexpr int NTHREADS = threads_for(NH);
    constexpr int SB = sbuffers_for(NH);
    static_assert(NH * SB * BN + NH * 128 <= 512, "tensor memory budget");
    constexpr int SW0 = first_softmax_warp(NH);
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + S::kQ;
    uint8_t *sK = smem + S::kK;
    uint8_t *sV = smem + S::kV;
    int32_t *crd = reinterpret_cast<int32_t *>(smem + S::kCrd);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint64_t *k_full = bars;
    uint64_t *k_empty = k_full + KS;
    uint64_t *v_full = k_empty + KS;
    uint64_t *v_empty = v_full + VS;
    uint64_t *s_full = v_empty + VS;      // [NH][SB]: QK of the tile in S buffer b done
    uint64_t *p_full = s_full + NH * SB;  // [NH][SB]: P of the tile written over S buffer b
    uint64_t *o_done = p_full + NH * SB;  // [NH][SB]: PV that read S buffer b done
    uint64_t *p_half = o_done + NH * SB;  // [NH][SB]: first half of that P written
    uint64_t *q_full = p_half + NH * SB;
    uint64_t *v_tail = q_full + 1;       // last V tile with its rows past the end zeroed
    uint64_t *mma_drain = v_tail + 1;    // [2 NH]: an issuer's MMAs done, after an abort
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *m_flag = reinterpret_cast<int *>(smem + S::kMisc + 16);  // merge: [ok, bad, zero]
    float *s_lse = reinterpret_cast<float *>(smem + S::kLse);   // [128 NH] log2-sum-exp
    float *s_fin = reinterpret_cast<float *>(smem + S::kFin);   // [128 NH] merged
    uint32_t *s_mask = reinterpret_cast<uint32_t *>(smem + S::kMask);  // contributing CTAs

    // tensor memory: S buffer (h, b) at columns [64 (SB h + b), +64); O of
    // half h at [256 + 128 h, +128); P goes over the first 32 columns of its S
    constexpr uint32_t kTmemCols = 512;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // KV heads vary fastest: the CTAs of one token range start together, so
    // the heads' slices of each token row are read from DRAM close in time
    const int g = blockIdx.x / p.row_blocks;
    const int rb = blockIdx.x % p.row_blocks;
    const int split = blockIdx.y;
    const int b = blockIdx.z;
    // One CTA per sequence owns its status word and stores it whole; other
    // CTAs only add SVF_DEV_TIMEOUT, which takes seconds to arise.
    const bool designated = g == 0 && rb == 0 && split == 0;
    if (!cluster_shape_is(1u, p.splits > 1 ? (uint32_t)p.splits : 1u, 1u)) {
        // not the cluster the merge addresses (the chunks of one unit along
        // y): the whole cluster leaves at once, touching no peer
        pdl_wait();
        if (threadIdx.x == 0) atomicOr(&p.status[b], SVF_DEV_BAD_CLUSTER);
        return;
    }
    // On-chip set-up first: it overlaps the previous kernel's tail.
    if (threadIdx.x == 0) {
        for (int s2 = 0; s2 < KS; ++s2) {
            mbar_init(&k_full[s2], 1);
            mbar_init(&k_empty[s2], NH);
        }
        for (int s2 = 0; s2 < VS; ++s2) {
            mbar_init(&v_full[s2], 1);
            mbar_init(&v_empty[s2], NH);
        }
        for (int k = 0; k < NH * SB; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 128);
            mbar_init(&o_done[k], 1);
            mbar_init(&p_half[k], 128);
        }
        mbar_init(q_full, 1);
        mbar_init(v_tail, 1);
        for (int k = 0; k < 2 * NH; ++k) mbar_init(&mma_drain[k], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1 && lane == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        if (p.q_tma) tma_prefetch_desc(&tmq);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_launch_dependents();

    uint64_t *s_anc = reinterpret_cast<uint64_t *>(smem + S::kAnc);
    if (p.parent) {
        // "EAGLE 演化史", § Tree Verification 详解, B: node i sees its
        // ancestors and itself. parent[] of the sequence into shared memory
        // with the tree check, then each thread walks one node's parent links
        // to the root (parent[i] < i bounds the walk). An invalid tree gives
        // every node only its own bit, as svf_tree_mask_build does. One CTA
        // per sequence writes the masks, depths and mask status out.
        int32_t *s_par = reinterpret_cast<int32_t *>(s_anc + 64);
        const int i = threadIdx.x;
        int badt = 0;
        if (i < p.N) {
            const int pp = p.parent[(size_t)b * p.N + i];
            s_par[i] = pp;
            badt = i == 0 ? pp != -1 : (pp < 0 || pp >= i);
        }
        badt = __syncthreads_or(badt);
        if (i < p.N) {
            uint64_t word = 1ull << i;
            int d = 0;
            if (!badt) {
                d = -1;
                word = 0;
                for (int a = i; a != -1; a = s_par[a]) {
                    word |= 1ull << a;
                    ++d;
                }
            }
            s_anc[i] = word;
            if (designated) {
                if (p.anc_out) p.anc_out[(size_t)b * p.N + i] = word;
                if (p.depth_out) p.depth_out[(size_t)b * p.N + i] = d;
            }
        }
        if (designated && i == 0 && p.mask_status)
            p.mask_status[b] = badt ? SVF_DEV_BAD_PARENT : 0;
        __syncthreads();
    }

    const int L = p.seq_lens[b];
    const long long T = (long long)L + p.N;
    const bool len_ok = L >= 0 && T <= (long long)p.max_pages * p.page_size;
    const int ntiles = len_ok ? (int)((T + BN - 1) / BN) : 0;
    // this sequence's tiles in equal shares over the cluster's CTAs
    const int chunk = (ntiles + p.splits - 1) / p.splits;
    const int j0 = split * chunk;
    const int j1 = min(j0 + chunk, ntiles);
    const int n = j1 - j0;
    if (n <= 0 && p.splits == 1) {
        // No tile here. The first chunk reports a bad length; with a single
        // chunk this CTA owns final outputs, which are zeros then.
        tc_fence_before();
        __syncthreads();
        if (warp == 2) {
            tc_fence_after();
            tmem_dealloc(*tmem_slot, kTmemCols);
        }
        if (designated && threadIdx.x == 0) p.status[b] = SVF_DEV_BAD_LENGTH;
        if (p.splits == 1 && threadIdx.x < 128 * NH) {
            const int R = rb * 128 * NH + threadIdx.x;
            if (R < p.M) {
                const size_t row = ((size_t)b * p.N + R / p.G) * p.Hq + g * p.G + R % p.G;
                const uint4 z = make_uint4(0, 0, 0, 0);
                for (int k = 0; k < HD / 8; ++k)
                    *reinterpret_cast<uint4 *>(p.out + row * HD + 8 * k) = z;
                if (p.lse) p.lse[row] = 0.0f;
            }
        }
        return;
    }

    int bad = 0;
    const uint32_t tmem = *tmem_slot;
    if (n <= 0) {
        // an empty chunk of a cluster: it only takes part in the merge; the
        // first chunk is never empty unless the length is bad
        if (designated && threadIdx.x == 0) p.status[b] = SVF_DEV_BAD_LENGTH;
        if (warp >= SW0) s_lse[threadIdx.x - 32 * SW0] = -INFINITY;
        tc_fence_before();
        __syncthreads();
    } else {
    // ---- set-up: barriers, Q, tensor memory, box coordinates
    const int ps = p.page_size;
    const int box_rows = ps < MAX_BOX_ROWS ? ps : MAX_BOX_ROWS;
    const int bpt = BN / box_rows;  // TMA boxes per tile and 64-dim half
    if (threadIdx.x == 0) {
        if (p.q_tma) {
            // rows (node, head) of this block: box = 64 dims x G heads x 128/G nodes
            mbar_arrive_expect_tx(q_full, NH * HALF_BYTES);
            const int nodes = 128 / p.G;
            for (int hh = 0; hh < NH; ++hh)
                for (int dh = 0; dh < 2; ++dh)
                    tma_load_4d(sQ + hh * HALF_BYTES + dh * Q_COL_BYTES, &tmq, dh * 64, g * p.G,
                                (rb * NH + hh) * nodes, b, q_full);
        }
    }
    if (!p.q_tma && warp >= SW0) {
        // Q rows -> shared memory by the softmax threads (K-major, 128-byte
        // swizzle: 16-byte chunk c of row r lands at chunk c ^ (r % 8)).
        const int tid = threadIdx.x - 32 * SW0;
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
            *reinterpret_cast<uint4 *>(sQ + hh * HALF_BYTES + dh * Q_COL_BYTES + r * 128 +
                                       ((c8 ^ (r & 7)) << 4)) = v[k];
        }
        fence_proxy_async_smem();
    }
    // Starting slot of every box of this chunk: a slot past the cache (which
    // TMA fills with zeros) for boxes past the sequence or with a page id
    // outside the cache. Every index fits in 32 bits (num_pages * page_size
    // <= INT_MAX).
    int bad_seq = 0;
    {
        const int oob = p.num_pages * ps;
        const int32_t *__restrict__ pt = p.page_table + (size_t)b * p.max_pages;
        if (designated) {
            // every page the sequence uses, for its status word
            const int npg = (int)((T + ps - 1) / ps);
            for (int i = threadIdx.x; i < npg; i += NTHREADS) {
                const int id = __ldg(pt + i);
                if (id < 0 || id >= p.num_pages) bad_seq = 1;
            }
        }
        for (int idx = threadIdx.x; idx < n * bpt; idx += NTHREADS) {
            const long long t0 = (long long)(j0 + idx / bpt) * BN + (idx % bpt) * box_rows;
            int c = oob;
            if (t0 < T) {
                const int page = (int)(t0 / ps);
                const int id = __ldg(pt + page);
                if (id < 0 || id >= p.num_pages) bad = 1;
                else c = id * ps + (int)(t0 - (long long)page * ps);
            }
            crd[idx] = c;
        }
    }
    bad_seq = __syncthreads_or(bad_seq);
    if (designated && threadIdx.x == 0) p.status[b] = bad_seq ? SVF_DEV_BAD_PAGE : 0;
    tc_fence_before();
    bad = __syncthreads_or(bad);
    tc_fence_after();

    if (warp <= 1) {
        // ------------------------------------------------------------ producers
        // Warp 0 streams K, warp 1 streams V, each into its ring as soon as a
        // stage is free; lane x < bpt issues box x of both 64-dim halves.
        const bool is_k = warp == 0;
        const CUtensorMap *map = is_k ? &tmk : &tmv;
        uint8_t *ring = is_k ? sK : sV;
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *empty = is_k ? k_empty : v_empty;
        const int stages = is_k ? KS : VS;
        int j = 0;  // tiles issued
        for (; j < n; ++j) {
            const int st = j % stages, use = j / stages;
            if (use > 0 && !warp_wait(&empty[st], (uint32_t)((use - 1) & 1), abort_flag, p.wait_ns)) break;
            if (lane == 0) mbar_arrive_expect_tx(&full[st], TILE_BYTES);
            if (lane < bpt) {
                const int c = crd[j * bpt + lane];
#pragma unroll
                for (int dh = 0; dh < 2; ++dh)
                    tma_load_3d(ring + st * TILE_BYTES + dh * KV_COL_BYTES + lane * box_rows * 128,
                                map, dh * 64, g, c, &full[st]);
            }
            __syncwarp();
        }
        const int kj = is_k ? j : 0, vj = is_k ? 0 : j;
        // V rows past the sequence end may hold anything (NaN included, and
        // P = 0 does not cancel NaN): zero them in the last tile, then let the
        // PV issuers in through v_tail.
        const long long tbl = (long long)(j0 + n - 1) * BN;
        if (!is_k && tbl + BN > T && vj == n) {
            const int jl = n - 1;
            if (warp_wait(&v_full[jl % VS], (uint32_t)((jl / VS) & 1), abort_flag, p.wait_ns)) {
                const int r0 = (int)(T - tbl);
                uint8_t *vs = sV + (jl % VS) * TILE_BYTES;
                for (int idx = lane; idx < (BN - r0) * 16; idx += 32) {
                    const int r = r0 + (idx >> 4), c = idx & 15;
                    *reinterpret_cast<uint4 *>(vs + (c >> 3) * KV_COL_BYTES + r * 128 +
                                               (c & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(v_tail);
            }
        }
        if (lane == 0) {
            // Never leave with copies in flight: wait (bounded, ignoring the
            // abort flag) for the last fill of every stage that was loaded.
            volatile int never = 0;
            for (int st = 0; st < KS && st < kj; ++st)
                mbar_wait_for(&k_full[st], ((kj - 1 - st) / KS) & 1, &never, kWaitDeadlineNs);
            for (int st = 0; st < VS && st < vj; ++st)
                mbar_wait_for(&v_full[st], ((vj - 1 - st) / VS) & 1, &never, kWaitDeadlineNs);
            if (is_k && p.q_tma) mbar_wait_for(q_full, 0, &never, kWaitDeadlineNs);
        }
    } else if (warp <= 1 + NH) {
        // ------------------------------------------------------------ QK issuer, half h
        // S_h,b = Q_h K^T for every tile, into the buffer whose previous PV is done.
        const int h = warp - 2;
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BN, false, false);
        const uint32_t aQ = smem_u32(sQ) + h * HALF_BYTES, aK = smem_u32(sK);
        bool ok = !p.q_tma || warp_wait(q_full, 0, abort_flag, p.wait_ns);
        for (int t = 0; ok && t < n; ++t) {
            const int bb = t % SB;
            if (!(ok = warp_wait(&k_full[t % KS], (uint32_t)((t / KS) & 1), abort_flag, p.wait_ns))) break;
            if (t >= SB) {
                // PV(t - SB) of this half read P from this S buffer
                const int pj = t - SB;
                if (!(ok = warp_wait(&o_done[h * SB + bb], (uint32_t)((pj / SB) & 1), abort_flag, p.wait_ns)))
                    break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t d = tmem + (uint32_t)((h * SB + bb) * BN);
                const uint32_t kst = aK + (t % KS) * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t oq = (kk >> 2) * Q_COL_BYTES + (kk & 3) * 32;
                    const uint32_t ok_ = (kk >> 2) * KV_COL_BYTES + (kk & 3) * 32;
                    umma_ss(d, smem_desc_sw128(aQ + oq, 16, 1024),
                            smem_desc_sw128(kst + ok_, 16, 1024), idesc_qk, kk > 0);
                }
                umma_commit(&s_full[h * SB + bb]);
                umma_commit(&k_empty[t % KS]);
            }
            __syncwarp();
        }
    } else if (warp <= 1 + 2 * NH) {
        // ------------------------------------------------------------ PV issuer, half h
        // O_h += P_h,b V for every tile once its softmax is done.
        const int h = warp - 2 - NH;
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD, false, true);
        const uint32_t aV = smem_u32(sV);
        bool ok = true;
        for (int j = 0; ok && j < n; ++j) {
            const int bb = j % SB;
            const bool tail = (long long)(j0 + j) * BN + BN > T;  // the sequence's last tile
            ok = tail ? warp_wait(v_tail, 0, abort_flag, p.wait_ns)
                      : warp_wait(&v_full[j % VS], (uint32_t)((j / VS) & 1), abort_flag, p.wait_ns);
            if (!ok) break;
            // P arrives in two halves of 32 tokens; the first half's K-steps
            // go in while the softmax still computes the second
            const uint32_t d = tmem + 256 + h * 128;
            const uint32_t a = tmem + (uint32_t)((h * SB + bb) * BN);
            const uint32_t vst = aV + (j % VS) * TILE_BYTES;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint64_t *pb = part == 0 ? &p_half[h * SB + bb] : &p_full[h * SB + bb];
                if (!(ok = warp_wait(pb, (uint32_t)((j / SB) & 1), abort_flag, p.wait_ns))) break;
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int k2 = 0; k2 < BN / 32; ++k2) {
                        const int kk = part * (BN / 32) + k2;
                        umma_ts(d, a + kk * 8, smem_desc_sw128(vst + kk * 2048, KV_COL_BYTES, 1024),
                                idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) {
                umma_commit(&o_done[h * SB + bb]);
                umma_commit(&v_empty[j % VS]);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int h = (warp - SW0) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int R = rb * 128 * NH + h * 128 + r;
        const bool row_valid = R < p.M;
        const int node = row_valid ? R / p.G : 0;
        const int hq = g * p.G + (row_valid ? R % p.G : 0);
        const uint64_t anc =
            row_valid ? (p.parent ? s_anc[node] : p.anc[(size_t)b * p.N + node]) : 0ull;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + 256 + h * 128;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int bb = j % SB;
            const uint32_t bph = (uint32_t)((j / SB) & 1);
            const uint32_t tS = tmem + lane_off + (uint32_t)((h * SB + bb) * BN);
            if (!(ok = warp_wait(&s_full[h * SB + bb], bph, abort_flag, p.wait_ns))) break;
            tc_fence_after();
            uint32_t v[BN];
            tmem_ld32(tS, v);
            tmem_ld32(tS + 32, v + 32);
            tmem_wait_ld();
            const long long tbase = (long long)(j0 + j) * BN;
            if (tbase + BN > L) {
                // this tile reaches the tree: ancestors only
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const uint32_t vis = visible_bits(tbase + 32 * c2 - L, anc);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        v[32 * c2 + c] = ((vis >> c) & 1u) ? v[32 * c2 + c] : 0xff800000u;
                }
            }
            float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 8) {
                m0 = fmax3(m0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
                m1 = fmax3(m1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
                m2 = fmax3(m2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
                m3 = fmax3(m3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
            }
            const float mx = fmax3(m0, m1, fmaxf(m2, m3)) * sl2;
            // lazy rescale: move the reference max only when it grows by > 2^8
            const bool need = mx > m_ref + kRescaleThreshold;
            if (__any_sync(FULL, need)) {
                const float alpha = need ? ex2_approx(m_ref - mx) : 1.0f;
                if (need) {
                    l *= alpha;
                    m_ref = mx;
                }
                if (j > 0) {
                    // O is final up to PV(j - 1) of this half
                    const int pj = j - 1;
                    if (!(ok = warp_wait(&o_done[h * SB + pj % SB], (uint32_t)((pj / SB) & 1),
                                         abort_flag, p.wait_ns)))
                        break;
                    tc_fence_after();
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
            // P = 2^(s*scale - m_ref) as bf16 pairs over the first 32 S
            // columns, in two halves of 32 tokens (the PV issuer starts on the
            // first); even and odd columns are summed in the two lanes of r
            const float mneg = m_ref == -INFINITY ? 0.0f : -m_ref;
            const float2 sc2 = make_float2(sl2, sl2), mn2 = make_float2(mneg, mneg);
            float2 r = make_float2(0.0f, 0.0f);
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                const float2 x = ffma2(make_float2(__uint_as_float(v[2 * c]),
                                                   __uint_as_float(v[2 * c + 1])), sc2, mn2);
                const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                r = fadd2(r, pp);
                pk[c] = pack_bf16x2(pp.x, pp.y);
                if (c == BN / 4 - 1) {
                    tmem_st16(tS, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&p_half[h * SB + bb]);
                }
            }
            tmem_st16(tS + BN / 4, pk + BN / 4);
            tmem_wait_st();
            l += r.x + r.y;
            tc_fence_before();
            mbar_arrive(&p_full[h * SB + bb]);
        }
        // epilogue: O of this half after its last PV
        if (ok) ok = warp_wait(&o_done[h * SB + (n - 1) % SB], (uint32_t)(((n - 1) / SB) & 1),
                               abort_flag, p.wait_ns);
        tc_fence_after();
        if (p.splits > 1) {
            // the merge reads O from tensor memory later; publish this row's
            // log2-sum-exp and the normalisation 1/l
            s_lse[h * 128 + r] = (ok && l > 0.0f) ? m_ref + __log2f(l) : -INFINITY;
            s_fin[h * 128 + r] = l > 0.0f ? 1.0f / l : 0.0f;
        }
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        const float lse_v = l > 0.0f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        const size_t row = ((size_t)b * p.N + node) * p.Hq + hq;
#pragma unroll 1
        for (int c64 = 0; c64 < 2 && p.splits == 1; ++c64) {
            uint32_t o[64];
            if (ok) {
                tmem_ld32(tO + c64 * 64, o);
                tmem_ld32(tO + c64 * 64 + 32, o + 32);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) o[c] = 0;
            }
            if (row_valid) {
                {
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
                }
            }
        }
        if (row_valid && p.splits == 1 && p.lse) p.lse[row] = lse_v;
    }

    tc_fence_before();
    __syncthreads();
    }  // n > 0

    if (*abort_flag) {
        // a wait gave up: let every MMA an issuer started finish before the
        // rings are reused or tensor memory is released
        if (warp >= 2 && warp < SW0 && lane == 0) {
            volatile int never = 0;
            umma_commit(&mma_drain[warp - 2]);
            mbar_wait_for(&mma_drain[warp - 2], 0, &never, kWaitDeadlineNs);
        }
        tc_fence_before();
        __syncthreads();
    }

    if (p.splits > 1) {
        // ---- merge of the cluster's chunks through distributed shared memory
        const uint32_t rank = cluster_ctarank();
        const int S2 = p.splits;
        constexpr int RB = 128 * NH;
        float4 *sO = reinterpret_cast<float4 *>(sK);  // [RB][32] normalised O rows, swizzled
        if (threadIdx.x == 0) {
            m_flag[0] = *abort_flag ? 0 : 1;
            m_flag[1] = bad;
        }
        if (warp >= SW0) {
            // the softmax role's row: half h, TMEM lane quarter (warp & 3);
            // s_lse holds its log2-sum-exp (-inf: no column here) and s_fin
            // 1 / l from the epilogue. Tensor-memory loads are warp-wide.
            const int lr = ((warp - SW0) >> 2) * 128 + (warp & 3) * 32 + lane;
            const bool contrib = n > 0 && s_lse[lr] != -INFINITY;
            tc_fence_after();
            if (__any_sync(FULL, contrib)) {
                const float inv = contrib ? s_fin[lr] : 0.0f;
                const uint32_t tO = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 256 +
                                    (uint32_t)((lr >> 7) * 128);
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o[32];
                    tmem_ld32(tO + c4 * 32, o);
                    tmem_wait_ld();
                    if (contrib) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            sO[lr * 32 + ((c4 * 8 + k) ^ (lr & 31))] =
                                make_float4(__uint_as_float(o[4 * k]) * inv,
                                            __uint_as_float(o[4 * k + 1]) * inv,
                                            __uint_as_float(o[4 * k + 2]) * inv,
                                            __uint_as_float(o[4 * k + 3]) * inv);
                    }
                }
            }
        }
        tc_fence_before();
        cluster_arrive();
        cluster_wait();
        // rows lr = rank + o S of this row block. First the merge weights of
        // each row, from the cluster's log-sum-exps (into the free Q area)
        float *wgt = reinterpret_cast<float *>(sQ);  // [nrows][kMaxSplits]
        const int nrows = (RB - (int)rank + S2 - 1) / S2;
        if (threadIdx.x == 0) {
            int fl[2 * kMaxSplits];
#pragma unroll
            for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                fl[2 * s2] = s2 < S2 ? ld_dsmem_s32(cluster_map(&m_flag[0], (uint32_t)s2)) : 1;
                fl[2 * s2 + 1] = s2 < S2 ? ld_dsmem_s32(cluster_map(&m_flag[1], (uint32_t)s2)) : 0;
            }
            int zero = len_ok ? 0 : 1;
#pragma unroll
            for (int s2 = 0; s2 < kMaxSplits; ++s2) zero |= (fl[2 * s2] == 0) | (fl[2 * s2 + 1] != 0);
            m_flag[2] = zero;
        }
        for (int o = threadIdx.x; o < nrows; o += NTHREADS) {
            const int lr = (int)rank + o * S2;
            float lv[kMaxSplits];
#pragma unroll
            for (int s2 = 0; s2 < kMaxSplits; ++s2)
                lv[s2] = s2 < S2 ? ld_dsmem_f32(cluster_map(&s_lse[lr], (uint32_t)s2)) : -INFINITY;
            float lmax = -INFINITY;
#pragma unroll
            for (int s2 = 0; s2 < kMaxSplits; ++s2) lmax = fmaxf(lmax, lv[s2]);
            float W = 0.0f;
#pragma unroll
            for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                lv[s2] = lv[s2] == -INFINITY ? 0.0f : ex2_approx(lv[s2] - lmax);
                W += lv[s2];
            }
            const float winv = W > 0.0f ? 1.0f / W : 0.0f;
#pragma unroll
            for (int s2 = 0; s2 < kMaxSplits; ++s2) wgt[o * kMaxSplits + s2] = lv[s2] * winv;
            s_mask[o] = __float_as_uint(W > 0.0f ? lmax + __log2f(W) : -INFINITY);
        }
        __syncthreads();
        // then 16 bytes of a row per thread: the row's chunk from every CTA
        // that saw the row, loaded together
        const bool zero = m_flag[2] != 0;
        for (int it = threadIdx.x; it < nrows * 32; it += NTHREADS) {
            const int o = it >> 5;
            const int lr = (int)rank + o * S2;
            const int c = it & 31;
            const int Rg = rb * RB + lr;
            if (Rg >= p.M) continue;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!zero) {
                const uint32_t src = smem_u32(&sO[lr * 32 + (c ^ (lr & 31))]);
                float4 v[kMaxSplits];
                float w[kMaxSplits];
#pragma unroll
                for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                    w[s2] = s2 < S2 ? wgt[o * kMaxSplits + s2] : 0.0f;
                    v[s2] = w[s2] > 0.0f ? ld_dsmem_v4(cluster_map_addr(src, (uint32_t)s2))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int s2 = 0; s2 < kMaxSplits; ++s2) {
                    acc.x = fmaf(w[s2], v[s2].x, acc.x);
                    acc.y = fmaf(w[s2], v[s2].y, acc.y);
                    acc.z = fmaf(w[s2], v[s2].z, acc.z);
                    acc.w = fmaf(w[s2], v[s2].w, acc.w);
                }
            }
            const size_t row = ((size_t)b * p.N + Rg / p.G) * p.Hq + g * p.G + Rg % p.G;
            uint2 w2;
            w2.x = pack_bf16x2(acc.x, acc.y);
            w2.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(p.out + row * HD + c * 4) = w2;
            if (c == 0 && p.lse)
                p.lse[row] = zero ? 0.0f : __uint_as_float(s_mask[o]) * 0.69314718055994531f;
        }
        // no CTA leaves while a peer may still read its shared memory
        cluster_arrive();
        cluster_wait();
    }

    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(&p.status[b], SVF_DEV_TIMEOUT);
    // With a single chunk this CTA wrote final outputs: a sequence with a bad
    // page gets zeros (every CTA of the sequence saw the same page table).
    if (p.splits == 1 && bad && warp >= SW0) {
        const int h = (warp - SW0) >> 2;
        const int R = rb * 128 * NH + h * 128 + (warp & 3) * 32 + lane;
        if (R < p.M) {
            const size_t row = ((size_t)b * p.N + R / p.G) * p.Hq + g * p.G + R % p.G;
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int k = 0; k < HD / 8; ++k)
                *reinterpret_cast<uint4 *>(p.out + row * HD + 8 * k) = z;
            if (p.lse) p.lse[row] = 0.0f;
        }
    }
}

// ---------------------------------------------------------------- host side

// Largest number of clusters of `splits` CTAs of the kernel for NH halves
// that can be resident at once (one CTA per SM; a cluster's CTAs share a
// GPC, so not every SM takes part for every cluster size).
static int resident_ctas(int NH, int splits) {
    static int cache[3][tc::kMaxSplits + 1] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    static int cached_dev = -1;
    if (cached_dev != dev) {
        for (auto &row : cache)
            for (int &v : row) v = 0;
        cached_dev = dev;
    }
    int &slot = cache[NH][splits];
    if (slot > 0) return slot;
    const int C = num_sms();
    int n = C;
    if (splits > 1) {
        const int smem = NH == 1 ? TcSmem<1>::kDynamic : TcSmem<2>::kDynamic;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)splits, (unsigned)C);
        cfg.blockDim = dim3(tc::threads_for(NH));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = (unsigned)splits;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        cudaError_t e;
        if (NH == 1) {
            cudaFuncSetAttribute(attn_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            e = cudaOccupancyMaxActiveClusters(&clusters, attn_tc_kernel<1>, &cfg);
        } else {
            cudaFuncSetAttribute(attn_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            e = cudaOccupancyMaxActiveClusters(&clusters, attn_tc_kernel<2>, &cfg);
        }
        n = (e == cudaSuccess && clusters > 0) ? clusters * splits : (C / splits) * splits;
    }
    slot = n;
    return n;
}

// Chunks per (sequence, KV head, row block) = the cluster size S. A wave is
// as many CTAs as can be resident for that cluster size, and each CTA costs
// its tiles plus a fixed cost (plus the merge when S > 1), with at most
// CMAX_TILES tiles per chunk. The lengths are on the device, so the host
// rates each S on two length profiles and averages them: every sequence at
// the page table's capacity (waves x the longest chunk), and lengths spread
// evenly below it (the longest chunk, or the total work spread over the
// resident CTAs, whichever is larger). Each cluster then splits its own
// sequence's tiles evenly, so shorter sequences simply finish sooner.
int attn_tc_splits(int B, int N, int Hq, int Hkv, int max_pages, int page_size) {
    const int G = Hq / Hkv;
    const int M = N * G;
    const int NH = row_halves(M);
    const int row_blocks = (M + 128 * NH - 1) / (128 * NH);
    const long long units = (long long)B * Hkv * row_blocks;
    const long long kv_max = (long long)max_pages * page_size;
    const int tiles = (int)((kv_max + tc::BN - 1) / tc::BN);
    double best = 1e300;
    int best_s = 1;
    for (int s = 1; s <= tc::kMaxSplits; ++s) {
        const int per_cta = (tiles + s - 1) / s;
        if (per_cta > tc::CMAX_TILES) continue;
        // chunks of a few tiles cost more in merge and co-scheduling than
        // they save
        if (s > 1 && per_cta < tc::kMinChunkTiles) break;
        const int cap = resident_ctas(NH, s);
        const double fixed = tc::kFixedTiles + (s > 1 ? tc::kMergeTiles : 0.0);
        const long long waves = (units * s + cap - 1) / cap;
        const double t_full = (double)waves * (per_cta + fixed);
        const double longest = per_cta + fixed;
        const double spread = (double)units * s * (0.5 * per_cta + fixed) / cap;
        const double t_spread = longest > spread ? longest : spread;
        const double t = 0.5 * (t_full + t_spread);
        if (t < best - 1e-9) {
            best = t;
            best_s = s;
        }
    }
    return best_s;
}

bool attn_tc_supported(int max_pages, int page_size) {
    const long long kv_max = (long long)max_pages * page_size;
    const int tiles = (int)((kv_max + tc::BN - 1) / tc::BN);
    return tiles <= tc::kMaxSplits * tc::CMAX_TILES;
}

// No workspace: chunks merge on chip.
size_t attn_tc_workspace_bytes(int, int, int, int, int, int) { return 0; }

static std::atomic<long long> g_attn_wait_ns{0};
static std::atomic<int> g_attn_force_splits{0};

void attn_tc_set_wait_ns(long long ns) { g_attn_wait_ns.store(ns > 0 ? ns : 0); }
long long attn_tc_wait_ns() { return g_attn_wait_ns.load(); }
void attn_tc_force_splits(int s) {
    g_attn_force_splits.store(s > 0 && s <= tc::kMaxSplits ? s : 0);
}
int attn_tc_forced_splits() { return g_attn_force_splits.load(); }

int launch_attn_tc(const AttnArgs &a, void *, size_t, cudaStream_t stream) {
    const int G = a.Hq / a.Hkv;
    const int M = a.N * G;
    const int NH = row_halves(M);
    const int row_blocks = (M + 128 * NH - 1) / (128 * NH);
    if (!attn_tc_supported(a.max_pages, a.page_size)) return SVF_ERR_UNSUPPORTED;
    int splits = attn_tc_splits(a.B, a.N, a.Hq, a.Hkv, a.max_pages, a.page_size);
    const int forced = g_attn_force_splits.load();
    if (forced > 0) {
        const long long kv_max = (long long)a.max_pages * a.page_size;
        const int tiles = (int)((kv_max + tc::BN - 1) / tc::BN);
        splits = forced;
        while ((tiles + splits - 1) / splits > tc::CMAX_TILES) ++splits;
    }

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
    const long long wns = g_attn_wait_ns.load();
    p.wait_ns = wns > 0 ? (unsigned long long)wns : kWaitDeadlineNs;
    p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.status = a.status;
    p.parent = a.parent;
    p.anc_out = a.anc_out;
    p.depth_out = a.depth_out;
    p.mask_status = a.mask_status;

    dim3 grid(a.Hkv * row_blocks, splits, a.B);
    const unsigned cl = splits > 1 ? (unsigned)splits : 0u;
    if (NH == 1) {
        const int smem = TcSmem<1>::kDynamic;
        cudaFuncSetAttribute(attn_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (launch_pdl_cluster_y(attn_tc_kernel<1>, grid, dim3(tc::threads_for(1)), smem, stream,
                                 cl, tmk, tmv, tmq, p) != cudaSuccess)
            return SVF_ERR_LAUNCH;
    } else {
        const int smem = TcSmem<2>::kDynamic;
        cudaFuncSetAttribute(attn_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (launch_pdl_cluster_y(attn_tc_kernel<2>, grid, dim3(tc::threads_for(2)), smem, stream,
                                 cl, tmk, tmv, tmq, p) != cudaSuccess)
            return SVF_ERR_LAUNCH;
    }
    if (cudaGetLastError() != cudaSuccess) return SVF_ERR_LAUNCH;
    return SVF_OK;
}

}  // namespace svf
