// attn_sk.cu -- tree attention as one persistent stream of tiles per SM
// (bf16, head_dim 128, 5th-generation tensor cores).
//
// "EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree Verification 详解, A-B:
// one target pass verifies the whole tree; node i sees the cached prefix and
// tree positions L_b + j for j an ancestor of i (or i). § D.2 sizes the cost
// as O(N·P) reads of the prefix, so the work is a stream of K/V tiles, and
// the way to its roofline is to keep every SM streaming for the whole call.
//
// The per-tile pipeline and the warp roles are those of attn_tc.cu (a K and a
// V producer, a QK and a PV issuer per 128-row half, four softmax warps per
// half; S and O in tensor memory, P written over S). What differs is the
// work decomposition. A unit is (sequence, KV head, row block); its tiles are
// the 64-token blocks of prefix + tree. The CTAs form groups of Hkv, one CTA
// per KV head, and a group's CTAs stream the same token ranges side by side
// (each token row of the cache holds all heads, so they read it from DRAM
// together). The (sequence, row block) pairs' tiles are laid end to end
// (sequence-major) and group c of C takes tiles [cT/C, (c+1)T/C): every CTA
// streams the same number of tiles whatever the batch, the lengths or the
// number of units, and no wave is left half full. A CTA's share is a run of
// segments, each a contiguous part of one unit. At a segment boundary the QK
// issuers load the next unit's Q, the PV issuers restart O, and the softmax
// warps write the finished segment out:
//   - a unit that lies inside one CTA is written as final output;
//   - a unit split between CTAs (only a CTA's first and last segment can be)
//     is published by each piece as normalised fp32 rows and their
//     log2-sum-exps in the workspace, and counted in the unit's arrival
//     counter. After its own tiles every CTA merges a share of the rows of
//     the split units it took part in, once all their pieces arrived:
//     out = sum_k w_k O_k with w_k = 2^(lse_k - max) / sum.
// The launch is cooperative (every CTA resident while another waits for it),
// and every wait is bounded. The counters are zero between calls: the last
// CTA to finish a unit's merge puts them back to zero (the workspace is
// zero-filled once, before its first use).
#include <string.h>

#include <atomic>

#include "attn_tc_common.cuh"
#include "internal.h"

namespace svf {

namespace sk {
// K/V ring depths as in attn_tc.cu: Q (32 KB per half) plus 9 (two halves)
// or 11 (one half) stages of 16 KB.
__host__ __device__ constexpr int kstages_for(int NH) { return NH == 1 ? 5 : 4; }
__host__ __device__ constexpr int vstages_for(int NH) { return NH == 1 ? 6 : 5; }
constexpr int kLookahead = 4;         // page-table entries are read this many tiles ahead
constexpr int kMinTilesPerCta = 8;    // small calls use fewer CTAs than SMs
constexpr int kBarSoftmax = 1;        // named barrier of the softmax warps
constexpr unsigned long long kMergeDeadlineNs = 5000000000ull;  // > any pipeline wait
}  // namespace sk

struct SkParams {
    const int32_t *page_table;
    const int32_t *seq_lens;
    const uint64_t *anc;
    int B, N, Hq, Hkv, G, M;
    int num_pages, page_size, max_pages;
    int row_blocks;
    float scale_log2;
    unsigned long long wait_ns;  // deadline of the pipeline waits
    __nv_bfloat16 *out;
    float *lse;
    int32_t *status;
    const int32_t *parent;  // non-null: masks from parent[] (N <= 64), written out below
    uint64_t *anc_out;
    int32_t *depth_out;
    int32_t *mask_status;
    float4 *part;     // [2 C][32][128 NH]: a piece's normalised rows, 16-byte chunk-major
    float *part_lse;  // [2 C][128 NH]: its rows' log2-sum-exp (-inf: no visible column)
    int *part_flags;  // [2 C]: bit 0 a page id outside the cache, bit 1 a wait gave up
    int *counters;    // [B][Hkv][row_blocks][2]: pieces published, merges done (zero between calls)
};

template <int NH>
struct SkSmem {
    static constexpr int kKS = sk::kstages_for(NH);
    static constexpr int kVS = sk::vstages_for(NH);
    static constexpr int kSB = tc::sbuffers_for(NH);
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + NH * tc::HALF_BYTES;
    static constexpr int kV = kK + kKS * tc::TILE_BYTES;
    static constexpr int kBar = kV + kVS * tc::TILE_BYTES;
    static constexpr int kNumBars = 2 * kKS + 2 * kVS + 4 * NH * kSB + 3 * NH + kVS + 2 * NH;
    static constexpr int kMisc = kBar + ((kNumBars * 8 + 127) / 128) * 128;
    static constexpr int kPar = kMisc + 256;     // parent[] of the segment's sequence [2][64]
    static constexpr int kDes = kPar + 2 * 64 * 4;  // parent[] for the designated build [64]
    static constexpr int kBytes = kDes + 64 * 4;
    static constexpr int kDynamic = kBytes + 1024;  // slack to align the base to 1 KB
    static_assert(kDynamic <= 227 * 1024, "shared memory budget");
    // the merge's weights go in the Q area, the set-up scan in the K ring
    static_assert(NH * tc::HALF_BYTES >= 4 * (256 + 2 * 1024), "merge weights fit in Q");
};

// One segment: the part [x0, x1) of the tile space that this CTA's group
// takes of row block k of sequence b (for this CTA's KV head), whose tiles
// start at index pu.
struct SkSeg {
    long long pu, x0, x1;
    int b, k, t, L;  // t: tiles per unit of the sequence, L: its prefix length
};

struct SkJob {  // a split unit this CTA merges a share of
    long long pu;
    int b, k, F, kf;  // F pieces (groups); this CTA's group holds piece kf
    int pad[2];
};

__device__ __forceinline__ int sk_tiles(const SkParams &p, int L) {
    const long long T = (long long)L + p.N;
    return (L >= 0 && T <= (long long)p.max_pages * p.page_size) ? (int)((T + tc::BN - 1) / tc::BN)
                                                                 : 0;
}

// First tile of group c's share and the group whose share holds tile x.
__device__ __forceinline__ long long sk_start(int c, long long T, int C) {
    return (long long)c * T / C;
}
__device__ __forceinline__ int sk_cta_of(long long x, long long T, int C) {
    return (int)(((x + 1) * (long long)C - 1) / T);
}

__device__ __forceinline__ bool sk_first(const SkParams &p, SkSeg &g, int b0, long long pb0,
                                         long long s, long long e) {
    if (s >= e) return false;
    g.b = b0;
    g.L = __ldg(p.seq_lens + b0);
    g.t = sk_tiles(p, g.L);
    if (g.t <= 0) return false;
    g.k = (int)((s - pb0) / g.t);
    g.pu = pb0 + (long long)g.k * g.t;
    g.x0 = s;
    g.x1 = min(g.pu + g.t, e);
    return true;
}

// The next segment (false past the end of the share). Sequences without
// tiles (a bad length) hold no unit in the tile space and are skipped.
__device__ __forceinline__ bool sk_next(const SkParams &p, SkSeg &g, long long e) {
    if (g.x1 >= e) return false;
    const long long x = g.x1;
    if (++g.k == p.row_blocks) {
        g.k = 0;
        do {
            ++g.b;
            g.L = __ldg(p.seq_lens + g.b);
            g.t = sk_tiles(p, g.L);
        } while (g.t == 0 && g.b + 1 < p.B);
    }
    g.pu = x;
    g.x0 = x;
    g.x1 = min(x + g.t, e);
    return g.t > 0;
}

__device__ __forceinline__ int named_bar_or(int id, int n, int pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(n)
        : "memory");
    return (int)r;
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("barrier.cta.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Status word, masks and (for a bad length) zero outputs of sequence bd, by
// the nst softmax threads (thread st). The tree check and the parent walks
// are those of svf_tree_mask_build ("EAGLE 演化史", § Tree Verification
// 详解, B: a node sees its ancestors and itself).
__device__ void sk_designated(const SkParams &p, int bd, int st, int nst, int32_t *spar) {
    const int L = __ldg(p.seq_lens + bd);
    const long long Tq = (long long)L + p.N;
    const bool len_ok = L >= 0 && Tq <= (long long)p.max_pages * p.page_size;
    int bad_pg = 0;
    if (len_ok) {
        const long long npg = (Tq + p.page_size - 1) / p.page_size;
        const int32_t *pt = p.page_table + (size_t)bd * p.max_pages;
        for (long long i = st; i < npg; i += nst) {
            const int id = __ldg(pt + i);
            if (id < 0 || id >= p.num_pages) bad_pg = 1;
        }
    }
    int bad_tree = 0;
    if (p.parent && st < p.N) {
        const int pp = __ldg(p.parent + (size_t)bd * p.N + st);
        spar[st] = pp;
        bad_tree = st == 0 ? pp != -1 : (pp < 0 || pp >= st);
    }
    bad_pg = named_bar_or(sk::kBarSoftmax, nst, bad_pg);
    if (p.parent) bad_tree = named_bar_or(sk::kBarSoftmax, nst, bad_tree);
    if (st == 0) p.status[bd] = !len_ok ? SVF_DEV_BAD_LENGTH : (bad_pg ? SVF_DEV_BAD_PAGE : 0);
    if (p.parent) {
        if (st < p.N) {
            uint64_t word = 1ull << st;
            int d = 0;
            if (!bad_tree) {
                d = -1;
                word = 0;
                for (int a = st; a != -1; a = spar[a]) {
                    word |= 1ull << a;
                    ++d;
                }
            }
            if (p.anc_out) p.anc_out[(size_t)bd * p.N + st] = word;
            if (p.depth_out) p.depth_out[(size_t)bd * p.N + st] = d;
        }
        if (st == 0 && p.mask_status) p.mask_status[bd] = bad_tree ? SVF_DEV_BAD_PARENT : 0;
    }
    if (!len_ok) {
        // no tile of this sequence is in the tile space: its outputs are zeros
        const long long rows = (long long)p.N * p.Hq;
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (long long i = st; i < rows * (tc::HD / 8); i += nst) {
            const long long row = (long long)bd * rows + i / (tc::HD / 8);
            reinterpret_cast<uint4 *>(p.out + row * tc::HD)[i % (tc::HD / 8)] = z;
        }
        if (p.lse)
            for (long long i = st; i < rows; i += nst) p.lse[(long long)bd * rows + i] = 0.0f;
    }
    named_bar_sync(sk::kBarSoftmax, nst);  // spar is reused by the next sequence
}

template <int NH>
__global__ void __launch_bounds__(tc::threads_for(NH), 1)
    attn_sk_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmq, SkParams p) {
    using S = SkSmem<NH>;
    using namespace tc;
    constexpr int KS = S::kKS;
    constexpr int VS = S::kVS;
    constexpr int SB = S::kSB;
    constexpr int NTHREADS = threads_for(NH);
    constexpr int NWARPS = NTHREADS / 32;
    constexpr int SW0 = first_softmax_warp(NH);
    constexpr int RB = 128 * NH;
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(NH * SB * BN + NH * 128 <= 512, "tensor memory budget");
    static_assert(NWARPS <= 32, "one warp scans the warp totals");
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
    uint64_t *s_full = v_empty + VS;      // [NH][SB]: QK of the tile in S buffer b done
    uint64_t *p_full = s_full + NH * SB;  // [NH][SB]: P of the tile written over S buffer b
    uint64_t *o_done = p_full + NH * SB;  // [NH][SB]: PV that read S buffer b done
    uint64_t *p_half = o_done + NH * SB;  // [NH][SB]: first half of that P written
    uint64_t *q_full = p_half + NH * SB;  // [NH]: the segment's Q half landed
    uint64_t *q_free = q_full + NH;       // [NH]: the segment's QKs done (Q may be replaced)
    uint64_t *o_free = q_free + NH;       // [NH]: the segment's O read out (O may restart)
    uint64_t *v_zero = o_free + NH;       // [VS]: half 0 zeroed the rows past the end
    uint64_t *mma_drain = v_zero + VS;    // [2 NH]: an issuer's MMAs done, after an abort
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *m_ok = reinterpret_cast<int *>(smem + S::kMisc + 8);
    int *njobs = reinterpret_cast<int *>(smem + S::kMisc + 12);
    long long *info = reinterpret_cast<long long *>(smem + S::kMisc + 16);  // T, s, e, pb0
    int *info_i = reinterpret_cast<int *>(smem + S::kMisc + 48);           // b0, C, group
    SkJob *jobs = reinterpret_cast<SkJob *>(smem + S::kMisc + 64);         // [2]
    int32_t *s_par = reinterpret_cast<int32_t *>(smem + S::kPar);
    int32_t *s_des = reinterpret_cast<int32_t *>(smem + S::kDes);

    // tensor memory: S buffer (h, b) at columns [64 (SB h + b), +64); O of
    // half h at [256 + 128 h, +128); P goes over the first 32 columns of its S
    constexpr uint32_t kTmemCols = 512;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int hd = c % p.Hkv;  // this CTA's KV head

    // On-chip set-up first: it overlaps the previous kernel's tail.
    if (threadIdx.x == 0) {
        for (int s2 = 0; s2 < KS; ++s2) {
            mbar_init(&k_full[s2], 1);
            mbar_init(&k_empty[s2], NH);
        }
        for (int s2 = 0; s2 < VS; ++s2) {
            mbar_init(&v_full[s2], 1);
            mbar_init(&v_empty[s2], NH);
            mbar_init(&v_zero[s2], 1);
        }
        for (int k = 0; k < NH * SB; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], 128);
            mbar_init(&o_done[k], 1);
            mbar_init(&p_half[k], 128);
        }
        for (int h = 0; h < NH; ++h) {
            mbar_init(&q_full[h], 1);
            mbar_init(&q_free[h], 1);
            mbar_init(&o_free[h], 128);
        }
        for (int k = 0; k < 2 * NH; ++k) mbar_init(&mma_drain[k], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1 && lane == 0) {
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
        tma_prefetch_desc(&tmq);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_launch_dependents();

    // ---- the tile space: tiles of every sequence's units, sequence-major.
    // Thread i sums a contiguous block of sequences; a block-wide scan gives
    // each block's first tile and the total T.
    {
        long long *wsum = reinterpret_cast<long long *>(sK);  // [NWARPS]; the ring is idle
        const long long lo = (long long)p.B * threadIdx.x / NTHREADS;
        const long long hi = (long long)p.B * (threadIdx.x + 1) / NTHREADS;
        long long mine = 0;
        for (long long b = lo; b < hi; ++b) mine += sk_tiles(p, __ldg(p.seq_lens + b));
        mine *= p.row_blocks;
        long long incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const long long w = lane < NWARPS ? wsum[lane] : 0;
            long long wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long v = __shfl_up_sync(FULL, wi, o);
                if (lane >= o) wi += v;
            }
            __syncwarp();
            if (lane < NWARPS) wsum[lane] = wi - w;
            if (lane == 31) info[0] = wi;
        }
        __syncthreads();
        const long long T = info[0];
        const long long first = wsum[warp] + incl - mine;
        // groups of Hkv CTAs; fewer groups than fit when the work is small
        long long Cl = T / sk::kMinTilesPerCta;
        const long long groups = gridDim.x / p.Hkv;
        Cl = Cl < 1 ? 1 : (Cl > groups ? groups : Cl);
        const int C = (int)Cl;
        const int grp = c / p.Hkv;
        const long long s = grp < C && T > 0 ? sk_start(grp, T, C) : T;
        const long long e = grp < C && T > 0 ? sk_start(grp + 1, T, C) : T;
        if (s < e && first <= s && s < first + mine) {
            // this thread's block holds tile s: find its sequence
            long long pb = first;
            for (long long b = lo; b < hi; ++b) {
                const long long tb = (long long)sk_tiles(p, __ldg(p.seq_lens + b)) * p.row_blocks;
                if (s < pb + tb) {
                    info[3] = pb;
                    info_i[0] = (int)b;
                    break;
                }
                pb += tb;
            }
        }
        if (threadIdx.x == 0) {
            info[1] = s;
            info[2] = e;
            info_i[1] = C;
            info_i[2] = grp;
        }
        __syncthreads();
    }
    // the tile space's constants stay in shared memory: the roles read them
    // at segment boundaries only (registers are scarce with two halves)
    volatile long long *vinfo = info;
    volatile int *vinfo_i = info_i;
#define SK_T (vinfo[0])
#define SK_S (vinfo[1])
#define SK_E (vinfo[2])
#define SK_PB0 (vinfo[3])
#define SK_B0 (vinfo_i[0])
#define SK_C (vinfo_i[1])
#define SK_GRP (vinfo_i[2])
    const uint32_t tmem = *tmem_slot;
    tc_fence_after();

    if (warp <= 1) {
        // ------------------------------------------------------------ producers
        // Warp 0 streams K, warp 1 streams V, each into its ring as soon as a
        // stage is free; lane x < bpt issues box x of both 64-dim halves. Each
        // lane reads its box's page-table entry kLookahead tiles ahead.
        constexpr int LA = sk::kLookahead;
        const bool is_k = warp == 0;
        const CUtensorMap *map = is_k ? &tmk : &tmv;
        uint8_t *ring = is_k ? sK : sV;
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *empty = is_k ? k_empty : v_empty;
        const int stages = is_k ? KS : VS;
        const int ps = p.page_size;
        const int box_rows = ps < MAX_BOX_ROWS ? ps : MAX_BOX_ROWS;
        const int bpt = BN / box_rows;
        const int oob = p.num_pages * ps;  // a slot past the cache: TMA fills zeros
        long long issued = 0;
        SkSeg gi, ga;
        if (sk_first(p, gi, SK_B0, SK_PB0, SK_S, SK_E)) {
            ga = gi;
            const long long s = SK_S, n = SK_E - s;
            // page id (raw; -1: no token) and slot offset of this lane's box of tile x
            auto fetch = [&](long long x, int &id, int &off) {
                while (x >= ga.x1) sk_next(p, ga, SK_E);
                const long long tok = (x - ga.pu) * BN + (long long)lane * box_rows;
                id = -1;
                off = 0;
                if (lane < bpt && tok < (long long)ga.L + p.N) {
                    const int page = (int)(tok / ps);
                    off = (int)(tok - (long long)page * ps);
                    id = __ldg(p.page_table + (size_t)ga.b * p.max_pages + page);
                }
            };
            int cid[LA], coff[LA];
#pragma unroll
            for (int q = 0; q < LA; ++q) {
                cid[q] = -1;
                coff[q] = 0;
                if (q < n) fetch(s + q, cid[q], coff[q]);
            }
            bool ok = true;
            for (long long j0 = 0; ok && j0 < n; j0 += LA) {
#pragma unroll
                for (int q = 0; q < LA; ++q) {
                    const long long j = j0 + q;
                    if (!ok || j >= n) break;
                    while (s + j >= gi.x1) sk_next(p, gi, SK_E);
                    const int st = (int)(j % stages);
                    const long long use = j / stages;
                    if (use > 0 &&
                        !(ok = warp_wait(&empty[st], (uint32_t)((use - 1) & 1), abort_flag, p.wait_ns)))
                        break;
                    const int crd = (cid[q] < 0 || cid[q] >= p.num_pages) ? oob : cid[q] * ps + coff[q];
                    if (lane == 0) mbar_arrive_expect_tx(&full[st], TILE_BYTES);
                    if (lane < bpt) {
#pragma unroll
                        for (int dh = 0; dh < 2; ++dh)
                            tma_load_3d(ring + st * TILE_BYTES + dh * KV_COL_BYTES + lane * box_rows * 128,
                                        map, dh * 64, hd, crd, &full[st]);
                    }
                    __syncwarp();
                    ++issued;
                    cid[q] = -1;
                    coff[q] = 0;
                    if (j + LA < n) fetch(s + j + LA, cid[q], coff[q]);
                }
            }
        }
        if (lane == 0) {
            // Never leave with copies in flight: wait (bounded, ignoring the
            // abort flag) for the last fill of every stage that was loaded.
            volatile int never = 0;
            for (int st = 0; st < stages && st < issued; ++st)
                mbar_wait_for(&full[st], (uint32_t)(((issued - 1 - st) / stages) & 1), &never,
                              kWaitDeadlineNs);
        }
    } else if (warp <= 1 + NH) {
        // ------------------------------------------------------------ QK issuer, half h
        // Per segment: this half's Q rows of the unit by TMA once the previous
        // segment's QKs are done, then S_h,b = Q_h K^T for every tile into
        // the buffer whose previous PV is done.
        const int h = warp - 2;
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BN, false, false);
        const uint32_t aQ = smem_u32(sQ) + h * HALF_BYTES, aK = smem_u32(sK);
        const int nodes = 128 / p.G;
        SkSeg g;
        bool more = sk_first(p, g, SK_B0, SK_PB0, SK_S, SK_E), ok = true, q_pending = false;
        long long j = 0;
        int segi = 0;
        while (more) {
            if (segi > 0 &&
                !(ok = warp_wait(&q_free[h], (uint32_t)((segi - 1) & 1), abort_flag, p.wait_ns)))
                break;
            if (lane == 0) {
                const int rb = g.k;
                mbar_arrive_expect_tx(&q_full[h], HALF_BYTES);
#pragma unroll
                for (int dh = 0; dh < 2; ++dh)
                    tma_load_4d(sQ + h * HALF_BYTES + dh * Q_COL_BYTES, &tmq, dh * 64, hd * p.G,
                                (rb * NH + h) * nodes, g.b, &q_full[h]);
            }
            __syncwarp();
            q_pending = true;
            if (!(ok = warp_wait(&q_full[h], (uint32_t)(segi & 1), abort_flag, p.wait_ns))) break;
            q_pending = false;
            const long long n = g.x1 - g.x0;
            for (long long jl = 0; jl < n; ++jl, ++j) {
                const int bb = (int)(j % SB);
                if (!(ok = warp_wait(&k_full[j % KS], (uint32_t)((j / KS) & 1), abort_flag, p.wait_ns)))
                    break;
                if (j >= SB) {
                    // PV(j - SB) of this half read P from this S buffer
                    const long long pj = j - SB;
                    if (!(ok = warp_wait(&o_done[h * SB + bb], (uint32_t)((pj / SB) & 1), abort_flag,
                                         p.wait_ns)))
                        break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d = tmem + (uint32_t)((h * SB + bb) * BN);
                    const uint32_t kst = aK + (uint32_t)(j % KS) * TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t oq = (kk >> 2) * Q_COL_BYTES + (kk & 3) * 32;
                        const uint32_t ok_ = (kk >> 2) * KV_COL_BYTES + (kk & 3) * 32;
                        umma_ss(d, smem_desc_sw128(aQ + oq, 16, 1024),
                                smem_desc_sw128(kst + ok_, 16, 1024), idesc_qk, kk > 0);
                    }
                    umma_commit(&s_full[h * SB + bb]);
                    umma_commit(&k_empty[j % KS]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&q_free[h]);
            __syncwarp();
            ++segi;
            more = sk_next(p, g, SK_E);
        }
        if (q_pending && lane == 0) {
            volatile int never = 0;
            mbar_wait_for(&q_full[h], (uint32_t)(segi & 1), &never, kWaitDeadlineNs);
        }
    } else if (warp <= 1 + 2 * NH) {
        // ------------------------------------------------------------ PV issuer, half h
        // O_h += P_h,b V for every tile once its softmax is done; the first
        // tile of a segment restarts O once the previous segment's O was read.
        const int h = warp - 2 - NH;
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD, false, true);
        const uint32_t aV = smem_u32(sV);
        SkSeg g;
        bool more = sk_first(p, g, SK_B0, SK_PB0, SK_S, SK_E), ok = true;
        long long j = 0;
        int segi = 0;
        uint32_t zpar = 0;  // half 1: parity of the next zeroing signal, per V stage
        while (more && ok) {
            const long long n = g.x1 - g.x0;
            const long long Tq = (long long)g.L + p.N;
            for (long long jl = 0; jl < n; ++jl, ++j) {
                const int bb = (int)(j % SB);
                const int vs = (int)(j % VS);
                if (!(ok = warp_wait(&v_full[vs], (uint32_t)((j / VS) & 1), abort_flag, p.wait_ns)))
                    break;
                const long long t0 = (g.x0 - g.pu + jl) * BN;
                if (t0 + BN > Tq) {
                    // The sequence's last tile. V rows past its end may hold
                    // anything (NaN included, and P = 0 does not cancel NaN):
                    // half 0 zeroes them before either half reads the stage.
                    if (NH == 1 || h == 0) {
                        const int r0 = (int)(Tq - t0);
                        uint8_t *vsm = sV + vs * TILE_BYTES;
                        for (int idx = lane; idx < (BN - r0) * 16; idx += 32) {
                            const int r = r0 + (idx >> 4), c16 = idx & 15;
                            *reinterpret_cast<uint4 *>(vsm + (c16 >> 3) * KV_COL_BYTES + r * 128 +
                                                       (c16 & 7) * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (NH == 2 && lane == 0) mbar_arrive(&v_zero[vs]);
                    } else {
                        if (!(ok = warp_wait(&v_zero[vs], (zpar >> vs) & 1u, abort_flag, p.wait_ns)))
                            break;
                        zpar ^= 1u << vs;
                    }
                }
                if (jl == 0 && segi > 0 &&
                    !(ok = warp_wait(&o_free[h], (uint32_t)((segi - 1) & 1), abort_flag, p.wait_ns)))
                    break;
                // P arrives in two halves of 32 tokens; the first half's K-steps
                // go in while the softmax still computes the second
                const uint32_t d = tmem + 256 + h * 128;
                const uint32_t a = tmem + (uint32_t)((h * SB + bb) * BN);
                const uint32_t vst = aV + (uint32_t)vs * TILE_BYTES;
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
                                    idesc_pv, (jl > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) {
                    umma_commit(&o_done[h * SB + bb]);
                    umma_commit(&v_empty[vs]);
                }
                __syncwarp();
            }
            ++segi;
            more = sk_next(p, g, SK_E);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int h = (warp - SW0) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int lr = h * 128 + r;                 // row of the CTA's row block
        const int st = threadIdx.x - 32 * SW0;       // 0 .. RB - 1
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + 256 + h * 128;
        const float sl2 = p.scale_log2;

        // Status words and masks: a sequence with tiles gets them from the
        // CTA that holds its first tile, at the start of that segment (so a
        // timeout bit this CTA ORs in later cannot be overwritten); one with
        // no tile (a bad length) from CTA b mod grid, with its zero outputs.
        for (int bd = c; bd < p.B; bd += gridDim.x)
            if (sk_tiles(p, __ldg(p.seq_lens + bd)) == 0) sk_designated(p, bd, st, RB, s_des);

        // The segment is kept in shared memory (one thread steps it, double
        // buffered by segment parity): registers are scarce in this role.
        SkSeg *sseg = reinterpret_cast<SkSeg *>(smem + S::kMisc + 128);  // [2]
        bool ok = true;  // false once a wait gave up: later segments skip their tiles
        int j = 0;       // tiles of this CTA so far
        for (int segi = 0;; ++segi) {
            volatile SkSeg *cur = sseg + (segi & 1);
            if (st == 0) {
                SkSeg g;
                bool more;
                if (segi == 0) {
                    more = sk_first(p, g, SK_B0, SK_PB0, SK_S, SK_E);
                } else {
                    const volatile SkSeg *pv = sseg + ((segi - 1) & 1);
                    g.pu = pv->pu; g.x0 = pv->x0; g.x1 = pv->x1;
                    g.b = pv->b; g.k = pv->k; g.t = pv->t; g.L = pv->L;
                    more = sk_next(p, g, SK_E);
                }
                cur->pu = g.pu; cur->x0 = g.x0; cur->x1 = g.x1;
                cur->b = g.b; cur->k = g.k; cur->L = g.L;
                cur->t = more ? g.t : 0;
            }
            named_bar_sync(sk::kBarSoftmax, RB);
            if (cur->t == 0) break;
            const int gb = cur->b, gk = cur->k;
            if (hd == 0 && gk == 0 && cur->x0 == cur->pu) sk_designated(p, gb, st, RB, s_des);
            const int gkv = hd, rb = gk;
            const int R = rb * RB + lr;
            const bool row_valid = R < p.M;
            const int node = row_valid ? R / p.G : 0;
            const int hq = gkv * p.G + (row_valid ? R % p.G : 0);
            const int L = cur->L;
            const int Tq = L + p.N;
            const int n = (int)(cur->x1 - cur->x0);
            const int tin0 = (int)(cur->x0 - cur->pu);
            // a page id outside the cache among this segment's tiles zeroes
            // the unit's output (the sequence's status word says so)
            int seg_bad = 0;
            {
                const int ps = p.page_size;
                const int tok1 = min((tin0 + n) * BN, Tq);
                const int pg1 = (tok1 + ps - 1) / ps;
                const int32_t *pt = p.page_table + (size_t)gb * p.max_pages;
                for (int pg = tin0 * BN / ps + st; pg < pg1; pg += RB) {
                    const int id = __ldg(pt + pg);
                    if (id < 0 || id >= p.num_pages) seg_bad = 1;
                }
            }
            int32_t *spar = s_par + (segi & 1) * 64;
            int tree_bad = 0;
            if (p.parent && st < p.N) {
                const int pp = __ldg(p.parent + (size_t)gb * p.N + st);
                spar[st] = pp;
                tree_bad = st == 0 ? pp != -1 : (pp < 0 || pp >= st);
            }
            seg_bad = named_bar_or(sk::kBarSoftmax, RB, seg_bad);
            uint64_t anc = 0;
            if (p.parent) {
                // the ancestor mask of this row's node, as svf_tree_mask_build
                // builds it (an invalid tree: every node sees only itself)
                tree_bad = named_bar_or(sk::kBarSoftmax, RB, tree_bad);
                if (row_valid) {
                    if (tree_bad) {
                        anc = 1ull << node;
                    } else {
                        for (int a = node; a != -1; a = spar[a]) anc |= 1ull << a;
                    }
                }
            } else if (row_valid) {
                anc = __ldg(p.anc + (size_t)gb * p.N + node);
            }

            float m_ref = -INFINITY, l = 0.0f;
            for (int jl = 0; ok && jl < n; ++jl, ++j) {
                const int bb = j % SB;
                const uint32_t bph = (uint32_t)((j / SB) & 1);
                const uint32_t tS = tmem + lane_off + (uint32_t)((h * SB + bb) * BN);
                if (!(ok = warp_wait(&s_full[h * SB + bb], bph, abort_flag, p.wait_ns))) break;
                tc_fence_after();
                uint32_t v[BN];
                tmem_ld32(tS, v);
                tmem_ld32(tS + 32, v + 32);
                tmem_wait_ld();
                const int tbase = (tin0 + jl) * BN;
                if (tbase + BN > L) {
                    // this tile reaches the tree: ancestors only
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const uint32_t vis = visible_bits(tbase + 32 * c2 - L, anc);
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc)
                            v[32 * c2 + cc] = ((vis >> cc) & 1u) ? v[32 * c2 + cc] : 0xff800000u;
                    }
                }
                float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < BN; cc += 8) {
                    m0 = fmax3(m0, __uint_as_float(v[cc]), __uint_as_float(v[cc + 1]));
                    m1 = fmax3(m1, __uint_as_float(v[cc + 2]), __uint_as_float(v[cc + 3]));
                    m2 = fmax3(m2, __uint_as_float(v[cc + 4]), __uint_as_float(v[cc + 5]));
                    m3 = fmax3(m3, __uint_as_float(v[cc + 6]), __uint_as_float(v[cc + 7]));
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
                    if (jl > 0) {
                        // O is final up to PV(j - 1) of this half
                        const int pj = j - 1;
                        if (!(ok = warp_wait(&o_done[h * SB + pj % SB], (uint32_t)((pj / SB) & 1),
                                             abort_flag, p.wait_ns)))
                            break;
                        tc_fence_after();
                        // in 16-column pieces: S is still live in registers
#pragma unroll 1
                        for (int c8 = 0; c8 < 8; ++c8) {
                            uint32_t o[16];
                            tmem_ld16(tO + c8 * 16, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int cc = 0; cc < 16; ++cc)
                                o[cc] = __float_as_uint(__uint_as_float(o[cc]) * alpha);
                            tmem_st16(tO + c8 * 16, o);
                        }
                        tmem_wait_st();
                    }
                }
                // P = 2^(s*scale - m_ref) as bf16 pairs over the first 32 S
                // columns, in two halves of 32 tokens (the PV issuer starts on the
                // first); even and odd columns are summed in the two lanes of r
                const float mneg = m_ref == -INFINITY ? 0.0f : -m_ref;
                const float2 sc2 = make_float2(sl2, sl2), mn2 = make_float2(mneg, mneg);
                float2 rs = make_float2(0.0f, 0.0f);
                uint32_t pk[BN / 2];
#pragma unroll
                for (int cc = 0; cc < BN / 2; ++cc) {
                    const float2 x = ffma2(make_float2(__uint_as_float(v[2 * cc]),
                                                       __uint_as_float(v[2 * cc + 1])), sc2, mn2);
                    const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    rs = fadd2(rs, pp);
                    pk[cc] = pack_bf16x2(pp.x, pp.y);
                    if (cc == BN / 4 - 1) {
                        tmem_st16(tS, pk);
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(&p_half[h * SB + bb]);
                    }
                }
                tmem_st16(tS + BN / 4, pk + BN / 4);
                tmem_wait_st();
                l += rs.x + rs.y;
                tc_fence_before();
                mbar_arrive(&p_full[h * SB + bb]);
            }
            // ---- epilogue of the segment: O of this half after its last PV
            if (ok && n > 0)
                ok = warp_wait(&o_done[h * SB + (j - 1) % SB], (uint32_t)(((j - 1) / SB) & 1),
                               abort_flag, p.wait_ns);
            tc_fence_after();
            const long long gpu_ = cur->pu;
            const int cf = sk_cta_of(gpu_, SK_T, SK_C), cl = sk_cta_of(gpu_ + cur->t - 1, SK_T, SK_C);
            const int slot = 2 * c + (cur->x0 == SK_S ? 0 : 1);  // 0: this CTA's first segment
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            if (cf == cl) {
                // the whole unit is in this CTA: final output (zeros for a
                // sequence with a bad page or after a wait gave up)
                const bool zero = !ok || seg_bad;
                const float lse_v = (l > 0.0f && !zero) ? (m_ref + __log2f(l)) * 0.69314718055994531f
                                                        : (zero ? 0.0f : -INFINITY);
                const size_t row = ((size_t)gb * p.N + node) * p.Hq + hq;
#pragma unroll 1
                for (int c64 = 0; c64 < 2; ++c64) {
                    uint32_t o[64];
                    if (!zero) {
                        tmem_ld32(tO + c64 * 64, o);
                        tmem_ld32(tO + c64 * 64 + 32, o + 32);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int cc = 0; cc < 64; ++cc) o[cc] = 0;
                    }
                    if (row_valid) {
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
                if (row_valid && p.lse) p.lse[row] = lse_v;
            } else {
                // one piece of a split unit: publish the normalised rows and
                // their log2-sum-exp in this CTA's slot (0: its first segment)
                float4 *dst = p.part + (size_t)slot * 32 * RB;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t o[32];
                    if (ok) {
                        tmem_ld32(tO + c4 * 32, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) o[cc] = 0;
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        __stcg(dst + (size_t)(c4 * 8 + k) * RB + lr,
                               make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                           __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv));
                }
                __stcg(p.part_lse + (size_t)slot * RB + lr,
                       (ok && l > 0.0f) ? m_ref + __log2f(l) : -INFINITY);
                __threadfence();
            }
            // O may restart for the next segment
            tc_fence_before();
            mbar_arrive(&o_free[h]);
            if (cf != cl) {
                // every row of the piece is written: count it in the unit
                named_bar_sync(sk::kBarSoftmax, RB);
                if (st == 0) {
                    __stcg(p.part_flags + slot, (seg_bad ? 1 : 0) | (*abort_flag ? 2 : 0));
                    __threadfence();
                    atomicAdd(p.counters + 2 * (((size_t)gb * p.Hkv + hd) * p.row_blocks + gk), 1);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait gave up: let every MMA an issuer started finish before
        // tensor memory is released
        if (warp >= 2 && warp < SW0 && lane == 0) {
            volatile int never = 0;
            umma_commit(&mma_drain[warp - 2]);
            mbar_wait_for(&mma_drain[warp - 2], 0, &never, kWaitDeadlineNs);
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }

    // ---- the split units this CTA took part in: its last segment and its
    // first (a CTA's middle segments are whole units)
    if (threadIdx.x == 0) {
        int nj = 0;
        SkSeg g, first, last;
        if (sk_first(p, g, SK_B0, SK_PB0, SK_S, SK_E)) {
            first = g;
            last = g;
            while (sk_next(p, g, SK_E)) last = g;
            auto add = [&](long long pu, int b, int k, int t) {
                const int cf = sk_cta_of(pu, SK_T, SK_C), cl = sk_cta_of(pu + t - 1, SK_T, SK_C);
                if (cl > cf) {
                    jobs[nj].pu = pu;
                    jobs[nj].b = b;
                    jobs[nj].k = k;
                    jobs[nj].F = cl - cf + 1;
                    jobs[nj].kf = SK_GRP - cf;
                    ++nj;
                }
            };
            add(last.pu, last.b, last.k, last.t);
            if (first.x0 != last.x0) add(first.pu, first.b, first.k, first.t);
            if (*abort_flag)
                for (int b = first.b; b <= last.b; ++b) atomicOr(&p.status[b], SVF_DEV_TIMEOUT);
        }
        *njobs = nj;
    }
    __syncthreads();
    const int nj = *njobs;
    for (int jb = 0; jb < nj; ++jb) {
        const SkJob J = jobs[jb];
        int *cnt = p.counters + 2 * (((size_t)J.b * p.Hkv + hd) * p.row_blocks + J.k);
        if (threadIdx.x == 0) {
            // every piece of the unit published (bounded: a piece's CTA
            // publishes even after its own waits gave up)
            int got = ld_acquire_gpu(cnt) >= J.F;
            const unsigned long long t0 = globaltimer_ns();
            while (!got) {
                __nanosleep(128);
                got = ld_acquire_gpu(cnt) >= J.F;
                if (!got && globaltimer_ns() - t0 > sk::kMergeDeadlineNs) break;
            }
            *m_ok = got;
        }
        __syncthreads();
        const int cf = SK_GRP - J.kf;
        const long long s_cf = sk_start(cf, SK_T, SK_C);
        // slot of piece f: this head's CTA of group cf + f, slot 0 if the unit
        // is that CTA's first segment
        auto slot_of = [&](int f) {
            return 2 * ((cf + f) * p.Hkv + hd) + ((f == 0 && s_cf < J.pu) ? 1 : 0);
        };
        int zero = !*m_ok, timed_out = !*m_ok;
        for (int f = threadIdx.x; f < J.F; f += NTHREADS) {
            const int fl = __ldcg(p.part_flags + slot_of(f));
            zero |= fl != 0;
            timed_out |= (fl & 2) != 0;
        }
        zero = __syncthreads_or(zero);
        timed_out = __syncthreads_or(timed_out);
        const int rb = J.k, gkv = hd;
        const int RBv = min(RB, p.M - rb * RB);
        const int r0 = (int)((long long)J.kf * RBv / J.F);
        const int r1 = (int)((long long)(J.kf + 1) * RBv / J.F);
        const int nr = r1 - r0;
        // weights of every row of this share (Q's shared memory is free)
        float *wgt = reinterpret_cast<float *>(sQ);   // [nr][F]
        float *mlse = wgt + nr * J.F;                  // [nr] merged log2-sum-exp
        for (int i = threadIdx.x; i < nr && !zero; i += NTHREADS) {
            float lmax = -INFINITY;
            for (int f = 0; f < J.F; ++f) {
                const float lv = __ldcg(p.part_lse + (size_t)slot_of(f) * RB + r0 + i);
                wgt[i * J.F + f] = lv;
                lmax = fmaxf(lmax, lv);
            }
            float W = 0.0f;
            for (int f = 0; f < J.F; ++f) {
                const float lv = wgt[i * J.F + f];
                const float w = lv == -INFINITY ? 0.0f : ex2_approx(lv - lmax);
                wgt[i * J.F + f] = w;
                W += w;
            }
            const float winv = W > 0.0f ? 1.0f / W : 0.0f;
            for (int f = 0; f < J.F; ++f) wgt[i * J.F + f] *= winv;
            mlse[i] = W > 0.0f ? lmax + __log2f(W) : -INFINITY;
        }
        __syncthreads();
        // then 16 bytes of a row per thread, rows fastest (the pieces' rows
        // are chunk-major, so a warp reads 512 contiguous bytes per piece)
        for (int it = threadIdx.x; it < nr * 32; it += NTHREADS) {
            const int i = it % nr, c4 = it / nr;
            const int Rg = rb * RB + r0 + i;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!zero) {
                int f = 0;
                for (; f + 4 <= J.F; f += 4) {
                    float4 v4[4];
                    float w4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        w4[q] = wgt[i * J.F + f + q];
                        v4[q] = w4[q] > 0.0f ? __ldcg(p.part + ((size_t)slot_of(f + q) * 32 + c4) * RB + r0 + i)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc.x = fmaf(w4[q], v4[q].x, acc.x);
                        acc.y = fmaf(w4[q], v4[q].y, acc.y);
                        acc.z = fmaf(w4[q], v4[q].z, acc.z);
                        acc.w = fmaf(w4[q], v4[q].w, acc.w);
                    }
                }
                for (; f < J.F; ++f) {
                    const float w = wgt[i * J.F + f];
                    if (w > 0.0f) {
                        const float4 v = __ldcg(p.part + ((size_t)slot_of(f) * 32 + c4) * RB + r0 + i);
                        acc.x = fmaf(w, v.x, acc.x);
                        acc.y = fmaf(w, v.y, acc.y);
                        acc.z = fmaf(w, v.z, acc.z);
                        acc.w = fmaf(w, v.w, acc.w);
                    }
                }
            }
            const size_t row = ((size_t)J.b * p.N + Rg / p.G) * p.Hq + gkv * p.G + Rg % p.G;
            uint2 w2;
            w2.x = pack_bf16x2(acc.x, acc.y);
            w2.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(p.out + row * HD + c4 * 4) = w2;
            if (c4 == 0 && p.lse)
                p.lse[row] = zero ? 0.0f : mlse[i] * 0.69314718055994531f;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            if (timed_out) atomicOr(&p.status[J.b], SVF_DEV_TIMEOUT);
            // the last merger of the unit puts its counters back to zero
            __threadfence();
            if (atomicAdd(cnt + 1, 1) == J.F - 1) {
                cnt[0] = 0;
                cnt[1] = 0;
            }
        }
        __syncthreads();
    }
}

#undef SK_T
#undef SK_S
#undef SK_E
#undef SK_PB0
#undef SK_B0
#undef SK_C
#undef SK_GRP

// ---------------------------------------------------------------- host side

bool attn_sk_supported(int Hq, int Hkv) {
    const int G = Hq / Hkv;
    // Q by TMA only; one group of Hkv CTAs at least
    return G >= 1 && G <= 128 && (G & (G - 1)) == 0 && Hkv <= num_sms();
}

// Workspace: the pieces' rows, log-sum-exps and flags (two slots per SM,
// each sized for two halves whatever the call) and then one pair of
// counters per unit. Only the counters' length depends on the call, and they
// start at the same offset for every call, so a workspace that one shape
// left with zero counters is ready for any other shape that fits in it.
struct SkLayout {
    size_t part, part_lse, part_flags, counters, total;
};

static SkLayout sk_layout(int B, int N, int Hq, int Hkv) {
    const int G = Hq / Hkv;
    const int M = N * G;
    const int RB = 128 * row_halves(M);
    const int row_blocks = (M + RB - 1) / RB;
    const size_t C = (size_t)num_sms();
    constexpr size_t kRows = 256;  // rows of a slot for two halves
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    SkLayout l;
    l.part = 0;
    l.part_lse = up(2 * C * 32 * kRows * sizeof(float4));
    l.part_flags = l.part_lse + up(2 * C * kRows * sizeof(float));
    l.counters = l.part_flags + up(2 * C * sizeof(int));
    l.total = l.counters + up((size_t)B * Hkv * row_blocks * 2 * sizeof(int));
    return l;
}

size_t attn_sk_workspace_bytes(int B, int N, int Hq, int Hkv) {
    if (!attn_sk_supported(Hq, Hkv)) return 0;
    return sk_layout(B, N, Hq, Hkv).total;
}

template <int NH>
static cudaError_t launch_sk(dim3 grid, cudaStream_t stream, const CUtensorMap &tmk,
                             const CUtensorMap &tmv, const CUtensorMap &tmq, const SkParams &p) {
    const int smem = SkSmem<NH>::kDynamic;
    cudaFuncSetAttribute(attn_sk_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(tc::threads_for(NH));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // cooperative with programmatic dependent launch where the driver takes
    // the pair, cooperative alone where it does not (remembered)
    static std::atomic<int> pdl_ok{1};
    if (pdl_ok.load()) {
        cfg.numAttrs = 2;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_sk_kernel<NH>, tmk, tmv, tmq, p);
        if (e != cudaErrorInvalidValue && e != cudaErrorNotSupported) return e;
        cudaGetLastError();
        pdl_ok.store(0);
    }
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_sk_kernel<NH>, tmk, tmv, tmq, p);
}

static std::atomic<int> g_attn_kernel{0};

void attn_set_kernel(int which) { g_attn_kernel.store(which >= 0 && which <= 2 ? which : 0); }

// 1: chunks merged in clusters (attn_tc.cu), 2: persistent (this file), -1:
// the persistent kernel was asked for without a large enough workspace.
// The persistent kernel pays a longer start (the tile space is scanned on
// the device) and a merge through L2 at the end, ~15-20 us together, against
// the cluster kernel's per-CTA prologue and on-chip merge and its last
// partial wave. Measured on this part (CUDA events, full clock): 70B layer
// (1728 tiles per CTA) 1718-1746 against 1786-1805 us; EAGLE-2 (27 tiles per
// CTA) 68-72 against 46-50 us; paged chain (30) 66 against 50 us; binary
// tree (8) 29 against 19 us. So it is taken when every CTA would stream at
// least kPersistentTiles tiles with the page tables full.
int attn_choose_kernel(const AttnArgs &a, const void *workspace, size_t ws_bytes) {
    constexpr long long kPersistentTiles = 256;
    const bool sk_ok = attn_sk_supported(a.Hq, a.Hkv);
    const bool ws_ok = sk_ok && workspace && ws_bytes >= attn_sk_workspace_bytes(a.B, a.N, a.Hq, a.Hkv);
    const int forced = g_attn_kernel.load();
    if (attn_tc_forced_splits() > 0 || forced == 1) return 1;
    if (forced == 2) return ws_ok ? 2 : -1;
    if (!ws_ok) return 1;
    const int M = a.N * (a.Hq / a.Hkv);
    const int RB = 128 * row_halves(M);
    const long long row_blocks = (M + RB - 1) / RB;
    const long long tiles = ((long long)a.max_pages * a.page_size + tc::BN - 1) / tc::BN;
    const long long groups = num_sms() / a.Hkv;
    const long long per_cta = (long long)a.B * row_blocks * tiles / (groups > 0 ? groups : 1);
    return per_cta >= kPersistentTiles ? 2 : 1;
}

int launch_attn_sk(const AttnArgs &a, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    const int G = a.Hq / a.Hkv;
    const int M = a.N * G;
    const int NH = row_halves(M);
    const int row_blocks = (M + 128 * NH - 1) / (128 * NH);
    if (!attn_sk_supported(a.Hq, a.Hkv)) return SVF_ERR_UNSUPPORTED;
    const SkLayout lay = sk_layout(a.B, a.N, a.Hq, a.Hkv);
    if (!workspace || ws_bytes < lay.total) return SVF_ERR_WORKSPACE;
    CUtensorMap tmk, tmv, tmq;
    if (!make_kv_map(&tmk, a.k_cache, a.num_pages, a.page_size, a.Hkv) ||
        !make_kv_map(&tmv, a.v_cache, a.num_pages, a.page_size, a.Hkv) ||
        !make_q_map(&tmq, a.q, a.B, a.N, a.Hq, G))
        return SVF_ERR_LAUNCH;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SkParams p;
    p.page_table = a.page_table;
    p.seq_lens = a.seq_lens;
    p.anc = a.anc;
    p.B = a.B; p.N = a.N; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.M = M;
    p.num_pages = a.num_pages; p.page_size = a.page_size; p.max_pages = a.max_pages;
    p.row_blocks = row_blocks;
    const float scale = a.sm_scale > 0.0f ? a.sm_scale : 1.0f / sqrtf((float)a.D);
    p.scale_log2 = scale * 1.4426950408889634f;
    const long long wns = attn_tc_wait_ns();
    p.wait_ns = wns > 0 ? (unsigned long long)wns : kWaitDeadlineNs;
    p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.status = a.status;
    p.parent = a.parent;
    p.anc_out = a.anc_out;
    p.depth_out = a.depth_out;
    p.mask_status = a.mask_status;
    p.counters = reinterpret_cast<int *>(ws + lay.counters);
    p.part = reinterpret_cast<float4 *>(ws + lay.part);
    p.part_lse = reinterpret_cast<float *>(ws + lay.part_lse);
    p.part_flags = reinterpret_cast<int *>(ws + lay.part_flags);

    // one CTA per SM, all resident (cooperative launch)
    const dim3 grid((unsigned)num_sms());
    cudaError_t e = NH == 1 ? launch_sk<1>(grid, stream, tmk, tmv, tmq, p)
                            : launch_sk<2>(grid, stream, tmk, tmv, tmq, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SVF_ERR_LAUNCH;
    }
    return SVF_OK;
}

}  // namespace svf
