// kv_commit.cu -- keep the accepted path's K/V and roll back the rest.
//
// "EAGLE-4 Technical Deepdive", § EAGLE-4 verification trees and harness:
// once a tree is verified, the accepted continuation stays in the KV cache and
// the rejected nodes' entries are released. "EAGLE 演化史", § D.2: every tree
// node wrote its own K/V during the verification pass, so those entries must
// be rolled back (page by page in EAGLE's paged cache).
//
// Token t of sequence b sits in page page_table[b][t / ps], slot t % ps, and
// tree node j is token L_b + j. The committed sequence is
//   token L_b + k  <-  token L_b + path[k],   k = 0 .. accept_len,
// for K and V, every head and every layer. A root path in BFS order has
// strictly increasing entries with path[k] >= k, so a copy that walks k
// upwards never overwrites a row it has yet to read: rows L_b + path[k'] with
// k' > k lie past token L_b + k. Each thread owns one 16-byte column of the K
// or V rows of one (layer, sequence) and walks it down the path in that order,
// reading a batch of sources before writing their destinations; a source of
// the batch that is also one of its destinations is read before it is
// written. No two threads touch the same address, so no barrier is needed.
// A row with path[k] == k is already in place and does not move.
//
// Bound: HBM (or L2 for a cache the attention pass just read). Algorithmic
// bytes: 2 (K, V) x 2 (read, write) x rows moved x Hkv x D x element size per
// layer, where a row moves when path[k] != k.
#include "common.cuh"
#include "internal.h"

namespace svf {

namespace {

constexpr int kCommitThreads = 256;
constexpr int kBatch = 8;

// Checks one sequence; every CTA of the sequence reaches the same answer.
__device__ int commit_status(const int32_t *pt, const int32_t *pb, int len, int L, int N,
                             int ps, int max_pages, int num_pages) {
    int st = 0;
    if (len < 0 || len > N - 1) {
        st |= SVF_DEV_BAD_PATH;
    } else {
        for (int k = threadIdx.x; k <= len; k += blockDim.x) {
            const int cur = pb[k];
            const bool bad = (k == 0) ? (cur != 0) : (cur <= pb[k - 1] || cur >= N);
            if (bad) st |= SVF_DEV_BAD_PATH;
        }
    }
    if (L < 0 || (long long)L + N > (long long)max_pages * ps) {
        st |= SVF_DEV_BAD_LENGTH;
    } else {
        const int p0 = L / ps, p1 = (int)(((long long)L + N - 1) / ps);
        for (int i = p0 + (int)threadIdx.x; i <= p1; i += blockDim.x) {
            const int page = pt[i];
            if (page < 0 || page >= num_pages) st |= SVF_DEV_BAD_PAGE;
        }
    }
    return st;
}

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(
    uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache, long long layer_stride_bytes,
    int num_pages, int ps, const int32_t *__restrict__ page_table, int max_pages,
    const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ path,
    const int32_t *__restrict__ accept_len, int N, int row_chunks, int32_t *__restrict__ new_seq_lens,
    int32_t *__restrict__ freed, int max_free, int32_t *__restrict__ n_freed,
    int32_t *__restrict__ status) {
    extern __shared__ int s_rows[];  // [2][N]: source and destination rows of each move
    __shared__ int s_bits;
    const int b = blockIdx.x;
    const int layer = blockIdx.y;
    if (threadIdx.x == 0) s_bits = 0;
    pdl_wait();
    pdl_launch_dependents();
    const int32_t *pt = page_table + (size_t)b * max_pages;
    const int32_t *pb = path + (size_t)b * N;
    const int L = seq_lens[b];
    const int len = accept_len[b];
    __syncthreads();
    const int mine = commit_status(pt, pb, len, L, N, ps, max_pages, num_pages);
    if (mine) atomicOr(&s_bits, mine);
    __syncthreads();
    const int st = s_bits;
    const int new_len = st ? L : L + len + 1;
    if (layer == 0) {
        // the sequence's designated CTA writes its scalar outputs
        const int first = (new_len + ps - 1) / ps;
        const int end = st ? first : (int)(((long long)L + N + ps - 1) / ps);
        if (threadIdx.x == 0) {
            status[b] = st;
            new_seq_lens[b] = new_len;
            if (n_freed) n_freed[b] = end - first;
        }
        if (freed)
            for (int i = threadIdx.x; i < max_free; i += blockDim.x)
                freed[(size_t)b * max_free + i] = (first + i < end) ? pt[first + i] : -1;
    }
    if (st || len == 0) return;
    // rows (page * ps + slot) of the source and destination of k = 1 .. len
    for (int k = 1 + (int)threadIdx.x; k <= len; k += blockDim.x) {
        const long long ts = (long long)L + pb[k], td = (long long)L + k;
        s_rows[k - 1] = pt[ts / ps] * ps + (int)(ts % ps);
        s_rows[N + k - 1] = pt[td / ps] * ps + (int)(td % ps);
    }
    __syncthreads();
    const size_t row_bytes = (size_t)row_chunks * 16;
    for (int c = threadIdx.x; c < 2 * row_chunks; c += blockDim.x) {
        const bool is_v = c >= row_chunks;
        uint8_t *base = (is_v ? v_cache : k_cache) + (size_t)layer * layer_stride_bytes +
                        (size_t)(is_v ? c - row_chunks : c) * 16;
        for (int m0 = 0; m0 < len; m0 += kBatch) {
            uint4 buf[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (m0 + u < len && s_rows[m0 + u] != s_rows[N + m0 + u])
                    buf[u] = *reinterpret_cast<const uint4 *>(base + (size_t)s_rows[m0 + u] * row_bytes);
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (m0 + u < len && s_rows[m0 + u] != s_rows[N + m0 + u])
                    *reinterpret_cast<uint4 *>(base + (size_t)s_rows[N + m0 + u] * row_bytes) = buf[u];
        }
    }
}

}  // namespace

cudaError_t launch_kv_commit(const KvCommitArgs &a, cudaStream_t stream) {
    const int row_chunks = (int)((size_t)a.Hkv * a.D * a.elem_size / 16);
    return launch_pdl(kv_commit_kernel, dim3((unsigned)a.B, (unsigned)a.num_layers),
                      dim3(kCommitThreads), (size_t)2 * a.N * sizeof(int), stream, 0u,
                      reinterpret_cast<uint8_t *>(a.k_cache), reinterpret_cast<uint8_t *>(a.v_cache),
                      a.layer_stride * (long long)a.elem_size, a.num_pages, a.page_size,
                      a.page_table, a.max_pages, a.seq_lens, a.path, a.accept_len, a.N, row_chunks,
                      a.new_seq_lens, a.freed_pages, a.max_free, a.n_freed, a.status);
}

}  // namespace svf
