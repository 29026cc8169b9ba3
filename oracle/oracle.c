/*
 * oracle.c -- plain, slow, fp64 CPU oracle for one-pass tree verification.
 *
 * TEST INFRASTRUCTURE ONLY. Tests, the smoke check and the benchmark's CPU
 * baseline call it; the product path never does. It shares no code, header,
 * table or helper with the CUDA library, and it follows the definitions on the
 * pages literally, with no blocking, fusion or reordering:
 *
 *   oracle_tree_mask   "EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree
 *                      Verification 详解, B (the tree is flattened in BFS
 *                      order; a node sees only its ancestors, never siblings or
 *                      cousins) and G step 3 (the 7-node worked tree).
 *   oracle_tree_attn   same page, § A and § B (one target pass over prefix +
 *                      tree; each node attends to the prefix, its ancestors and
 *                      itself; its output equals running prompt + root->node
 *                      path as an ordinary causal sequence).
 *   oracle_kv_commit   "EAGLE-4 Technical Deepdive", § EAGLE-4 verification
 *                      trees and harness (after verification keep the
 *                      accepted continuation, free the rejected KV entries)
 *                      and "EAGLE 演化史", § D.2 (every tree node writes its
 *                      own K/V; rejected nodes' entries must not stay in the
 *                      cache, which is rolled back page by page).
 *   oracle_spec_accept "Eagle vs DFlash", speculative sampling rule (accept
 *                      x with probability min(1, p(x)/q(x)); on rejection
 *                      sample from normalize(max(0, p - q))); "EAGLE 演化史"
 *                      § C (walk from the root, children in order, residual
 *                      after each rejected sibling, sample from the residual
 *                      when every child is rejected, longest accepted path)
 *                      and § G steps 5-6 (worked walk with a bonus token).
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   - N counts nodes including the root; node 0 is the root, whose KV is at
 *     logical position L_b, and node j's KV is at L_b + j.
 *   - head h reads KV head h / (Hq / Hkv); the softmax scale is given.
 *   - a sequence with an invalid parent[] gets status bit 1; its masks hold
 *     only each node's own bit (depth 0), and the acceptance outputs are "no
 *     result" (-1 everywhere, accept_len 0).
 *   - siblings are tried in ascending node index; the draft distribution for
 *     a child is the draft softmax at its parent, and only the target side is
 *     replaced by the residual after a rejection.
 *   - accept iff u * q(x) < p~(x); a residual with zero mass leaves p~ as it
 *     was; the bonus token is the smallest k whose cumulative p~ exceeds
 *     u * sum(p~), else the last k with p~(k) > 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BAD_PARENT 1
#define ORACLE_BAD_TOKEN 2
#define ORACLE_BAD_PAGE 4
#define ORACLE_BAD_LENGTH 8
#define ORACLE_BAD_PATH 32

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* A parent array is a BFS-flattened tree: node 0 is the root (parent -1) and
 * every other node's parent comes before it. */
static int tree_is_valid(const int32_t *parent, int N) {
    if (N < 1 || parent[0] != -1) return 0;
    for (int i = 1; i < N; ++i)
        if (parent[i] < 0 || parent[i] >= i) return 0;
    return 1;
}

/* is node j on the root->i path (j == i included)?  Walks parent links up. */
static int is_ancestor_or_self(const int32_t *parent, int j, int i) {
    for (int a = i; a != -1; a = parent[a])
        if (a == j) return 1;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O1: ancestor bitmasks and depths.                                         */
/* anc is [B, N, W] with W = ceil(N / 64); bit j of anc[b, i] is set iff node */
/* j is an ancestor of node i or i itself.                                    */
/* ------------------------------------------------------------------------ */
int oracle_tree_mask(const int32_t *parent, int B, int N, uint64_t *anc,
                     int32_t *depth, int32_t *status) {
    if (B < 0 || N < 0) return -1;
    const int W = (N + 63) / 64;
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (size_t)b * N;
        const int ok = tree_is_valid(par, N);
        status[b] = ok ? 0 : ORACLE_BAD_PARENT;
        for (int i = 0; i < N; ++i) {
            uint64_t *row = anc + ((size_t)b * N + i) * W;
            for (int w = 0; w < W; ++w) row[w] = 0;
            if (!ok) {
                row[i / 64] |= (uint64_t)1 << (i % 64);
                if (depth) depth[(size_t)b * N + i] = 0;
                continue;
            }
            int d = -1;
            for (int a = i; a != -1; a = par[a]) {
                row[a / 64] |= (uint64_t)1 << (a % 64);
                ++d;
            }
            if (depth) depth[(size_t)b * N + i] = d;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O2: tree attention, fp64.                                                 */
/*   q   [B, N, Hq, D]    (float32 values; bf16 inputs arrive widened)       */
/*   k,v [B, Tcap, Hkv, D] logical token order: token t of sequence b is at   */
/*                         [b, t]; the prefix is t < L_b, node j is L_b + j   */
/*   rows: nrows triples (b, i, h) to compute, or NULL for every (b, i, h) in */
/*         that order; out [nrows, D], lse [nrows].                           */
/* For row (b, i, h) with g = h / (Hq / Hkv) the visible tokens are           */
/* t < L_b and L_b + j for j an ancestor of i or i itself:                    */
/*   s_t = scale * <q, k_t>,  o = sum_t softmax(s)_t v_t,  lse = log sum e^s. */
/* ------------------------------------------------------------------------ */
int oracle_tree_attn(const float *q, const float *k, const float *v, int Tcap,
                     const int32_t *seq_lens, const int32_t *parent,
                     int B, int N, int Hq, int Hkv, int D, double scale,
                     const int32_t *rows, int nrows, double *out, double *lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return -1;
    const int G = Hq / Hkv;
    const long total = rows ? nrows : (long)B * N * Hq;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < total; ++r) {
        int b, i, h;
        if (rows) {
            b = rows[3 * r]; i = rows[3 * r + 1]; h = rows[3 * r + 2];
        } else {
            b = (int)(r / ((long)N * Hq)); i = (int)((r / Hq) % N); h = (int)(r % Hq);
        }
        if (b < 0 || b >= B || i < 0 || i >= N || h < 0 || h >= Hq) { err = 1; continue; }
        const int g = h / G;
        const int L = seq_lens[b];
        const int32_t *par = parent + (size_t)b * N;
        const int valid = tree_is_valid(par, N);
        const int T = L + N;
        if (T > Tcap) { err = 1; continue; }
        const float *qv = q + (((size_t)b * N + i) * Hq + h) * D;
        double *s = (double *)malloc(sizeof(double) * T);
        char *vis = (char *)malloc(T);
        for (int t = 0; t < T; ++t) {
            if (t < L) vis[t] = 1;
            else {
                int j = t - L;
                vis[t] = valid ? (char)is_ancestor_or_self(par, j, i) : (char)(j == i);
            }
        }
        double m = -INFINITY;
        for (int t = 0; t < T; ++t) {
            if (!vis[t]) continue;
            const float *kt = k + (((size_t)b * Tcap + t) * Hkv + g) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += (double)qv[d] * (double)kt[d];
            s[t] = scale * acc;
            if (s[t] > m) m = s[t];
        }
        double Z = 0.0;
        for (int t = 0; t < T; ++t)
            if (vis[t]) Z += exp(s[t] - m);
        double *o = out + (size_t)r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int t = 0; t < T; ++t) {
            if (!vis[t]) continue;
            const double w = exp(s[t] - m) / Z;
            const float *vt = v + (((size_t)b * Tcap + t) * Hkv + g) * D;
            for (int d = 0; d < D; ++d) o[d] += w * (double)vt[d];
        }
        if (lse) lse[r] = m + log(Z);
        free(s);
        free(vis);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* O3: acceptance walk over the tree, fp64.                                  */
/* ------------------------------------------------------------------------ */

/* p = softmax(row): m = max, e = exp(l - m), p = e / sum(e). */
static void softmax64(const float *row, int V, double *p) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if ((double)row[v] > m) m = (double)row[v];
    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp((double)row[v] - m);
        Z += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= Z;
}

/*
 * Inputs:  target, draft [B, N, V] logits (softmax at temperature 1);
 *          tokens [B, N] (tokens[b][c] is node c's draft token; the root's is
 *          not tested); parent [B, N]; u_accept [B, N] (u of node c tests c);
 *          u_bonus [B].
 * Outputs: accept_len [B]   accepted draft tokens (root excluded);
 *          path [B, N]      root first, then the accepted nodes, -1 padded;
 *          out_tokens [B,N] accepted draft tokens then the bonus, -1 padded;
 *          ratio [B, N]     p~(x)/q(x) for every tested node, NaN otherwise;
 *          accept_margin [B,N]  |u q(x) - p~(x)| / max(u q(x), p~(x)) for
 *                           tested nodes, NaN otherwise (how near a tie the
 *                           decision was);
 *          bonus_margin [B] distance of u*sum(p~) to the nearer edge of the
 *                           chosen token's CDF interval, divided by sum(p~);
 *          n_rejects [B]    rejected children of the node the bonus is drawn
 *                           at (0: drawn from that node's target softmax);
 *          status [B]       bit 1 bad parent[], bit 2 token outside [0, V).
 *          probe_cdf [B,3]  if probe_token is given: for k = probe_token[b]
 *                           (skipped when -1), the normalised cumulative
 *                           p~ before k and through k, and u_bonus[b] -- so a
 *                           caller can check that a token k picked elsewhere
 *                           lies on the inverse-CDF crossing.
 * Any of ratio / accept_margin / bonus_margin / n_rejects / probe_* may be NULL.
 */
int oracle_spec_accept(const float *target, const float *draft, const int32_t *tokens,
                       const int32_t *parent, const float *u_accept, const float *u_bonus,
                       int B, int N, int V, int32_t *accept_len, int32_t *path,
                       int32_t *out_tokens, double *ratio, double *accept_margin,
                       double *bonus_margin, int32_t *n_rejects, int32_t *status,
                       const int32_t *probe_token, double *probe_cdf) {
    if (B < 0 || N < 0 || V <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (size_t)b * N;
        const int32_t *tok = tokens + (size_t)b * N;
        int st = 0;
        if (!tree_is_valid(par, N)) st |= ORACLE_BAD_PARENT;
        for (int c = 1; c < N; ++c)
            if (tok[c] < 0 || tok[c] >= V) st |= ORACLE_BAD_TOKEN;
        status[b] = st;
        for (int c = 0; c < N; ++c) {
            path[(size_t)b * N + c] = -1;
            out_tokens[(size_t)b * N + c] = -1;
            if (ratio) ratio[(size_t)b * N + c] = NAN;
            if (accept_margin) accept_margin[(size_t)b * N + c] = NAN;
        }
        accept_len[b] = 0;
        if (bonus_margin) bonus_margin[b] = NAN;
        if (n_rejects) n_rejects[b] = 0;
        if (st != 0 || N == 0) continue;

        double *pt = (double *)malloc(sizeof(double) * V); /* p~ at the current node */
        double *qd = (double *)malloc(sizeof(double) * V); /* draft softmax at the current node */
        double *res = (double *)malloc(sizeof(double) * V);

        int cur = 0, len = 0, rejects = 0;
        path[(size_t)b * N] = 0;
        softmax64(target + ((size_t)b * N + cur) * V, V, pt);
        for (;;) {
            int has_child = 0, moved = 0;
            rejects = 0;
            for (int c = cur + 1; c < N && !moved; ++c) {
                if (par[c] != cur) continue;
                if (!has_child) {
                    softmax64(draft + ((size_t)b * N + cur) * V, V, qd);
                    has_child = 1;
                }
                const int x = tok[c];
                const double u = (double)u_accept[(size_t)b * N + c];
                const double qx = qd[x], px = pt[x];
                if (ratio) ratio[(size_t)b * N + c] = px / qx;
                if (accept_margin) {
                    double hi = u * qx > px ? u * qx : px;
                    accept_margin[(size_t)b * N + c] = hi > 0 ? fabs(u * qx - px) / hi : 0.0;
                }
                if (u * qx < px) {
                    /* accepted: move to c; its target softmax is the new p~ */
                    ++len;
                    path[(size_t)b * N + len] = c;
                    out_tokens[(size_t)b * N + len - 1] = x;
                    cur = c;
                    softmax64(target + ((size_t)b * N + cur) * V, V, pt);
                    moved = 1;
                } else {
                    /* rejected: p~ <- normalize(max(0, p~ - q)), try the next sibling */
                    double S = 0.0;
                    for (int v = 0; v < V; ++v) {
                        res[v] = pt[v] - qd[v] > 0.0 ? pt[v] - qd[v] : 0.0;
                        S += res[v];
                    }
                    if (S > 0.0)
                        for (int v = 0; v < V; ++v) pt[v] = res[v] / S;
                    ++rejects;
                }
            }
            if (!moved) break;
        }
        /* bonus: inverse CDF of p~ at u_bonus */
        double tot = 0.0;
        for (int v = 0; v < V; ++v) tot += pt[v];
        const double thr = (double)u_bonus[b] * tot;
        double cum = 0.0, prev = 0.0;
        int pick = -1;
        for (int v = 0; v < V; ++v) {
            prev = cum;
            cum += pt[v];
            if (cum > thr) { pick = v; break; }
        }
        double margin;
        if (pick < 0) {
            for (int v = V - 1; v >= 0; --v)
                if (pt[v] > 0.0) { pick = v; break; }
            margin = 0.0;
        } else {
            double a = thr - prev, c2 = cum - thr;
            margin = (a < c2 ? a : c2) / tot;
        }
        if (probe_token && probe_cdf && probe_token[b] >= 0 && probe_token[b] < V) {
            double before = 0.0;
            for (int v = 0; v < probe_token[b]; ++v) before += pt[v];
            probe_cdf[3 * (size_t)b] = before / tot;
            probe_cdf[3 * (size_t)b + 1] = (before + pt[probe_token[b]]) / tot;
            probe_cdf[3 * (size_t)b + 2] = (double)u_bonus[b];
        }
        out_tokens[(size_t)b * N + len] = pick;
        accept_len[b] = len;
        if (bonus_margin) bonus_margin[b] = margin;
        if (n_rejects) n_rejects[b] = rejects;
        free(pt);
        free(qd);
        free(res);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O5: commit the accepted path's K/V (rollback of the rejected nodes).     */
/*   k_cache, v_cache: num_layers caches of [num_pages, page_size, Hkv, D]   */
/*     elements of elem_size bytes, layer l starting layer_stride elements   */
/*     after layer l-1. Token t of sequence b sits in page                   */
/*     page_table[b][t / page_size], slot t % page_size; the tree's node j   */
/*     is token L_b + j.                                                     */
/*   path [B, N], accept_len [B]: the acceptance walk's result (root first). */
/* For each layer and each sequence, the K/V rows of tokens                  */
/*   L_b + path[0], L_b + path[1], ..., L_b + path[accept_len]              */
/* are read, and then written to tokens L_b, L_b + 1, ..., L_b + accept_len. */
/* new_seq_lens[b] = L_b + accept_len + 1. The pages at table indices        */
/* ceil(new_len / ps) .. ceil((L_b + N) / ps) - 1 held only rejected nodes;  */
/* their ids go to freed[b][0..] in that order (-1 after them), the count to */
/* n_freed[b].                                                               */
/* A sequence with a bad path (accept_len outside [0, N-1], path[0] != 0, or */
/* a path index outside (path[k-1], N)), a bad length (L_b < 0 or           */
/* L_b + N beyond its page table) or a bad page (a page of tokens            */
/* [L_b, L_b + N) outside [0, num_pages)) is left untouched: status bits,    */
/* new_seq_lens[b] = L_b, no freed pages.                                    */
/* ------------------------------------------------------------------------ */
int oracle_kv_commit(uint8_t *k_cache, uint8_t *v_cache, int elem_size, int num_layers,
                     long long layer_stride, int num_pages, int page_size,
                     const int32_t *page_table, int max_pages, const int32_t *seq_lens,
                     const int32_t *path, const int32_t *accept_len, int B, int N, int Hkv,
                     int D, int32_t *new_seq_lens, int32_t *freed, int max_free,
                     int32_t *n_freed, int32_t *status) {
    if (B < 0 || N < 1 || Hkv < 1 || D < 1 || page_size < 1 || max_pages < 1 || num_layers < 1 ||
        (elem_size != 2 && elem_size != 4))
        return -1;
    const size_t row_bytes = (size_t)Hkv * D * elem_size;
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        const int32_t *pt = page_table + (size_t)b * max_pages;
        const int32_t *pb = path + (size_t)b * N;
        const int len = accept_len[b];
        int st = 0;
        if (len < 0 || len > N - 1 || pb[0] != 0) {
            st |= ORACLE_BAD_PATH;
        } else {
            for (int k = 1; k <= len; ++k)
                if (pb[k] <= pb[k - 1] || pb[k] >= N) st |= ORACLE_BAD_PATH;
        }
        if (L < 0 || (long long)L + N > (long long)max_pages * page_size) {
            st |= ORACLE_BAD_LENGTH;
        } else {
            for (long long t = L; t < (long long)L + N; ++t) {
                const int page = pt[t / page_size];
                if (page < 0 || page >= num_pages) st |= ORACLE_BAD_PAGE;
            }
        }
        status[b] = st;
        if (freed)
            for (int i = 0; i < max_free; ++i) freed[(size_t)b * max_free + i] = -1;
        if (n_freed) n_freed[b] = 0;
        if (st) {
            new_seq_lens[b] = L;
            continue;
        }
        const int new_len = L + len + 1;
        new_seq_lens[b] = new_len;
        /* read every source row first, then write the destinations */
        uint8_t *buf = (uint8_t *)malloc(row_bytes * (size_t)(len + 1) * 2);
        for (int l = 0; l < num_layers; ++l) {
            uint8_t *kl = k_cache + (size_t)l * layer_stride * elem_size;
            uint8_t *vl = v_cache + (size_t)l * layer_stride * elem_size;
            for (int k = 0; k <= len; ++k) {
                const long long t = (long long)L + pb[k];
                const size_t off = ((size_t)pt[t / page_size] * page_size + t % page_size) * row_bytes;
                memcpy(buf + (size_t)(2 * k) * row_bytes, kl + off, row_bytes);
                memcpy(buf + (size_t)(2 * k + 1) * row_bytes, vl + off, row_bytes);
            }
            for (int k = 0; k <= len; ++k) {
                const long long t = (long long)L + k;
                const size_t off = ((size_t)pt[t / page_size] * page_size + t % page_size) * row_bytes;
                memcpy(kl + off, buf + (size_t)(2 * k) * row_bytes, row_bytes);
                memcpy(vl + off, buf + (size_t)(2 * k + 1) * row_bytes, row_bytes);
            }
        }
        free(buf);
        const int first = (new_len + page_size - 1) / page_size;
        const int end = (int)(((long long)L + N + page_size - 1) / page_size);
        int cnt = 0;
        for (int i = first; i < end; ++i) {
            if (freed && cnt < max_free) freed[(size_t)b * max_free + cnt] = pt[i];
            ++cnt;
        }
        if (n_freed) n_freed[b] = cnt;
    }
    return 0;
}
