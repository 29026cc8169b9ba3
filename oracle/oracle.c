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
 *   oracle_spec_accept_greedy  "Eagle vs DFlash", § A fair evaluation
 *                      protocol (greedy decoding must reproduce a target-only
 *                      run): at temperature 0 the target emits its argmax, so
 *                      a draft node is accepted iff its token is the argmax of
 *                      its parent's target row, and the bonus token is the
 *                      argmax at the last accepted node.
 *   oracle_spec_accept_onehot  the sampling rule of oracle_spec_accept with
 *                      q = one-hot(candidate token) for every child, the form
 *                      that stays lossless for deterministic (top-k) siblings.
 *   oracle_eagle2_*    "EAGLE 演化史", § E.2 (a node's value is the product
 *                      of draft confidences on its root path; expand the
 *                      top-k frontier nodes by value into their top-k draft
 *                      tokens each round; rerank all nodes by value and keep
 *                      the top N, a connected subtree) and § E.3 (one worked
 *                      expansion step); "The EAGLE Family", EAGLE-2 (expand,
 *                      then rerank and flatten for verification).
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

/* ------------------------------------------------------------------------ */
/* O6: acceptance variants that read only target rows.                      */
/* ------------------------------------------------------------------------ */

/* Validity of one sequence, as for oracle_spec_accept; resets its outputs. */
static int variant_reset(const int32_t *par, const int32_t *tok, int N, int V, int32_t *path,
                         int32_t *out_tokens, double *ratio, double *accept_margin) {
    int st = 0;
    if (!tree_is_valid(par, N)) st |= ORACLE_BAD_PARENT;
    for (int c = 1; c < N; ++c)
        if (tok[c] < 0 || tok[c] >= V) st |= ORACLE_BAD_TOKEN;
    for (int c = 0; c < N; ++c) {
        path[c] = -1;
        out_tokens[c] = -1;
        if (ratio) ratio[c] = NAN;
        if (accept_margin) accept_margin[c] = NAN;
    }
    return st;
}

/* Greedy: a = argmax of the current node's target logits (the lowest index
 * among equal maxima); accept the first child (ascending index) whose token
 * is a and continue there; stop when no child carries a. The bonus token is
 * the last a. Outputs as for oracle_spec_accept. */
int oracle_spec_accept_greedy(const float *target, const int32_t *tokens, const int32_t *parent,
                              int B, int N, int V, int32_t *accept_len, int32_t *path,
                              int32_t *out_tokens, int32_t *status) {
    if (B < 0 || N < 1 || V <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (size_t)b * N;
        const int32_t *tok = tokens + (size_t)b * N;
        int32_t *pb = path + (size_t)b * N, *ob = out_tokens + (size_t)b * N;
        const int st = variant_reset(par, tok, N, V, pb, ob, NULL, NULL);
        status[b] = st;
        accept_len[b] = 0;
        if (st) continue;
        int cur = 0, len = 0;
        pb[0] = 0;
        for (;;) {
            const float *row = target + ((size_t)b * N + cur) * V;
            int a = 0;
            for (int v = 1; v < V; ++v)
                if (row[v] > row[a]) a = v;
            int next = -1;
            for (int c = cur + 1; c < N; ++c)
                if (par[c] == cur && tok[c] == a) {
                    next = c;
                    break;
                }
            if (next < 0) {
                ob[len] = a;
                break;
            }
            ++len;
            pb[len] = next;
            ob[len - 1] = a;
            cur = next;
        }
        accept_len[b] = len;
    }
    return 0;
}

/* One-hot candidates: the sampling rule with q_c = one-hot(x_c) for child c.
 * With p~ the current target distribution (softmax of the node's row, then
 * residuals), child c is accepted iff u_c * q_c(x_c) = u_c < p~(x_c); on a
 * rejection p~ <- normalize(max(0, p~ - one-hot(x_c))), i.e. x_c loses its
 * mass; when every child is rejected, or at a leaf, the bonus token is the
 * inverse CDF of p~ at u_bonus (smallest k whose cumulative p~ exceeds
 * u * sum(p~), else the last k with p~(k) > 0). ratio = p~(x)/q(x) = p~(x);
 * margins as for oracle_spec_accept. */
int oracle_spec_accept_onehot(const float *target, const int32_t *tokens, const int32_t *parent,
                              const float *u_accept, const float *u_bonus, int B, int N, int V,
                              int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                              double *ratio, double *accept_margin, double *bonus_margin,
                              int32_t *status) {
    if (B < 0 || N < 1 || V <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (size_t)b * N;
        const int32_t *tok = tokens + (size_t)b * N;
        int32_t *pb = path + (size_t)b * N, *ob = out_tokens + (size_t)b * N;
        double *rb = ratio ? ratio + (size_t)b * N : NULL;
        double *mb = accept_margin ? accept_margin + (size_t)b * N : NULL;
        const int st = variant_reset(par, tok, N, V, pb, ob, rb, mb);
        status[b] = st;
        accept_len[b] = 0;
        if (bonus_margin) bonus_margin[b] = NAN;
        if (st) continue;
        double *pt = (double *)malloc(sizeof(double) * V);
        int cur = 0, len = 0;
        pb[0] = 0;
        softmax64(target + ((size_t)b * N + cur) * V, V, pt);
        for (;;) {
            int moved = 0;
            for (int c = cur + 1; c < N && !moved; ++c) {
                if (par[c] != cur) continue;
                const int x = tok[c];
                const double u = (double)u_accept[(size_t)b * N + c];
                const double px = pt[x];
                if (rb) rb[c] = px;
                if (mb) {
                    const double hi = u > px ? u : px;
                    mb[c] = hi > 0 ? fabs(u - px) / hi : 0.0;
                }
                if (u < px) {
                    ++len;
                    pb[len] = c;
                    ob[len - 1] = x;
                    cur = c;
                    softmax64(target + ((size_t)b * N + cur) * V, V, pt);
                    moved = 1;
                } else {
                    /* p~ <- normalize(max(0, p~ - one-hot(x))) */
                    double S = 0.0;
                    for (int v = 0; v < V; ++v) {
                        const double r = pt[v] - (v == x ? 1.0 : 0.0);
                        pt[v] = r > 0.0 ? r : 0.0;
                        S += pt[v];
                    }
                    if (S > 0.0)
                        for (int v = 0; v < V; ++v) pt[v] /= S;
                }
            }
            if (!moved) break;
        }
        double tot = 0.0;
        for (int v = 0; v < V; ++v) tot += pt[v];
        const double thr = (double)u_bonus[b] * tot;
        double cum = 0.0, prev = 0.0;
        int pick = -1;
        for (int v = 0; v < V; ++v) {
            prev = cum;
            cum += pt[v];
            if (cum > thr) {
                pick = v;
                break;
            }
        }
        double margin = 0.0;
        if (pick < 0) {
            for (int v = V - 1; v >= 0; --v)
                if (pt[v] > 0.0) {
                    pick = v;
                    break;
                }
        } else {
            const double a = thr - prev, c2 = cum - thr;
            margin = (a < c2 ? a : c2) / tot;
        }
        ob[len] = pick;
        accept_len[b] = len;
        if (bonus_margin) bonus_margin[b] = margin;
        free(pt);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O8: EAGLE-2 dynamic tree construction, fp64.                              */
/* A pool per sequence holds every node created so far, by creation id      */
/* (cid): parent cid (-1 for the root), depth, token and value. The root is  */
/* cid 0 with value 1. One expansion round takes the draft logits row of    */
/* each frontier node (frontier[b][r], -1 entries only at the end), creates */
/* for each its top-k draft tokens (by probability, ties to the lower id)   */
/* as children with value = parent value * confidence, the confidence being */
/* the draft softmax probability of the child's token, numbered in order of */
/* frontier position then rank; the next frontier is the top-k of the new   */
/* children by (value desc, cid asc), -1 padded. select_gap[b] reports the */
/* relative gap between the last selected and the first unselected value   */
/* (+inf when nothing was left out), so a caller can tell near ties.        */
/* ------------------------------------------------------------------------ */
int oracle_eagle2_expand(const float *rows, int B, int R, int V, int k, const int32_t *frontier,
                         int C, int32_t *pool_parent, int32_t *pool_depth, int32_t *pool_token,
                         double *pool_value, int32_t *pool_count, int32_t *next_frontier,
                         double *select_gap) {
    if (B < 0 || R < 1 || V < 1 || k < 1 || k > V || C < 1) return -1;
    for (int b = 0; b < B; ++b) {
        int32_t *pp = pool_parent + (size_t)b * C, *pd = pool_depth + (size_t)b * C;
        int32_t *pt = pool_token + (size_t)b * C;
        double *pv = pool_value + (size_t)b * C;
        const int first = pool_count[b];
        int cnt = first;
        double *prob = (double *)malloc(sizeof(double) * V);
        char *taken = (char *)malloc((size_t)V);
        for (int r = 0; r < R; ++r) {
            const int f = frontier[(size_t)b * R + r];
            if (f < 0) break;
            softmax64(rows + ((size_t)b * R + r) * V, V, prob);
            memset(taken, 0, (size_t)V);
            for (int i = 0; i < k; ++i) {
                int best = -1;
                for (int v = 0; v < V; ++v)
                    if (!taken[v] && (best < 0 || prob[v] > prob[best])) best = v;
                taken[best] = 1;
                if (cnt < C) {
                    pp[cnt] = f;
                    pd[cnt] = pd[f] + 1;
                    pt[cnt] = best;
                    pv[cnt] = pv[f] * prob[best];
                }
                ++cnt;
            }
        }
        if (cnt > C) cnt = C;
        pool_count[b] = cnt;
        /* next frontier: top-k of the new children by (value desc, cid asc) */
        char *sel = (char *)calloc((size_t)(cnt - first) + 1, 1);
        double last = INFINITY;
        for (int i = 0; i < k; ++i) {
            int best = -1;
            for (int c = first; c < cnt; ++c)
                if (!sel[c - first] && (best < 0 || pv[c] > pv[best])) best = c;
            next_frontier[(size_t)b * k + i] = best;
            if (best >= 0) {
                sel[best - first] = 1;
                last = pv[best];
            }
        }
        double gap = INFINITY;
        for (int c = first; c < cnt; ++c)
            if (!sel[c - first] && last > 0.0) {
                const double g = (last - pv[c]) / last;
                if (g < gap) gap = g;
            }
        if (select_gap) select_gap[b] = gap;
        free(sel);
        free(prob);
        free(taken);
    }
    return 0;
}

/* Rerank and flatten: keep the root and the n_nodes - 1 best other nodes by */
/* (value desc, depth asc, cid asc); number them in BFS order, level by     */
/* level, a level ordered by (parent's new index, value desc, cid asc).     */
/* Outputs [B, n_nodes]: parent (new indices, -1 for the root), token,      */
/* value, cid; -1 / 0 padded when the pool holds fewer nodes. n_out[b] is  */
/* the number of nodes kept, cut_gap[b] the relative gap between the last   */
/* kept and the first dropped value (+inf when nothing was dropped), and   */
/* connected[b] 1 if every kept node's parent was kept.                     */
int oracle_eagle2_finalize(int B, int C, const int32_t *pool_parent, const int32_t *pool_depth,
                           const int32_t *pool_token, const double *pool_value,
                           const int32_t *pool_count, int n_nodes, int32_t *parent,
                           int32_t *token, double *value, int32_t *cid, int32_t *n_out,
                           double *cut_gap, int32_t *connected) {
    if (B < 0 || C < 1 || n_nodes < 1) return -1;
    for (int b = 0; b < B; ++b) {
        const int32_t *pp = pool_parent + (size_t)b * C, *pd = pool_depth + (size_t)b * C;
        const int32_t *pt = pool_token + (size_t)b * C;
        const double *pv = pool_value + (size_t)b * C;
        const int cnt = pool_count[b];
        int32_t *ob_p = parent + (size_t)b * n_nodes, *ob_t = token + (size_t)b * n_nodes;
        int32_t *ob_c = cid + (size_t)b * n_nodes;
        double *ob_v = value + (size_t)b * n_nodes;
        for (int i = 0; i < n_nodes; ++i) {
            ob_p[i] = -1;
            ob_t[i] = -1;
            ob_c[i] = -1;
            ob_v[i] = 0.0;
        }
        char *kept = (char *)calloc((size_t)cnt, 1);
        kept[0] = 1;
        int nk = 1;
        double last = INFINITY;
        while (nk < n_nodes) {
            int best = -1;
            for (int c = 1; c < cnt; ++c) {
                if (kept[c]) continue;
                if (best < 0 || pv[c] > pv[best] || (pv[c] == pv[best] && pd[c] < pd[best]))
                    best = c;
            }
            if (best < 0) break;
            kept[best] = 1;
            last = pv[best];
            ++nk;
        }
        double gap = INFINITY;
        for (int c = 1; c < cnt; ++c)
            if (!kept[c] && last > 0.0 && last < INFINITY) {
                const double g = (last - pv[c]) / last;
                if (g < gap) gap = g;
            }
        int conn = 1;
        for (int c = 1; c < cnt; ++c)
            if (kept[c] && !kept[pp[c]]) conn = 0;
        /* BFS numbering */
        int *newidx = (int *)malloc(sizeof(int) * (size_t)cnt);
        char *placed = (char *)calloc((size_t)cnt, 1);
        for (int c = 0; c < cnt; ++c) newidx[c] = -1;
        newidx[0] = 0;
        placed[0] = 1;
        ob_p[0] = -1;
        ob_t[0] = pt[0];
        ob_v[0] = pv[0];
        ob_c[0] = 0;
        int at = 1;
        for (int d = 1; at < nk; ++d) {
            for (;;) {
                int best = -1;
                for (int c = 1; c < cnt; ++c) {
                    if (!kept[c] || placed[c] || pd[c] != d || newidx[pp[c]] < 0) continue;
                    if (best < 0) {
                        best = c;
                        continue;
                    }
                    const int a1 = newidx[pp[c]], a0 = newidx[pp[best]];
                    if (a1 < a0 || (a1 == a0 && (pv[c] > pv[best] ||
                                                 (pv[c] == pv[best] && c < best))))
                        best = c;
                }
                if (best < 0) break;
                placed[best] = 1;
                newidx[best] = at;
                ob_p[at] = newidx[pp[best]];
                ob_t[at] = pt[best];
                ob_v[at] = pv[best];
                ob_c[at] = best;
                ++at;
            }
            if (d > C) break;
        }
        n_out[b] = at;
        if (cut_gap) cut_gap[b] = gap;
        if (connected) connected[b] = conn;
        free(kept);
        free(newidx);
        free(placed);
    }
    return 0;
}

/*
 * LM head. "The EAGLE Family: Speculating in Feature Space", § Why predict
 * features instead of tokens?: the target's next-token distribution is
 * softmax(W_LM h_t), the LM head being a fixed linear map of the last hidden
 * state. "EAGLE 演化史", § D.2, puts the verify pass's bandwidth cost here:
 * one vocabulary-sized product per tree node.
 *
 * Inputs:  h [R, H] (one hidden state per tree node, R = B * N), W [V, H]
 *          (row v = the LM-head weights of token v); bf16 values arrive
 *          widened exactly to float.
 * Output:  logits [R, V] fp64: sum over k of h[r][k] * W[v][k], accumulated
 *          in fp64 in increasing k.
 */
int oracle_lm_head(const float *h, const float *W, int R, int H, int V, double *logits) {
    if (R < 0 || H < 1 || V < 1) return -1;
#pragma omp parallel for schedule(static)
    for (long long rv = 0; rv < (long long)R * V; ++rv) {
        const long long r = rv / V, v = rv % V;
        const float *hr = h + r * H, *wv = W + v * H;
        double s = 0.0;
        for (int k = 0; k < H; ++k) s += (double)hr[k] * (double)wv[k];
        logits[rv] = s;
    }
    return 0;
}
