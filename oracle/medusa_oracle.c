/*
 * medusa_oracle.c -- plain, slow CPU oracle of the Medusa decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the bench may load this library.  It shares no code, header,
 * table or constant with the CUDA library; it is written from the method's
 * definition, in float64, one obvious loop at a time.
 *
 * Sources, cited by page title and section:
 *   [MH]  "Medusa Heads" glossary page (Arabic and Portuguese editions), sections
 *         "How heads predict later tokens" and "Tree attention and acceptance".
 *   [SD]  "Giai ma dau co: doan truoc roi kiem mot luot" (speculative decoding
 *         e-book page), sections "Why a round always yields exactly k + 1
 *         tokens" and "Faster without changing the result".
 *
 * Every input is decoded exactly (bf16 -> float -> double) and all arithmetic is
 * double unless a comment says otherwise.  Readings of points the pages leave
 * open are stated where they are used.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_ENOMEM (-2)

/* dtype codes of this oracle's interface: 0 = float32, 1 = bf16 bit patterns. */
static double load(const void* base, int dtype, size_t i) {
    if (dtype == 0) return (double)((const float*)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* O1: Medusa heads [MH, "How heads predict later tokens"].                   */
/* Head k reads the last hidden state h and computes                          */
/*   logits_k = W2_k (h + SiLU(W1_k h + b1_k)),   SiLU(x) = x * sigmoid(x),    */
/* with W1_k a hidden x hidden linear layer with bias and W2_k a bias-free    */
/* hidden -> vocab projection, both stored [out, in] like a linear layer.     */
/* ------------------------------------------------------------------------- */
int oracle_heads_logits(const void* h, const void* w1, const void* b1, const void* w2,
                        int dtype, int B, int K, int H, int V,
                        double* z_out /* [B,K,H] or NULL */, double* logits /* [B,K,V] */) {
    if (B < 0 || K < 0 || H <= 0 || V <= 0 || !h || !w1 || !b1 || !w2 || !logits)
        return OR_EINVAL;
    double* z = (double*)malloc((size_t)H * sizeof(double));
    if (!z) return OR_ENOMEM;
    for (int b = 0; b < B; ++b) {
        for (int k = 0; k < K; ++k) {
            for (int i = 0; i < H; ++i) {
                double u = load(b1, dtype, (size_t)k * H + i);
                for (int j = 0; j < H; ++j)
                    u += load(w1, dtype, ((size_t)k * H + i) * H + j) * load(h, dtype, (size_t)b * H + j);
                double silu = u / (1.0 + exp(-u));
                z[i] = load(h, dtype, (size_t)b * H + i) + silu;
                if (z_out) z_out[((size_t)b * K + k) * H + i] = z[i];
            }
            for (int v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int i = 0; i < H; ++i)
                    acc += load(w2, dtype, ((size_t)k * V + v) * H + i) * z[i];
                logits[((size_t)b * K + k) * V + v] = acc;
            }
        }
    }
    free(z);
    return OR_OK;
}

/* The lm_head's own next-token logits: lm_head h, the "+1" prediction that the
 * heads start from when W1 = b1 = 0 and W2 = lm_head [MH]. */
int oracle_lm_head_logits(const void* h, const void* lm, int dtype, int B, int H, int V,
                          double* logits /* [B,V] */) {
    if (!h || !lm || !logits || H <= 0 || V <= 0) return OR_EINVAL;
    for (int b = 0; b < B; ++b)
        for (int v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int i = 0; i < H; ++i)
                acc += load(lm, dtype, (size_t)v * H + i) * load(h, dtype, (size_t)b * H + i);
            logits[(size_t)b * V + v] = acc;
        }
    return OR_OK;
}

/* Top-k of one row: the k largest values, larger value first, lower index first
 * among equal values.  Done as k passes of "take the best not yet taken". */
int oracle_topk(const double* x, int n, int k, int32_t* idx, double* val) {
    if (!x || n <= 0 || k <= 0 || k > n || !idx) return OR_EINVAL;
    unsigned char* taken = (unsigned char*)calloc((size_t)n, 1);
    if (!taken) return OR_ENOMEM;
    for (int t = 0; t < k; ++t) {
        int best = -1;
        for (int v = 0; v < n; ++v) {
            if (taken[v]) continue;
            if (best < 0 || x[v] > x[best]) best = v; /* strict: keeps the lower index on ties */
        }
        taken[best] = 1;
        idx[t] = best;
        if (val) val[t] = x[best];
    }
    free(taken);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* O2: candidate tree [MH, "Tree attention and acceptance"].                  */
/* The heads' top guesses combine into candidate continuations that share     */
/* prefixes: a node is a tuple of ranks (r_1..r_d), r_k being a rank in head  */
/* k's top-k list, and its parent is (r_1..r_{d-1}).  Canonical node order    */
/* (a reading; the pages fix none): the root first, then by depth, then by    */
/* rank tuple in lexicographic order.                                         */
/* ------------------------------------------------------------------------- */
static int tuple_cmp(const int32_t* a, const int32_t* b, int maxd) {
    int da = 0, db = 0;
    while (da < maxd && a[da] >= 0) ++da;
    while (db < maxd && b[db] >= 0) ++db;
    if (da != db) return da < db ? -1 : 1;
    for (int i = 0; i < da; ++i)
        if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
    return 0;
}

static int tuple_len(const int32_t* a, int maxd) {
    int d = 0;
    while (d < maxd && a[d] >= 0) ++d;
    return d;
}

/* paths: P rank tuples of max_depth entries each, padded with -1 after the last
 * rank.  Every prefix of every tuple becomes a node.  Outputs (capacity
 * cap_nodes nodes, cap_paths retrieve rows):
 *   parent[N], depth[N], rank[N] (rank of the last head; -1 for the root),
 *   mask[N*W] (bit m of row i set iff node m is node i or an ancestor of it),
 *   retrieve[n_paths*(max_depth+1)]: for each leaf, in leaf index order, the
 *   node indices from the root to the leaf, padded with -1. */
int oracle_tree_layout(const int32_t* paths, int P, int max_depth, int cap_nodes, int cap_paths,
                       int32_t* parent, int32_t* depth, int32_t* rank, uint64_t* mask,
                       int32_t* retrieve, int* N_out, int* W_out, int* n_paths_out) {
    if (!paths || P < 0 || max_depth <= 0 || !parent || !depth || !rank || !N_out || !W_out)
        return OR_EINVAL;
    /* Validate: ranks >= 0 before the padding, -1 after it. */
    for (int p = 0; p < P; ++p) {
        int d = tuple_len(paths + (size_t)p * max_depth, max_depth);
        for (int i = d; i < max_depth; ++i)
            if (paths[(size_t)p * max_depth + i] != -1) return OR_EINVAL;
    }
    /* Collect every prefix (lengths 0..d) of every tuple. */
    size_t cap = 1 + (size_t)P * max_depth;
    int32_t* nodes = (int32_t*)malloc(cap * max_depth * sizeof(int32_t));
    if (!nodes) return OR_ENOMEM;
    size_t n = 0;
    for (int i = 0; i < max_depth; ++i) nodes[i] = -1; /* the root: empty tuple */
    n = 1;
    for (int p = 0; p < P; ++p) {
        const int32_t* t = paths + (size_t)p * max_depth;
        int d = tuple_len(t, max_depth);
        for (int len = 1; len <= d; ++len) {
            int32_t* dst = nodes + n * max_depth;
            for (int i = 0; i < max_depth; ++i) dst[i] = i < len ? t[i] : -1;
            ++n;
        }
    }
    /* Sort canonically (insertion sort: slow and plain), then drop duplicates. */
    int32_t* tmp = (int32_t*)malloc((size_t)max_depth * sizeof(int32_t));
    if (!tmp) { free(nodes); return OR_ENOMEM; }
    for (size_t i = 1; i < n; ++i) {
        memcpy(tmp, nodes + i * max_depth, (size_t)max_depth * sizeof(int32_t));
        size_t j = i;
        while (j > 0 && tuple_cmp(nodes + (j - 1) * max_depth, tmp, max_depth) > 0) {
            memcpy(nodes + j * max_depth, nodes + (j - 1) * max_depth, (size_t)max_depth * sizeof(int32_t));
            --j;
        }
        memcpy(nodes + j * max_depth, tmp, (size_t)max_depth * sizeof(int32_t));
    }
    free(tmp);
    size_t u = 0;
    for (size_t i = 0; i < n; ++i) {
        if (u > 0 && tuple_cmp(nodes + (u - 1) * max_depth, nodes + i * max_depth, max_depth) == 0) continue;
        if (u != i) memcpy(nodes + u * max_depth, nodes + i * max_depth, (size_t)max_depth * sizeof(int32_t));
        ++u;
    }
    n = u;
    if ((int)n > cap_nodes) { free(nodes); return OR_EINVAL; }
    int N = (int)n, W = (N + 63) / 64;
    /* parent = the node whose tuple is this tuple without its last rank */
    for (int i = 0; i < N; ++i) {
        const int32_t* t = nodes + (size_t)i * max_depth;
        int d = tuple_len(t, max_depth);
        depth[i] = d;
        rank[i] = d > 0 ? t[d - 1] : -1;
        parent[i] = -1;
        if (d == 0) continue;
        for (int j = 0; j < N; ++j) {
            const int32_t* s = nodes + (size_t)j * max_depth;
            if (tuple_len(s, max_depth) != d - 1) continue;
            int same = 1;
            for (int e = 0; e < d - 1; ++e) same &= (s[e] == t[e]);
            if (same) { parent[i] = j; break; }
        }
    }
    free(nodes);
    if (mask) {
        memset(mask, 0, (size_t)N * W * sizeof(uint64_t));
        for (int i = 0; i < N; ++i)
            for (int a = i; a >= 0; a = parent[a])
                mask[(size_t)i * W + a / 64] |= (uint64_t)1 << (a % 64);
    }
    int np = 0;
    for (int i = 0; i < N; ++i) {
        int has_child = 0;
        for (int j = 0; j < N; ++j) has_child |= (parent[j] == i);
        if (has_child) continue;
        if (retrieve) {
            if (np >= cap_paths) return OR_EINVAL;
            int32_t* row = retrieve + (size_t)np * (max_depth + 1);
            for (int e = 0; e <= max_depth; ++e) row[e] = -1;
            for (int a = i; a >= 0; a = parent[a]) row[depth[a]] = a;
        }
        ++np;
    }
    *N_out = N;
    *W_out = W;
    if (n_paths_out) *n_paths_out = np;
    return OR_OK;
}

/* Sparse tree: the n_nodes - 1 "most accurate combinations" [MH, "Tree attention
 * and acceptance"], with the accuracy of a rank tuple (r_1..r_d) read as the
 * product over its heads of head_p^k * rank_p^(r_k) (head k, rank r, ranks
 * counted from 0).  The product equals head_p^(d(d+1)/2) * rank_p^(sum r);
 * tuples are ranked by that value, larger first, then by depth, then
 * lexicographically.  Every factor is below 1, so the chosen set contains the
 * prefix of each of its tuples.  Tuples range over depth 1..max_depth and ranks
 * 0..max_rank-1.  Output: n_nodes - 1 tuples (max_depth entries, -1 padded) in
 * canonical node order. */
typedef struct { double key; int32_t t[16]; int d; } sp_item;

static int sp_better(const sp_item* a, const sp_item* b) {
    /* Equal (depth, rank sum) means an equal accuracy; only then tie-break. */
    if (a->key != b->key) return a->key > b->key;
    if (a->d != b->d) return a->d < b->d;
    for (int i = 0; i < a->d; ++i)
        if (a->t[i] != b->t[i]) return a->t[i] < b->t[i];
    return 0;
}

int oracle_sparse_tree_paths(int n_nodes, int max_depth, int max_rank, double head_p, double rank_p,
                             int32_t* paths_out /* [(n_nodes-1)*max_depth] */) {
    if (n_nodes < 1 || max_depth < 1 || max_depth > 16 || max_rank < 1 || !paths_out) return OR_EINVAL;
    if (!(head_p > 0 && head_p < 1 && rank_p > 0 && rank_p < 1)) return OR_EINVAL;
    size_t total = 0, cnt = 1;
    for (int d = 1; d <= max_depth; ++d) { cnt *= (size_t)max_rank; total += cnt; if (total > 50000000) return OR_EINVAL; }
    if ((size_t)(n_nodes - 1) > total) return OR_EINVAL;
    sp_item* all = (sp_item*)malloc(total * sizeof(sp_item));
    if (!all) return OR_ENOMEM;
    size_t n = 0;
    for (int d = 1; d <= max_depth; ++d) {
        int32_t t[16] = {0};
        for (;;) {
            sp_item* it = &all[n++];
            it->d = d;
            int sum = 0;
            for (int i = 0; i < 16; ++i) it->t[i] = i < d ? t[i] : -1;
            for (int i = 0; i < d; ++i) sum += t[i];
            /* log of head_p^(d(d+1)/2) * rank_p^sum, the same expression for every tuple */
            it->key = (double)(d * (d + 1) / 2) * log(head_p) + (double)sum * log(rank_p);
            int pos = d - 1;
            while (pos >= 0 && ++t[pos] == max_rank) { t[pos] = 0; --pos; }
            if (pos < 0) break;
        }
    }
    /* Selection: n_nodes-1 passes of "take the best not yet taken". */
    unsigned char* taken = (unsigned char*)calloc(n, 1);
    int32_t* chosen = (int32_t*)malloc((size_t)(n_nodes > 1 ? n_nodes - 1 : 1) * sizeof(int32_t));
    if (!taken || !chosen) { free(all); free(taken); free(chosen); return OR_ENOMEM; }
    for (int c = 0; c < n_nodes - 1; ++c) {
        long best = -1;
        for (size_t i = 0; i < n; ++i)
            if (!taken[i] && (best < 0 || sp_better(&all[i], &all[best]))) best = (long)i;
        taken[best] = 1;
        chosen[c] = (int32_t)best;
    }
    /* canonical order: by depth, then lexicographic */
    for (int i = 1; i < n_nodes - 1; ++i) {
        int32_t x = chosen[i];
        int j = i;
        while (j > 0) {
            const sp_item* a = &all[chosen[j - 1]];
            const sp_item* b = &all[x];
            int gt = a->d != b->d ? a->d > b->d : 0;
            if (a->d == b->d)
                for (int e = 0; e < a->d; ++e)
                    if (a->t[e] != b->t[e]) { gt = a->t[e] > b->t[e]; break; }
            if (!gt) break;
            chosen[j] = chosen[j - 1];
            --j;
        }
        chosen[j] = x;
    }
    for (int c = 0; c < n_nodes - 1; ++c)
        for (int i = 0; i < max_depth; ++i)
            paths_out[(size_t)c * max_depth + i] = i < 16 ? all[chosen[c]].t[i] : -1;
    free(all); free(taken); free(chosen);
    return OR_OK;
}

/* Candidate tokens [MH, "Tree attention and acceptance"]: the root holds the
 * base model's own next token; node i of depth d >= 1 holds the token at rank
 * rank_i of head d's top-k list (head k scores position t + k + 1, so head d
 * fills depth d). */
int oracle_build_tree(const int32_t* topk_idx /* [B,K,topk] */, const int32_t* root_tok /* [B] */,
                      const int32_t* depth, const int32_t* rank, int B, int K, int topk, int N,
                      int32_t* cand /* [B,N] */) {
    if (!topk_idx || !root_tok || !depth || !rank || !cand) return OR_EINVAL;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < N; ++i) {
            if (depth[i] == 0) { cand[(size_t)b * N + i] = root_tok[b]; continue; }
            if (depth[i] > K || rank[i] < 0 || rank[i] >= topk) return OR_EINVAL;
            cand[(size_t)b * N + i] = topk_idx[((size_t)b * K + depth[i] - 1) * topk + rank[i]];
        }
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* O3: tree attention [MH, "Tree attention and acceptance"]: every candidate  */
/* is appended to the input at once and may see only its tree ancestors.      */
/* Query i of sequence b attends to the prefix keys [0, L_b) and to the tree  */
/* keys at slots L_b + m for every m with bit m of mask row i set.  Textbook  */
/* softmax(scale * q.k) v over that key set, two passes (max, then sums).     */
/* rows: optional list of (b, i, hq) triples to compute; NULL = all, in       */
/* [B,N,Hq] order.  out: [n_rows, D].                                         */
/* ------------------------------------------------------------------------- */
int oracle_tree_attention(const void* q, const void* kc, const void* vc, const int32_t* kv_len,
                          const uint64_t* mask, int dtype, int B, int N, int Hq, int Hkv, int D,
                          int Lmax, double scale, const int32_t* rows, int n_rows, double* out) {
    if (!q || !kc || !vc || !kv_len || !mask || !out || Hkv <= 0 || Hq % Hkv) return OR_EINVAL;
    int W = (N + 63) / 64;
    int total = rows ? n_rows : B * N * Hq;
    double* s = (double*)malloc((size_t)(Lmax + N) * sizeof(double));
    if (!s) return OR_ENOMEM;
    for (int r = 0; r < total; ++r) {
        int b, i, hq;
        if (rows) { b = rows[3 * r]; i = rows[3 * r + 1]; hq = rows[3 * r + 2]; }
        else { b = r / (N * Hq); i = (r / Hq) % N; hq = r % Hq; }
        int hk = hq / (Hq / Hkv);
        int L = kv_len[b];
        if (L < 0 || L + N > Lmax) { free(s); return OR_EINVAL; }
        size_t qoff = (((size_t)b * N + i) * Hq + hq) * D;
        size_t kvbase = ((size_t)b * Hkv + hk) * Lmax;
        /* allowed keys: slots [0, L) and L + m for tree ancestors m */
        int nk = 0;
        double mx = -INFINITY;
        for (int j = 0; j < L + N; ++j) {
            int allowed = j < L || ((mask[(size_t)i * W + (j - L) / 64] >> ((j - L) % 64)) & 1);
            if (!allowed) continue;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += load(q, dtype, qoff + d) * load(kc, dtype, (kvbase + j) * D + d);
            s[nk++] = scale * dot;
            (void)0;
        }
        for (int t = 0; t < nk; ++t) if (s[t] > mx) mx = s[t];
        double den = 0.0;
        for (int t = 0; t < nk; ++t) den += exp(s[t] - mx);
        for (int d = 0; d < D; ++d) out[(size_t)r * D + d] = 0.0;
        int t = 0;
        for (int j = 0; j < L + N; ++j) {
            int allowed = j < L || ((mask[(size_t)i * W + (j - L) / 64] >> ((j - L) % 64)) & 1);
            if (!allowed) continue;
            double w = exp(s[t++] - mx) / den;
            for (int d = 0; d < D; ++d) out[(size_t)r * D + d] += w * load(vc, dtype, (kvbase + j) * D + d);
        }
    }
    free(s);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* O4: acceptance on the tree [MH, "Tree attention and acceptance"].          */
/* The verifier's logits row of node u scores the token that follows u.       */
/* Greedy: a candidate is accepted when it equals the model's top choice      */
/*   after its parent (argmax of the parent's row, lowest token on ties).     */
/* Typical (the entropy-tied threshold; its form is this build's reading):    */
/*   P = softmax(row / T), H = -sum P ln P, tau = min(eps, delta * exp(-H));  */
/*   the candidate is accepted when P(candidate) > tau of its parent's row.   */
/* A node counts only if its parent counts (the root always does).  The       */
/* longest accepted branch ends at the deepest accepted node, lowest index on */
/* ties; accept_len = its depth, and the round's extra token is the argmax of */
/* its row ([SD, "Why a round always yields exactly k + 1 tokens"]).          */
/* ------------------------------------------------------------------------- */
int oracle_verify_tree(const float* logits, const int32_t* cand, const int32_t* parent, const int32_t* depth,
                       int B, int N, int V, int Dmax, int mode, double T, double eps, double delta,
                       int32_t* accept_len, int32_t* best_node, int32_t* path_nodes, int32_t* next_tok,
                       int32_t* argmax_out /* [B,N] or NULL */, double* tau_out /* [B,N] or NULL */,
                       double* pcand_out /* [B,N]: P_parent(cand) (typical) or NULL */,
                       uint8_t* accepted_out /* [B,N] or NULL */) {
    if (!logits || !cand || !parent || !depth || !accept_len || !best_node || !path_nodes || !next_tok)
        return OR_EINVAL;
    if (mode != 0 && mode != 1) return OR_EINVAL;
    int32_t* amax = (int32_t*)malloc((size_t)N * sizeof(int32_t));
    double* tau = (double*)malloc((size_t)N * sizeof(double));
    uint8_t* acc = (uint8_t*)malloc((size_t)N);
    double* P = (double*)malloc((size_t)V * sizeof(double));
    double* pc = (double*)malloc((size_t)N * sizeof(double));
    if (!amax || !tau || !acc || !P || !pc) { free(amax); free(tau); free(acc); free(P); free(pc); return OR_ENOMEM; }
    for (int b = 0; b < B; ++b) {
        for (int u = 0; u < N; ++u) {
            const float* row = logits + ((size_t)b * N + u) * V;
            int a = 0;
            for (int v = 1; v < V; ++v) if (row[v] > row[a]) a = v;
            amax[u] = a;
            tau[u] = 0.0;
        }
        for (int j = 0; j < N; ++j) pc[j] = 0.0;
        if (mode == 1) {
            for (int u = 0; u < N; ++u) {
                const float* row = logits + ((size_t)b * N + u) * V;
                double mx = -INFINITY, den = 0.0, H = 0.0;
                for (int v = 0; v < V; ++v) if ((double)row[v] / T > mx) mx = (double)row[v] / T;
                for (int v = 0; v < V; ++v) { P[v] = exp((double)row[v] / T - mx); den += P[v]; }
                for (int v = 0; v < V; ++v) { P[v] /= den; if (P[v] > 0) H -= P[v] * log(P[v]); }
                double t = delta * exp(-H);
                tau[u] = eps < t ? eps : t;
                for (int j = 1; j < N; ++j)
                    if (parent[j] == u) pc[j] = P[cand[(size_t)b * N + j]];
            }
        }
        acc[0] = 1;
        for (int j = 1; j < N; ++j) { /* parents precede children in node order */
            int u = parent[j];
            int pass = mode == 0 ? (cand[(size_t)b * N + j] == amax[u]) : (pc[j] > tau[u]);
            acc[j] = (uint8_t)(acc[u] && pass);
        }
        int best = 0;
        for (int j = 1; j < N; ++j)
            if (acc[j] && depth[j] > depth[best]) best = j; /* strict: lowest index on equal depth */
        accept_len[b] = depth[best];
        best_node[b] = best;
        next_tok[b] = amax[best];
        for (int e = 0; e <= Dmax; ++e) path_nodes[(size_t)b * (Dmax + 1) + e] = -1;
        for (int a = best; a >= 0; a = parent[a]) path_nodes[(size_t)b * (Dmax + 1) + depth[a]] = a;
        for (int u = 0; u < N; ++u) {
            if (argmax_out) argmax_out[(size_t)b * N + u] = amax[u];
            if (tau_out) tau_out[(size_t)b * N + u] = tau[u];
            if (pcand_out) pcand_out[(size_t)b * N + u] = pc[u];
            if (accepted_out) accepted_out[(size_t)b * N + u] = acc[u];
        }
    }
    free(amax); free(tau); free(acc); free(P); free(pc);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* O5: speculative sampling along a chain of gamma drafts                     */
/* [SD, "Faster without changing the result"; "Why a round always yields      */
/* exactly k + 1 tokens"].  Draft x_i ~ q_i is accepted with probability      */
/* min(1, p_i(x_i)/q_i(x_i)); at the first rejection a token is drawn from    */
/* max(0, p_i - q_i) normalised, and the round stops; if all gamma are        */
/* accepted, a bonus token is drawn from p_{gamma+1}.  k + 1 tokens result.   */
/*                                                                            */
/* Random numbers: SplitMix64 (Steele, Lea and Flood, 2014).  sm_next(s, n)   */
/* is the n-th output of the generator started from state s.                  */
/*   f(x)    = sm_next(x, 1)                                                  */
/*   row key = f(f(f(f(f(seed) ^ stream) ^ b) ^ round) ^ pos)                 */
/*   U(h)    = (h >> 40) / 2^24 in [0,1)  (accept uniforms: h = sm_next(row   */
/*             key, 1))                                                       */
/*   race uniforms: one output serves two vocab entries, h_m = sm_next(row    */
/*             key, m + 1) for entries 2m and 2m + 1; entry 2m takes bits     */
/*             40..63 and entry 2m + 1 bits 16..39:                           */
/*             Up_v = (bits_v + 1) / 2^24 in (0, 1]                           */
/* streams: 1 = accept uniform (v = 0), 2 = residual draw, 3 = bonus draw;   */
/* pos counts draft positions from 1.                                         */
/* Accept test: u * q_i(x_i) < p_i(x_i), exact in double (u has 24 bits).     */
/* Draw from weights w: argmin over w_v > 0 of -ln(Up_v) / w_v, lowest v      */
/* on ties (the exponential race); if no weight is positive, argmax of p_i.   */
/* ------------------------------------------------------------------------- */
#define SM_GAMMA 0x9E3779B97F4A7C15ULL
static uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}
static uint64_t sm_next(uint64_t state, uint64_t n) { return sm_mix(state + n * SM_GAMMA); }

uint64_t oracle_splitmix64(uint64_t state, uint64_t n) { return sm_next(state, n); }

uint64_t oracle_row_key(uint64_t seed, uint64_t stream, uint64_t b, uint64_t round, uint64_t pos) {
    uint64_t x = sm_next(seed, 1);
    x = sm_next(x ^ stream, 1);
    x = sm_next(x ^ b, 1);
    x = sm_next(x ^ round, 1);
    return sm_next(x ^ pos, 1);
}

static double unif(uint64_t h) { return (double)(h >> 40) * (1.0 / 16777216.0); }
/* Up_v of the race: two disjoint 24-bit fields of one generator output */
static double race_unif(uint64_t key, int v) {
    const uint64_t h = sm_next(key, (uint64_t)(v >> 1) + 1);
    const uint64_t bits = (v & 1) ? ((h >> 16) & 0xFFFFFFULL) : (h >> 40);
    return (double)(bits + 1) * (1.0 / 16777216.0);
}

/* exponential race over weights w[V]; returns the chosen token, and the gap
 * between the best and second-best keys relative to the best (for tie checks) */
static int race(const double* w, const float* p_fallback, int V, uint64_t key, double* rel_gap) {
    int best = -1;
    double k1 = INFINITY, k2 = INFINITY;
    for (int v = 0; v < V; ++v) {
        if (!(w[v] > 0.0)) continue;
        double kv = -log(race_unif(key, v)) / w[v];
        if (kv < k1) { k2 = k1; k1 = kv; best = v; }
        else if (kv < k2) k2 = kv;
    }
    if (best < 0) {
        best = 0;
        for (int v = 1; v < V; ++v) if (p_fallback[v] > p_fallback[best]) best = v;
        if (rel_gap) *rel_gap = INFINITY;
        return best;
    }
    if (rel_gap) *rel_gap = k1 > 0 ? (k2 - k1) / k1 : (k2 > 0 ? INFINITY : 0.0);
    return best;
}

int oracle_verify_chain(const float* p /* [B,gamma+1,V] */, const float* q /* [B,gamma,V] */,
                        const int32_t* draft /* [B,gamma] */, int B, int gamma, int V,
                        uint64_t seed, uint64_t round, int32_t* n_acc /* [B] */,
                        int32_t* out_tok /* [B,gamma+1] */, double* race_gap /* [B] or NULL */) {
    if (!p || (gamma > 0 && (!q || !draft)) || !n_acc || !out_tok || gamma < 0 || V <= 0) return OR_EINVAL;
    double* w = (double*)malloc((size_t)V * sizeof(double));
    if (!w) return OR_ENOMEM;
    for (int b = 0; b < B; ++b) {
        int k = 0;
        for (int e = 0; e <= gamma; ++e) out_tok[(size_t)b * (gamma + 1) + e] = -1;
        int rejected = 0;
        for (int i = 1; i <= gamma; ++i) {
            int x = draft[(size_t)b * gamma + i - 1];
            if (x < 0 || x >= V) { free(w); return OR_EINVAL; }
            double qi = q[((size_t)b * gamma + i - 1) * V + x];
            double pi = p[((size_t)b * (gamma + 1) + i - 1) * V + x];
            double u = unif(sm_next(oracle_row_key(seed, 1, (uint64_t)b, round, (uint64_t)i), 1));
            if (u * qi < pi) { out_tok[(size_t)b * (gamma + 1) + k] = x; ++k; continue; }
            /* first rejection at position i: draw from max(0, p_i - q_i) */
            const float* pr = p + ((size_t)b * (gamma + 1) + i - 1) * V;
            const float* qr = q + ((size_t)b * gamma + i - 1) * V;
            for (int v = 0; v < V; ++v) { double d = (double)pr[v] - (double)qr[v]; w[v] = d > 0 ? d : 0.0; }
            out_tok[(size_t)b * (gamma + 1) + k] =
                race(w, pr, V, oracle_row_key(seed, 2, (uint64_t)b, round, (uint64_t)i), race_gap ? &race_gap[b] : NULL);
            rejected = 1;
            break;
        }
        if (!rejected) { /* all gamma accepted: bonus token from p_{gamma+1} */
            const float* pr = p + ((size_t)b * (gamma + 1) + gamma) * V;
            for (int v = 0; v < V; ++v) w[v] = pr[v] > 0 ? (double)pr[v] : 0.0;
            out_tok[(size_t)b * (gamma + 1) + gamma] =
                race(w, pr, V, oracle_row_key(seed, 3, (uint64_t)b, round, (uint64_t)gamma + 1),
                     race_gap ? &race_gap[b] : NULL);
        }
        n_acc[b] = k;
    }
    free(w);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* O6: keep the accepted branch [MH, "Tree attention and acceptance"]: the    */
/* K/V rows of the root and the accepted nodes move to the contiguous slots   */
/* L_b .. L_b + a, kv_len grows by a + 1, and the hidden state of the last    */
/* accepted node is kept for the heads of the next round.  All rows are read  */
/* into a temporary before any is written, so overlapping moves are safe.     */
/* elem = bytes per element (4 fp32, 2 bf16).                                 */
/* ------------------------------------------------------------------------- */
/* O4s: typical acceptance with a sampled next token [MH, "Tree attention and */
/* acceptance": in sampling, Medusa uses typical acceptance].  The accepted   */
/* branch is the one oracle_verify_tree finds in typical mode; the token after */
/* it is drawn from the base model's distribution at the best node,           */
/* P = softmax(row / T), by the exponential race above with weights           */
/* w_v = exp(row_v / T - max / T) and row key stream 4, pos 0.                */
/* ------------------------------------------------------------------------- */
int oracle_verify_tree_sample(const float* logits, const int32_t* cand, const int32_t* parent,
                              const int32_t* depth, int B, int N, int V, int Dmax, double T, double eps,
                              double delta, uint64_t seed, uint64_t round, int32_t* accept_len,
                              int32_t* best_node, int32_t* path_nodes, int32_t* next_tok,
                              double* race_gap /* [B] or NULL */) {
    if (!(T > 0)) return OR_EINVAL;
    int rc = oracle_verify_tree(logits, cand, parent, depth, B, N, V, Dmax, 1, T, eps, delta, accept_len,
                                best_node, path_nodes, next_tok, NULL, NULL, NULL, NULL);
    if (rc != OR_OK) return rc;
    double* w = (double*)malloc((size_t)V * sizeof(double));
    if (!w) return OR_ENOMEM;
    for (int b = 0; b < B; ++b) {
        const float* row = logits + ((size_t)b * N + best_node[b]) * V;
        double mx = -INFINITY;
        for (int v = 0; v < V; ++v) if ((double)row[v] / T > mx) mx = (double)row[v] / T;
        for (int v = 0; v < V; ++v) w[v] = exp((double)row[v] / T - mx);
        next_tok[b] = race(w, row, V, oracle_row_key(seed, 4, (uint64_t)b, round, 0),
                           race_gap ? race_gap + b : NULL);
    }
    free(w);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
int oracle_kv_compact(void* kc, void* vc, int elem, int32_t* kv_len, const int32_t* path_nodes,
                      const int32_t* accept_len, const int32_t* best_node, const void* hidden_tree,
                      void* h_next, int B, int Hkv, int D, int Lmax, int N, int H, int Dmax,
                      int32_t* src_idx /* [B,Dmax+1] or NULL */) {
    if (!kc || !vc || !kv_len || !path_nodes || !accept_len || !best_node || (elem != 2 && elem != 4))
        return OR_EINVAL;
    size_t row = (size_t)D * elem;
    unsigned char* tmp = (unsigned char*)malloc((size_t)(Dmax + 1) * row);
    if (!tmp) return OR_ENOMEM;
    for (int b = 0; b < B; ++b) {
        int a = accept_len[b], L = kv_len[b];
        if (a < 0 || a > Dmax || L < 0 || L + N > Lmax) { free(tmp); return OR_EINVAL; }
        for (int i = 0; i <= a; ++i)
            if (path_nodes[(size_t)b * (Dmax + 1) + i] < 0 || path_nodes[(size_t)b * (Dmax + 1) + i] >= N) {
                free(tmp); return OR_EINVAL;
            }
        for (int c = 0; c < 2; ++c) {
            unsigned char* cache = (unsigned char*)(c == 0 ? kc : vc);
            for (int hk = 0; hk < Hkv; ++hk) {
                unsigned char* base = cache + ((size_t)b * Hkv + hk) * Lmax * row;
                for (int i = 0; i <= a; ++i)
                    memcpy(tmp + (size_t)i * row, base + (size_t)(L + path_nodes[(size_t)b * (Dmax + 1) + i]) * row, row);
                for (int i = 0; i <= a; ++i)
                    memcpy(base + (size_t)(L + i) * row, tmp + (size_t)i * row, row);
            }
        }
        if (src_idx)
            for (int i = 0; i <= Dmax; ++i)
                src_idx[(size_t)b * (Dmax + 1) + i] = i <= a ? L + path_nodes[(size_t)b * (Dmax + 1) + i] : -1;
        if (hidden_tree && h_next)
            memcpy((unsigned char*)h_next + (size_t)b * H * elem,
                   (const unsigned char*)hidden_tree + ((size_t)b * N + best_node[b]) * H * elem, (size_t)H * elem);
        kv_len[b] = L + a + 1;
    }
    free(tmp);
    return OR_OK;
}
