// tree.cu -- candidate tree ("Medusa Heads" glossary page, "Tree attention and
// acceptance": the heads' top guesses combine into candidate continuations
// that share prefixes and form a tree; a sparse tree of the most accurate
// combinations beats a dense one; each candidate may attend only to its
// ancestors).
//
// The node table (parent, depth, rank, ancestor bitmask, root-to-leaf paths) is
// static for a tree shape and is built once on the host.  Per step only the
// candidate tokens change: build_tree_kernel gathers them from the heads' top-k
// lists.
#include <math.h>

#include <algorithm>
#include <map>
#include <vector>

#include "common.cuh"

namespace medusa {
namespace {

using Tuple = std::vector<int32_t>;

// canonical order: by length, then lexicographic
bool canonical_less(const Tuple& a, const Tuple& b) {
    if (a.size() != b.size()) return a.size() < b.size();
    return a < b;
}

__global__ void build_tree_kernel(const int32_t* __restrict__ topk_idx,
                                  const int32_t* __restrict__ root_tok,
                                  const int32_t* __restrict__ depth,
                                  const int32_t* __restrict__ rank, int B, int K, int topk, int N,
                                  int32_t* __restrict__ cand) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * N) return;
    const int b = i / N, n = i - b * N;
    const int d = depth[n], r = rank[n];
    int32_t tok;
    if (d == 0)
        tok = root_tok[b];
    else if (d > K || r < 0 || r >= topk)
        tok = -1;
    else
        tok = topk_idx[((size_t)b * K + (d - 1)) * topk + r];
    cand[i] = tok;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_sparse_tree_paths(int n_nodes, int max_depth, int max_rank, double head_p,
                                        double rank_p, int32_t* paths_out) {
    if (n_nodes < 1 || max_depth < 1 || max_depth > 16 || max_rank < 1 || !paths_out)
        return fail(MEDUSA_ERR_INVALID_ARG, "sparse_tree_paths: bad sizes or null output");
    if (!(head_p > 0 && head_p < 1 && rank_p > 0 && rank_p < 1))
        return fail(MEDUSA_ERR_INVALID_ARG, "sparse_tree_paths: head_p and rank_p must lie in (0,1)");
    // Count candidates; refuse enumerations that would not fit comfortably in memory.
    double total = 0, cnt = 1;
    for (int d = 1; d <= max_depth; ++d) {
        cnt *= max_rank;
        total += cnt;
    }
    if (total > 2e7) return fail(MEDUSA_ERR_UNSUPPORTED, "sparse_tree_paths: %g candidate tuples", total);
    if (n_nodes - 1 > (long long)total)
        return fail(MEDUSA_ERR_INVALID_ARG, "sparse_tree_paths: only %g tuples for %d nodes", total,
                    n_nodes);
    struct Cand {
        int tri, sum;  // accuracy = head_p^tri * rank_p^sum, tri = d(d+1)/2
        double key;    // its logarithm
        Tuple t;
    };
    const double lh = log(head_p), lr = log(rank_p);
    std::vector<Cand> all;
    all.reserve((size_t)total);
    for (int d = 1; d <= max_depth; ++d) {
        Tuple t(d, 0);
        for (;;) {
            int sum = 0;
            for (int x : t) sum += x;
            const int tri = d * (d + 1) / 2;
            all.push_back(Cand{tri, sum, tri * lh + sum * lr, t});
            int pos = d - 1;
            while (pos >= 0 && ++t[pos] == max_rank) t[pos--] = 0;
            if (pos < 0) break;
        }
    }
    // Two tuples are equally accurate exactly when (tri, sum) agree; only then do
    // depth and lexicographic order decide.
    auto more_accurate = [](const Cand& a, const Cand& b) {
        if (a.tri != b.tri || a.sum != b.sum) return a.key > b.key;
        return canonical_less(a.t, b.t);
    };
    const size_t take = (size_t)(n_nodes - 1);
    std::partial_sort(all.begin(), all.begin() + take, all.end(), more_accurate);
    std::vector<Tuple> chosen;
    for (size_t i = 0; i < take; ++i) chosen.push_back(all[i].t);
    std::sort(chosen.begin(), chosen.end(), canonical_less);
    for (size_t i = 0; i < take; ++i)
        for (int e = 0; e < max_depth; ++e)
            paths_out[i * max_depth + e] = e < (int)chosen[i].size() ? chosen[i][e] : -1;
    return MEDUSA_OK;
}

extern "C" int medusa_tree_layout(const int32_t* rank_paths, int P, int max_depth, int cap_nodes,
                                  int cap_paths, int32_t* parent, int32_t* depth, int32_t* rank,
                                  uint64_t* mask, int32_t* retrieve, int* N_out, int* W_out,
                                  int* n_paths_out) {
    if ((!rank_paths && P > 0) || P < 0 || max_depth < 1 || !parent || !depth || !rank || !N_out ||
        !W_out)
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_layout: null pointer or bad size");
    std::vector<Tuple> nodes;
    nodes.push_back(Tuple());
    for (int p = 0; p < P; ++p) {
        const int32_t* row = rank_paths + (size_t)p * max_depth;
        int d = 0;
        while (d < max_depth && row[d] >= 0) ++d;
        for (int e = d; e < max_depth; ++e)
            if (row[e] != -1)
                return fail(MEDUSA_ERR_INVALID_ARG, "tree_layout: tuple %d is not -1 padded", p);
        for (int len = 1; len <= d; ++len) nodes.push_back(Tuple(row, row + len));
    }
    std::sort(nodes.begin(), nodes.end(), canonical_less);
    nodes.erase(std::unique(nodes.begin(), nodes.end()), nodes.end());
    const int N = (int)nodes.size();
    if (N > cap_nodes)
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_layout: %d nodes exceed capacity %d", N, cap_nodes);
    const int W = (N + 63) / 64;
    std::map<Tuple, int> index;
    for (int i = 0; i < N; ++i) index[nodes[i]] = i;
    std::vector<char> has_child(N, 0);
    for (int i = 0; i < N; ++i) {
        const Tuple& t = nodes[i];
        depth[i] = (int32_t)t.size();
        rank[i] = t.empty() ? -1 : t.back();
        parent[i] = t.empty() ? -1 : index[Tuple(t.begin(), t.end() - 1)];
        if (parent[i] >= 0) has_child[parent[i]] = 1;
    }
    if (mask) {
        for (int i = 0; i < N; ++i) {
            uint64_t* row = mask + (size_t)i * W;
            for (int w = 0; w < W; ++w) row[w] = 0;
            for (int a = i; a >= 0; a = parent[a]) row[a >> 6] |= 1ull << (a & 63);
        }
    }
    int np = 0;
    for (int i = 0; i < N; ++i) {
        if (has_child[i]) continue;
        if (retrieve) {
            if (np >= cap_paths)
                return fail(MEDUSA_ERR_INVALID_ARG, "tree_layout: more leaves than cap_paths %d",
                            cap_paths);
            int32_t* row = retrieve + (size_t)np * (max_depth + 1);
            for (int e = 0; e <= max_depth; ++e) row[e] = -1;
            for (int a = i; a >= 0; a = parent[a]) row[depth[a]] = a;
        }
        ++np;
    }
    *N_out = N;
    *W_out = W;
    if (n_paths_out) *n_paths_out = np;
    return MEDUSA_OK;
}

extern "C" int medusa_build_tree(const int32_t* topk_idx, const int32_t* root_tok,
                                 const int32_t* depth, const int32_t* rank, int B, int K, int topk,
                                 int N, int32_t* cand, void* stream) {
    if (!topk_idx || !root_tok || !depth || !rank || !cand)
        return fail(MEDUSA_ERR_INVALID_ARG, "build_tree: null pointer");
    if (B < 1 || K < 1 || topk < 1 || N < 1)
        return fail(MEDUSA_ERR_INVALID_ARG, "build_tree: sizes must be positive");
    const int total = B * N;
    cudaError_t e = launch(build_tree_kernel, dim3((total + 255) / 256), dim3(256), 0,
                           as_stream(stream), topk_idx, root_tok, depth, rank, B, K, topk, N, cand);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "build_tree: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}
