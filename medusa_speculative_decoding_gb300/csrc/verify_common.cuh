// verify_common.cuh -- what the tree-acceptance kernels share between the
// logits path (verify.cu) and the fused verification projection (project.cu):
// the per-(row, vocab chunk) statistics record and the acceptance launcher.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace medusa {

struct RowStat {      // per (row, vocab chunk)
    float maxv;       // largest logit
    int arg;          // its lowest index
    float m, s, a;    // x = logit/T: max, sum e^(x-m), sum e^(x-m) (x-m)
    float pad[3];
};

// merge softmax/entropy partial states (m, s, a)
__device__ __forceinline__ void merge_msa(float& m, float& s, float& a, float m2, float s2,
                                          float a2) {
    if (s2 == 0.f) return;
    if (s == 0.f) { m = m2; s = s2; a = a2; return; }
    const float mn = fmaxf(m, m2);
    const float c1 = expf(m - mn), c2 = expf(m2 - mn);
    a = c1 * (a + (m - mn) * s) + c2 * (a2 + (m2 - mn) * s2);
    s = c1 * s + c2 * s2;
    m = mn;
}

// One x = logit/T (already scaled) into the running (m, s, a) state.
__device__ __forceinline__ void take_msa(float& m, float& s, float& a, float xv) {
    if (!(xv > -INFINITY)) return;  // contributes no probability mass
    if (s == 0.f) {
        m = xv;
        s = 1.f;
        a = 0.f;
    } else if (xv > m) {
        const float c1 = expf(m - xv);
        a = c1 * (a + (m - xv) * s);
        s = c1 * s + 1.f;
        m = xv;
    } else {
        const float e = expf(xv - m);
        s += e;
        a += e * (xv - m);
    }
}

// Arguments of the acceptance kernel.  The candidate logit of node u (row
// parent(u), token cand[u]) is read from `logits` when given, else from
// child_logit[b*N + u].
struct AcceptArgs {
    const float* logits;       // [B,N,V] or nullptr
    const float* child_logit;  // [B*N] (when logits is nullptr)
    const int32_t* cand;
    const int32_t* parent;
    const int32_t* depth;
    int B, N, V, Dmax, nchunk;
    float inv_t, eps, delta;
    const RowStat* stats;     // [B*N][nchunk]
    const int* status;        // [nstatus]: any nonzero entry invalidates the statistics
    int nstatus;
    int32_t* accept_len;
    int32_t* best_node;
    int32_t* path_nodes;
    int32_t* next_tok;
};
constexpr int kAcceptThreads = 512;  // >= max nodes
int launch_accept_tree(bool typical, const AcceptArgs& a, cudaStream_t st);

// Per-row finish of the fused projection's statistics: merges the `splits`
// records of each of the `rows` rows into out[row] and, for typical
// acceptance, writes child_logit[b*N + u] = hidden[b, parent(u)] . lm[cand[b,u]]
// (bf16 rows of H elements, float32 sum; NaN where parent or token is invalid).
int launch_row_finish(bool typical, const RowStat* stats, int splits, int rows, int N, int V, int H,
                      const uint16_t* hidden, const uint16_t* lm, const int32_t* cand,
                      const int32_t* parent, RowStat* out, float* child_logit, cudaStream_t st);

}  // namespace medusa
