// compact.cu -- keep the accepted branch ("Medusa Heads" glossary page, "Tree
// attention and acceptance": the longest accepted branch is kept and its final
// hidden state feeds the heads in the next round).
//
// The K/V rows of the root and the accepted nodes move to the contiguous slots
// L_b .. L_b + a so the cache holds the accepted text in order.  A row's
// destination can be the source of a later row of the same head, so each block
// first reads every row it moves into shared memory and only then writes.
//   kv_compact_kernel : a cluster of CTAs per sequence; each CTA moves the rows
//                       of its share of the (cache, KV head) pairs, all of a
//                       pair's rows read before any is written, and gathers its
//                       share of h_next; after a cluster barrier (every CTA has
//                       read kv_len[b]) rank 0 advances kv_len[b]
#include "common.cuh"
#include "umma.cuh"

namespace medusa {
namespace {

constexpr int kCompactThreads = 256;
constexpr int kCompactCtas = 8;              // CTAs per sequence: one portable cluster
constexpr size_t kCompactSmem = 48 * 1024;   // staging buffer per CTA

// true iff sequence b's inputs are in range (otherwise it is left unchanged)
__device__ __forceinline__ bool seq_ok(const int32_t* kv_len, const int32_t* path_nodes,
                                       const int32_t* accept_len, const int32_t* best_node, int b,
                                       int N, int Lmax, int Dmax) {
    const int a = accept_len[b], L = kv_len[b], best = best_node[b];
    if (a < 0 || a > Dmax || L < 0 || L + N > Lmax || best < 0 || best >= N) return false;
    for (int i = 0; i <= a; ++i) {
        const int n = path_nodes[(size_t)b * (Dmax + 1) + i];
        if (n < 0 || n >= N) return false;
    }
    return true;
}

// Grid (C, B), cluster (C, 1, 1): CTA r of sequence b owns the (cache, KV head)
// pairs [r*2Hkv/C, (r+1)*2Hkv/C), moved in chunks that fit the staging buffer.
// Rows of different pairs never overlap, so only the rows of one pair need to
// be read before any of them is written.
__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, int32_t* __restrict__ kv_len,
    const int32_t* __restrict__ path_nodes, const int32_t* __restrict__ accept_len,
    const int32_t* __restrict__ best_node, const uint4* __restrict__ hidden_tree,
    uint4* __restrict__ h_next, int Hkv, int row16, int Lmax, int N, int h16, int Dmax,
    int32_t* __restrict__ src_idx) {
    extern __shared__ uint4 buf[];
    __shared__ int s_ok, s_a, s_L, s_best;
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y, rank = blockIdx.x, C = gridDim.x;
    if (threadIdx.x == 0) {
        s_ok = seq_ok(kv_len, path_nodes, accept_len, best_node, b, N, Lmax, Dmax);
        s_a = accept_len[b];
        s_L = kv_len[b];
        s_best = best_node[b];
    }
    __syncthreads();
    const bool ok = s_ok;
    const int a = s_a, L = s_L;
    const int32_t* path = path_nodes + (size_t)b * (Dmax + 1);
    if (src_idx && rank == 0)
        for (int i = threadIdx.x; i <= Dmax; i += blockDim.x)
            src_idx[(size_t)b * (Dmax + 1) + i] = !ok ? -2 : (i <= a ? L + path[i] : -1);
    if (ok) {
        if (hidden_tree && h_next) {
            const uint4* src = hidden_tree + ((size_t)b * N + s_best) * h16;
            const int e0 = rank * h16 / C, e1 = (rank + 1) * h16 / C;
            for (int i = e0 + threadIdx.x; i < e1; i += blockDim.x) h_next[(size_t)b * h16 + i] = src[i];
        }
        const int pairs = 2 * Hkv;
        const int p0 = rank * pairs / C, p1 = (rank + 1) * pairs / C;
        const int per_pair = (a + 1) * row16;  // uint4 per (cache, head)
        const int cap = max(1, (int)(kCompactSmem / sizeof(uint4)) / per_pair);
        for (int q0 = p0; q0 < p1; q0 += cap) {
            const int n = min(cap, p1 - q0) * per_pair;
#pragma unroll 4
            for (int t = threadIdx.x; t < n; t += blockDim.x) {
                const int pr = q0 + t / per_pair, r = t % per_pair;
                const int c = pr / Hkv, h = pr - c * Hkv, i = r / row16, e = r - i * row16;
                const uint4* cache = c ? vc : kc;
                const size_t row = ((size_t)b * Hkv + h) * Lmax + L + path[i];
                buf[t] = cache[row * row16 + e];
            }
            __syncthreads();
#pragma unroll 4
            for (int t = threadIdx.x; t < n; t += blockDim.x) {
                const int pr = q0 + t / per_pair, r = t % per_pair;
                const int c = pr / Hkv, h = pr - c * Hkv, i = r / row16, e = r - i * row16;
                uint4* cache = c ? vc : kc;
                const size_t row = ((size_t)b * Hkv + h) * Lmax + L + i;
                cache[row * row16 + e] = buf[t];
            }
            __syncthreads();
        }
    }
    // kv_len[b] changes only after every CTA of the sequence has read it
    umma::cluster_sync();
    if (ok && rank == 0 && threadIdx.x == 0) kv_len[b] = L + a + 1;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" int medusa_kv_compact(void* k_cache, void* v_cache, int32_t* kv_len,
                                 const int32_t* path_nodes, const int32_t* accept_len,
                                 const int32_t* best_node, const void* hidden_tree, void* h_next,
                                 medusa_dtype dtype, int B, int Hkv, int D, int Lmax, int N, int H,
                                 int Dmax, int32_t* src_idx, void* stream) {
    if (!k_cache || !v_cache || !kv_len || !path_nodes || !accept_len || !best_node)
        return fail(MEDUSA_ERR_INVALID_ARG, "kv_compact: null pointer");
    if ((hidden_tree == nullptr) != (h_next == nullptr))
        return fail(MEDUSA_ERR_INVALID_ARG, "kv_compact: hidden_tree and h_next go together");
    if (B < 1 || Hkv < 1 || D < 1 || Lmax < 1 || N < 1 || Dmax < 0 || (hidden_tree && H < 1))
        return fail(MEDUSA_ERR_INVALID_ARG, "kv_compact: bad sizes");
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_UNSUPPORTED, "kv_compact: unknown dtype %d", (int)dtype);
    const int elem = dtype == MEDUSA_F32 ? 4 : 2;
    if ((D * elem) % 16 || (hidden_tree && (H * elem) % 16))
        return fail(MEDUSA_ERR_UNSUPPORTED, "kv_compact: rows must be multiples of 16 bytes");
    if (!aligned16(k_cache) || !aligned16(v_cache) || (hidden_tree && (!aligned16(hidden_tree) || !aligned16(h_next))))
        return fail(MEDUSA_ERR_INVALID_ARG, "kv_compact: caches and hidden states must be 16-byte aligned");
    const int row16 = D * elem / 16;
    if ((size_t)(Dmax + 1) * row16 * sizeof(uint4) > kCompactSmem)
        return fail(MEDUSA_ERR_UNSUPPORTED, "kv_compact: Dmax %d with D %d does not fit the staging buffer",
                    Dmax, D);
    if (B > 65535) return fail(MEDUSA_ERR_UNSUPPORTED, "kv_compact: batch %d above 65535", B);
    cudaStream_t st = as_stream(stream);
    cudaFuncSetAttribute(kv_compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCompactSmem);
    cudaError_t e = launch_cluster(kv_compact_kernel, dim3(kCompactCtas, B), dim3(kCompactThreads),
                                   kCompactSmem, st, kCompactCtas,
                                   static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), kv_len,
                           path_nodes, accept_len, best_node, static_cast<const uint4*>(hidden_tree),
                           static_cast<uint4*>(h_next), Hkv, row16, Lmax, N,
                           hidden_tree ? H * elem / 16 : 0, Dmax, src_idx);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "kv_compact: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}
