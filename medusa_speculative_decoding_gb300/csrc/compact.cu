// compact.cu -- keep the accepted branch ("Medusa Heads" glossary page, "Tree
// attention and acceptance": the longest accepted branch is kept and its final
// hidden state feeds the heads in the next round).
//
// The K/V rows of the root and the accepted nodes move to the contiguous slots
// L_b .. L_b + a so the cache holds the accepted text in order.  A row's
// destination can be the source of a later row of the same head, so each block
// first reads every row it moves into shared memory and only then writes.
//   kv_compact_rows_kernel : grid (B, head groups); also gathers h_next and
//                            writes the source slots for sequence b
//   kv_len_update_kernel   : kv_len[b] += a + 1 (a separate launch: every block
//                            of the first kernel reads kv_len[b])
#include "common.cuh"

namespace medusa {
namespace {

constexpr int kCompactThreads = 256;
constexpr int kHeadsPerBlock = 8;

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

__global__ void __launch_bounds__(kCompactThreads) kv_compact_rows_kernel(
    uint4* __restrict__ kc, uint4* __restrict__ vc, const int32_t* __restrict__ kv_len,
    const int32_t* __restrict__ path_nodes, const int32_t* __restrict__ accept_len,
    const int32_t* __restrict__ best_node, const uint4* __restrict__ hidden_tree,
    uint4* __restrict__ h_next, int Hkv, int row16, int Lmax, int N, int h16, int Dmax,
    int32_t* __restrict__ src_idx) {
    extern __shared__ uint4 buf[];  // [2][heads][Dmax+1][row16]
    const int b = blockIdx.x;
    const int h0 = blockIdx.y * kHeadsPerBlock;
    const int nh = min(kHeadsPerBlock, Hkv - h0);
    const bool ok = seq_ok(kv_len, path_nodes, accept_len, best_node, b, N, Lmax, Dmax);
    if (blockIdx.y == 0 && src_idx) {
        for (int i = threadIdx.x; i <= Dmax; i += blockDim.x) {
            const int a = accept_len[b];
            src_idx[(size_t)b * (Dmax + 1) + i] =
                !ok ? -2 : (i <= a ? kv_len[b] + path_nodes[(size_t)b * (Dmax + 1) + i] : -1);
        }
    }
    if (!ok) return;
    const int a = accept_len[b], L = kv_len[b];
    const int32_t* path = path_nodes + (size_t)b * (Dmax + 1);
    if (blockIdx.y == 0 && hidden_tree && h_next) {
        const uint4* src = hidden_tree + ((size_t)b * N + best_node[b]) * h16;
        for (int i = threadIdx.x; i < h16; i += blockDim.x) h_next[(size_t)b * h16 + i] = src[i];
    }
    const int per_cache = nh * (a + 1) * row16;
    for (int t = threadIdx.x; t < 2 * per_cache; t += blockDim.x) {
        const int c = t / per_cache, r = t % per_cache;
        const int h = r / ((a + 1) * row16), i = (r / row16) % (a + 1), e = r % row16;
        const uint4* cache = c ? vc : kc;
        const size_t row = ((size_t)b * Hkv + h0 + h) * Lmax + L + path[i];
        buf[t] = cache[row * row16 + e];
    }
    __syncthreads();
    for (int t = threadIdx.x; t < 2 * per_cache; t += blockDim.x) {
        const int c = t / per_cache, r = t % per_cache;
        const int h = r / ((a + 1) * row16), i = (r / row16) % (a + 1), e = r % row16;
        uint4* cache = c ? vc : kc;
        const size_t row = ((size_t)b * Hkv + h0 + h) * Lmax + L + i;
        cache[row * row16 + e] = buf[t];
    }
}

__global__ void kv_len_update_kernel(int32_t* __restrict__ kv_len, const int32_t* __restrict__ path_nodes,
                                     const int32_t* __restrict__ accept_len,
                                     const int32_t* __restrict__ best_node, int B, int N, int Lmax,
                                     int Dmax) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    if (seq_ok(kv_len, path_nodes, accept_len, best_node, b, N, Lmax, Dmax)) kv_len[b] += accept_len[b] + 1;
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
    const size_t smem = (size_t)2 * kHeadsPerBlock * (Dmax + 1) * row16 * sizeof(uint4);
    if (smem > (size_t)max_smem_optin())
        return fail(MEDUSA_ERR_UNSUPPORTED, "kv_compact: Dmax %d needs %zu bytes of shared memory", Dmax, smem);
    cudaStream_t st = as_stream(stream);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(kv_compact_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(B, (Hkv + kHeadsPerBlock - 1) / kHeadsPerBlock);
    kv_compact_rows_kernel<<<grid, kCompactThreads, smem, st>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), kv_len, path_nodes, accept_len,
        best_node, static_cast<const uint4*>(hidden_tree), static_cast<uint4*>(h_next), Hkv, row16,
        Lmax, N, hidden_tree ? H * elem / 16 : 0, Dmax, src_idx);
    int rc = check_launch("kv_compact_rows");
    if (rc) return rc;
    kv_len_update_kernel<<<(B + 255) / 256, 256, 0, st>>>(kv_len, path_nodes, accept_len, best_node, B, N,
                                                            Lmax, Dmax);
    return check_launch("kv_len_update");
}
