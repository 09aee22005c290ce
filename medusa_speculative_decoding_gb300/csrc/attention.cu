// attention.cu -- tree attention ("Medusa Heads" glossary page, "Tree attention
// and acceptance": every candidate is appended to the input at once and the
// attention mask lets each candidate see only its ancestors, so all branches
// are scored in one pass against the KV cache).
//
// Query i of sequence b attends to the prefix keys [0, L_b) and to the tree
// keys L_b + m whose bit m is set in mask row i.  The KV cache dominates the
// bytes, so the bf16 kernel reads each KV tile once per (sequence, KV head,
// query block) and scores all of the block's tree queries against it:
//   tree_attn_bf16_kernel : split-KV over CTAs; per 64-key tile S = Q K^T and
//                           O += P V on tensor cores (mma.sync m16n8k16 bf16,
//                           float32 accumulate), online softmax in float32,
//                           ancestor bits tested only on tiles that reach the
//                           tree slots
//   attn_combine_kernel   : merges the per-split (max, sum, O) partials
//   tree_attn_f32_kernel  : float32 storage path (one warp per query row)
#include <float.h>

#include "common.cuh"

namespace medusa {
namespace {

constexpr int kBlockN = 64;  // keys per tile
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 bytes read -> the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, float32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Byte offset of element (row, col) in a [rows][D] bf16 tile whose 16-byte
// chunks are XOR-swizzled by (row & 7), so ldmatrix row groups hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int col) {
    const int chunk = (col >> 3) ^ (row & 7);
    return (uint32_t)((row * D + chunk * 8 + (col & 7)) * 2);
}

struct AttnArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* kv_len;
    const uint64_t* mask;
    float* out;
    float* part_o;   // [B,Hq,N,S,D]
    float* part_ml;  // [B,Hq,N,S,2]
    int B, N, Hq, Hkv, G, Lmax, W, S, chunk, qblocks;
    float scale_log2;
};

__device__ __forceinline__ int clamp_len(int L, int N, int Lmax) {
    return L < 0 ? 0 : (L > Lmax - N ? Lmax - N : L);
}

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) tree_attn_bf16_kernel(AttnArgs a) {
    constexpr int BM = 16 * NW;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* qs = smem;                                 // [BM][D]
    uint8_t* ks = smem + BM * D * 2;                    // [2][64][D]
    uint8_t* vs = ks + 2 * kBlockN * D * 2;             // [2][64][D]

    const int split = blockIdx.x;
    const int hk = blockIdx.y / a.qblocks, qb = blockIdx.y % a.qblocks;
    const int b = blockIdx.z;
    const int N = a.N, G = a.G;
    const int L = clamp_len(a.kv_len[b], N, a.Lmax);
    const int total = L + N;
    const int k_begin = split * a.chunk;
    if (k_begin >= total) return;  // this split holds no keys of sequence b
    const int k_end = min(total, k_begin + a.chunk);
    const int nblk = (k_end - k_begin + kBlockN - 1) / kBlockN;
    const int rows = N * G;
    const int row0 = qb * BM;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint16_t* kbase = a.k + ((size_t)b * a.Hkv + hk) * a.Lmax * D;
    const uint16_t* vbase = a.v + ((size_t)b * a.Hkv + hk) * a.Lmax * D;

    // Q tile: row r -> node r / G, query head hk * G + r % G
    for (int c = tid; c < BM * CH; c += NW * 32) {
        const int r = c / CH, ch = c % CH;
        const int gr = row0 + r;
        const bool ok = gr < rows;
        const int node = ok ? gr / G : 0, hq = hk * G + (ok ? gr % G : 0);
        const uint16_t* src = a.q + (((size_t)b * N + node) * a.Hq + hq) * D + ch * 8;
        cp_async16(smem_u32(qs) + swz<D>(r, ch * 8), src, ok);
    }
    auto load_kv = [&](int blk, int stage) {
        const int j0 = k_begin + blk * kBlockN;
        for (int c = tid; c < kBlockN * CH; c += NW * 32) {
            const int r = c / CH, ch = c % CH;
            const int j = j0 + r;
            const bool ok = j < k_end;
            const size_t off = (size_t)(ok ? j : 0) * D + ch * 8;
            const uint32_t o = swz<D>(r, ch * 8) + stage * kBlockN * D * 2;
            cp_async16(smem_u32(ks) + o, kbase + off, ok);
            cp_async16(smem_u32(vs) + o, vbase + off, ok);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // per-thread rows of the warp's 16-row slice: g and g + 8
    const int g = lane >> 2, q4 = lane & 3;
    const int wrow = warp * 16;
    int node_r[2];
    bool valid_r[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int gr = row0 + wrow + g + 8 * h;
        valid_r[h] = gr < rows;
        node_r[h] = valid_r[h] ? gr / G : 0;
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    uint32_t qa[D / 16][4];

    for (int blk = 0; blk < nblk; ++blk) {
        if (blk + 1 < nblk) {
            load_kv(blk + 1, (blk + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (blk == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = wrow + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int c = kk * 16 + 8 * (lane >> 4);
                ldsm_x4(smem_u32(qs) + swz<D>(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            }
        }
        const uint32_t kst = smem_u32(ks) + (blk & 1) * kBlockN * D * 2;
        const uint32_t vst = smem_u32(vs) + (blk & 1) * kBlockN * D * 2;

        // S = Q K^T over this tile (16 rows x 64 keys per warp)
        float s[kBlockN / 8][4];
#pragma unroll
        for (int i = 0; i < kBlockN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < kBlockN / 16; ++np) {
                const int key = np * 16 + (lane & 7) + 8 * (lane >> 4);
                const int c = kk * 16 + 8 * ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kst + swz<D>(key, c), b0, b1, b2, b3);
                mma_bf16(s[2 * np], qa[kk], b0, b1);
                mma_bf16(s[2 * np + 1], qa[kk], b2, b3);
            }
        }
        // scale, mask: prefix keys always visible; tree key L + m only if m is an
        // ancestor-or-self of the row's node; keys past this split's end never.
        const int j0 = k_begin + blk * kBlockN;
        const bool tree_tile = j0 + kBlockN > L;
#pragma unroll
        for (int nt = 0; nt < kBlockN / 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e >> 1;
                const int j = j0 + nt * 8 + q4 * 2 + (e & 1);
                bool ok = j < k_end;
                if (tree_tile && ok && j >= L) {
                    const int m = j - L;
                    ok = valid_r[h] &&
                         ((__ldg(a.mask + (size_t)node_r[h] * a.W + (m >> 6)) >> (m & 63)) & 1ull);
                }
                s[nt][e] = ok ? s[nt][e] * a.scale_log2 : -INFINITY;
            }
        }
        // online softmax (log2 domain); each row is spread over a quad of lanes
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float mx = m_r[h];
#pragma unroll
            for (int nt = 0; nt < kBlockN / 8; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * h], s[nt][2 * h + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float base = mx == -INFINITY ? 0.f : mx;
            corr[h] = exp2f(m_r[h] - base);
            m_r[h] = mx;
            float sum = 0.f;
#pragma unroll
            for (int nt = 0; nt < kBlockN / 8; ++nt) {
                s[nt][2 * h] = exp2f(s[nt][2 * h] - base);
                s[nt][2 * h + 1] = exp2f(s[nt][2 * h + 1] - base);
                sum += s[nt][2 * h] + s[nt][2 * h + 1];
            }
            l_r[h] = l_r[h] * corr[h] + sum;
        }
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= corr[0];
            o[i][1] *= corr[0];
            o[i][2] *= corr[1];
            o[i][3] *= corr[1];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int c = dp * 16 + 8 * (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vst + swz<D>(key, c), b0, b1, b2, b3);
                mma_bf16(o[2 * dp], pa, b0, b1);
                mma_bf16(o[2 * dp + 1], pa, b2, b3);
            }
        }
        __syncthreads();  // the stage read here is refilled by the next iteration's load
    }

    // row sums: combine the quad's partial sums
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
        l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
    }
    const int S = gridDim.x;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (!valid_r[h]) continue;
        const int gr = row0 + wrow + g + 8 * h;
        const int node = gr / G, hq = hk * G + gr % G;
        if (S == 1) {
            const float inv = l_r[h] > 0.f ? 1.f / l_r[h] : 0.f;
            float* dst = a.out + (((size_t)b * N + node) * a.Hq + hq) * D;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                const int col = i * 8 + q4 * 2;
                *reinterpret_cast<float2*>(dst + col) =
                    make_float2(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
            }
        } else {
            const size_t prow = (((size_t)b * a.Hq + hq) * N + node) * S + split;
            float* dst = a.part_o + prow * D;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                const int col = i * 8 + q4 * 2;
                *reinterpret_cast<float2*>(dst + col) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
            }
            if (q4 == 0) {
                a.part_ml[prow * 2] = m_r[h];
                a.part_ml[prow * 2 + 1] = l_r[h];
            }
        }
    }
}

// One warp per (b, node, query head): merge the splits that hold keys.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= a.B * a.N * a.Hq) return;
    const int b = row / (a.N * a.Hq), node = (row / a.Hq) % a.N, hq = row % a.Hq;
    const int L = clamp_len(a.kv_len[b], a.N, a.Lmax);
    const int S = a.S;
    const int active = min(S, (L + a.N + a.chunk - 1) / a.chunk);
    const size_t prow = (((size_t)b * a.Hq + hq) * a.N + node) * S;
    float mx = -INFINITY;
    for (int s = lane; s < active; s += 32) mx = fmaxf(mx, a.part_ml[(prow + s) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float base = mx == -INFINITY ? 0.f : mx;
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float l = 0.f;
    for (int s = 0; s < active; ++s) {
        const float ms = a.part_ml[(prow + s) * 2], ls = a.part_ml[(prow + s) * 2 + 1];
        if (ls == 0.f) continue;
        const float w = exp2f(ms - base);
        l += ls * w;
        const float* src = a.part_o + (prow + s) * D;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += src[lane + 32 * i] * w;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* dst = a.out + (((size_t)b * a.N + node) * a.Hq + hq) * D;
#pragma unroll
    for (int i = 0; i < PER; ++i) dst[lane + 32 * i] = acc[i] * inv;
}

// float32 storage: one warp per (b, node, query head), keys in order, online softmax.
template <int D>
__global__ void __launch_bounds__(256) tree_attn_f32_kernel(const float* __restrict__ q,
                                                            const float* __restrict__ k,
                                                            const float* __restrict__ v,
                                                            const int32_t* __restrict__ kv_len,
                                                            const uint64_t* __restrict__ mask,
                                                            int B, int N, int Hq, int Hkv, int Lmax,
                                                            int W, float scale,
                                                            float* __restrict__ out) {
    constexpr int PER = D / 32;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= B * N * Hq) return;
    const int b = row / (N * Hq), node = (row / Hq) % N, hq = row % Hq;
    const int hk = hq / (Hq / Hkv);
    const int L = clamp_len(kv_len[b], N, Lmax);
    float qv[PER], acc[PER];
    const float* qp = q + (((size_t)b * N + node) * Hq + hq) * D;
#pragma unroll
    for (int i = 0; i < PER; ++i) { qv[i] = qp[lane + 32 * i]; acc[i] = 0.f; }
    const float* kb = k + ((size_t)b * Hkv + hk) * Lmax * D;
    const float* vb = v + ((size_t)b * Hkv + hk) * Lmax * D;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < L + N; ++j) {
        if (j >= L) {
            const int t = j - L;
            if (!((mask[(size_t)node * W + (t >> 6)] >> (t & 63)) & 1ull)) continue;
        }
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) d = fmaf(qv[i], kb[(size_t)j * D + lane + 32 * i], d);
        d = warp_sum(d) * scale;
        const float mn = fmaxf(m, d);
        const float c = expf(m - mn), p = expf(d - mn);
        l = l * c + p;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = acc[i] * c + p * vb[(size_t)j * D + lane + 32 * i];
        m = mn;
    }
    float* dst = out + (((size_t)b * N + node) * Hq + hq) * D;
#pragma unroll
    for (int i = 0; i < PER; ++i) dst[lane + 32 * i] = acc[i] / l;
}

struct AttnPlan {
    int NW, qblocks, S, chunk;
    size_t smem, off_o, off_ml, ws_bytes;
};

AttnPlan plan_attention(int B, int N, int Hq, int Hkv, int D, int Lmax) {
    AttnPlan p{};
    const int rows = N * (Hq / Hkv);
    p.NW = rows <= 64 ? 4 : 8;
    const int BM = 16 * p.NW;
    p.qblocks = (rows + BM - 1) / BM;
    p.smem = (size_t)BM * D * 2 + 4 * (size_t)kBlockN * D * 2;
    const long long units = (long long)B * Hkv * p.qblocks;
    const int target = 2 * sm_count();
    const int max_splits = (Lmax + kBlockN - 1) / kBlockN;
    long long s = (target + units - 1) / units;
    if (s < 1) s = 1;
    if (s > max_splits) s = max_splits;
    if (s > 64) s = 64;
    int chunk = (int)((Lmax + s - 1) / s);
    chunk = (chunk + kBlockN - 1) / kBlockN * kBlockN;
    p.chunk = chunk;
    p.S = (Lmax + chunk - 1) / chunk;
    size_t off = 0;
    p.off_o = off;
    if (p.S > 1) {
        off = align_up(off + (size_t)B * Hq * N * p.S * D * sizeof(float), 256);
        p.off_ml = off;
        off = align_up(off + (size_t)B * Hq * N * p.S * 2 * sizeof(float), 256);
    }
    p.ws_bytes = off;
    return p;
}

int check_attn(int B, int N, int Hq, int Hkv, int D, int Lmax) {
    if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Lmax < 1)
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_attention: sizes must be positive");
    if ((D != 64 && D != 128) || N > 512 || Hq % Hkv || N * (Hq / Hkv) > 4096 || N > Lmax)
        return fail(MEDUSA_ERR_UNSUPPORTED,
                    "tree_attention: unsupported shape (N=%d Hq=%d Hkv=%d D=%d Lmax=%d)", N, Hq,
                    Hkv, D, Lmax);
    return MEDUSA_OK;
}

template <int D>
int launch_bf16(AttnArgs& a, const AttnPlan& p, cudaStream_t st) {
    dim3 grid(p.S, a.Hkv * p.qblocks, a.B);
    if (p.NW == 4) {
        auto kern = tree_attn_bf16_kernel<D, 4>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        kern<<<grid, 128, p.smem, st>>>(a);
    } else {
        auto kern = tree_attn_bf16_kernel<D, 8>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        kern<<<grid, 256, p.smem, st>>>(a);
    }
    int rc = check_launch("tree_attention");
    if (rc || p.S == 1) return rc;
    const int rows = a.B * a.N * a.Hq;
    attn_combine_kernel<D><<<(rows + 7) / 8, 256, 0, st>>>(a);
    return check_launch("attn_combine");
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_tree_attention_workspace(int B, int N, int Hq, int Hkv, int D, int Lmax) {
    if (check_attn(B, N, Hq, Hkv, D, Lmax)) return 0;
    return plan_attention(B, N, Hq, Hkv, D, Lmax).ws_bytes;
}

extern "C" int medusa_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* kv_len, const uint64_t* mask,
                                     medusa_dtype dtype, int B, int N, int Hq, int Hkv, int D,
                                     int Lmax, float scale, float* out, void* ws, size_t ws_bytes,
                                     void* stream) {
    int rc = check_attn(B, N, Hq, Hkv, D, Lmax);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !kv_len || !mask || !out)
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_attention: null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_attention: q, caches and out must be 16-byte aligned");
    const int W = (N + 63) / 64;
    cudaStream_t st = as_stream(stream);
    if (dtype == MEDUSA_F32) {
        const int rows = B * N * Hq;
        if (D == 64)
            tree_attn_f32_kernel<64><<<(rows + 7) / 8, 256, 0, st>>>(
                (const float*)q, (const float*)k_cache, (const float*)v_cache, kv_len, mask, B, N,
                Hq, Hkv, Lmax, W, scale, out);
        else
            tree_attn_f32_kernel<128><<<(rows + 7) / 8, 256, 0, st>>>(
                (const float*)q, (const float*)k_cache, (const float*)v_cache, kv_len, mask, B, N,
                Hq, Hkv, Lmax, W, scale, out);
        return check_launch("tree_attention_f32");
    }
    if (dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_UNSUPPORTED, "tree_attention: unknown dtype %d", (int)dtype);
    AttnPlan p = plan_attention(B, N, Hq, Hkv, D, Lmax);
    if (p.ws_bytes > 0 && (!ws || ws_bytes < p.ws_bytes))
        return fail(MEDUSA_ERR_WORKSPACE, "tree_attention: workspace of %zu bytes needed, %zu given",
                    p.ws_bytes, ws ? ws_bytes : (size_t)0);
    if (p.ws_bytes > 0 && !aligned16(ws))
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_attention: ws must be 16-byte aligned");
    AttnArgs a{};
    a.q = (const uint16_t*)q;
    a.k = (const uint16_t*)k_cache;
    a.v = (const uint16_t*)v_cache;
    a.kv_len = kv_len;
    a.mask = mask;
    a.out = out;
    a.part_o = p.S > 1 ? (float*)((char*)ws + p.off_o) : nullptr;
    a.part_ml = p.S > 1 ? (float*)((char*)ws + p.off_ml) : nullptr;
    a.B = B; a.N = N; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.Lmax = Lmax; a.W = W;
    a.S = p.S; a.chunk = p.chunk; a.qblocks = p.qblocks;
    a.scale_log2 = scale * kLog2e;
    return D == 64 ? launch_bf16<64>(a, p, st) : launch_bf16<128>(a, p, st);
}
