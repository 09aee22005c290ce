// heads.cu -- Medusa heads and per-head top-k ("Medusa Heads" glossary page,
// "How heads predict later tokens": head k reads the last hidden state h and
// scores position t + k + 1 through one residual SiLU layer and a vocab
// projection).
//
// At decode batch sizes both products read weights that are used once per
// step, so the heads are bound by HBM bandwidth.  bf16 batches of 3 to 64 run
// on the tensor cores (heads_umma.cu); everything else (batches 1-2, and float32
// up to batch 8) runs here, on CUDA cores, as matrix-vector products:
//   K1 heads_w1_silu : z[b,k,:] = h[b] + SiLU(W1_k h[b] + b1_k)   (float32 z);
//                      the K*H rows of W1 are split evenly over the warps of
//                      one wave of CTAs
//   K2 heads_w2_topk : logits = W2_k z, streamed over vocab slices; each CTA keeps
//                      its slice's logits in shared memory and emits its top-k;
//                      the last CTA of a head merges the head's slice lists
//                      into the final sorted top-k
// Each warp walks a few weight rows at once with 16-byte loads (lanes stride
// over the hidden dimension); the vectors z / h live in shared memory as float32
// and are read once per group of rows.  K2 is launched as a programmatic
// dependent of K1 and prefetches its first W2 rows into L2 before it waits for z.
#include <float.h>
#include <limits.h>

#include <mutex>

#include "common.cuh"
#include "topk.cuh"

namespace medusa {

// tensor-core heads for bf16 batches of 3 to 64 (heads_umma.cu)
bool heads_umma_applies(int B, int K, int H, int V, int topk, bool bf16);
size_t heads_umma_workspace(int B, int K, int H, int V, int topk);
int launch_heads_umma(const void* h, const void* w1, const void* b1, const void* w2, int B, int K, int H,
                      int V, int topk, int32_t* topk_idx, float* topk_val, float* logits, char* ws,
                      cudaStream_t st);

namespace {

constexpr int kRows2 = 4;    // W2 rows a warp reduces together
constexpr int kUnroll2 = 2;  // 16-byte chunks per W2 row in flight per lane
constexpr int kRows1 = 2;    // W1 rows a warp reduces together (finer, for balance)
constexpr int kUnroll1 = 4;
constexpr int kPrefetchRows = 8;  // W2 rows per CTA prefetched into L2 before the wait

template <typename WT>
struct Elems { static constexpr int n = 16 / sizeof(WT); };

template <typename WT>
__device__ __forceinline__ float load_scalar(const WT* p, size_t i);
template <>
__device__ __forceinline__ float load_scalar<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_scalar<uint16_t>(const uint16_t* p, size_t i) {
    return bf16_to_f32(p[i]);
}

// Shared-memory layout of one float32 vector of H elements.  float32 weights:
// plain.  bf16 weights (16-byte chunks of 8 elements): elements 0-3 of chunk c
// sit at 4c and elements 4-7 at H/2 + 4c, so the lanes of a warp, which read
// consecutive chunks, read consecutive 16-byte words of each half (no bank
// conflicts).
template <typename WT>
__device__ __forceinline__ int xpos(int i, int H) {
    if (sizeof(WT) == 4) return i;
    return ((i >> 2) & 1) * (H >> 1) + ((i >> 3) << 2) + (i & 3);
}

// acc += dot(16-byte weight chunk c, x[chunk c]); xlo / xhi point at the
// chunk's two float4 halves (xhi unused for float32 weights)
template <typename WT>
__device__ __forceinline__ float dot_chunk(const uint4& w, const float* xlo, const float* xhi, float acc);
template <>
__device__ __forceinline__ float dot_chunk<uint16_t>(const uint4& w, const float* xlo, const float* xhi,
                                                     float acc) {
    const float4 a = *reinterpret_cast<const float4*>(xlo);
    const float4 b = *reinterpret_cast<const float4*>(xhi);
    acc = fmaf(bf16_lo(w.x), a.x, acc);
    acc = fmaf(bf16_hi(w.x), a.y, acc);
    acc = fmaf(bf16_lo(w.y), a.z, acc);
    acc = fmaf(bf16_hi(w.y), a.w, acc);
    acc = fmaf(bf16_lo(w.z), b.x, acc);
    acc = fmaf(bf16_hi(w.z), b.y, acc);
    acc = fmaf(bf16_lo(w.w), b.z, acc);
    acc = fmaf(bf16_hi(w.w), b.w, acc);
    return acc;
}
template <>
__device__ __forceinline__ float dot_chunk<float>(const uint4& w, const float* xlo, const float*, float acc) {
    const float4 a = *reinterpret_cast<const float4*>(xlo);
    acc = fmaf(__uint_as_float(w.x), a.x, acc);
    acc = fmaf(__uint_as_float(w.y), a.y, acc);
    acc = fmaf(__uint_as_float(w.z), a.z, acc);
    acc = fmaf(__uint_as_float(w.w), a.w, acc);
    return acc;
}

// Partial dot products of rows row0..row0+R-1 of W ([rows][H]) with the NB
// shared-memory vectors xs[b*H ..] (laid out as xpos says).  Rows past
// last_row repeat last_row (their results are discarded by the caller).  Each
// lane covers chunks lane, lane+32..
template <typename WT, int NB, int R, int U>
__device__ __forceinline__ void dot_rows(const WT* __restrict__ W, int row0, int last_row, int H,
                                         const float* __restrict__ xs, float (&acc)[R][NB],
                                         int lane) {
    constexpr int VEC = Elems<WT>::n;
    const int nchunk = H / VEC;
    const char* rp[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        int row = min(row0 + r, last_row);
        rp[r] = reinterpret_cast<const char*>(W + (size_t)row * H);
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
    }
    for (int c0 = lane; c0 < nchunk; c0 += 32 * U) {
        uint4 w[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
#pragma unroll
            for (int r = 0; r < R; ++r)
                w[u][r] = c < nchunk ? ld_stream16(rp[r] + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
            if (c < nchunk) {
                const float* xlo = xs + (size_t)c * 4;  // see xpos
                const float* xhi = xlo + (H >> 1);
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        acc[r][b] = dot_chunk<WT>(w[u][r], xlo + (size_t)b * H, xhi + (size_t)b * H, acc[r][b]);
            }
        }
    }
}

// Chunk c (16 bytes) of a vector into its shared-memory places (see xpos); xv
// is the vector's base in shared memory.
template <typename WT>
__device__ __forceinline__ void store_chunk(const uint4& w, float* xv, int c, int H);
template <>
__device__ __forceinline__ void store_chunk<uint16_t>(const uint4& w, float* xv, int c, int H) {
    *reinterpret_cast<float4*>(xv + 4 * c) = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    *reinterpret_cast<float4*>(xv + (H >> 1) + 4 * c) =
        make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
}
template <>
__device__ __forceinline__ void store_chunk<float>(const uint4& w, float* xv, int c, int) {
    *reinterpret_cast<float4*>(xv + 4 * c) =
        make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w));
}

// The NB vectors src[b*H .. b*H + H) as float32 into dst[b*H ..] (xpos
// layout), with 16-byte loads when src is aligned (H is a multiple of 8, dst
// 16-byte aligned).  The loads are cached in L2 only: src may have been
// written by the previous kernel on the stream.
template <typename WT>
__device__ __forceinline__ void load_vector_to_smem(const WT* src, float* dst, int NB, int H) {
    constexpr int VEC = Elems<WT>::n;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        const int per = H / VEC;
#pragma unroll 4
        for (int c = threadIdx.x; c < NB * per; c += blockDim.x) {
            const int b = c / per;
            store_chunk<WT>(__ldcg(s4 + c), dst + (size_t)b * H, c - b * per, H);
        }
    } else {
        for (int i = threadIdx.x; i < NB * H; i += blockDim.x) {
            const int b = i / H, j = i - b * H;
            dst[(size_t)b * H + xpos<WT>(j, H)] = load_scalar<WT>(src, i);
        }
    }
}

// K1: z[b,k,i] = h[b,i] + SiLU(sum_j W1[k,i,j] h[b,j] + b1[k,i]).
// W1 is walked as K*H consecutive rows (row k*H + i); each warp of the grid
// takes an equal contiguous range of kRows1-row groups, so one wave of CTAs
// finishes together.  Block 0 also zeroes the per-head counters that K2 uses to
// elect the CTA that merges a head's slice lists.
template <typename WT, int NB, int THREADS>
__global__ void __launch_bounds__(THREADS) heads_w1_silu_kernel(
    const WT* __restrict__ h, const WT* __restrict__ w1, const WT* __restrict__ b1, int K, int H,
    float* __restrict__ z, unsigned* __restrict__ done) {
    extern __shared__ __align__(16) float xs[];  // [NB][H]
    pdl_wait();  // h may come from the previous kernel (the last round's compaction)
    if (blockIdx.x == 0)
        for (int k = threadIdx.x; k < K; k += THREADS) done[k] = 0u;
    load_vector_to_smem<WT>(h, xs, NB, H);
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long groups = (long long)K * H / kRows1;
    const long long nwarps = (long long)gridDim.x * (THREADS / 32);
    const long long gw = (long long)blockIdx.x * (THREADS / 32) + warp;
    const long long g0 = gw * groups / nwarps, g1 = (gw + 1) * groups / nwarps;
    for (long long g = g0; g < g1; ++g) {
        const int row = (int)(g * kRows1);  // kRows1 divides H: a group never spans heads
        const int k = row / H, i0 = row - k * H;
        float acc[kRows1][NB];
        dot_rows<WT, NB, kRows1, kUnroll1>(w1, row, row + kRows1 - 1, H, xs, acc, lane);
#pragma unroll
        for (int r = 0; r < kRows1; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float s = warp_sum(acc[r][b]);
                if (lane == ((r * NB + b) & 31)) {
                    const int i = i0 + r;
                    const float u = s + load_scalar<WT>(b1, (size_t)k * H + i);
                    const float silu = u / (1.f + expf(-u));
                    z[((size_t)b * K + k) * H + i] = xs[(size_t)b * H + xpos<WT>(i, H)] + silu;
                }
            }
    }
}

// K2: logits of one vocab slice of head k, then the slice's top-k per sequence.
// The last CTA of head k to finish (elected with an atomic counter that K1
// zeroed) merges the head's S slice lists into the final sorted top-k.
template <typename WT, int NB, int THREADS>
__global__ void __launch_bounds__(THREADS) heads_w2_topk_kernel(
    const WT* __restrict__ w2, const float* __restrict__ z, int K, int H, int V, int rows_per_cta,
    int topk, float* __restrict__ logits, float* __restrict__ cval, int* __restrict__ cidx,
    unsigned* __restrict__ done, int32_t* __restrict__ topk_idx, float* __restrict__ topk_val) {
    extern __shared__ __align__(16) float sm[];
    float* xs = sm;                       // [NB][H]
    float* lg = sm + (size_t)NB * H;      // [NB][rows_per_cta]
    __shared__ bool s_last;
    const int s = blockIdx.x, S = gridDim.x, k = blockIdx.y;
    const int v0 = s * rows_per_cta;
    const int v1 = min(V, v0 + rows_per_cta);
    const WT* wk = w2 + (size_t)k * V * H;
    // W2 does not depend on the previous kernel: start pulling this CTA's first
    // rows into L2 while K1 finishes.
    if (threadIdx.x == 0) {
        const int pr = min(kPrefetchRows, v1 - v0);
        const size_t bytes = (size_t)pr * H * sizeof(WT);
        if ((bytes & 15) == 0 && bytes > 0)
            prefetch_l2_bulk(wk + (size_t)v0 * H, (uint32_t)bytes);
    }
    pdl_wait();
    {
        // z rows are 16-byte aligned (H % 8 == 0); L2-only loads, K1 wrote them.
        // float4 j holds elements 4j..4j+3 (xpos layout: half j & 1 of chunk j / 2)
        const int h4 = H / 4;
#pragma unroll 4
        for (int c = threadIdx.x; c < NB * h4; c += THREADS) {
            const int b = c / h4, j = c - b * h4;
            const int dst = sizeof(WT) == 4 ? 4 * j : (j & 1) * (H >> 1) + 4 * (j >> 1);
            *reinterpret_cast<float4*>(xs + (size_t)b * H + dst) =
                __ldcg(reinterpret_cast<const float4*>(z + ((size_t)b * K + k) * H) + j);
        }
    }
    __syncthreads();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int g = v0 + warp * kRows2; g < v1; g += (THREADS / 32) * kRows2) {
        float acc[kRows2][NB];
        dot_rows<WT, NB, kRows2, kUnroll2>(wk, g, v1 - 1, H, xs, acc, lane);
#pragma unroll
        for (int r = 0; r < kRows2; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float sum = warp_sum(acc[r][b]);
                const int v = g + r;
                if (v < v1 && lane == ((r * NB + b) & 31)) {
                    lg[(size_t)b * rows_per_cta + (v - v0)] = sum;
                    if (logits) logits[((size_t)b * K + k) * V + v] = sum;
                }
            }
    }
    __syncthreads();
    const int n = v1 - v0;
    for (int b = warp; b < NB; b += THREADS / 32) {
        const float* row = lg + (size_t)b * rows_per_cta;
        float* ov = cval + (((size_t)b * K + k) * S + s) * topk;
        int* oi = cidx + (((size_t)b * K + k) * S + s) * topk;
        warp_select_topk(
            n, topk, [&](int j, float& x, int& xi) { x = row[j]; xi = v0 + j; },
            [&](int t, float v, int i) { ov[t] = v; oi[t] = i; }, lane);
    }
    // Elect the last CTA of head k: make this CTA's lists visible, then count.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&done[k], 1u) == (unsigned)(S - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Merge the S lists of each sequence, staged in shared memory when they fit.
    const int m = S * topk;
    for (int b = warp; b < NB; b += THREADS / 32) {
        const size_t base = ((size_t)b * K + k) * S * topk;
        int32_t* oi = topk_idx + ((size_t)b * K + k) * topk;
        float* ov = topk_val ? topk_val + ((size_t)b * K + k) * topk : nullptr;
        // the vectors and slice logits are no longer needed: sequence b stages
        // its lists in its own (H + rows_per_cta)-float share of shared memory
        const bool staged = 2 * m <= H + rows_per_cta;
        float* sv = sm + (size_t)b * (H + rows_per_cta);
        int* si = reinterpret_cast<int*>(sv + m);
        if (staged) {
            for (int j = lane; j < m; j += 32) {
                sv[j] = __ldcg(cval + base + j);
                si[j] = __ldcg(cidx + base + j);
            }
            __syncwarp();
        }
        warp_select_topk(
            m, topk,
            [&](int j, float& x, int& xi) {
                if (staged) { x = sv[j]; xi = si[j]; }
                else { x = __ldcg(cval + base + j); xi = __ldcg(cidx + base + j); }
            },
            [&](int t, float v, int i) {
                oi[t] = i;
                if (ov) ov[t] = v;
            },
            lane);
    }
}

struct HeadsPlan {
    int threads;       // 256 or 512
    int rows2;         // K2 vocab rows per CTA
    int S;             // K2 slices per head
    size_t smem1, smem2;
    size_t off_z, off_val, off_idx, off_done, ws_bytes;
};

HeadsPlan plan_heads(int B, int K, int H, int V, int topk) {
    HeadsPlan p{};
    if (B > 8) {  // tensor cores only
        p.ws_bytes = heads_umma_workspace(B, K, H, V, topk);
        return p;
    }
    const size_t xbytes = (size_t)B * H * sizeof(float);
    const bool big = xbytes > 64 * 1024;
    p.threads = big ? 512 : 256;
    const int per_sm = big ? 1 : 2;
    const int target = sm_count() * per_sm;
    // K2: vocab slices so that K * S fills one wave; each slice >= topk rows
    int s0 = target / K;
    if (s0 < 1) s0 = 1;
    int r2 = (V + s0 - 1) / s0;
    // a slice's logits live in shared memory next to the vectors
    const long long room = ((long long)max_smem_optin() - 1024 - (long long)xbytes) / ((long long)B * 4);
    if (room > 0 && r2 > room) r2 = (int)room;
    if (r2 < topk) r2 = topk;
    p.rows2 = r2;
    p.S = (V + r2 - 1) / r2;
    p.smem1 = xbytes;
    p.smem2 = xbytes + (size_t)B * r2 * sizeof(float);
    size_t off = 0;
    p.off_z = off;
    off = align_up(off + (size_t)B * K * H * sizeof(float), 256);
    p.off_val = off;
    off = align_up(off + (size_t)B * K * p.S * topk * sizeof(float), 256);
    p.off_idx = off;
    off = align_up(off + (size_t)B * K * p.S * topk * sizeof(int), 256);
    p.off_done = off;
    off = align_up(off + (size_t)K * sizeof(unsigned), 256);
    p.ws_bytes = off;
    if (heads_umma_applies(B, K, H, V, topk, true)) {
        const size_t u = heads_umma_workspace(B, K, H, V, topk);
        if (u > p.ws_bytes) p.ws_bytes = u;
    }
    return p;
}

template <typename WT, int NB, int THREADS>
int launch_heads(const void* h, const void* w1, const void* b1, const void* w2, int K, int H, int V,
                 int topk, int32_t* topk_idx, float* topk_val, float* logits, char* ws,
                 const HeadsPlan& p, cudaStream_t st) {
    float* z = reinterpret_cast<float*>(ws + p.off_z);
    float* cval = reinterpret_cast<float*>(ws + p.off_val);
    int* cidx = reinterpret_cast<int*>(ws + p.off_idx);
    unsigned* done = reinterpret_cast<unsigned*>(ws + p.off_done);
    auto k1 = heads_w1_silu_kernel<WT, NB, THREADS>;
    auto k2 = heads_w2_topk_kernel<WT, NB, THREADS>;
    if (p.smem1 > 48 * 1024)
        cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem1);
    if (p.smem2 > 48 * 1024)
        cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem2);
    // K1 grid: one wave of at most two CTAs per SM (no more warps than row
    // groups).  The rest of each SM stays free for K2's CTAs, which launch as
    // programmatic dependents while K1 runs: they load their set-up and warm L2
    // with their first W2 rows before K1 ends (batch-1 step: 268 -> 265 us
    // against a full K1 wave of four CTAs per SM).
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k1, THREADS, p.smem1) != cudaSuccess || occ < 1)
        occ = 1;
    long long grid1 = (long long)sm_count() * (occ < 2 ? occ : 2);
    const long long groups = (long long)K * H / kRows1;
    const long long max_ctas = (groups + THREADS / 32 - 1) / (THREADS / 32);
    if (grid1 > max_ctas) grid1 = max_ctas;
    cudaError_t e = launch(k1, dim3((unsigned)grid1), dim3(THREADS), p.smem1, st,
                           static_cast<const WT*>(h), static_cast<const WT*>(w1),
                           static_cast<const WT*>(b1), K, H, z, done);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_w1_silu: launch failed: %s", cudaGetErrorString(e));
    e = launch(k2, dim3(p.S, K), dim3(THREADS), p.smem2, st, static_cast<const WT*>(w2),
               static_cast<const float*>(z), K, H, V, p.rows2, topk, logits, cval, cidx, done,
               topk_idx, topk_val);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_w2_topk: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

template <typename WT, int NB>
int dispatch_threads(const void* h, const void* w1, const void* b1, const void* w2, int K, int H,
                     int V, int topk, int32_t* ti, float* tv, float* lg, char* ws,
                     const HeadsPlan& p, cudaStream_t st) {
    if (p.threads == 512)
        return launch_heads<WT, NB, 512>(h, w1, b1, w2, K, H, V, topk, ti, tv, lg, ws, p, st);
    return launch_heads<WT, NB, 256>(h, w1, b1, w2, K, H, V, topk, ti, tv, lg, ws, p, st);
}

template <typename WT>
int dispatch_batch(int B, const void* h, const void* w1, const void* b1, const void* w2, int K,
                   int H, int V, int topk, int32_t* ti, float* tv, float* lg, char* ws,
                   const HeadsPlan& p, cudaStream_t st) {
    switch (B) {
#define MEDUSA_CASE(n) \
    case n: return dispatch_threads<WT, n>(h, w1, b1, w2, K, H, V, topk, ti, tv, lg, ws, p, st);
        MEDUSA_CASE(1) MEDUSA_CASE(2) MEDUSA_CASE(3) MEDUSA_CASE(4)
        MEDUSA_CASE(5) MEDUSA_CASE(6) MEDUSA_CASE(7) MEDUSA_CASE(8)
#undef MEDUSA_CASE
    }
    return fail(MEDUSA_ERR_UNSUPPORTED, "heads_topk: batch %d not in [1, 8]", B);
}

int check_heads_shapes(int B, int K, int H, int V, int topk) {
    if (B < 1 || K < 1 || H < 1 || V < 1 || topk < 1)
        return fail(MEDUSA_ERR_INVALID_ARG, "heads_topk: sizes must be positive (B=%d K=%d H=%d V=%d topk=%d)",
                    B, K, H, V, topk);
    // batches 9-64 exist only on the tensor cores (bf16, H % 128 == 0)
    const bool wide_ok = B > 8 && B <= 64 && heads_umma_applies(B, K, H, V, topk, true);
    if ((B > 8 && !wide_ok) || K > 64 || H < 8 || H > 16384 || H % 8 || (B <= 8 && (long long)B * H > 49152) ||
        topk > 16 || topk > V)
        return fail(MEDUSA_ERR_UNSUPPORTED,
                    "heads_topk: unsupported shape (B=%d K=%d H=%d V=%d topk=%d): need K<=64, "
                    "8<=H<=16384, H%%8==0, topk<=16, topk<=V, and B<=8 with B*H<=49152, or B<=64 "
                    "for bf16 with H%%128==0",
                    B, K, H, V, topk);
    return MEDUSA_OK;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_heads_topk_workspace(int B, int K, int H, int V, int topk) {
    if (check_heads_shapes(B, K, H, V, topk)) return 0;
    return plan_heads(B, K, H, V, topk).ws_bytes;
}

extern "C" int medusa_heads_topk(const void* h, const void* w1, const void* b1, const void* w2,
                                 medusa_dtype dtype, int B, int K, int H, int V, int topk,
                                 int32_t* topk_idx, float* topk_val, float* logits, void* ws,
                                 size_t ws_bytes, void* stream) {
    int rc = check_heads_shapes(B, K, H, V, topk);
    if (rc) return rc;
    if (!h || !w1 || !b1 || !w2 || !topk_idx)
        return fail(MEDUSA_ERR_INVALID_ARG, "heads_topk: null input or output pointer");
    if (!aligned16(w1) || !aligned16(w2))
        return fail(MEDUSA_ERR_INVALID_ARG, "heads_topk: w1 and w2 must be 16-byte aligned");
    if (dtype != MEDUSA_F32 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_UNSUPPORTED, "heads_topk: unknown dtype %d", (int)dtype);
    if (B > 8 && dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_UNSUPPORTED, "heads_topk: batches above 8 need bf16 (batch %d)", B);
    HeadsPlan p = plan_heads(B, K, H, V, topk);
    if (!ws || ws_bytes < p.ws_bytes)
        return fail(MEDUSA_ERR_WORKSPACE, "heads_topk: workspace of %zu bytes needed, %zu given",
                    p.ws_bytes, ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(MEDUSA_ERR_INVALID_ARG, "heads_topk: ws must be 16-byte aligned");
    if (p.smem2 > (size_t)max_smem_optin())
        return fail(MEDUSA_ERR_UNSUPPORTED, "heads_topk: %zu bytes of shared memory needed", p.smem2);
    cudaStream_t st = as_stream(stream);
    char* w = static_cast<char*>(ws);
    if (heads_umma_applies(B, K, H, V, topk, dtype == MEDUSA_BF16)) {
        if (!aligned16(h)) return fail(MEDUSA_ERR_INVALID_ARG, "heads_topk: h must be 16-byte aligned");
        return launch_heads_umma(h, w1, b1, w2, B, K, H, V, topk, topk_idx, topk_val, logits, w, st);
    }
    if (dtype == MEDUSA_BF16)
        return dispatch_batch<uint16_t>(B, h, w1, b1, w2, K, H, V, topk, topk_idx, topk_val, logits,
                                        w, p, st);
    return dispatch_batch<float>(B, h, w1, b1, w2, K, H, V, topk, topk_idx, topk_val, logits, w, p,
                                 st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of medusa_heads_topk.
//
// Some callers cannot call cudaMalloc: a plugin or custom operator inside a
// host inference engine that owns all device memory and hands its operators no
// workspace, or a process whose device memory is entirely reserved by a pool
// it may not grow.  For them medusa_heads_topk_static takes its scratch (the
// float32 z vectors and the per-slice top-k candidates) from one file-scope
// device array of MEDUSA_HEADS_STATIC_SCRATCH_BYTES instead of a caller buffer.
// Every GPU that loads this library reserves that array until the process
// exits.  Host code never passes the array's name to a kernel (in host code it
// is only a stand-in symbol): the device address comes from
// cudaGetSymbolAddress with that device current.  The address is cached per
// device together with the unique ID of the CUDA context it was looked up in;
// a call made in another context (after cudaDeviceReset, or under a context the
// caller created) looks it up again, so a stale address is never used.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_heads_static_scratch[MEDUSA_HEADS_STATIC_SCRATCH_BYTES];

namespace medusa {
namespace {
std::mutex g_static_mu;
void* g_static_ptr[64];
unsigned long long g_static_ctx[64];

int static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(MEDUSA_ERR_CUDA, "heads_topk_static: cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64)
        return fail(MEDUSA_ERR_UNSUPPORTED, "heads_topk_static: device index %d above 63", dev);
    unsigned long long ctx = 0;
    int rc = current_context_id(&ctx);
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev] || ctx == 0 || g_static_ctx[dev] != ctx) {
        // the lookup also initialises the device's primary context when none
        // is current yet
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_heads_static_scratch);
        if (e != cudaSuccess || !p)
            return fail(MEDUSA_ERR_CUDA, "heads_topk_static: cudaGetSymbolAddress failed: %s",
                        cudaGetErrorString(e));
        if (ctx == 0 && (rc = current_context_id(&ctx)) != 0) return rc;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = ctx;
    }
    *out = g_static_ptr[dev];
    return MEDUSA_OK;
}
}  // namespace
}  // namespace medusa

extern "C" int medusa_heads_topk_static(const void* h, const void* w1, const void* b1,
                                        const void* w2, medusa_dtype dtype, int B, int K, int H,
                                        int V, int topk, int32_t* topk_idx, float* topk_val,
                                        float* logits, void* stream) {
    int rc = check_heads_shapes(B, K, H, V, topk);
    if (rc) return rc;
    const size_t need = plan_heads(B, K, H, V, topk).ws_bytes;
    if (need > (size_t)MEDUSA_HEADS_STATIC_SCRATCH_BYTES)
        return fail(MEDUSA_ERR_UNSUPPORTED,
                    "heads_topk_static: these shapes need %zu bytes of scratch, above the static "
                    "maximum of %zu bytes; use medusa_heads_topk with a caller workspace",
                    need, (size_t)MEDUSA_HEADS_STATIC_SCRATCH_BYTES);
    void* ws = nullptr;
    rc = static_scratch(&ws);
    if (rc) return rc;
    // No scratch byte needs to start at zero: the call writes every byte whose
    // value it uses (z before the vocab pass, the slice lists before the merge;
    // on the tensor-core path the padding rows of the z planes are loaded but
    // feed only accumulator columns that are never read).
    return medusa_heads_topk(h, w1, b1, w2, dtype, B, K, H, V, topk, topk_idx, topk_val, logits, ws,
                             (size_t)MEDUSA_HEADS_STATIC_SCRATCH_BYTES, stream);
}
