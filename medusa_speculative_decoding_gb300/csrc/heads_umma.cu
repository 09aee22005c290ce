// heads_umma.cu -- Medusa heads on the tensor cores for batches of 4 to 8
// ("Medusa Heads" glossary page, "How heads predict later tokens": head k
// computes W2_k (h + SiLU(W1_k h + b1_k)) from the last hidden state h).
//
// At a batch of one or two the heads are matrix-vector products and stay on
// CUDA cores (heads.cu).  From a batch of four, every weight element feeds 4-8
// products and the CUDA-core path runs out of issue slots and shared-memory
// bandwidth before HBM does, so the same products run as skinny GEMMs on
// tcgen05: the weights are the M = 128 operand (K-major, streamed by TMA), the
// batch's vectors the N operand, accumulators in TMEM.
//   heads_w1_umma_kernel : D[128 W1 rows x 16] = W1 . h^T (h is bf16, exact);
//                          epilogue z = h + SiLU(D + b1) in float32, written as
//                          three bf16 planes z = hi + mid + lo (the split keeps
//                          24 significant bits, as many as float32)
//   heads_w2_umma_kernel : D[128 vocab rows x N] = W2 . [hi; mid; lo]^T with N =
//                          3B rounded up to 16; the logit of sequence b is the
//                          sum of its three columns.  Each CTA takes a run of
//                          (head, 128-row vocab tile) items, keeps every tile's
//                          top-k per sequence, reduces each head's run to one
//                          list, and the last CTA of a head merges the head's
//                          lists into the final sorted top-k.
// Roles (192 threads): warp 0 TMA producer, warp 1 TMEM allocation and MMA
// issue, warps 2-5 epilogue (warp w reads TMEM lanes 32*(w%4) ..).  Every wait
// is bounded; a CTA that gives up marks the call's status word and writes -1
// into the top-k lists it owns.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "tmap.cuh"
#include "topk.cuh"
#include "umma.cuh"

namespace medusa {
namespace {

constexpr int kUM = 128;                 // weight rows per tile (MMA M)
constexpr int kUK = 64;                  // hidden elements per stage
constexpr int kUThreads = 192;
constexpr int kUA = kUM * kUK * 2;       // 16 KB of weight rows per stage
constexpr int kUBmax = 32 * kUK * 2;     // 4 KB of activation rows per stage (N <= 32)
constexpr int kUStage = kUA + kUBmax;
constexpr int kUMaxItems = 16;           // W2 items one CTA may own
constexpr int kUMaxB = 8;
constexpr int kUTopk = 16;
constexpr long long kUWait = 1ll << 31;  // ~1 s at 2 GHz
// W1: two CTAs per SM (its 160-200 tiles then need no second round); W2: one
// CTA per SM with a deeper ring, so each SM's share of the 128-row items is
// within one item of the mean
constexpr int kW1Stages = 5, kW2Stages = 8;

// ring | barriers | tmem slot, flags | (W2 only) tile logits and run staging
template <int STAGES, bool STAGING>
struct UmmaSmem {
    static constexpr int kStages = STAGES;
    static constexpr int kBars = 2 * STAGES + 4 + 1;
    static constexpr int kOffBar = STAGES * kUStage;
    static constexpr int kOffMisc = kOffBar + kBars * 8;
    static constexpr int kOffLgt = kOffMisc + 32;                           // float [8][128]
    static constexpr int kOffRunV = kOffLgt + (STAGING ? kUMaxB * kUM * 4 : 0);
    static constexpr int kRun = STAGING ? kUMaxB * kUMaxItems * kUTopk * 4 : 0;
    static constexpr int kOffRunI = kOffRunV + kRun;
    static constexpr int kBytes = kOffRunI + kRun + 1024;
};
using W1Smem = UmmaSmem<kW1Stages, false>;
using W2Smem = UmmaSmem<kW2Stages, true>;

// Shared pipeline: warp 0 streams A (weights) and B (activations) slices for
// each item, warp 1 issues the MMAs into one of two TMEM accumulators, the
// epilogue warps call epi(item, tmem column base) once per item and release the
// accumulator.  Returns false (on every thread) if a wait gave up.
template <typename Sm, typename Coords, typename Epi>
__device__ __forceinline__ bool umma_pipeline(uint8_t* base, uint32_t tmem, int nitems, int nkb, int N,
                                              const CUtensorMap* tma, const CUtensorMap* tmb,
                                              Coords coords, Epi epi) {
    using namespace umma;
    const uint32_t sbase = smem_addr(base);
    const uint32_t bar0 = sbase + Sm::kOffBar;
    auto full = [&](int i) { return bar0 + 8 * i; };
    auto empty = [&](int i) { return bar0 + 8 * (Sm::kStages + i); };
    auto d_full = [&](int i) { return bar0 + 8 * (2 * Sm::kStages + i); };
    auto d_empty = [&](int i) { return bar0 + 8 * (2 * Sm::kStages + 2 + i); };
    const uint32_t drain = bar0 + 8 * (2 * Sm::kStages + 4);
    volatile int* fail_flag = reinterpret_cast<volatile int*>(base + Sm::kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bbytes = (uint32_t)N * kUK * 2;
    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < nitems && ok; ++it) {
                int ay, by;
                coords(it, ay, by);
                for (int kb = 0; kb < nkb; ++kb, ++issued) {
                    const int st = issued % Sm::kStages;
                    if (issued >= Sm::kStages && !mbar_wait(empty(st), ((issued / Sm::kStages) - 1) & 1, kUWait)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + st * kUStage, sb = sa + kUA;
                    mbar_expect_tx(full(st), (uint32_t)kUA + bbytes);
                    tma_load_2d(sa, tma, kb * kUK, ay, full(st));
                    tma_load_2d(sb, tmb, kb * kUK, by, full(st));
                }
            }
            if (!ok) *fail_flag = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kUM, N, 0, 0);
            bool ok = true;
            int it2 = 0;
            for (int it = 0; it < nitems && ok; ++it) {
                const int buf = it & 1;
                if (it >= 2 && !mbar_wait(d_empty(buf), ((it / 2) - 1) & 1, kUWait)) {
                    ok = false;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(buf * 32);
                for (int kb = 0; kb < nkb; ++kb, ++it2) {
                    const int st = it2 % Sm::kStages;
                    if (!mbar_wait(full(st), (it2 / Sm::kStages) & 1, kUWait)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t sa = sbase + st * kUStage, sb = sa + kUA;
#pragma unroll
                    for (int ks = 0; ks < kUK / 16; ++ks)
                        mma_bf16(d, desc_sw128(sa + ks * 32, 16, 1024), desc_sw128(sb + ks * 32, 16, 1024),
                                 idesc, (kb | ks) != 0);
                    commit(empty(st));
                }
                if (ok) commit(d_full(buf));
            }
            if (!ok) *fail_flag = 1;
            commit(drain);  // every MMA issued here completes before TMEM is released
            if (!mbar_wait(drain, 0, kUWait)) *fail_flag = 1;
        }
    } else {
        bool ok = true;
        for (int it = 0; it < nitems; ++it) {
            const int buf = it & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(d_full(buf), (it / 2) & 1, kUWait));
            if (!ok) break;
            fence_after_sync();
            epi(it, (uint32_t)(buf * 32));
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty(buf));
        }
        if (!ok && lane == 0) *fail_flag = 1;
    }
    fence_before_sync();
    __syncthreads();
    const bool failed = *fail_flag != 0;
    if (failed && warp == 0 && lane == 0)  // let copies in flight land first
        for (int i = max(0, issued - Sm::kStages); i < issued; ++i)
            mbar_wait(full(i % Sm::kStages), (i / Sm::kStages) & 1, kUWait);
    return !failed;
}

template <typename Sm>
__device__ __forceinline__ void umma_setup(uint8_t* base, uint32_t* tmem_out) {
    using namespace umma;
    const uint32_t bar0 = smem_addr(base) + Sm::kOffBar;
    uint32_t* slot = reinterpret_cast<uint32_t*>(base + Sm::kOffMisc);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * Sm::kStages; ++i) mbar_init(bar0 + 8 * i, 1);
        mbar_init(bar0 + 8 * (2 * Sm::kStages + 0), 1);
        mbar_init(bar0 + 8 * (2 * Sm::kStages + 1), 1);
        mbar_init(bar0 + 8 * (2 * Sm::kStages + 2), 4);  // one arrival per epilogue warp
        mbar_init(bar0 + 8 * (2 * Sm::kStages + 3), 4);
        mbar_init(bar0 + 8 * (2 * Sm::kStages + 4), 1);
        *reinterpret_cast<volatile int*>(base + Sm::kOffMisc + 4) = 0;
        mbar_init_fence();
    }
    if ((threadIdx.x >> 5) == 1) tmem_alloc(slot, 64);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    *tmem_out = *slot;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

// z = h + SiLU(W1 h + b1) for 128 rows of W1 per item; items are the K*H/128
// row tiles, dealt evenly over the grid.
__global__ void __launch_bounds__(kUThreads, 2) heads_w1_umma_kernel(
    const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmh,
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ b1, int B, int K, int H,
    uint16_t* __restrict__ zp, unsigned* __restrict__ done, int* __restrict__ status) {
    using namespace umma;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint32_t tmem;
    umma_setup<W1Smem>(base, &tmem);
    pdl_wait();  // h may come from the previous kernel (the last round's compaction)
    if (blockIdx.x == 0) {
        for (int k = threadIdx.x; k < K; k += blockDim.x) done[k] = 0u;
        if (threadIdx.x == 0) *status = 0;
    }
    pdl_trigger();
    const int tiles = K * H / kUM;
    const int i0 = (int)((long long)blockIdx.x * tiles / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * tiles / gridDim.x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
    auto coords = [&](int it, int& ay, int& by) { ay = (i0 + it) * kUM; by = 0; };
    auto epi = [&](int it, uint32_t col) {
        const int row = (i0 + it) * kUM + q * 32 + lane;  // W1 row k*H + i
        const int k = row / H, i = row - k * H;
        float d[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + col, d);
        tmem_wait_ld();
        const float bias = bf16_to_f32(b1[(size_t)k * H + i]);
#pragma unroll
        for (int b = 0; b < kUMaxB; ++b) {
            if (b < B) {
                const float u = d[b] + bias;
                const float z = bf16_to_f32(h[(size_t)b * H + i]) + u / (1.f + expf(-u));
                const uint16_t hi = f32_to_bf16_rn(z);
                const float r1 = z - bf16_to_f32(hi);
                const uint16_t mid = f32_to_bf16_rn(r1);
                const uint16_t lo = f32_to_bf16_rn(r1 - bf16_to_f32(mid));
                uint16_t* zk = zp + (size_t)k * 3 * B * H;
                zk[((size_t)0 * B + b) * H + i] = hi;
                zk[((size_t)1 * B + b) * H + i] = mid;
                zk[((size_t)2 * B + b) * H + i] = lo;
            }
        }
    };
    const bool ok = umma_pipeline<W1Smem>(base, tmem, i1 - i0, H / kUK, 16, &tmw, &tmh, coords, epi);
    if (!ok && threadIdx.x == 0) atomicExch(status, 1);
    if (warp == 1) {
        fence_after_sync();
        tmem_dealloc(tmem, 64);
    }
}

struct W2Args {
    int B, K, H, V, T, topk, N;
    int items;          // K * T
    float* logits;      // [B][K][V] or nullptr
    float* run_val;     // [K][grid][B][topk]
    int* run_idx;
    unsigned* done;     // [K]
    int* status;
    int32_t* topk_idx;  // [B][K][topk]
    float* topk_val;    // or nullptr
};

// first and one-past-last CTA whose item range meets head k (items dealt evenly)
__device__ __forceinline__ void head_ctas(int k, int T, int items, int grid, int& c0, int& c1) {
    // CTA c owns items [c*items/grid, (c+1)*items/grid)
    const long long a = (long long)k * T, z = (long long)(k + 1) * T;  // head k's items [a, z)
    c0 = (int)((a * grid) / items);
    while (c0 > 0 && (long long)c0 * items / grid > a) --c0;
    while ((long long)(c0 + 1) * items / grid <= a) ++c0;
    c1 = (int)(((z - 1) * grid) / items);
    while ((long long)(c1 + 1) * items / grid <= z - 1) ++c1;
    while (c1 > 0 && (long long)c1 * items / grid > z - 1) --c1;
    ++c1;
}

template <int NB>
__global__ void __launch_bounds__(kUThreads, 1) heads_w2_umma_kernel(
    const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmz, W2Args a) {
    using namespace umma;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* lgt = reinterpret_cast<float*>(base + W2Smem::kOffLgt);
    float* runv = reinterpret_cast<float*>(base + W2Smem::kOffRunV);
    int* runi = reinterpret_cast<int*>(base + W2Smem::kOffRunI);
    __shared__ int s_last;
    uint32_t tmem;
    umma_setup<W2Smem>(base, &tmem);
    pdl_wait();  // the z planes come from heads_w1_umma_kernel
    pdl_trigger();
    const int c = blockIdx.x, grid = gridDim.x;
    const int i0 = (int)((long long)c * a.items / grid), i1 = (int)((long long)(c + 1) * a.items / grid);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
    constexpr int B = NB;
    const int T = a.T, topk = a.topk;
    const int ew = warp - 2;  // epilogue warp 0..3
    auto coords = [&](int it, int& ay, int& by) {
        const int g = i0 + it, k = g / T, t = g - k * T;
        ay = k * a.V + t * kUM;
        by = k * 3 * B;
    };
    // Writes head k's run (items [r0, r1) of this CTA, staged in runv/runi) as
    // one top-k list per sequence, then merges the head if this CTA is last.
    auto finish_run = [&](int k, int nstaged) {
        for (int b = ew; b < B; b += 4) {
            float* ov = a.run_val + (((size_t)k * grid + c) * B + b) * topk;
            int* oi = a.run_idx + (((size_t)k * grid + c) * B + b) * topk;
            const float* sv = runv + b * kUMaxItems * kUTopk;
            const int* si = runi + b * kUMaxItems * kUTopk;
            warp_select_topk(
                nstaged, topk, [&](int j, float& x, int& xi) { x = sv[j]; xi = si[j]; },
                [&](int t, float v, int i) { ov[t] = v; oi[t] = i; }, lane);
        }
        __threadfence();
        named_barrier_or(1, 128, false);
        int h0, h1;
        head_ctas(k, T, a.items, grid, h0, h1);
        if (ew == 0 && lane == 0) s_last = atomicAdd(&a.done[k], 1u) == (unsigned)(h1 - h0 - 1);
        named_barrier_or(1, 128, false);
        if (!s_last) return;
        __threadfence();
        const int m = (h1 - h0) * topk;
        for (int b = ew; b < B; b += 4) {
            int32_t* oi = a.topk_idx + ((size_t)b * a.K + k) * topk;
            float* ov = a.topk_val ? a.topk_val + ((size_t)b * a.K + k) * topk : nullptr;
            warp_merge_topk<kUTopk>(
                m, topk,
                [&](int j, float& x, int& xi) {
                    const int cc = h0 + j / topk, e = j - (j / topk) * topk;
                    const size_t o = (((size_t)k * grid + cc) * B + b) * topk + e;
                    x = __ldcg(a.run_val + o);
                    xi = __ldcg(a.run_idx + o);
                },
                [&](int t, float v, int i) {
                    oi[t] = i;
                    if (ov) ov[t] = v;
                },
                lane);
        }
    };
    int run_k = -1, nstaged = 0;
    auto epi = [&](int it, uint32_t col) {
        const int g = i0 + it, k = g / T, t = g - k * T;
        if (k != run_k) {
            if (run_k >= 0) finish_run(run_k, nstaged);
            run_k = k;
            nstaged = 0;
        }
        const int vl = q * 32 + lane, v = t * kUM + vl;
        float d[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + col, d);
        tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const float x = v < a.V ? d[b] + d[B + b] + d[2 * B + b] : -INFINITY;
            lgt[b * kUM + vl] = x;
            if (a.logits && v < a.V) a.logits[((size_t)b * a.K + k) * a.V + v] = x;
        }
        named_barrier_or(1, 128, false);
        for (int b = ew; b < B; b += 4) {
            float* sv = runv + b * kUMaxItems * kUTopk + nstaged;
            int* si = runi + b * kUMaxItems * kUTopk + nstaged;
            const float* row = lgt + b * kUM;
            warp_select_topk(
                kUM, topk, [&](int j, float& x, int& xi) { x = row[j]; xi = t * kUM + j; },
                [&](int tt, float vv, int ii) { sv[tt] = vv; si[tt] = ii; }, lane);
        }
        nstaged += topk;
        named_barrier_or(1, 128, false);
    };
    // a failure of the first kernel leaves the z planes undefined
    const bool ok1 = __syncthreads_or(*(volatile int*)a.status != 0) == 0;
    bool ok = ok1 && umma_pipeline<W2Smem>(base, tmem, i1 - i0, a.H / kUK, a.N, &tmw, &tmz, coords, epi);
    if (ok && warp >= 2 && run_k >= 0) finish_run(run_k, nstaged);
    if (!ok) {
        // every list of the heads this CTA touches is marked invalid
        if (threadIdx.x == 0) atomicExch(a.status, 1);
        const int k0 = i0 / T, k1 = (i1 - 1) / T;
        const int n = (k1 - k0 + 1) * B * topk;
        for (int j = threadIdx.x; j < n; j += blockDim.x) {
            const int e = j % topk, b = (j / topk) % B, k = k0 + j / (topk * B);
            a.topk_idx[((size_t)b * a.K + k) * topk + e] = -1;
        }
    }
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, 64);
    }
}

int bf16_rows_map(CUtensorMap* m, const void* p, int H, long long rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(MEDUSA_ERR_CUDA, "heads_topk: cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {(cuuint32_t)kUK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MEDUSA_ERR_CUDA, "heads_topk: tensor map encode failed (%d)", (int)r);
    return MEDUSA_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// W2 items are dealt over one CTA per SM
int umma_grid() { return sm_count(); }

bool heads_umma_applies(int B, int K, int H, int V, int topk, bool bf16) {
    const int grid = umma_grid();
    const int T = (V + kUM - 1) / kUM;
    return bf16 && B >= 4 && B <= kUMaxB && H % kUM == 0 && topk <= kUTopk &&
           ((long long)K * T + grid - 1) / grid <= kUMaxItems && (long long)K * V < (1ll << 31) &&
           W2Smem::kBytes <= max_smem_optin();
}

size_t heads_umma_workspace(int B, int K, int H, int V, int topk) {
    const int grid = umma_grid();
    size_t off = align_up((size_t)K * 3 * B * H * 2, 256);                 // z planes
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);            // run values
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);            // run indices
    off = align_up(off + (size_t)K * 4, 256);                              // done counters
    return align_up(off + 16, 256);                                        // status
}

int launch_heads_umma(const void* h, const void* w1, const void* b1, const void* w2, int B, int K, int H,
                      int V, int topk, int32_t* topk_idx, float* topk_val, float* logits, char* ws,
                      cudaStream_t st) {
    const int grid = umma_grid();
    const int T = (V + kUM - 1) / kUM;
    const int N = (3 * B + 15) / 16 * 16;
    uint16_t* zp = reinterpret_cast<uint16_t*>(ws);
    size_t off = align_up((size_t)K * 3 * B * H * 2, 256);
    float* run_val = reinterpret_cast<float*>(ws + off);
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);
    int* run_idx = reinterpret_cast<int*>(ws + off);
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);
    unsigned* done = reinterpret_cast<unsigned*>(ws + off);
    off = align_up(off + (size_t)K * 4, 256);
    int* status = reinterpret_cast<int*>(ws + off);
    CUtensorMap tw1, th, tw2, tz;
    int rc = bf16_rows_map(&tw1, w1, H, (long long)K * H, kUM);
    if (!rc) rc = bf16_rows_map(&th, h, H, B, 16);
    if (!rc) rc = bf16_rows_map(&tw2, w2, H, (long long)K * V, kUM);
    if (!rc) rc = bf16_rows_map(&tz, zp, H, (long long)K * 3 * B, N);
    if (rc) return rc;
    cudaFuncSetAttribute(heads_w1_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, W1Smem::kBytes);
    auto k2 = B == 4 ? heads_w2_umma_kernel<4> : B == 5 ? heads_w2_umma_kernel<5> : B == 6 ? heads_w2_umma_kernel<6>
            : B == 7 ? heads_w2_umma_kernel<7> : heads_w2_umma_kernel<8>;
    cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, W2Smem::kBytes);
    const int tiles1 = K * H / kUM;
    cudaError_t e = launch(heads_w1_umma_kernel, dim3(min(2 * grid, tiles1)), dim3(kUThreads), (size_t)W1Smem::kBytes, st,
                           tw1, th, static_cast<const uint16_t*>(h), static_cast<const uint16_t*>(b1), B, K, H,
                           zp, done, status);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_w1_umma: launch failed: %s", cudaGetErrorString(e));
    W2Args a{};
    a.B = B; a.K = K; a.H = H; a.V = V; a.T = T; a.topk = topk; a.N = N;
    a.items = K * T;
    a.logits = logits;
    a.run_val = run_val;
    a.run_idx = run_idx;
    a.done = done;
    a.status = status;
    a.topk_idx = topk_idx;
    a.topk_val = topk_val;
    e = launch(k2, dim3(min(grid, a.items)), dim3(kUThreads), (size_t)W2Smem::kBytes, st, tw2, tz, a);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_w2_umma: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

}  // namespace medusa
