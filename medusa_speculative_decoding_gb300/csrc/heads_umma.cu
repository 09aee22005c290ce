// heads_umma.cu -- Medusa heads on the tensor cores for batches of 3 to 64
// ("Medusa Heads" glossary page, "How heads predict later tokens": head k
// computes W2_k (h + SiLU(W1_k h + b1_k)) from the last hidden state h).
//
// At a batch of one or two the heads are matrix-vector products and stay on
// CUDA cores (heads.cu).  From a batch of three, every weight element feeds
// 3-64 products and the CUDA-core path runs out of issue slots and shared-memory
// bandwidth before HBM does, so the same products run as skinny GEMMs on
// tcgen05: the weights are the M = 128 operand (K-major, streamed by TMA), the
// batch's vectors the N operand, accumulators in TMEM.  The batch is padded to
// Bp, a multiple of 16.
//   heads_w1_umma_kernel : D[128 W1 rows x Bp] = W1 . h^T (h is bf16, exact);
//                          epilogue z = h + SiLU(D + b1) in float32, written as
//                          three bf16 planes z = hi + mid + lo (the split keeps
//                          24 significant bits, as many as float32)
//   heads_w2_umma_kernel : D[128 vocab rows x 3 Bp] = W2 . [hi; mid; lo]^T, the
//                          planes at columns [0, Bp), [Bp, 2Bp), [2Bp, 3Bp); the
//                          logit of sequence b is the sum of its three columns.
//                          Each CTA takes a run of (head, 128-row vocab tile)
//                          items and keeps every sequence's top-k over its run
//                          (a tile enters the list only where one of its logits
//                          beats the list's last entry)
//   heads_merge_kernel   : merges every head's run lists into the sorted top-k
// Roles of the two tensor-core kernels (192 threads): warp 0 TMA producer, warp
// 1 TMEM allocation and MMA issue, warps 2-5 epilogue (warp w reads TMEM lanes
// 32*(w%4) ..).  Every wait is bounded; every CTA writes its own status slot
// (nonzero if a wait gave up), and the merge then writes -1 into every top-k
// list of a call in which any slot is set.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "tmap.cuh"
#include "topk.cuh"
#include "umma.cuh"

namespace medusa {
namespace {

MEDUSA_WAIT_CONTROL()

constexpr int kUM = 128;                 // weight rows per tile (MMA M)
constexpr int kUK = 64;                  // hidden elements per stage
constexpr int kUThreads = 192;
constexpr int kUA = kUM * kUK * 2;       // 16 KB of weight rows per stage
constexpr int kUMinB = 3, kUMaxB = 64;    // batches on the tensor cores
constexpr int kUTopk = 16;
constexpr int kUSmemCap = 227 * 1024;    // opt-in shared memory per CTA
constexpr long long kUWait = kDefaultWaitCycles;  // drain waits (~1 s at 2 GHz)

// ring of STAGES x (16 KB weights + BBYTES activations) | barriers | tmem slot,
// flags | EXTRA bytes of epilogue staging.  Accumulator buffer i sits at TMEM
// column i * ACC; the CTA allocates TMEMC columns.
template <int STAGES, int BBYTES, int ACC, int TMEMC, int EXTRA>
struct UmmaSmem {
    static constexpr int kStages = STAGES;
    static constexpr int kStage = kUA + BBYTES;
    static constexpr int kAcc = ACC;
    static constexpr int kTmemCols = TMEMC;
    static constexpr int kBars = 2 * STAGES + 4 + 1;
    static constexpr int kOffBar = STAGES * kStage;
    static constexpr int kOffMisc = kOffBar + kBars * 8;
    static constexpr int kOffExtra = kOffMisc + 32;
    static constexpr int kBytes = kOffExtra + EXTRA + 1024;
    static_assert(kStage % 1024 == 0, "stages start on 1024-byte swizzle atoms");
};
// W1: Bp <= 64 activation rows per stage, two CTAs per SM (the K*H/128 row tiles
// then need no second round)
using W1Smem = UmmaSmem<4, kUMaxB * kUK * 2, 64, 128, 0>;

// W2 at a batch padded to BP: N = 3 BP rows of z planes per stage (one CTA per
// SM, as many stages as fit); tile logits float [BP][129] (one padding word per
// row), and one sorted list of 16 (value, index) pairs per sequence [BP][16]
// (values, then indices)
constexpr int kLgtStride = kUM + 1;
constexpr int kEpi = 128;      // epilogue threads
constexpr int kRebuildAt = 6;  // more candidates than this: rebuild instead of inserting
template <int BP>
struct W2Cfg {
    static constexpr int kN = 3 * BP;
    static constexpr int kBBytes = kN * kUK * 2;
    static constexpr int kLgt = (BP * kLgtStride * 4 + 15) / 16 * 16;
    static constexpr int kList = BP * kUTopk * 8;
    static constexpr int kExtra = kLgt + kList;
    static constexpr int kFit = (kUSmemCap - kExtra - 2048) / (kUA + kBBytes);
    static constexpr int kStages = kFit < 8 ? kFit : 8;
    using Sm = UmmaSmem<kStages, kBBytes, 256, 512, kExtra>;
    static_assert(BP <= 64 && kN <= 256 && kStages >= 3 && Sm::kBytes <= kUSmemCap, "W2 configuration");
};

// One warp keeps a sorted list of kUTopk (value, index) pairs, best first (the
// order of `better`), as entry j in lane j (lanes from kUTopk on hold empty
// entries).  Inserting a pair shifts the worse entries down one lane.
__device__ __forceinline__ void wl_insert(float& ev, int& ei, float cv, int ci, int lane) {
    const unsigned worse = __ballot_sync(0xffffffffu, better(cv, ci, ev, ei));  // a suffix of lanes
    const int p = __ffs(worse) - 1;
    const float uv = __shfl_up_sync(0xffffffffu, ev, 1);
    const int ui = __shfl_up_sync(0xffffffffu, ei, 1);
    if (worse != 0u) {
        if (lane > p) { ev = uv; ei = ui; }
        else if (lane == p) { ev = cv; ei = ci; }
    }
}

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
    // limit of the first waits; the drain waits keep kUWait
    const long long lim = g_wait_limit;
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
                    if (issued >= Sm::kStages && !mbar_wait(empty(st), ((issued / Sm::kStages) - 1) & 1, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + st * Sm::kStage, sb = sa + kUA;
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
                if (it >= 2 && !mbar_wait(d_empty(buf), ((it / 2) - 1) & 1, lim)) {
                    ok = false;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(buf * Sm::kAcc);
                for (int kb = 0; kb < nkb; ++kb, ++it2) {
                    const int st = it2 % Sm::kStages;
                    if (!mbar_wait(full(st), (it2 / Sm::kStages) & 1, lim)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t sa = sbase + st * Sm::kStage, sb = sa + kUA;
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
            ok = __all_sync(0xffffffffu, mbar_wait(d_full(buf), (it / 2) & 1, lim));
            if (!ok) break;
            fence_after_sync();
            epi(it, (uint32_t)(buf * Sm::kAcc));
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
    if (failed && threadIdx.x == 0) atomicExch(&g_wait_gave_up, 1);
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
    if ((threadIdx.x >> 5) == 1) tmem_alloc(slot, Sm::kTmemCols);
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
// row tiles, dealt evenly over the grid.  N1 activation rows (the batch padded
// to 16) per MMA; the planes of head k are [3][Bz][H] with Bz the padded batch
// (padding rows are never written and only ever feed accumulator columns that
// nothing reads).
template <typename Sm>
__global__ void __launch_bounds__(kUThreads, 2) heads_w1_umma_kernel(
    const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmh,
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ b1, int B, int K, int H, int N1, int Bz,
    uint16_t* __restrict__ zp, int* __restrict__ status) {
    using namespace umma;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint32_t tmem;
    umma_setup<Sm>(base, &tmem);
    pdl_wait();  // h may come from the previous kernel (the last round's compaction)
    pdl_trigger();
    const int tiles = K * H / kUM;
    const int i0 = (int)((long long)blockIdx.x * tiles / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * tiles / gridDim.x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
    auto coords = [&](int it, int& ay, int& by) { ay = (i0 + it) * kUM; by = 0; };
    auto epi = [&](int it, uint32_t col) {
        const int row = (i0 + it) * kUM + q * 32 + lane;  // W1 row k*H + i
        const int k = row / H, i = row - k * H;
        const float bias = bf16_to_f32(b1[(size_t)k * H + i]);
        uint16_t* zk = zp + (size_t)k * 3 * Bz * H;
#pragma unroll 1
        for (int b0 = 0; b0 < B; b0 += 8) {
            float d[8];
            tmem_ld8(tmem + ((uint32_t)(q * 32) << 16) + col + (uint32_t)b0, d);
            tmem_wait_ld();
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) {
                const int b = b0 + bb;
                if (b < B) {
                    const float u = d[bb] + bias;
                    const float z = bf16_to_f32(h[(size_t)b * H + i]) + u / (1.f + expf(-u));
                    const uint16_t hi = f32_to_bf16_rn(z);
                    const float r1 = z - bf16_to_f32(hi);
                    const uint16_t mid = f32_to_bf16_rn(r1);
                    const uint16_t lo = f32_to_bf16_rn(r1 - bf16_to_f32(mid));
                    zk[((size_t)0 * Bz + b) * H + i] = hi;
                    zk[((size_t)1 * Bz + b) * H + i] = mid;
                    zk[((size_t)2 * Bz + b) * H + i] = lo;
                }
            }
        }
    };
    const bool ok = umma_pipeline<Sm>(base, tmem, i1 - i0, H / kUK, N1, &tmw, &tmh, coords, epi);
    if (threadIdx.x == 0) status[blockIdx.x] = ok ? 0 : 1;  // this CTA's own slot: no race, no reset
    if (warp == 1) {
        fence_after_sync();
        tmem_dealloc(tmem, Sm::kTmemCols);
    }
}

struct W2Args {
    int B, K, H, V, T, topk;
    int items;          // K * T
    float* logits;      // [B][K][V] or nullptr
    float* run_val;     // [K][grid][B][topk]
    int* run_idx;
    const int* status1;  // [n1]: one slot per CTA of the W1 kernel, nonzero if it gave up
    int n1;
    int* status2;        // [grid of the W2 kernel]: the same for the W2 kernel
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

// The batch padded to BP.  Epilogue warp w owns sequences w, w + 4, ..:
// it keeps each one's sorted top-k over the items of the CTA's current head run
// as a list in shared memory.  Per item the warp tests the sequence's 128
// logits against the list's entry topk - 1 (four compares per lane and a
// ballot); a few that beat it are inserted one by one with lane shuffles, and
// when more do (always on a run's first item) the list is rebuilt from list and
// tile by passes that pop the best of the lanes' sorted registers.  At the end of a run the lists are published to
// run_val / run_idx; heads_merge_kernel then merges every head's run lists.
template <int BP>
__global__ void __launch_bounds__(kUThreads, 1) heads_w2_umma_kernel(
    const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmz, W2Args a) {
    using namespace umma;
    using Cfg = W2Cfg<BP>;
    using Sm = typename Cfg::Sm;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    float* lgt = reinterpret_cast<float*>(base + Sm::kOffExtra);               // [BP][129]
    float* lvs = reinterpret_cast<float*>(base + Sm::kOffExtra + Cfg::kLgt);  // [BP][16]
    int* lis = reinterpret_cast<int*>(lvs + BP * kUTopk);
    uint32_t tmem;
    umma_setup<Sm>(base, &tmem);
    pdl_wait();  // the z planes come from heads_w1_umma_kernel
    pdl_trigger();
    const int c = blockIdx.x, grid = gridDim.x;
    const int i0 = (int)((long long)c * a.items / grid), i1 = (int)((long long)(c + 1) * a.items / grid);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
    const int B = a.B, T = a.T, topk = a.topk;
    const int ew = warp - 2;  // epilogue warp 0..3
    auto coords = [&](int it, int& ay, int& by) {
        const int g = i0 + it, k = g / T, t = g - k * T;
        ay = k * a.V + t * kUM;
        by = k * 3 * BP;
    };
    auto clear_lists = [&]() {
        for (int sq = ew; sq < B; sq += 4)
            if (lane < kUTopk) { lvs[sq * kUTopk + lane] = -INFINITY; lis[sq * kUTopk + lane] = INT_MAX; }
        __syncwarp();
    };
    // head k's run is complete: publish every sequence's list, clear the lists
    auto finish_run = [&](int k) {
        for (int sq = ew; sq < B; sq += 4) {
            if (lane < topk) {
                const size_t o = (((size_t)k * grid + c) * B + sq) * topk + lane;
                a.run_val[o] = lvs[sq * kUTopk + lane];
                a.run_idx[o] = lis[sq * kUTopk + lane];
            }
        }
        __syncwarp();
        clear_lists();
    };
    if (warp >= 2) clear_lists();
    int run_k = -1;
    auto epi = [&](int it, uint32_t col) {
        const int g = i0 + it, k = g / T, t = g - k * T;
        if (k != run_k) {
            if (run_k >= 0) finish_run(run_k);
            run_k = k;
        }
        const int vl = q * 32 + lane, v = t * kUM + vl;
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + col;
        for (int b0 = 0; b0 < B; b0 += 16) {
            float dh[16], dm[16], dl[16];
            tmem_ld16(ta + (uint32_t)b0, dh);
            tmem_ld16(ta + (uint32_t)(BP + b0), dm);
            tmem_ld16(ta + (uint32_t)(2 * BP + b0), dl);
            tmem_wait_ld();
#pragma unroll
            for (int bb = 0; bb < 16; ++bb) {
                const int b = b0 + bb;
                if (b < B) {
                    const float x = v < a.V ? dh[bb] + dm[bb] + dl[bb] : -INFINITY;
                    lgt[b * kLgtStride + vl] = x;
                    if (a.logits && v < a.V) a.logits[((size_t)b * a.K + k) * a.V + v] = x;
                }
            }
        }
        named_barrier_or(1, kEpi, false);
        for (int sq = ew; sq < B; sq += 4) {
            const float* row = lgt + sq * kLgtStride;
            float* Lv = lvs + sq * kUTopk;
            int* Li = lis + sq * kUTopk;
            float ev = lane < kUTopk ? Lv[lane] : -INFINITY;
            int ei = lane < kUTopk ? Li[lane] : INT_MAX;
            float tv = __shfl_sync(0xffffffffu, ev, topk - 1);
            int ti = __shfl_sync(0xffffffffu, ei, topk - 1);
            float x[kUM / 32];
            unsigned m = 0;
#pragma unroll
            for (int u = 0; u < kUM / 32; ++u) {
                x[u] = row[lane + 32 * u];
                if (better(x[u], t * kUM + lane + 32 * u, tv, ti)) m |= 1u << u;
            }
            const int ncand = __reduce_add_sync(0xffffffffu, __popc(m));
            if (ncand == 0) continue;
            if (ncand > kRebuildAt) {
                // many candidates: rebuild the list from list and tile.  Each
                // lane sorts its four tile logits and its list entry; each pass
                // takes the best head across the warp into lane `tt` and the
                // lane that held it pops it.
                float cv[kUM / 32 + 1];
                int ci[kUM / 32 + 1];
#pragma unroll
                for (int u = 0; u < kUM / 32; ++u) { cv[u] = x[u]; ci[u] = t * kUM + lane + 32 * u; }
                cv[kUM / 32] = ev;
                ci[kUM / 32] = ei;
#pragma unroll
                for (int i = 1; i <= kUM / 32; ++i)
#pragma unroll
                    for (int j = i; j > 0; --j)
                        if (better(cv[j], ci[j], cv[j - 1], ci[j - 1])) {
                            const float tv0 = cv[j];
                            const int ti0 = ci[j];
                            cv[j] = cv[j - 1];
                            ci[j] = ci[j - 1];
                            cv[j - 1] = tv0;
                            ci[j - 1] = ti0;
                        }
                float nv = -INFINITY;
                int ni = INT_MAX;
                for (int tt = 0; tt < topk; ++tt) {
                    float bv = cv[0];
                    int bi = ci[0];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
                    }
                    if (lane == tt) { nv = bv; ni = bi; }
                    if (cv[0] == bv && ci[0] == bi) {
#pragma unroll
                        for (int e = 0; e < kUM / 32; ++e) { cv[e] = cv[e + 1]; ci[e] = ci[e + 1]; }
                        cv[kUM / 32] = -INFINITY;
                        ci[kUM / 32] = INT_MAX;
                    }
                }
                ev = nv;
                ei = ni;
            } else {
#pragma unroll
                for (int u = 0; u < kUM / 32; ++u) {
                    unsigned bal = __ballot_sync(0xffffffffu, (m >> u) & 1u);
                    while (bal) {
                        const int src = __ffs(bal) - 1;
                        bal &= bal - 1;
                        const float cv = __shfl_sync(0xffffffffu, x[u], src);
                        const int ci = t * kUM + src + 32 * u;
                        if (!better(cv, ci, tv, ti)) continue;  // the list moved on meanwhile
                        wl_insert(ev, ei, cv, ci, lane);
                        tv = __shfl_sync(0xffffffffu, ev, topk - 1);
                        ti = __shfl_sync(0xffffffffu, ei, topk - 1);
                    }
                }
            }
            __syncwarp();
            if (lane < kUTopk) { Lv[lane] = ev; Li[lane] = ei; }
            __syncwarp();
        }
        named_barrier_or(1, kEpi, false);
    };
    // a failure of the first kernel leaves the z planes undefined
    int bad1 = 0;
    for (int i = threadIdx.x; i < a.n1; i += blockDim.x) bad1 |= a.status1[i];
    const bool ok1 = __syncthreads_or(bad1) == 0;
    bool ok = ok1 && umma_pipeline<Sm>(base, tmem, i1 - i0, a.H / kUK, Cfg::kN, &tmw, &tmz, coords, epi);
    if (ok && warp >= 2 && run_k >= 0) finish_run(run_k);
    if (threadIdx.x == 0) a.status2[blockIdx.x] = ok ? 0 : 1;
    if (!ok) {
        const int k0 = i0 / T, k1 = (i1 - 1) / T;
        const int n = (k1 - k0 + 1) * B * topk;
        for (int j = threadIdx.x; j < n; j += blockDim.x) {
            const int ee = j % topk, b = (j / topk) % B, k = k0 + j / (topk * B);
            a.topk_idx[((size_t)b * a.K + k) * topk + ee] = -1;
        }
    }
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, Sm::kTmemCols);
    }
}

// One warp per (head, sequence) merges the run lists of the CTAs
// whose items met the head (grid2 = the W2 kernel's grid) into the sorted
// top-k.  If an earlier kernel of the call gave up a wait, every list is -1.
__global__ void __launch_bounds__(128) heads_merge_kernel(W2Args a, int grid2) {
    pdl_wait();  // the run lists come from heads_w2_umma_kernel
    pdl_trigger();
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= a.K * a.B) return;
    const int k = w / a.B, b = w - (w / a.B) * a.B, topk = a.topk;
    int32_t* oi = a.topk_idx + ((size_t)b * a.K + k) * topk;
    float* ov = a.topk_val ? a.topk_val + ((size_t)b * a.K + k) * topk : nullptr;
    int bad = 0;
    for (int i = lane; i < grid2; i += 32) bad |= a.status2[i];
    if (__any_sync(0xffffffffu, bad != 0)) {
        if (lane < topk) oi[lane] = -1;
        return;
    }
    int h0, h1;
    head_ctas(k, a.T, a.items, grid2, h0, h1);
    warp_merge_topk<kUTopk>(
        (h1 - h0) * topk, topk,
        [&](int j, float& x, int& xi) {
            const int cc = h0 + j / topk, e = j - (j / topk) * topk;
            const size_t o = (((size_t)k * grid2 + cc) * a.B + b) * topk + e;
            x = a.run_val[o];
            xi = a.run_idx[o];
        },
        [&](int t, float v, int i) {
            oi[t] = i;
            if (ov) ov[t] = v;
        },
        lane);
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

// the batch padded to a multiple of 16
static int pad16(int B) { return (B + 15) / 16 * 16; }

static int w2_smem(int Bp) {
    switch (Bp) {
        case 16: return W2Cfg<16>::Sm::kBytes;
        case 32: return W2Cfg<32>::Sm::kBytes;
        case 48: return W2Cfg<48>::Sm::kBytes;
        default: return W2Cfg<64>::Sm::kBytes;
    }
}

bool heads_umma_applies(int B, int K, int H, int V, int topk, bool bf16) {
    return bf16 && B >= kUMinB && B <= kUMaxB && H % kUM == 0 && topk <= kUTopk &&
           (long long)K * V < (1ll << 31) && w2_smem(pad16(B)) <= max_smem_optin() &&
           W1Smem::kBytes <= max_smem_optin();
}

size_t heads_umma_workspace(int B, int K, int H, int V, int topk) {
    const int grid = umma_grid();
    size_t off = align_up((size_t)K * 3 * pad16(B) * H * 2, 256);      // z planes
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);            // run values
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);            // run indices
    return align_up(off + (size_t)3 * grid * 4, 256);                      // per-CTA status slots
}

template <int BP>
cudaError_t launch_w2(const CUtensorMap& tw2, const CUtensorMap& tz, const W2Args& a, int grid, cudaStream_t st) {
    auto k2 = heads_w2_umma_kernel<BP>;
    constexpr int smem = W2Cfg<BP>::Sm::kBytes;
    cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return launch(k2, dim3(grid), dim3(kUThreads), (size_t)smem, st, tw2, tz, a);
}

int launch_heads_umma(const void* h, const void* w1, const void* b1, const void* w2, int B, int K, int H,
                      int V, int topk, int32_t* topk_idx, float* topk_val, float* logits, char* ws,
                      cudaStream_t st) {
    const int grid = umma_grid();
    const int T = (V + kUM - 1) / kUM;
    const int Bp = pad16(B);  // z plane rows per head, and the W1 MMA's N
    uint16_t* zp = reinterpret_cast<uint16_t*>(ws);
    size_t off = align_up((size_t)K * 3 * Bp * H * 2, 256);
    float* run_val = reinterpret_cast<float*>(ws + off);
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);
    int* run_idx = reinterpret_cast<int*>(ws + off);
    off = align_up(off + (size_t)K * grid * B * topk * 4, 256);
    int* status = reinterpret_cast<int*>(ws + off);  // W1 slots [0, g1), then W2 slots [g1, g1 + g2)
    CUtensorMap tw1, th, tw2, tz;
    int rc = bf16_rows_map(&tw1, w1, H, (long long)K * H, kUM);
    if (!rc) rc = bf16_rows_map(&th, h, H, B, Bp);
    if (!rc) rc = bf16_rows_map(&tw2, w2, H, (long long)K * V, kUM);
    if (!rc) rc = bf16_rows_map(&tz, zp, H, (long long)K * 3 * Bp, 3 * Bp);
    if (rc) return rc;
    const int tiles1 = K * H / kUM;
    auto k1 = heads_w1_umma_kernel<W1Smem>;
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, W1Smem::kBytes);
    const int g1 = min(2 * grid, tiles1);
    cudaError_t e = launch(k1, dim3(g1), dim3(kUThreads), (size_t)W1Smem::kBytes, st, tw1, th,
                           static_cast<const uint16_t*>(h), static_cast<const uint16_t*>(b1), B, K, H, Bp, Bp, zp,
                           status);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_w1_umma: launch failed: %s", cudaGetErrorString(e));
    W2Args a{};
    a.B = B; a.K = K; a.H = H; a.V = V; a.T = T; a.topk = topk;
    a.items = K * T;
    a.logits = logits;
    a.run_val = run_val;
    a.run_idx = run_idx;
    a.status1 = status;
    a.n1 = g1;
    a.status2 = status + g1;
    a.topk_idx = topk_idx;
    a.topk_val = topk_val;
    const int g2 = min(grid, a.items);
    e = Bp == 16 ? launch_w2<16>(tw2, tz, a, g2, st)
      : Bp == 32 ? launch_w2<32>(tw2, tz, a, g2, st)
      : Bp == 48 ? launch_w2<48>(tw2, tz, a, g2, st)
                 : launch_w2<64>(tw2, tz, a, g2, st);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_w2_umma: launch failed: %s", cudaGetErrorString(e));
    e = launch(heads_merge_kernel, dim3((K * B + 3) / 4), dim3(128), 0, st, a, g2);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "heads_merge: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

}  // namespace medusa
