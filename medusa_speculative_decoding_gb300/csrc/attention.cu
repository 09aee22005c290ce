// attention.cu -- tree attention ("Medusa Heads" glossary page, "Tree attention
// and acceptance": every candidate is appended to the input at once and the
// attention mask lets each candidate see only its ancestors, so all branches
// are scored in one pass against the KV cache).
//
// Query i of sequence b attends to the prefix keys [0, L_b) and to the tree
// keys L_b + m whose bit m is set in mask row i.  The KV cache dominates the
// bytes, so the bf16 kernel reads each KV tile once per (sequence, KV head,
// block of 128 tree queries) and scores all of the block's queries against it
// on the fifth-generation tensor cores (tcgen05, accumulators in TMEM):
//   tree_attn_umma_kernel : split-KV over a cluster of CTAs; per 128-key tile
//                           S = Q K^T and O += P V as tcgen05.mma (bf16 in,
//                           float32 out) fed by TMA; online softmax in float32;
//                           ancestor bits tested only on tiles that reach the
//                           tree slots; split partials merged in the cluster
//   tree_attn_f32_kernel  : float32 storage path (one warp per query row)
#include <float.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tmap.cuh"
#include "umma.cuh"

namespace medusa {
namespace {

MEDUSA_WAIT_CONTROL()

constexpr int kBlockN = 128;  // keys per tile
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 bytes read -> the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}


// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// (a0, a1) * b + c on the paired float32 pipe
__device__ __forceinline__ void fma_pair(float a0, float a1, float b, float c, float& d0, float& d1) {
    asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %4};\nmov.b64 rc, {%5, %5};\n"
        "fma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (s0, s1) += the two bf16 halves of w (low, high), exactly
__device__ __forceinline__ void add_bf16_pair(float& s0, float& s1, uint32_t w) {
    asm("{\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %2;\nadd.rn.f32.bf16 %0, lo, %0;\nadd.rn.f32.bf16 %1, hi, %1;\n}"
        : "+f"(s0), "+f"(s1) : "r"(w));
}

// Visibility of keys c0 .. c0 + 31 to one query row, as a bit mask (bit e: key
// c0 + e): the key lies in [klo, k_end) and, if it is a tree key (>= Lb), the
// row's ancestor mask holds its tree position; prefix keys are visible to every
// row.  The mask row's bits for the chunk are taken with one funnel shift.
__device__ __forceinline__ uint32_t key_visibility32(int c0, int klo, int k_end, int Lb, bool valid,
                                                     const uint64_t* mrow, int W) {
    uint32_t vm = 0xffffffffu;
    const int lo = klo - c0;  // bits below lo: keys before the range
    if (lo > 0) vm = lo >= 32 ? 0u : vm & (0xffffffffu << lo);
    const int hi = k_end - c0;  // bits from hi on: keys past its end
    if (hi < 32) vm = hi <= 0 ? 0u : vm & (0xffffffffu >> (32 - hi));
    const int off = c0 - Lb;  // tree position of bit 0 (negative: prefix keys come first)
    if (off > -32) {
        uint32_t tree = 0;
        if (valid) {
            const int p = max(off, 0);  // first tree position in the chunk
            const int wi = p >> 6, sh = p & 63;
            const uint64_t w0 = wi < W ? __ldg(mrow + wi) : 0ull;
            const uint64_t w1 = wi + 1 < W ? __ldg(mrow + wi + 1) : 0ull;
            const uint64_t bits = sh ? (w0 >> sh) | (w1 << (64 - sh)) : w0;  // bit j: position p + j
            tree = off >= 0 ? (uint32_t)bits : (uint32_t)(bits << (-off));
        }
        const uint32_t prefix = off >= 0 ? 0u : 0xffffffffu >> (32 + off);  // bits below -off
        vm &= prefix | tree;
    }
    return vm;
}

struct AttnArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* kv_len;
    const uint64_t* mask;
    float* out;
    int B, N, Hq, Hkv, G, Lmax, W, S, chunk, qblocks;
    int q_tma;   // Q tile loaded by TMA
    int spread;  // query blocks of <= 64 rows spread over the TMEM lane quarters
    float scale_log2;
};

__device__ __forceinline__ int clamp_len(int L, int N, int Lmax) {
    return L < 0 ? 0 : (L > Lmax - N ? Lmax - N : L);
}

// ---------------------------------------------------------------------------
// tcgen05 kernel.  One CTA per (KV split, KV head x block of 128 tree queries,
// sequence); the CTAs of one (head, query block) split the keys and form a
// thread-block cluster.  Query row r lives in TMEM lane r.
//
// A block of at most 64 query rows is spread 16 rows per TMEM lane quarter so
// that all four SM sub-partitions share the softmax.
//
// Warp roles (576 threads):
//   warps 0-15  softmax: thread (r, q), q = tid / 128, owns 32 of the 128
//               scores of TMEM lane r in every tile and D/4 of its output
//               columns; the four owners of a row exchange their maxima
//               through shared memory (one named barrier per tile)
//   warp 16     MMA: lane 0 issues every tcgen05.mma and commit
//   warp 17     TMA: lane 0 loads Q and streams K and V tiles into two 2-deep
//               rings
// Per 128-key tile j (keys [k_j, k_j + 128)):
//   S_j = Q K_j^T       tcgen05.mma into TMEM S buffer j & 1      (s_full)
//   softmax             row max, P_j = exp2(S_j*scale*log2e - m) as bf16
//                       written back over S buffer j & 1        (p_full)
//   O += P_j V_j        tcgen05.mma, A = P_j from TMEM, into the TMEM
//                       accumulator                             (o_done)
// The MMA lane issues PV_{j-1} and S_{j+1} while the softmax warps work on tile
// j.  Every ring stage has a full barrier (TMA bytes landed) and an empty
// barrier (the MMA that read it completed), so no wait can fall two phases
// behind.  The last tile of a split is shifted back to end at the split's last
// key, so no row past it is read; keys the shift brings back are masked.  The
// reference max moves only when a row max grows by more than 2^8 (log2
// domain); O and the row sums are rescaled in TMEM then.  Split partials (O,
// max, sum) are merged across the cluster: after a cluster barrier every CTA
// stores each row's partial into the shared memory of the CTA that owns the
// row (rows are dealt round-robin), and after a second barrier each CTA merges
// its rows from its own shared memory.
// Every wait is bounded; a CTA that gives up writes NaN.
// ---------------------------------------------------------------------------
constexpr int kUmmaM = 128;
constexpr int kSoftmaxWarps = 16;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = kSoftmaxWarps, kTmaWarp = kSoftmaxWarps + 1;
constexpr int kAttnThreads = kSoftmaxThreads + 64;
constexpr int kRing = 2;       // K and V ring depth
constexpr int kMaxSplits = 8;  // portable cluster size
constexpr float kRescaleThreshold = 8.f;
constexpr long long kWaitCycles = kDefaultWaitCycles;  // drain waits (~1 s at 2 GHz)

template <int D>
struct AttnSmem {
    static constexpr int kQ = kUmmaM * D * 2;
    static constexpr int kTile = kBlockN * D * 2;  // one K or V tile
    static constexpr int kOffK = kQ;
    static constexpr int kOffV = kOffK + kRing * kTile;
    static constexpr int kOffRed = kOffV + kRing * kTile;     // float [2][4][128]
    static constexpr int kOffBar = kOffRed + 2 * 4 * 128 * 4;
    // kfull[kRing] vfull[kRing] kempty[kRing] vempty[kRing] s_full[2] o_done[2]
    // p_full[2] qfull drain
    static constexpr int kNumBar = 4 * kRing + 8;
    static constexpr int kOffMisc = kOffBar + kNumBar * 8;    // tmem slot, flag
    // query blocks of <= 64 rows: a receive area of its own for the split
    // partials (O [slots][D], then (max, sum) [slots]), so partials can arrive
    // while this CTA still streams tiles
    static constexpr int kRecvSlots = 64 + kMaxSplits;
    static constexpr int kOffRecv = (kOffMisc + 16 + 15) / 16 * 16;
    static constexpr int kRecvBytes = kRecvSlots * (D + 2) * 4;
    static constexpr int kBytes = kOffRecv + kRecvBytes + 1024;  // + alignment slack
    // after the tile loop the K/V rings receive the partials of the rows this
    // CTA owns: float O [kMaxSplits][rows_per_owner][D], then (max, sum)
    static constexpr int kOffPartO = kOffK;
    static constexpr int kOffPartML = kOffK + (kUmmaM + kMaxSplits) * D * 4;
    static_assert((kUmmaM + kMaxSplits) * (D + 2) * 4 <= 2 * kRing * kTile, "partials fit the rings");
};

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) tree_attn_umma_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const __grid_constant__ CUtensorMap tmq, AttnArgs a) {
    using namespace umma;
    using L = AttnSmem<D>;
    constexpr int CH = D / 8;          // 16-byte chunks per row
    constexpr int TMEM_COLS = 512;     // O: D columns at 0; S buffers at 128 and 256
    constexpr uint32_t kSCol = 128;
    constexpr int SW = kBlockN / 4;    // scores per softmax thread (32)
    constexpr int QW = D / 4;          // output columns per softmax thread
    extern __shared__ uint8_t smem_raw[];

    const int split = blockIdx.x, S = gridDim.x;
    const int hk = blockIdx.y / a.qblocks, qb = blockIdx.y % a.qblocks;
    const int N = a.N, G = a.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = tid & (kUmmaM - 1), q = (tid >> 7) & 3;

    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t* base = smem_raw + pad;
    const uint32_t base_a = smem_addr(base);
    const uint32_t qs_a = base_a, ks_a = base_a + L::kOffK, vs_a = base_a + L::kOffV;
    float* red = reinterpret_cast<float*>(base + L::kOffRed);
    const uint32_t bar_a = base_a + L::kOffBar;
    const uint32_t kfull0 = bar_a, vfull0 = kfull0 + 8 * kRing, kempty0 = vfull0 + 8 * kRing,
                   vempty0 = kempty0 + 8 * kRing, s_full0 = vempty0 + 8 * kRing,
                   o_done0 = s_full0 + 16, p_full0 = o_done0 + 16, qfull = p_full0 + 16, drain = qfull + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);
    volatile int* flag = reinterpret_cast<volatile int*>(base + L::kOffMisc + 4);
    // limit of the first waits (input tiles, MMA results, free buffers); the
    // drain waits below keep kWaitCycles
    const long long lim = g_wait_limit;
    // loads the TMA lane has issued: Q, and the K and V tiles below these counts
    bool q_issued = false;
    int issued_k = 0, issued_v = 0;

    // Set-up that reads no input runs before the dependency wait, overlapping
    // the previous kernel: barriers, tensor-map prefetch, TMEM, and (batch 1)
    // an L2 warm-up of this split's K and V rows.
    if (warp == kTmaWarp && lane == 0) {
        for (int i = 0; i < L::kNumBar; ++i) mbar_init(bar_a + 8 * i, 1);
        mbar_init(p_full0, kSoftmaxWarps);
        mbar_init(p_full0 + 8, kSoftmaxWarps);
        mbar_init_fence();
        *flag = 0;
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        if (a.q_tma) prefetch_tmap(&tmq);
        if (a.B == 1) {
            // the rows come from the split's nominal range (no input is read
            // before the dependency wait); a prefetch is only a hint
            const size_t head = (size_t)hk * a.Lmax;
            for (int t = 0; t * kBlockN < a.chunk; ++t) {
                const int key0 = split * a.chunk + t * kBlockN;
                if (key0 >= a.Lmax) break;
                const uint32_t bytes = (uint32_t)min(kBlockN, a.Lmax - key0) * D * 2;
                prefetch_l2_bulk(a.k + (head + key0) * D, bytes);
                prefetch_l2_bulk(a.v + (head + key0) * D, bytes);
            }
        }
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    // Blocks of <= 64 query rows merge their split partials through a receive
    // area of their own: arrive on the cluster barrier now, wait before the
    // first remote store (which must not precede the peers' start).
    const bool early_merge = S > 1 && a.spread != 0;
    if (early_merge) cluster_arrive_relaxed();
    pdl_wait();
    pdl_trigger();
    // Sequences are taken longest first: blockIdx.z is a rank in the order of
    // decreasing KV length (ties by index), so the CTAs launched first carry
    // the most work and the short sequences fill the tail of the grid.
    __shared__ int s_seq;
    int b = blockIdx.z;
    if (a.B > 1 && a.B <= kAttnThreads) {
        const int t = threadIdx.x;
        if (t < a.B) {
            const int Lt = clamp_len(a.kv_len[t], N, a.Lmax);
            int rank = 0;
            for (int j = 0; j < a.B; ++j) {
                const int Lj = clamp_len(a.kv_len[j], N, a.Lmax);
                rank += (Lj > Lt || (Lj == Lt && j < t)) ? 1 : 0;
            }
            if (rank == (int)blockIdx.z) s_seq = t;
        }
        __syncthreads();
        b = s_seq;
    }
    const int Lb = clamp_len(a.kv_len[b], N, a.Lmax);
    const int total = Lb + N;
    const int k_begin = split * a.chunk;
    const int k_end = min(total, k_begin + a.chunk);
    const int ntiles = k_begin < total ? (k_end - k_begin + kBlockN - 1) / kBlockN : 0;
    const int rows = N * G;
    const int row0 = qb * kUmmaM;
    const int nblk = min(rows - row0, kUmmaM);  // query rows in this block
    // A block of at most 64 rows is spread over the four TMEM lane quarters (16
    // rows each) so all four SM sub-partitions share the softmax; otherwise
    // block row i is TMEM lane i.
    const bool spread = a.spread != 0;
    auto qrow_of = [&](int m) -> int {  // TMEM lane -> block row, -1 for padding
        const int i = spread ? (((m & 31) < 16) ? 16 * (m >> 5) + (m & 15) : -1) : m;
        return (i >= 0 && i < nblk) ? i : -1;
    };

    auto tile_lo = [&](int t) { return k_begin + t * kBlockN; };
    auto tile_start = [&](int t) { return min(k_begin + t * kBlockN, k_end - kBlockN); };
    const int zrow = b * a.Hkv + hk;

    if (warp == kTmaWarp && lane == 0) {
        // Q and the first K/V tiles, while the softmax warps set up
        if (a.q_tma && ntiles > 0) {  // Q rows (node, group member) x D
            q_issued = true;
            if (spread) {  // block rows 16g .. 16g+15 -> TMEM lanes 32g .. 32g+15
                mbar_expect_tx(qfull, 4 * 16 * D * 2);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        tma_load_4d(qs_a + x * kUmmaM * 128 + g * 32 * 128, &tmq, x * 64, hk * G,
                                    (row0 + 16 * g) / G, b, qfull);
            } else {
                mbar_expect_tx(qfull, L::kQ);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_4d(qs_a + x * kUmmaM * 128, &tmq, x * 64, hk * G, row0 / G, b, qfull);
            }
        }
        for (int t = 0; t < kRing && t < ntiles; ++t) {
            issued_k = issued_v = t + 1;
            mbar_expect_tx(kfull0 + 8 * t, L::kTile);
            mbar_expect_tx(vfull0 + 8 * t, L::kTile);
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
                tma_load_3d(ks_a + t * L::kTile + x * kBlockN * 128, &tmk, x * 64, tile_start(t), zrow, kfull0 + 8 * t);
                tma_load_3d(vs_a + t * L::kTile + x * kBlockN * 128, &tmv, x * 64, tile_start(t), zrow, vfull0 + 8 * t);
            }
        }
    }
    // Q tile without TMA (group size not dividing 128): row rr -> node rr / G,
    // query head hk * G + rr % G; padding rows are zero
    if (!a.q_tma && warp < kSoftmaxWarps) {
        for (int c = tid; c < kUmmaM * CH; c += kSoftmaxThreads) {
            const int m = c / CH, ch = c % CH;  // TMEM lane m = MMA row m
            const int i = qrow_of(m);
            const bool ok = i >= 0;
            const int gr = row0 + max(i, 0);
            const int node = gr / G, hq = hk * G + gr % G;
            cp_async16(qs_a + sw128_offset(m, ch, kUmmaM),
                       a.q + (((size_t)b * N + (ok ? node : 0)) * a.Hq + (ok ? hq : 0)) * D + ch * 8, ok);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_async_smem();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    float m_ref = -INFINITY, l = 0.f;
    bool bad = false;
    if (warp == kMmaWarp) {
        // -------------------------------- MMA lane --------------------------------
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kUmmaM, kBlockN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16(kUmmaM, D, 0, 1);
            // descriptors of the first k-step; later k-steps add byte offsets >> 4
            // to the start-address field
            const uint64_t dq0 = desc_sw128(qs_a, 16, 1024);
            const uint64_t dk0 = desc_sw128(ks_a, 16, 1024);
            const uint64_t dv0 = desc_sw128(vs_a, kBlockN * 128, 1024);
            bool fail = false;
            auto wait = [&](uint32_t bar, uint32_t parity) {
                if (fail) return false;
                if (!mbar_wait(bar, parity, lim)) { fail = true; *flag = 1; return false; }
                return true;
            };
            auto issue_s = [&](int t) {  // S_t = Q K_t^T into S buffer t & 1
                const uint64_t dk = dk0 + (uint64_t)(((t % kRing) * L::kTile) >> 4);
                const uint32_t d = tmem + kSCol + (t & 1) * kBlockN;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t qo = ((ks >> 2) * (kUmmaM * 128) + (ks & 3) * 32) >> 4;
                    const uint32_t ko = ((ks >> 2) * (kBlockN * 128) + (ks & 3) * 32) >> 4;
                    mma_bf16(d, dq0 + qo, dk + ko, idesc_s, ks > 0);
                }
                commit(s_full0 + 8 * (t & 1));
                commit(kempty0 + 8 * (t % kRing));
            };
            auto issue_pv = [&](int t) {  // O += P_t V_t, P_t in TMEM over S buffer t & 1
                const uint64_t dv = dv0 + (uint64_t)(((t % kRing) * L::kTile) >> 4);
                const uint32_t pa = tmem + kSCol + (t & 1) * kBlockN;
#pragma unroll
                for (int ks = 0; ks < kBlockN / 16; ++ks)
                    mma_bf16_ta(tmem, pa + ks * 8, dv + ((ks * 2048) >> 4), idesc_pv,
                                (t > 0 || ks > 0) ? 1u : 0u);
                commit(o_done0 + 8 * (t & 1));
                commit(vempty0 + 8 * (t % kRing));
            };
            if ((!a.q_tma || wait(qfull, 0)) && wait(kfull0, 0)) issue_s(0);
            for (int i = 0; i <= ntiles && !fail; ++i) {
                if (i >= 1) {  // PV of tile i-1 once its P is written and its V has landed
                    const int t = i - 1;
                    if (!wait(p_full0 + 8 * (t & 1), (t >> 1) & 1)) break;
                    if (!wait(vfull0 + 8 * (t % kRing), (t / kRing) & 1)) break;
                    fence_after_sync();
                    issue_pv(t);
                }
                if (i + 1 < ntiles) {  // S of tile i+1 (its S buffer was read by softmax i-1)
                    const int t = i + 1;
                    if (!wait(kfull0 + 8 * (t % kRing), (t / kRing) & 1)) break;
                    issue_s(t);
                }
            }
        }
    } else if (warp == kTmaWarp) {
        // -------------------------------- TMA lane --------------------------------
        // (a CTA that gives up lets the loads issued here land after the
        // block-wide barrier below, before it frees TMEM and leaves)
        if (lane == 0) {
            for (int t = kRing; t < ntiles; ++t) {
                // stage t % kRing held tile t - kRing: wait for the MMAs that read it
                const uint32_t par = (uint32_t)((t / kRing - 1) & 1);
                if (!mbar_wait(kempty0 + 8 * (t % kRing), par, lim)) { *flag = 1; break; }
                mbar_expect_tx(kfull0 + 8 * (t % kRing), L::kTile);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(ks_a + (t % kRing) * L::kTile + x * kBlockN * 128, &tmk, x * 64, tile_start(t),
                                zrow, kfull0 + 8 * (t % kRing));
                issued_k = t + 1;
                if (!mbar_wait(vempty0 + 8 * (t % kRing), par, lim)) { *flag = 1; break; }
                mbar_expect_tx(vfull0 + 8 * (t % kRing), L::kTile);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(vs_a + (t % kRing) * L::kTile + x * kBlockN * 128, &tmv, x * 64, tile_start(t),
                                zrow, vfull0 + 8 * (t % kRing));
                issued_v = t + 1;
            }
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        const int qi = qrow_of(r);            // query-block row of TMEM lane r, or -1
        const bool valid = qi >= 0;
        const int grow = row0 + max(qi, 0);
        const bool warp_valid = __any_sync(0xffffffffu, valid);
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int node = valid ? grow / G : 0;
        const uint64_t* mrow = a.mask + (size_t)node * a.W;
        bool fail = false;
        for (int j = 0; j < ntiles; ++j) {
            bool ok = !fail && mbar_wait(s_full0 + 8 * (j & 1), (uint32_t)((j >> 1) & 1), lim);
            ok = __all_sync(0xffffffffu, ok);
            fence_after_sync();
            float sv[SW];
            float mt = -INFINITY;
            const int kt = tile_start(j), klo = tile_lo(j);
            if (warp_valid && ok) {
                tmem_ld32(tmem + lane_off + kSCol + (j & 1) * kBlockN + q * SW, sv);
                tmem_wait_ld();
                const int c0 = kt + q * SW;  // key of sv[0]
                if (kt == klo && kt + kBlockN <= min(k_end, Lb)) {  // plain prefix tile
                    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                    for (int i = 0; i < SW; i += 4) {
                        m0 = fmax3(m0, sv[i], sv[i + 1]);
                        m1 = fmax3(m1, sv[i + 2], sv[i + 3]);
                    }
                    mt = fmaxf(m0, m1);
                } else {
                    const uint32_t vm = key_visibility32(c0, klo, k_end, Lb, valid, mrow, a.W);
#pragma unroll
                    for (int i = 0; i < SW; i += 2) {
                        sv[i] = (vm >> i) & 1u ? sv[i] : -INFINITY;
                        sv[i + 1] = (vm >> (i + 1)) & 1u ? sv[i + 1] : -INFINITY;
                        mt = fmax3(mt, sv[i], sv[i + 1]);
                    }
                }
                // raw scores are scaled inside the exponent's FMA below; the
                // scale is positive, so the row maximum scales the same way
                mt *= a.scale_log2;
            }
            float* rj = red + (j & 1) * 4 * 128;
            rj[q * 128 + r] = mt;
            if (named_barrier_or(1, kSoftmaxThreads, !ok)) { fail = true; break; }
            mt = fmaxf(fmaxf(rj[r], rj[128 + r]), fmaxf(rj[256 + r], rj[384 + r]));
            float corr = 1.f;
            bool rescale = false;
            if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescaleThreshold)) {
                if (m_ref != -INFINITY && j > 0) { corr = exp2f(m_ref - mt); rescale = true; }
                m_ref = mt;
            }
            l *= corr;
            if (warp_valid && __any_sync(0xffffffffu, rescale)) {
                // O must hold PV_{j-1} before it is rescaled (warp-collective TMEM access)
                ok = mbar_wait(o_done0 + 8 * ((j - 1) & 1), (uint32_t)(((j - 1) >> 1) & 1), lim);
                ok = __all_sync(0xffffffffu, ok);
                fence_after_sync();
                if (ok) {
                    const uint32_t ta = tmem + lane_off + q * QW;
                    if constexpr (QW == 32) {
                        float ov[32];
                        tmem_ld32(ta, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= corr;
                        tmem_st32(ta, ov);
                    } else {
                        float ov[16];
                        tmem_ld16(ta, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) ov[i] *= corr;
                        tmem_st16(ta, ov);
                    }
                    tmem_wait_st();
                } else {
                    fail = true;
                }
            }
            if (warp_valid) {
                // P_j (bf16, two per column) over the first 32 columns of S buffer
                // j & 1: every owner has read its scores before the barrier above
                const float mr = m_ref == -INFINITY ? 0.f : m_ref;
                uint32_t pk[SW / 2];
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int e = 0; e < SW / 2; ++e) {
                    float t0, t1;
                    fma_pair(sv[2 * e], sv[2 * e + 1], a.scale_log2, -mr, t0, t1);
                    pk[e] = pack_bf16(exp2_approx(t0), exp2_approx(t1));
                    // the row sum adds the bf16 values PV multiplies, so the
                    // output is an exactly normalised average of the values
                    add_bf16_pair(s0, s1, pk[e]);
                }
                const float psum = s0 + s1;
                tmem_st16u(tmem + lane_off + kSCol + (j & 1) * kBlockN + q * (SW / 2), pk);
                tmem_wait_st();
                l += psum;
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full0 + 8 * (j & 1));
        }
        bool ok = !fail;
        if (ok && ntiles > 0)
            ok = mbar_wait(o_done0 + 8 * ((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1), lim);
        float* rl = red + (ntiles & 1) * 4 * 128;
        rl[q * 128 + r] = l;
        bad = named_barrier_or(1, kSoftmaxThreads, !ok);
        l = rl[r] + rl[128 + r] + rl[256 + r] + rl[384 + r];
        fence_after_sync();
    }
    bad = __syncthreads_or(bad);
    bad = bad || *flag != 0;  // every write to the flag precedes the barrier
    if (bad) {
        // Gave up: let everything this CTA started complete before its tensor
        // memory is freed and it leaves (default-limit waits).  The MMA lane
        // commits once more, which tracks every MMA it issued; the TMA lane
        // waits for Q and for the last kRing K and V tiles it requested (older
        // tiles completed before their stage was requested again).
        if (warp == kMmaWarp && lane == 0) {
            commit(drain);
            mbar_wait(drain, 0, kWaitCycles);
        }
        if (warp == kTmaWarp && lane == 0) {
            if (q_issued) mbar_wait(qfull, 0, kWaitCycles);
            for (int t = max(0, issued_k - kRing); t < issued_k; ++t)
                mbar_wait(kfull0 + 8 * (t % kRing), (uint32_t)((t / kRing) & 1), kWaitCycles);
            for (int t = max(0, issued_v - kRing); t < issued_v; ++t)
                mbar_wait(vfull0 + 8 * (t % kRing), (uint32_t)((t / kRing) & 1), kWaitCycles);
        }
        if (tid == 0) atomicExch(&g_wait_gave_up, 1);
    }

    // ------------------------------ epilogue ------------------------------
    float ov[QW];
#pragma unroll
    for (int i = 0; i < QW; ++i) ov[i] = 0.f;
    const int qi = qrow_of(r);
    const int grow = row0 + max(qi, 0);
    const bool valid = warp < kSoftmaxWarps && qi >= 0;
    if (warp < kSoftmaxWarps && __any_sync(0xffffffffu, valid) && ntiles > 0) {
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        if constexpr (QW == 32) tmem_ld32(tmem + lane_off + q * QW, ov);
        else tmem_ld16(tmem + lane_off + q * QW, ov);
        tmem_wait_ld();
    }
    if (S == 1 && valid) {
        const int node = grow / G, hq = hk * G + grow % G;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* dst = a.out + (((size_t)b * N + node) * a.Hq + hq) * D + q * QW;
#pragma unroll
        for (int i = 0; i < QW; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                bad ? make_float4(NAN, NAN, NAN, NAN)
                    : make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
    if (S == 1) return;

    // ------------------ merge the cluster's split partials ------------------
    // row r belongs to CTA r % S and is its (r / S)-th row; split s of it goes to
    // slot [s][r / S] of the owner's receive area.  Blocks of <= 64 rows have a
    // receive area of their own (the cluster barrier was arrived at before the
    // tile loop, so its wait here only checks that every peer has started);
    // larger blocks receive in the owner's rings, free once every CTA of the
    // cluster has left its tile loop.
    const int own_rows = early_merge ? (64 + S - 1) / S : (kUmmaM + S - 1) / S;
    float* part_o = reinterpret_cast<float*>(base + (early_merge ? L::kOffRecv : L::kOffPartO));
    float* part_ml = early_merge ? part_o + (size_t)L::kRecvSlots * D : reinterpret_cast<float*>(base + L::kOffPartML);
    if (early_merge) cluster_wait();
    else cluster_sync();
    if (valid) {
        const int owner = qi % S, slot = split * own_rows + qi / S;
        const uint32_t po = cluster_map(smem_addr(part_o + (size_t)slot * D + q * QW), owner);
#pragma unroll
        for (int i = 0; i < QW; i += 4)
            st_cluster_f32x4(po + i * 4, make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]));
        if (q == 0)
            st_cluster_f32x2(cluster_map(smem_addr(part_ml + 2 * slot), owner), bad ? NAN : (ntiles > 0 ? m_ref : -INFINITY),
                             bad ? NAN : (ntiles > 0 ? l : 0.f));
    }
    cluster_sync();  // all partials delivered
    const int me = (int)cluster_rank();
    const int nvalid = min(rows - row0, kUmmaM);
    const int nmine = nvalid > me ? (nvalid - me + S - 1) / S : 0;
    constexpr int C4 = D / 4;
    for (int idx = tid; idx < nmine * C4; idx += kAttnThreads) {
        const int lr = idx / C4, c4 = idx % C4;
        float mx = -INFINITY;
        bool nan_seen = false;
        for (int sp = 0; sp < S; ++sp) {
            const float ls = part_ml[2 * (sp * own_rows + lr) + 1];
            if (ls != ls) nan_seen = true;
            else if (ls > 0.f) mx = fmaxf(mx, part_ml[2 * (sp * own_rows + lr)]);
        }
        const float basem = mx == -INFINITY ? 0.f : mx;
        float lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < S; ++sp) {
            const int slot = sp * own_rows + lr;
            const float ls = part_ml[2 * slot + 1];
            if (!(ls > 0.f)) continue;
            const float w = exp2f(part_ml[2 * slot] - basem);
            lsum += ls * w;
            const float4 o = *reinterpret_cast<const float4*>(part_o + (size_t)slot * D + c4 * 4);
            acc.x += o.x * w; acc.y += o.y * w; acc.z += o.z * w; acc.w += o.w * w;
        }
        const float inv = nan_seen ? NAN : (lsum > 0.f ? 1.f / lsum : 0.f);
        const int gr = row0 + lr * S + me;
        const int node = gr / G, hq = hk * G + gr % G;
        *reinterpret_cast<float4*>(a.out + (((size_t)b * N + node) * a.Hq + hq) * D + c4 * 4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// ---------------------------------------------------------------------------
// Two-stream tcgen05 kernel, for query blocks whose keys are not split across
// CTAs (a block of at most 64 query rows is spread 16 rows per TMEM lane
// quarter, as in the cluster kernel).  The block's key tiles are cut in two
// halves, each an independent online softmax (a "stream") with its own TMEM
// accumulator O_s and score buffer S_s; the two partial results are merged at
// the end.  The
// tensor core alternates between the streams, so one stream's softmax runs
// while the other's MMAs do, and each softmax thread owns a whole query row:
// no row statistic crosses threads inside the tile loop.
//
// Warp roles (320 threads):
//   warps 0-3, 4-7  softmax of stream 0, 1: thread r of the warpgroup owns TMEM
//                   lane r (block row r), all 128 scores of each of its
//                   stream's tiles, and half of the row's output columns
//   warp 8          MMA: lane 0 issues every tcgen05.mma and commit
//   warp 9          TMA: lane 0 loads Q and streams K and V tiles into two
//                   3-deep rings in the order the MMAs consume them
// Tiles are consumed in the order u = 0, 1, 2, ...; u = 2i + s is stream s's
// tile i (key tile i for s = 0, key tile nA + i for s = 1, nA = ceil(tiles/2)).
// TMEM (512 columns): O_0 at 0, O_1 at 128, S_0 at 256, S_1 at 384; P_s is
// written as bf16 over the first 64 columns of S_s.  For u = 0, 1, 2, ... the
// MMA lane issues PV(u) and then S(u + 2), so the commit of S_s(i) also covers
// PV_s(i - 1): a stream's softmax may rescale O_s once its scores are in.
// Every wait is bounded; a CTA that gives up writes NaN.
// ---------------------------------------------------------------------------
constexpr int kDualThreads = 320;
constexpr int kDualSoftmaxWarps = 8;
constexpr int kDualMmaWarp = 8, kDualTmaWarp = 9;
constexpr int kDualRing = 3;

template <int D>
struct DualSmem {
    static constexpr int kQ = kUmmaM * D * 2;
    static constexpr int kTile = kBlockN * D * 2;  // one K or V tile
    static constexpr int kOffK = kQ;
    static constexpr int kOffV = kOffK + kDualRing * kTile;
    static constexpr int kOffBar = kOffV + kDualRing * kTile;
    // kfull[R] vfull[R] kempty[R] vempty[R] s_full[2] o_done[2] p_full[2] qfull drain
    static constexpr int kNumBar = 4 * kDualRing + 8;
    static constexpr int kOffMisc = kOffBar + kNumBar * 8;  // tmem slot, flag
    static constexpr int kBytes = kOffMisc + 16 + 1024;     // + alignment slack
    // after the tile loop the K ring holds the streams' row statistics,
    // float (max, sum) [2][128]
    static_assert(2 * kUmmaM * 2 * 4 <= kDualRing * kTile, "row statistics fit the K ring");
};

template <int D>
__global__ void __launch_bounds__(kDualThreads, 1) tree_attn_dual_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
    const __grid_constant__ CUtensorMap tmq, AttnArgs a) {
    using namespace umma;
    using L = DualSmem<D>;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    constexpr int TMEM_COLS = 512;
    constexpr uint32_t kOCol = 128, kSCol = 256;  // O_s at 128 s, S_s at 256 + 128 s
    constexpr int R = kDualRing;
    extern __shared__ uint8_t smem_raw[];

    const int hk = blockIdx.y / a.qblocks, qb = blockIdx.y % a.qblocks;
    const int N = a.N, G = a.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = tid & (kUmmaM - 1);
    const int strm = (warp >> 2) & 1;  // stream of a softmax warp

    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t* base = smem_raw + pad;
    const uint32_t base_a = smem_addr(base);
    const uint32_t qs_a = base_a, ks_a = base_a + L::kOffK, vs_a = base_a + L::kOffV;
    const uint32_t bar_a = base_a + L::kOffBar;
    const uint32_t kfull0 = bar_a, vfull0 = kfull0 + 8 * R, kempty0 = vfull0 + 8 * R, vempty0 = kempty0 + 8 * R,
                   s_full0 = vempty0 + 8 * R, o_done0 = s_full0 + 16, p_full0 = o_done0 + 16,
                   qfull = p_full0 + 16, drain = qfull + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);
    volatile int* flag = reinterpret_cast<volatile int*>(base + L::kOffMisc + 4);
    const long long lim = g_wait_limit;
    bool q_issued = false;
    int issued_k = 0, issued_v = 0;

    if (warp == kDualTmaWarp && lane == 0) {
        for (int i = 0; i < L::kNumBar; ++i) mbar_init(bar_a + 8 * i, 1);
        mbar_init(p_full0, 4);
        mbar_init(p_full0 + 8, 4);
        mbar_init_fence();
        *flag = 0;
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        if (a.q_tma) prefetch_tmap(&tmq);
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    pdl_wait();
    pdl_trigger();
    // sequences longest first (blockIdx.z is a rank by decreasing KV length)
    __shared__ int s_seq;
    int b = blockIdx.z;
    if (a.B > 1 && a.B <= kDualThreads) {
        const int t = threadIdx.x;
        if (t < a.B) {
            const int Lt = clamp_len(a.kv_len[t], N, a.Lmax);
            int rank = 0;
            for (int j = 0; j < a.B; ++j) {
                const int Lj = clamp_len(a.kv_len[j], N, a.Lmax);
                rank += (Lj > Lt || (Lj == Lt && j < t)) ? 1 : 0;
            }
            if (rank == (int)blockIdx.z) s_seq = t;
        }
        __syncthreads();
        b = s_seq;
    }
    const int Lb = clamp_len(a.kv_len[b], N, a.Lmax);
    const int k_end = Lb + N;  // every key of the sequence: prefix, then the tree
    const int ntiles = (k_end + kBlockN - 1) / kBlockN;
    const int nA = (ntiles + 1) / 2, nB = ntiles / 2;
    const int rows = N * G;
    const int row0 = qb * kUmmaM;
    const int nblk = min(rows - row0, kUmmaM);
    // A block of at most 64 rows is spread 16 rows per TMEM lane quarter, so
    // all four SM sub-partitions share the softmax; otherwise block row i is
    // TMEM lane i.
    const bool spread = a.spread != 0;
    auto qrow_of = [&](int m) -> int {  // TMEM lane -> block row, -1 for padding
        const int i = spread ? (((m & 31) < 16) ? 16 * (m >> 5) + (m & 15) : -1) : m;
        return (i >= 0 && i < nblk) ? i : -1;
    };
    // the last tile ends at the last key (keys it brings back are masked)
    auto tile_lo = [&](int t) { return t * kBlockN; };
    auto tile_start = [&](int t) { return min(t * kBlockN, k_end - kBlockN); };
    auto key_tile = [&](int u) { return (u & 1) ? nA + (u >> 1) : (u >> 1); };
    const int zrow = b * a.Hkv + hk;

    if (warp == kDualTmaWarp && lane == 0) {
        if (a.q_tma && ntiles > 0) {
            q_issued = true;
            if (spread) {  // block rows 16g .. 16g+15 -> TMEM lanes 32g .. 32g+15
                mbar_expect_tx(qfull, 4 * 16 * D * 2);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        tma_load_4d(qs_a + x * kUmmaM * 128 + g * 32 * 128, &tmq, x * 64, hk * G,
                                    (row0 + 16 * g) / G, b, qfull);
            } else {
                mbar_expect_tx(qfull, L::kQ);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_4d(qs_a + x * kUmmaM * 128, &tmq, x * 64, hk * G, row0 / G, b, qfull);
            }
        }
        for (int u = 0; u < R && u < ntiles; ++u) {
            issued_k = issued_v = u + 1;
            mbar_expect_tx(kfull0 + 8 * u, L::kTile);
            mbar_expect_tx(vfull0 + 8 * u, L::kTile);
            const int ks = tile_start(key_tile(u));
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
                tma_load_3d(ks_a + u * L::kTile + x * kBlockN * 128, &tmk, x * 64, ks, zrow, kfull0 + 8 * u);
                tma_load_3d(vs_a + u * L::kTile + x * kBlockN * 128, &tmv, x * 64, ks, zrow, vfull0 + 8 * u);
            }
        }
    }
    // Q tile without TMA (group size not dividing 128); padding rows are zero
    if (!a.q_tma && warp < kDualSoftmaxWarps) {
        for (int c = tid; c < kUmmaM * CH; c += kDualSoftmaxWarps * 32) {
            const int m = c / CH, ch = c % CH;  // TMEM lane m = MMA row m
            const int i = qrow_of(m);
            const bool ok = i >= 0;
            const int gr = row0 + max(i, 0);
            const int node = gr / G, hq = hk * G + gr % G;
            cp_async16(qs_a + sw128_offset(m, ch, kUmmaM),
                       a.q + (((size_t)b * N + (ok ? node : 0)) * a.Hq + (ok ? hq : 0)) * D + ch * 8, ok);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_async_smem();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    float m_ref = -INFINITY, l = 0.f;
    bool gave_up = false;
    if (warp == kDualMmaWarp) {
        // -------------------------------- MMA lane --------------------------------
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kUmmaM, kBlockN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16(kUmmaM, D, 0, 1);
            const uint64_t dq0 = desc_sw128(qs_a, 16, 1024);
            const uint64_t dk0 = desc_sw128(ks_a, 16, 1024);
            const uint64_t dv0 = desc_sw128(vs_a, kBlockN * 128, 1024);
            bool fail = false;
            auto wait = [&](uint32_t bar, uint32_t parity) {
                if (fail) return false;
                if (!mbar_wait(bar, parity, lim)) { fail = true; *flag = 1; return false; }
                return true;
            };
            auto issue_s = [&](int u) {  // S_s(i) = Q K_u^T into S buffer s = u & 1
                const uint64_t dk = dk0 + (uint64_t)(((u % R) * L::kTile) >> 4);
                const uint32_t d = tmem + kSCol + (u & 1) * 128;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t qo = ((ks >> 2) * (kUmmaM * 128) + (ks & 3) * 32) >> 4;
                    const uint32_t ko = ((ks >> 2) * (kBlockN * 128) + (ks & 3) * 32) >> 4;
                    mma_bf16(d, dq0 + qo, dk + ko, idesc_s, ks > 0);
                }
                commit(s_full0 + 8 * (u & 1));
                commit(kempty0 + 8 * (u % R));
            };
            auto issue_pv = [&](int u) {  // O_s += P_s(i) V_u
                const int s = u & 1, i = u >> 1;
                const uint64_t dv = dv0 + (uint64_t)(((u % R) * L::kTile) >> 4);
                const uint32_t pa = tmem + kSCol + s * 128;
#pragma unroll
                for (int ks = 0; ks < kBlockN / 16; ++ks)
                    mma_bf16_ta(tmem + s * kOCol, pa + ks * 8, dv + ((ks * 2048) >> 4), idesc_pv,
                                (i > 0 || ks > 0) ? 1u : 0u);
                if (u + 2 >= ntiles) commit(o_done0 + 8 * s);  // the stream's last PV
                commit(vempty0 + 8 * (u % R));
            };
            if (!a.q_tma || wait(qfull, 0))
                for (int u = 0; u < 2 && u < ntiles; ++u) {
                    if (!wait(kfull0 + 8 * (u % R), (uint32_t)((u / R) & 1))) break;
                    issue_s(u);
                }
            for (int u = 0; u < ntiles && !fail; ++u) {
                if (!wait(p_full0 + 8 * (u & 1), (uint32_t)((u >> 1) & 1))) break;
                if (!wait(vfull0 + 8 * (u % R), (uint32_t)((u / R) & 1))) break;
                fence_after_sync();
                issue_pv(u);
                if (u + 2 < ntiles) {
                    if (!wait(kfull0 + 8 * ((u + 2) % R), (uint32_t)(((u + 2) / R) & 1))) break;
                    issue_s(u + 2);
                }
            }
        }
    } else if (warp == kDualTmaWarp) {
        // -------------------------------- TMA lane --------------------------------
        if (lane == 0) {
            for (int u = R; u < ntiles; ++u) {
                // stage u % R held tile u - R: wait for the MMAs that read it
                const uint32_t par = (uint32_t)((u / R - 1) & 1);
                const int ks = tile_start(key_tile(u));
                if (!mbar_wait(kempty0 + 8 * (u % R), par, lim)) { *flag = 1; break; }
                mbar_expect_tx(kfull0 + 8 * (u % R), L::kTile);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(ks_a + (u % R) * L::kTile + x * kBlockN * 128, &tmk, x * 64, ks, zrow,
                                kfull0 + 8 * (u % R));
                issued_k = u + 1;
                if (!mbar_wait(vempty0 + 8 * (u % R), par, lim)) { *flag = 1; break; }
                mbar_expect_tx(vfull0 + 8 * (u % R), L::kTile);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_3d(vs_a + (u % R) * L::kTile + x * kBlockN * 128, &tmv, x * 64, ks, zrow,
                                vfull0 + 8 * (u % R));
                issued_v = u + 1;
            }
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        const int s = strm;
        const int ns = s ? nB : nA;
        const int qi = qrow_of(r);
        const bool valid = qi >= 0;
        const bool warp_valid = __any_sync(0xffffffffu, valid);
        const int grow = row0 + max(qi, 0);
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + kSCol + s * 128, tO = tmem + lane_off + s * kOCol;
        const uint64_t* mrow = a.mask + (size_t)(grow / G) * a.W;
        bool fail = false;
        for (int i = 0; i < ns; ++i) {
            bool ok = mbar_wait(s_full0 + 8 * s, (uint32_t)(i & 1), lim);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { fail = true; break; }
            fence_after_sync();
            if (warp_valid) {
                const int t = s ? nA + i : i;
                const int kt = tile_start(t), klo = tile_lo(t);
                float sv[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sv[c]);
                tmem_wait_ld();
                float mt;
                if (kt == klo && kt + kBlockN <= min(k_end, Lb)) {  // plain prefix tile
                    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            m0 = fmax3(m0, sv[c][e], sv[c][e + 1]);
                            m1 = fmax3(m1, sv[c][e + 2], sv[c][e + 3]);
                        }
                    mt = fmaxf(m0, m1);
                } else {
                    mt = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t vm = key_visibility32(kt + 32 * c, klo, k_end, Lb, valid, mrow, a.W);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            sv[c][e] = (vm >> e) & 1u ? sv[c][e] : -INFINITY;
                            sv[c][e + 1] = (vm >> (e + 1)) & 1u ? sv[c][e + 1] : -INFINITY;
                            mt = fmax3(mt, sv[c][e], sv[c][e + 1]);
                        }
                    }
                }
                // raw scores are scaled inside the exponent's FMA below; the
                // scale is positive, so the row maximum scales the same way
                mt *= a.scale_log2;
                float corr = 1.f;
                bool rescale = false;
                if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescaleThreshold)) {
                    if (m_ref != -INFINITY) { corr = exp2f(m_ref - mt); rescale = true; }
                    m_ref = mt;
                }
                const float mr = m_ref == -INFINITY ? 0.f : m_ref;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float t0, t1;
                        fma_pair(sv[c][2 * e], sv[c][2 * e + 1], a.scale_log2, -mr, t0, t1);
                        pk[e] = pack_bf16(exp2_approx(t0), exp2_approx(t1));
                        // the row sum adds the bf16 values PV multiplies
                        add_bf16_pair(s0, s1, pk[e]);
                    }
                    tmem_st16u(tS + 16 * c, pk);
                }
                l = l * corr + (s0 + s1);
                if (__any_sync(0xffffffffu, rescale)) {
                    // O_s holds PV_s(i - 1): its commit preceded this tile's scores
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float ov[32];
                        tmem_ld32(tO + 32 * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] *= corr;
                        tmem_st32(tO + 32 * c, ov);
                    }
                }
                tmem_wait_st();
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full0 + 8 * s);
        }
        bool ok = !fail;
        if (ok && ns > 0) ok = mbar_wait(o_done0 + 8 * s, 0, lim);
        gave_up = !ok;
    }
    bool bad = __syncthreads_or(gave_up);
    bad = bad || *flag != 0;  // every write to the flag precedes the barrier
    if (bad) {
        // Gave up: let everything this CTA started complete before its tensor
        // memory is freed and it leaves (default-limit waits).
        if (warp == kDualMmaWarp && lane == 0) {
            commit(drain);
            mbar_wait(drain, 0, kWaitCycles);
        }
        if (warp == kDualTmaWarp && lane == 0) {
            if (q_issued) mbar_wait(qfull, 0, kWaitCycles);
            for (int u = max(0, issued_k - R); u < issued_k; ++u)
                mbar_wait(kfull0 + 8 * (u % R), (uint32_t)((u / R) & 1), kWaitCycles);
            for (int u = max(0, issued_v - R); u < issued_v; ++u)
                mbar_wait(vfull0 + 8 * (u % R), (uint32_t)((u / R) & 1), kWaitCycles);
        }
        if (tid == 0) atomicExch(&g_wait_gave_up, 1);
    }

    // ------------------------------ epilogue ------------------------------
    // The streams swap (max, sum) through the K ring, free now: every MMA
    // completed (both streams' last commits were waited for) and every tile
    // that landed was consumed.
    float* xch = reinterpret_cast<float*>(base + L::kOffK);
    if (warp < kDualSoftmaxWarps && !bad) {
        xch[2 * (strm * kUmmaM + r)] = m_ref;
        xch[2 * (strm * kUmmaM + r) + 1] = l;
    }
    __syncthreads();
    if (warp < kDualSoftmaxWarps && ntiles > 0) {
        const int qi = qrow_of(r);
        const bool valid = qi >= 0;
        const int grow = row0 + max(qi, 0);
        const int node = grow / G, hq = hk * G + grow % G;
        float* dst = a.out + (((size_t)b * N + node) * a.Hq + hq) * D + strm * (D / 2);
        if (bad) {
            if (valid)
                for (int e = 0; e < D / 2; e += 4)
                    *reinterpret_cast<float4*>(dst + e) = make_float4(NAN, NAN, NAN, NAN);
        } else if (__any_sync(0xffffffffu, valid)) {
            const float mA = xch[2 * r], lA = xch[2 * r + 1];
            const float mB = xch[2 * (kUmmaM + r)], lB = xch[2 * (kUmmaM + r) + 1];
            const float mx = fmaxf(lA > 0.f ? mA : -INFINITY, lB > 0.f ? mB : -INFINITY);
            const float mb = mx == -INFINITY ? 0.f : mx;
            const float wA = lA > 0.f ? exp2f(mA - mb) : 0.f, wB = lB > 0.f ? exp2f(mB - mb) : 0.f;
            const float den = lA * wA + lB * wB;
            const float inv = den > 0.f ? 1.f / den : 0.f;
            const float cA = wA * inv, cB = wB * inv;
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                const uint32_t col = strm * (D / 2) + 32 * c;
                float oa[32], ob[32];
                tmem_ld32(tmem + lane_off + col, oa);
                if (nB > 0) tmem_ld32(tmem + lane_off + kOCol + col, ob);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float4 o;
                        o.x = oa[e] * cA + (cB > 0.f ? ob[e] * cB : 0.f);
                        o.y = oa[e + 1] * cA + (cB > 0.f ? ob[e + 1] * cB : 0.f);
                        o.z = oa[e + 2] * cA + (cB > 0.f ? ob[e + 2] * cB : 0.f);
                        o.w = oa[e + 3] * cA + (cB > 0.f ? ob[e + 3] * cB : 0.f);
                        *reinterpret_cast<float4*>(dst + 32 * c + e) = o;
                    }
                }
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
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
    pdl_wait();
    pdl_trigger();
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
    int qblocks, S, chunk;
    size_t smem;
};

// Splits of the key range: the grid is (S, Hkv * qblocks, B) CTAs of kUmmaM
// query rows each, one CTA per SM; the S CTAs of a (head, query block) form a
// cluster.  S trades wave quantisation against each CTA's fixed set-up; the
// split plan assumes the caches are mostly full (keys up to Lmax).
AttnPlan plan_attention(int B, int N, int Hq, int Hkv, int D, int Lmax) {
    AttnPlan p{};
    const int rows = N * (Hq / Hkv);
    p.qblocks = (rows + kUmmaM - 1) / kUmmaM;
    p.smem = D == 128 ? (size_t)AttnSmem<128>::kBytes : (size_t)AttnSmem<64>::kBytes;
    const long long units = (long long)B * Hkv * p.qblocks;
    const long long target = (long long)sm_count();
    const int max_tiles = (Lmax + kBlockN - 1) / kBlockN;
    // cost in tile times: a CTA takes its set-up (about kSetupTiles tiles:
    // TMEM, barriers, Q, pipeline fill) plus its tiles.  With fewer units than SMs every wave runs CTAs of one size; with
    // at least as many units as SMs (batches, taken longest first) the CTAs
    // pack the SMs, so the cost is the larger of one CTA and an even share.
    constexpr int kSetupTiles = 4;
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= max_tiles && s <= kMaxSplits; ++s) {
        const long long per_cta = kSetupTiles + (max_tiles + s - 1) / s;
        long long cost;
        if (B > 1 && units >= target) {
            const long long share = (units * s * per_cta + target - 1) / target;
            cost = share > per_cta ? share : per_cta;
        } else {
            cost = (units * s + target - 1) / target * per_cta;
        }
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; }
    }
    int chunk = (Lmax + best - 1) / best;
    chunk = (chunk + kBlockN - 1) / kBlockN * kBlockN;
    p.chunk = chunk;
    p.S = (Lmax + chunk - 1) / chunk;
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

// [B*Hkv][Lmax][D] bf16 cache as a 3-D tensor, boxes of 64 keys x 64 elements,
// 128-byte swizzle (the shared-memory layout the MMA descriptors expect).
int kv_tensor_map(CUtensorMap* m, const void* cache, int D, int Lmax, int BH) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(MEDUSA_ERR_CUDA, "tree_attention: cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Lmax, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Lmax * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kBlockN, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MEDUSA_ERR_CUDA, "tree_attention: tensor map encode failed (%d)", (int)r);
    return MEDUSA_OK;
}

// q [B][N][Hq][D] as a 4-D tensor (D, Hq, N, B); a box of 64 x G x (box_rows/G)
// x 1 holds box_rows consecutive rows (node, group member) of a query block.
int q_tensor_map(CUtensorMap* m, const void* q, int D, int Hq, int N, int B, int G, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(MEDUSA_ERR_CUDA, "tree_attention: cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2, (cuuint64_t)N * Hq * D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(box_rows / G), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MEDUSA_ERR_CUDA, "tree_attention: q tensor map encode failed (%d)", (int)r);
    return MEDUSA_OK;
}

template <int D>
int launch_bf16(AttnArgs& a, const AttnPlan& p, cudaStream_t st) {
    CUtensorMap tmk, tmv, tmq;
    int rc = kv_tensor_map(&tmk, a.k, D, a.Lmax, a.B * a.Hkv);
    if (rc) return rc;
    rc = kv_tensor_map(&tmv, a.v, D, a.Lmax, a.B * a.Hkv);
    if (rc) return rc;
    const int rows = a.N * a.G;
    a.spread = rows <= kUmmaM / 2 ? 1 : 0;
    const int box_rows = a.spread ? 16 : kUmmaM;  // rows per TMA box
    a.q_tma = (a.G <= box_rows && box_rows % a.G == 0) ? 1 : 0;
    if (a.q_tma) {
        rc = q_tensor_map(&tmq, a.q, D, a.Hq, a.N, a.B, a.G, box_rows);
        if (rc) return rc;
    } else {
        tmq = tmk;  // unused
    }
    if (p.S == 1 && (size_t)DualSmem<D>::kBytes <= (size_t)max_smem_optin()) {
        // keys not split: two streams per CTA
        auto kern = tree_attn_dual_kernel<D>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DualSmem<D>::kBytes);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, a.Hkv * p.qblocks, a.B);
        cfg.blockDim = dim3(kDualThreads);
        cfg.dynamicSmemBytes = DualSmem<D>::kBytes;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, tmq, a);
        if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "tree_attention: launch failed: %s", cudaGetErrorString(e));
        return MEDUSA_OK;
    }
    auto kern = tree_attn_umma_kernel<D>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.S, a.Hkv * p.qblocks, a.B);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = p.S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, tmq, a);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "tree_attention: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_tree_attention_workspace(int B, int N, int Hq, int Hkv, int D, int Lmax) {
    (void)B; (void)N; (void)Hq; (void)Hkv; (void)D; (void)Lmax;
    return 0;  // split partials are merged on chip (thread-block cluster)
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
    if (!(scale > 0.f) || scale > 3.0e38f)
        return fail(MEDUSA_ERR_INVALID_ARG, "tree_attention: scale must be positive and finite");
    const int W = (N + 63) / 64;
    cudaStream_t st = as_stream(stream);
    if (dtype == MEDUSA_F32) {
        const int rows = B * N * Hq;
        auto kern = D == 64 ? tree_attn_f32_kernel<64> : tree_attn_f32_kernel<128>;
        cudaError_t e = launch(kern, dim3((rows + 7) / 8), dim3(256), 0, st, (const float*)q,
                               (const float*)k_cache, (const float*)v_cache, kv_len, mask, B, N, Hq,
                               Hkv, Lmax, W, scale, out);
        if (e != cudaSuccess)
            return fail(MEDUSA_ERR_CUDA, "tree_attention_f32: launch failed: %s", cudaGetErrorString(e));
        return MEDUSA_OK;
    }
    if (dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_UNSUPPORTED, "tree_attention: unknown dtype %d", (int)dtype);
    (void)ws;
    (void)ws_bytes;
    AttnPlan p = plan_attention(B, N, Hq, Hkv, D, Lmax);
    if (p.smem > (size_t)max_smem_optin())
        return fail(MEDUSA_ERR_UNSUPPORTED, "tree_attention: %zu bytes of shared memory needed", p.smem);
    AttnArgs a{};
    a.q = (const uint16_t*)q;
    a.k = (const uint16_t*)k_cache;
    a.v = (const uint16_t*)v_cache;
    a.kv_len = kv_len;
    a.mask = mask;
    a.out = out;
    a.B = B; a.N = N; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.Lmax = Lmax; a.W = W;
    a.S = p.S; a.chunk = p.chunk; a.qblocks = p.qblocks;
    a.scale_log2 = scale * kLog2e;
    return D == 64 ? launch_bf16<64>(a, p, st) : launch_bf16<128>(a, p, st);
}
