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
//   tree_attn_umma_kernel : split-KV over CTAs; per 64-key tile S = Q K^T and
//                           O += P V as tcgen05.mma (bf16 in, float32 out),
//                           online softmax in float32 with one query row per
//                           thread, ancestor bits tested only on tiles that
//                           reach the tree slots
//   attn_combine_kernel   : merges the per-split (max, sum, O) partials
//   tree_attn_f32_kernel  : float32 storage path (one warp per query row)
#include <float.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "umma.cuh"

namespace medusa {
namespace {

constexpr int kBlockN = 64;  // keys per tile
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

// ---------------------------------------------------------------------------
// tcgen05 kernel.  One CTA of 256 threads per (KV split, KV head x block of 128
// tree queries, sequence).  Query row r lives in TMEM lane r; threads r and
// r + 128 share it, each owning half of every 64-key score tile and half of
// the output columns.  Per tile j (keys [k_j, k_j + 64)):
//   S_j = Q K_j^T        tcgen05.mma, float32 in TMEM (two S buffers)
//   P_j = exp2(S_j * scale * log2e - m)   online softmax in registers, written
//                        as bf16 to one of two swizzled P buffers
//   O  += P_j V_j        tcgen05.mma, float32 accumulator in TMEM
// K and V tiles arrive by TMA (one thread, byte-counted mbarriers) into two
// 4-deep rings; S_{j+1} is issued before the softmax of tile j, so the tensor
// core overlaps the softmax.  The last tile of a split is shifted back to end
// exactly at the split's last key, so no row past it is ever read; keys the
// shift brings back are masked.  The reference max used for P moves only when
// the row max grows by more than 2^8 (log2 domain), and O and the row sum are
// rescaled in TMEM at that moment.
// ---------------------------------------------------------------------------
constexpr int kUmmaM = 128;
constexpr int kUmmaThreads = 256;
constexpr int kRingK = 4, kRingV = 4;
constexpr float kRescaleThreshold = 8.f;
constexpr long long kWaitCycles = 1ll << 31;  // ~1 s at 2 GHz

template <int D>
struct UmmaSmem {
    static constexpr int kQ = kUmmaM * D * 2;
    static constexpr int kTile = kBlockN * D * 2;  // one K or V tile
    static constexpr int kP = kUmmaM * kBlockN * 2;
    static constexpr int kOffK = kQ;
    static constexpr int kOffV = kOffK + kRingK * kTile;
    static constexpr int kOffP = kOffV + kRingV * kTile;
    static constexpr int kOffRed = kOffP + 2 * kP;       // float [2][128]
    static constexpr int kOffBar = kOffRed + 2 * 128 * 4;  // mbarriers
    static constexpr int kNumBar = 1 + 2 + kRingK + kRingV;
    static constexpr int kOffMisc = kOffBar + kNumBar * 8;  // tmem slot, flag
    static constexpr int kBytes = kOffMisc + 16 + 1024;     // + alignment slack
};

template <int D>
__global__ void __launch_bounds__(kUmmaThreads, 1) tree_attn_umma_kernel(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, AttnArgs a) {
    using namespace umma;
    using L = UmmaSmem<D>;
    constexpr int CH = D / 8;         // 16-byte chunks per row
    constexpr int TMEM_COLS = 256;    // O: D columns at 0; S buffers at 128 and 192
    constexpr uint32_t kSCol = 128;
    constexpr int HALF = kBlockN / 2;
    extern __shared__ uint8_t smem_raw[];

    const int split = blockIdx.x;
    const int hk = blockIdx.y / a.qblocks, qb = blockIdx.y % a.qblocks;
    const int b = blockIdx.z;
    const int N = a.N, G = a.G;
    pdl_wait();
    pdl_trigger();
    const int Lb = clamp_len(a.kv_len[b], N, a.Lmax);
    const int total = Lb + N;
    const int k_begin = split * a.chunk;
    if (k_begin >= total) return;  // no keys of sequence b in this split (uniform per CTA)
    const int k_end = min(total, k_begin + a.chunk);
    const int ntiles = (k_end - k_begin + kBlockN - 1) / kBlockN;
    const int rows = N * G;
    const int row0 = qb * kUmmaM;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int r = tid & (kUmmaM - 1), half = tid >> 7;

    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t* base = smem_raw + pad;
    const uint32_t base_a = smem_addr(base);
    const uint32_t qs_a = base_a, ks_a = base_a + L::kOffK, vs_a = base_a + L::kOffV,
                   ps_a = base_a + L::kOffP;
    float* red = reinterpret_cast<float*>(base + L::kOffRed);
    const uint32_t bar_a = base_a + L::kOffBar;
    const uint32_t mbS = bar_a, mbO0 = bar_a + 8;  // mbO[i] = mbO0 + 8 i
    const uint32_t kfull0 = bar_a + 24, vfull0 = kfull0 + 8 * kRingK;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kOffMisc);
    int* flag = reinterpret_cast<int*>(base + L::kOffMisc + 4);

    // key range of tile t: [tile_start, tile_start + 64); keys below tile_lo were
    // covered by an earlier tile (or another split)
    auto tile_lo = [&](int t) { return k_begin + t * kBlockN; };
    auto tile_start = [&](int t) { return min(k_begin + t * kBlockN, k_end - kBlockN); };
    const int zrow = b * a.Hkv + hk;
    auto load_k = [&](int t) {
        const uint32_t st = ks_a + (t % kRingK) * L::kTile, fb = kfull0 + 8 * (t % kRingK);
        mbar_expect_tx(fb, L::kTile);
#pragma unroll
        for (int x = 0; x < D / 64; ++x) tma_load_3d(st + x * kBlockN * 128, &tmk, x * 64, tile_start(t), zrow, fb);
    };
    auto load_v = [&](int t) {
        const uint32_t st = vs_a + (t % kRingV) * L::kTile, fb = vfull0 + 8 * (t % kRingV);
        mbar_expect_tx(fb, L::kTile);
#pragma unroll
        for (int x = 0; x < D / 64; ++x) tma_load_3d(st + x * kBlockN * 128, &tmv, x * 64, tile_start(t), zrow, fb);
    };

    if (tid == 0) {
        for (int i = 0; i < L::kNumBar; ++i) mbar_init(bar_a + 8 * i, 1);
        mbar_init_fence();
        *flag = 0;
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    // Q tile: row r -> node r / G, query head hk * G + r % G; padding rows are zero
    for (int c = tid; c < kUmmaM * CH; c += kUmmaThreads) {
        const int rr = c / CH, ch = c % CH;
        const int gr = row0 + rr;
        const bool ok = gr < rows;
        const int node = ok ? gr / G : 0, hq = hk * G + (ok ? gr % G : 0);
        cp_async16(qs_a + sw128_offset(rr, ch, kUmmaM),
                   a.q + (((size_t)b * N + node) * a.Hq + hq) * D + ch * 8, ok);
    }
    cp_async_commit();
    fence_before_sync();
    __syncthreads();  // barriers initialised, TMEM allocated
    fence_after_sync();
    int k_issued = 0, v_issued = 0;  // thread 0: K / V tiles requested so far
    if (tid == 0) {
        for (; k_issued < kRingK && k_issued < ntiles; ++k_issued) load_k(k_issued);
        for (; v_issued < kRingV && v_issued < ntiles; ++v_issued) load_v(v_issued);
    }
    cp_async_wait<0>();
    fence_async_smem();
    fence_before_sync();
    __syncthreads();  // Q resident and visible to the tensor core
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

    const int grow = row0 + r;
    const bool valid = grow < rows;
    const int node = valid ? grow / G : 0;
    const uint64_t* mrow = a.mask + (size_t)node * a.W;
    constexpr uint32_t idesc_s = idesc_bf16(kUmmaM, kBlockN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16(kUmmaM, D, 0, 1);

    // thread 0 only: S_t = Q K_t^T into S buffer t & 1, after K_t has landed
    auto issue_s = [&](int t) -> bool {
        if (!mbar_wait(kfull0 + 8 * (t % kRingK), (uint32_t)((t / kRingK) & 1), kWaitCycles)) return false;
        const uint32_t ka = ks_a + (t % kRingK) * L::kTile;
        const uint32_t d = tmem + kSCol + (t & 1) * kBlockN;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t ad = desc_sw128(qs_a + (ks >> 2) * (kUmmaM * 128) + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = desc_sw128(ka + (ks >> 2) * (kBlockN * 128) + (ks & 3) * 32, 16, 1024);
            mma_bf16(d, ad, bd, idesc_s, ks > 0);
        }
        commit(mbS);
        return true;
    };
    // thread 0 only: O += P_t V_t, after V_t has landed
    auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(vfull0 + 8 * (t % kRingV), (uint32_t)((t / kRingV) & 1), kWaitCycles)) return false;
        const uint32_t va = vs_a + (t % kRingV) * L::kTile;
        const uint32_t pa = ps_a + (t & 1) * L::kP;
#pragma unroll
        for (int ks = 0; ks < kBlockN / 16; ++ks) {
            const uint64_t ad = desc_sw128(pa + ks * 32, 16, 1024);
            const uint64_t bd = desc_sw128(va + ks * 2048, kBlockN * 128, 1024);
            mma_bf16(tmem, ad, bd, idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
        }
        commit(mbO0 + 8 * (t & 1));
        return true;
    };
    if (tid == 0 && !issue_s(0)) *flag = 1;

    float m_ref = -INFINITY, l = 0.f;
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
        // 1. S_j complete (K_j's stage is free again)
        bool ok = mbar_wait(mbS, (uint32_t)(j & 1), kWaitCycles);
        fence_after_sync();
        // 2. this half-row's 32 scores
        float sv[HALF];
        tmem_ld32(tmem + lane_off + kSCol + (j & 1) * kBlockN + half * HALF, sv);
        tmem_wait_ld();
        const int kt = tile_start(j), klo = tile_lo(j);
        const int c0 = kt + half * HALF;  // key of sv[0]
        float mt = -INFINITY;
        if (kt == klo && kt + kBlockN <= min(k_end, Lb)) {  // plain prefix tile
#pragma unroll
            for (int i = 0; i < HALF; ++i) { sv[i] *= a.scale_log2; mt = fmaxf(mt, sv[i]); }
        } else {
            uint64_t w0 = 0, w1 = 0;
            int mbase = 0;
            if (valid && c0 + HALF > Lb) {
                mbase = max(c0 - Lb, 0) & ~63;
                const int wi = mbase >> 6;
                w0 = wi < a.W ? __ldg(mrow + wi) : 0ull;
                w1 = wi + 1 < a.W ? __ldg(mrow + wi + 1) : 0ull;
            }
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
                const int key = c0 + i;
                bool vis = key >= klo && key < k_end;
                if (key >= Lb) {
                    const int m = key - Lb - mbase;  // in [0, 96)
                    vis = vis && valid && (((m < 64 ? w0 >> m : w1 >> (m - 64)) & 1ull) != 0);
                }
                sv[i] = vis ? sv[i] * a.scale_log2 : -INFINITY;
                mt = fmaxf(mt, sv[i]);
            }
        }
        red[half * 128 + r] = mt;
        // 3. thread 0 issues S_{j+1} (its K tile has landed) and refills K_j's stage
        if (tid == 0) {
            if (j + kRingK < ntiles) { load_k(j + kRingK); k_issued = j + kRingK + 1; }
            if (j + 1 < ntiles && !issue_s(j + 1)) *flag = 1;
        }
        bad = __syncthreads_or(!ok) || *flag;  // B1: row maxima exchanged
        if (bad) break;
        mt = fmaxf(mt, red[(half ^ 1) * 128 + r]);
        // 4. move the reference max when it grows by more than the threshold;
        //    O in TMEM must hold PV_{j-1} before it is rescaled
        float corr = 1.f;
        bool rescale = false;
        if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescaleThreshold)) {
            if (m_ref != -INFINITY && j > 0) { corr = exp2f(m_ref - mt); rescale = true; }
            m_ref = mt;
        }
        l *= corr;
        if (__any_sync(0xffffffffu, rescale)) {  // TMEM loads/stores are warp-collective
            ok = mbar_wait(mbO0 + 8 * ((j - 1) & 1), (uint32_t)(((j - 1) >> 1) & 1), kWaitCycles);
            fence_after_sync();
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < D / 2; cc += 32) {
                    float ov[32];
                    const uint32_t ta = tmem + lane_off + half * (D / 2) + cc;
                    tmem_ld32(ta, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= corr;
                    tmem_st32(ta, ov);
                }
                tmem_wait_st();
            }
        }
        // 5. P buffer j & 1 was last read by PV_{j-2}; its V stage is then free
        if (j >= 2) {
            ok = mbar_wait(mbO0 + 8 * (j & 1), (uint32_t)(((j - 2) >> 1) & 1), kWaitCycles) && ok;
            fence_after_sync();
            if (tid == 0 && j - 2 + kRingV < ntiles) { load_v(j - 2 + kRingV); v_issued = j - 2 + kRingV + 1; }
        }
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;
        uint8_t* prow = base + L::kOffP + (j & 1) * L::kP;
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < HALF / 8; ++c) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p0 = exp2f(sv[c * 8 + 2 * e] - mr);
                const float p1 = exp2f(sv[c * 8 + 2 * e + 1] - mr);
                psum += p0 + p1;
                pk[e] = pack_bf16(p0, p1);
            }
            *reinterpret_cast<uint4*>(prow + sw128_offset(r, half * (HALF / 8) + c, kUmmaM)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l += psum;
        // 6. P visible to the tensor core, then PV_j
        fence_async_smem();
        fence_before_sync();
        bad = __syncthreads_or(!ok);  // B2
        fence_after_sync();
        if (bad) break;
        if (tid == 0 && !issue_pv(j)) *flag = 1;
    }
    // drain: the last PV (and, on failure, whatever is in flight)
    bool ok = !bad && mbar_wait(mbO0 + 8 * ((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1), kWaitCycles);
    fence_after_sync();
    red[half * 128 + r] = l;
    bad = __syncthreads_or(!ok) || *flag;
    if (bad && tid == 0) {
        // give the tensor core and the TMA loads in flight a second bounded
        // chance to finish before TMEM is freed and the CTA leaves
        mbar_wait(mbO0 + 8 * ((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1), kWaitCycles);
        for (int t = max(0, k_issued - kRingK); t < k_issued; ++t)
            mbar_wait(kfull0 + 8 * (t % kRingK), (uint32_t)((t / kRingK) & 1), kWaitCycles);
        for (int t = max(0, v_issued - kRingV); t < v_issued; ++t)
            mbar_wait(vfull0 + 8 * (t % kRingV), (uint32_t)((t / kRingV) & 1), kWaitCycles);
    }
    __syncthreads();
    const float lt = l + red[(half ^ 1) * 128 + r];

    // epilogue: this thread's half of the O row (TMEM loads are warp-collective)
    const int hq = hk * G + grow % G;
    const int S = gridDim.x;
    float* dst = nullptr;
    float scale = 1.f;
    if (valid) {
        if (S == 1) {
            dst = a.out + (((size_t)b * N + node) * a.Hq + hq) * D;
            scale = lt > 0.f ? 1.f / lt : 0.f;
        } else {
            const size_t prow = (((size_t)b * a.Hq + hq) * N + node) * S + split;
            dst = a.part_o + prow * D;
            if (half == 0) {
                a.part_ml[prow * 2] = bad ? NAN : m_ref;
                a.part_ml[prow * 2 + 1] = bad ? NAN : lt;
            }
        }
    }
#pragma unroll
    for (int cc = 0; cc < D / 2; cc += 32) {
        float ov[32];
        const int col = half * (D / 2) + cc;
        tmem_ld32(tmem + lane_off + col, ov);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + col + i) =
                    bad ? make_float4(NAN, NAN, NAN, NAN)
                        : make_float4(ov[i] * scale, ov[i + 1] * scale, ov[i + 2] * scale, ov[i + 3] * scale);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// One warp per (b, node, query head): merge the splits that hold keys.  Lane s
// reads split s's (max, sum); the output columns are spread over the lanes and
// the splits' partial outputs are read four at a time.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a) {
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= a.B * a.N * a.Hq) return;
    const int b = row / (a.N * a.Hq), node = (row / a.Hq) % a.N, hq = row % a.Hq;
    const int L = clamp_len(a.kv_len[b], a.N, a.Lmax);
    const int S = a.S;
    const int active = min(S, (L + a.N + a.chunk - 1) / a.chunk);
    const size_t prow = (((size_t)b * a.Hq + hq) * a.N + node) * S;
    // split weights: lane s holds split s (and s + 32, ...)
    constexpr int kMaxSplitRegs = 2;  // S <= 64
    float ms[kMaxSplitRegs], ls[kMaxSplitRegs];
    float mx = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxSplitRegs; ++r) {
        const int s = lane + 32 * r;
        ms[r] = -INFINITY;
        ls[r] = 0.f;
        if (s < active) {
            const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (prow + s) * 2);
            ms[r] = ml.x;
            ls[r] = ml.y;
            if (ml.y > 0.f) mx = fmaxf(mx, ml.x);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float base = mx == -INFINITY ? 0.f : mx;
    float wl[kMaxSplitRegs], lsum = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxSplitRegs; ++r) {
        wl[r] = ls[r] > 0.f ? exp2f(ms[r] - base) : 0.f;
        lsum += ls[r] * wl[r];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < active; s0 += 4) {
        float w[4], v[4][PER];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int s = s0 + j;
            w[j] = __shfl_sync(0xffffffffu, (s >> 5) == 0 ? wl[0] : wl[1], s & 31);
            const float* src = a.part_o + (prow + min(s, active - 1)) * D;
#pragma unroll
            for (int i = 0; i < PER; ++i) v[j][i] = src[lane + 32 * i];
            if (s >= active) w[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < PER; ++i) acc[i] = fmaf(v[j][i], w[j], acc[i]);
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
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
    int qblocks, S, chunk, cps;
    size_t smem, off_o, off_ml, ws_bytes;
};

// Splits of the key range: the grid is (S, Hkv * qblocks, B) CTAs of kUmmaM
// query rows each.  S trades wave quantisation (one CTA per SM) against each
// CTA's fixed set-up; the split plan assumes the caches are mostly full (keys
// up to Lmax).
AttnPlan plan_attention(int B, int N, int Hq, int Hkv, int D, int Lmax) {
    AttnPlan p{};
    const int rows = N * (Hq / Hkv);
    p.qblocks = (rows + kUmmaM - 1) / kUmmaM;
    p.smem = D == 128 ? (size_t)UmmaSmem<128>::kBytes : (size_t)UmmaSmem<64>::kBytes;
    p.cps = 1;
    const long long units = (long long)B * Hkv * p.qblocks;
    const long long target = (long long)sm_count() * p.cps;
    const int max_splits = (Lmax + kBlockN - 1) / kBlockN;
    // cost in tile times: each wave takes the CTA's fixed set-up (about
    // kSetupTiles tiles: TMEM, barriers, Q, pipeline fill) plus its tiles
    constexpr int kSetupTiles = 4;
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= max_splits && s <= 64; ++s) {  // the combine holds <= 64 splits per row
        const long long waves = (units * s + target - 1) / target;
        const long long cost = waves * (kSetupTiles + (max_splits + s - 1) / s);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; }
    }
    int chunk = (Lmax + best - 1) / best;
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
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

template <int D>
int launch_bf16(AttnArgs& a, const AttnPlan& p, cudaStream_t st) {
    CUtensorMap tmk, tmv;
    int rc = kv_tensor_map(&tmk, a.k, D, a.Lmax, a.B * a.Hkv);
    if (rc) return rc;
    rc = kv_tensor_map(&tmv, a.v, D, a.Lmax, a.B * a.Hkv);
    if (rc) return rc;
    dim3 grid(p.S, a.Hkv * p.qblocks, a.B);
    auto kern = tree_attn_umma_kernel<D>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    cudaError_t e = launch(kern, grid, dim3(kUmmaThreads), p.smem, st, tmk, tmv, a);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "tree_attention: launch failed: %s", cudaGetErrorString(e));
    if (p.S == 1) return MEDUSA_OK;
    const int rows = a.B * a.N * a.Hq;
    e = launch(attn_combine_kernel<D>, dim3((rows + 7) / 8), dim3(256), 0, st, a);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "attn_combine: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
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
