// project.cu -- verification projection fused with tree acceptance ("Medusa
// Heads" glossary page, "Tree attention and acceptance": the base model scores
// every candidate of the tree in one pass; the verifier's next-token logits of
// tree node u are lm_head . hidden_u, and acceptance needs only per-row
// statistics of them).
//
// The [B*N, V] logits are never written to memory:
//   project_stats_kernel : CTA (vocab split s, block of 128 rows of the
//                          flattened [B*N] tree rows).  For each tile of tn
//                          tokens (tn in 128..256, chosen so the CTAs of one
//                          wave get equal work), D[128 rows x tn] = hidden .
//                          lm_head^T on the tensor cores (tcgen05.mma, bf16 in,
//                          float32 accumulate in TMEM, two D buffers); TMA
//                          streams 64-element slices of both operands through
//                          a 4-stage ring.  Epilogue threads (one per row) read
//                          D out of TMEM 32 columns at a time and fold them
//                          into the row's running argmax and, for typical
//                          acceptance, its softmax/entropy state.
//                          warp 0: TMA; warp 1: TMEM allocation and MMA issue;
//                          warps 2-5: epilogue (warp w reads TMEM lanes
//                          32*(w%4) .. 32*(w%4)+31)
//   row_finish_kernel    : (verify.cu) one warp per row: merges the splits'
//                          statistics and, for typical acceptance, computes the
//                          row's candidate logit as a dot product
//   accept_tree_kernel   : (verify.cu) tests the candidates and selects the
//                          longest accepted branch.
// Every wait is bounded; a CTA that gives up marks its status word and the
// acceptance kernel then writes -1 for every output.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "tmap.cuh"
#include "umma.cuh"
#include "verify_common.cuh"

namespace medusa {
namespace {

MEDUSA_WAIT_CONTROL()

constexpr int kPM = 128;      // tree rows per block (MMA M)
constexpr int kPN = 256;      // largest vocab tile (MMA N); the plan picks 128..256
constexpr int kPK = 64;       // hidden elements per stage (one 128-byte swizzle span)
constexpr int kPStages = 4;
constexpr int kPThreads = 192;
constexpr int kPA = kPM * kPK * 2;  // 16 KB of hidden rows per stage
constexpr int kPB = kPN * kPK * 2;  // 32 KB of lm_head rows per stage
constexpr int kPStage = kPA + kPB;
constexpr int kPBars = 2 * kPStages + 2 + 2 + 1;  // full, empty, d_full, d_empty, drain
constexpr int kPSmem = kPStages * kPStage + kPBars * 8 + 16 + 1024;
constexpr long long kPWait = kDefaultWaitCycles;  // drain waits (~1 s at 2 GHz)

struct ProjArgs {
    int rows;        // B * N
    int V;
    int nkb;         // hidden slices: ceil(H / 64)
    int tn;          // vocab tokens per tile, a multiple of 32 in [128, 256]
    int tiles;       // ceil(V / tn)
    int splits;      // vocab splits (gridDim.x)
    float inv_t;
    RowStat* stats;  // [rows][splits]
    int* status;     // [gridDim.y][splits]
};

template <bool TYPICAL>
__global__ void __launch_bounds__(kPThreads, 1) project_stats_kernel(
    const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb, ProjArgs a) {
    using namespace umma;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    uint8_t* base = smem_raw + pad;
    const uint32_t sbase = smem_addr(base);
    const uint32_t bar0 = sbase + kPStages * kPStage;
    auto full = [&](int i) { return bar0 + 8 * i; };
    auto empty = [&](int i) { return bar0 + 8 * (kPStages + i); };
    auto d_full = [&](int i) { return bar0 + 8 * (2 * kPStages + i); };
    auto d_empty = [&](int i) { return bar0 + 8 * (2 * kPStages + 2 + i); };
    const uint32_t drain = bar0 + 8 * (2 * kPStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kPStages * kPStage + kPBars * 8);
    volatile int* fail_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.x, nb = blockIdx.y;
    // limit of the first waits; the drain waits keep kPWait
    const long long lim = g_wait_limit;
    const int t0 = (int)((long long)s * a.tiles / a.splits);
    const int t1 = (int)((long long)(s + 1) * a.tiles / a.splits);
    const int ntiles = t1 - t0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(d_full(i), 1);
            mbar_init(d_empty(i), 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *fail_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 2 * kPN);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the hidden states may come from the previous kernel
    pdl_trigger();

    int issued = 0;  // TMA lane: loads issued
    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            for (int t = t0; t < t1 && ok; ++t)
                for (int kb = 0; kb < a.nkb; ++kb, ++issued) {
                    const int st = issued % kPStages;
                    if (issued >= kPStages &&
                        !mbar_wait(empty(st), ((issued / kPStages) - 1) & 1, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + st * kPStage, sb = sa + kPA;
                    mbar_expect_tx(full(st), (uint32_t)(kPA + a.tn * kPK * 2));
                    tma_load_2d(sa, &tma, kb * kPK, nb * kPM, full(st));
                    tma_load_2d(sb, &tmb, kb * kPK, t * a.tn, full(st));
                }
            if (!ok) *fail_flag = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kPM, a.tn, 0, 0);
            bool ok = true;
            int it = 0;
            for (int tl = 0; tl < ntiles && ok; ++tl) {
                const int buf = tl & 1;
                if (tl >= 2 && !mbar_wait(d_empty(buf), ((tl / 2) - 1) & 1, lim)) {
                    ok = false;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(buf * kPN);
                for (int kb = 0; kb < a.nkb; ++kb, ++it) {
                    const int st = it % kPStages;
                    if (!mbar_wait(full(st), (it / kPStages) & 1, lim)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t sa = sbase + st * kPStage, sb = sa + kPA;
#pragma unroll
                    for (int ks = 0; ks < kPK / 16; ++ks)
                        mma_bf16(d, desc_sw128(sa + ks * 32, 16, 1024), desc_sw128(sb + ks * 32, 16, 1024),
                                 idesc, (kb | ks) != 0);
                    commit(empty(st));  // the stage is free once these MMAs complete
                }
                if (ok) commit(d_full(buf));
            }
            if (!ok) *fail_flag = 1;
            // every MMA issued here completes before TMEM is released
            commit(drain);
            if (!mbar_wait(drain, 0, kPWait)) *fail_flag = 1;
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = nb * kPM + q * 32 + lane;
        // running argmax (bv, bi) and, for typical acceptance, the softmax state
        // of x = logit / T in base 2: m2 = max x*log2(e), s = sum 2^(x*log2e - m2),
        // a2 = sum 2^(..) (x*log2e - m2); a = a2 ln 2 in natural units
        float bv = -INFINITY, m2 = -INFINITY, ssum = 0.f, sa2 = 0.f;
        int bi = INT_MAX;
        const float k2 = a.inv_t * 1.4426950408889634f;
        bool ok = true;
        for (int tl = 0; tl < ntiles; ++tl) {
            const int buf = tl & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(d_full(buf), (tl / 2) & 1, lim));
            if (!ok) break;
            fence_after_sync();
            const int v0 = (t0 + tl) * a.tn;
#pragma unroll 1
            for (int c0 = 0; c0 < a.tn; c0 += 32) {
                float x[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kPN + c0), x);
                tmem_wait_ld();
                const int nv = min(32, a.V - (v0 + c0));  // columns past the vocab are padding
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j >= nv) x[j] = -INFINITY;
                // chunk maximum, then its lowest column; a later chunk only wins
                // with a strictly larger value (its tokens are larger)
                float cm = x[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) cm = fmaxf(cm, x[j]);
                if (cm > bv) {
                    int cj = 31;
#pragma unroll
                    for (int j = 31; j >= 0; --j)
                        if (x[j] == cm) cj = j;
                    bv = cm;
                    bi = v0 + c0 + cj;
                }
                if (TYPICAL && nv > 0) {
                    const float cm2 = cm * k2;
                    if (cm2 > m2) {  // move the reference to the chunk maximum
                        if (ssum > 0.f) {
                            const float c = umma::exp2_approx(m2 - cm2);
                            sa2 = c * (sa2 + (m2 - cm2) * ssum);
                            ssum *= c;
                        }
                        m2 = cm2;
                    }
                    float cs = 0.f, ca = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float d = fmaf(x[j], k2, -m2);  // -inf for padding: e = 0
                        const float e = umma::exp2_approx(d);
                        cs += e;
                        ca = fmaf(e, j < nv ? d : 0.f, ca);
                    }
                    ssum += cs;
                    sa2 += ca;
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_empty(buf));
        }
        const float m = m2 * 0.6931471805599453f, sa = sa2 * 0.6931471805599453f;
        if (!ok) {
            if (lane == 0) *fail_flag = 1;
        } else if (row < a.rows) {
            RowStat r;
            r.maxv = bv;
            r.arg = bi;
            r.m = m;
            r.s = ssum;
            r.a = sa;
            r.pad[0] = r.pad[1] = r.pad[2] = 0.f;
            a.stats[(size_t)row * a.splits + s] = r;
        }
    }
    fence_before_sync();
    __syncthreads();
    const bool failed = *fail_flag != 0;
    if (failed && warp == 0 && lane == 0) {
        // let the copies still in flight land before the CTA's shared memory goes
        for (int i = max(0, issued - kPStages); i < issued; ++i)
            mbar_wait(full(i % kPStages), (i / kPStages) & 1, kPWait);
    }
    if (threadIdx.x == 0) a.status[(size_t)nb * a.splits + s] = failed ? 1 : 0;
    if (failed && threadIdx.x == 0) atomicExch(&g_wait_gave_up, 1);
    if (warp == 1) {
        fence_after_sync();
        tmem_dealloc(tmem, 2 * kPN);
    }
}

// row-major [rows][H] bf16 as a 2-D tensor, boxes of box_rows x 64 elements,
// 128-byte swizzle (the shared-memory layout the MMA descriptors expect)
int rows_tensor_map(CUtensorMap* m, const void* p, int H, int rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(MEDUSA_ERR_CUDA, "verify_project_tree: cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {(cuuint32_t)kPK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MEDUSA_ERR_CUDA, "verify_project_tree: tensor map encode failed (%d)", (int)r);
    return MEDUSA_OK;
}

struct ProjPlan {
    int rows, nblocks, tn, tiles, splits, nkb;
    size_t off_status, off_final, off_cl, ws_bytes;
};

ProjPlan plan_project(int B, int N, int H, int V) {
    ProjPlan p{};
    p.rows = B * N;
    p.nblocks = (p.rows + kPM - 1) / kPM;
    p.nkb = (H + kPK - 1) / kPK;
    // One CTA per SM (the operand ring takes most of shared memory); each row
    // block gets `splits` CTAs.  The tile width is the one whose busiest CTA
    // has the fewest vocab columns (ties: the wider tile).
    const int per_block = sm_count() / p.nblocks;
    long long best = -1;
    for (int tn = kPN; tn >= 128; tn -= 32) {
        const int tiles = (V + tn - 1) / tn;
        const int splits = per_block < 1 ? 1 : (per_block > tiles ? tiles : per_block);
        const long long cols = (long long)((tiles + splits - 1) / splits) * tn;
        if (best < 0 || cols < best) {
            best = cols;
            p.tn = tn;
            p.tiles = tiles;
            p.splits = splits;
        }
    }
    p.off_status = align_up((size_t)p.rows * p.splits * sizeof(RowStat), 256);
    p.off_final = align_up(p.off_status + (size_t)p.nblocks * p.splits * sizeof(int), 256);
    p.off_cl = align_up(p.off_final + (size_t)p.rows * sizeof(RowStat), 256);
    p.ws_bytes = align_up(p.off_cl + (size_t)p.rows * sizeof(float), 256);
    return p;
}

int check_project_shapes(int B, int N, int H, int V) {
    if (B < 1 || N < 1 || H < 1 || V < 1)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_project_tree: sizes must be positive");
    if (N > kAcceptThreads || B > 65535 || (long long)B * N > 65535LL * kPM || H % 8 || H > 65536 ||
        V > (1 << 24))
        return fail(MEDUSA_ERR_UNSUPPORTED,
                    "verify_project_tree: unsupported shape (B=%d N=%d H=%d V=%d): need N<=%d, "
                    "B<=65535, H%%8==0, H<=65536, V<=2^24",
                    B, N, H, V, kAcceptThreads);
    return MEDUSA_OK;
}

}  // namespace
}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_verify_project_workspace(int B, int N, int H, int V) {
    if (check_project_shapes(B, N, H, V)) return 0;
    return plan_project(B, N, H, V).ws_bytes;
}

extern "C" int medusa_verify_project_tree(const void* hidden_tree, const void* lm_head,
                                          medusa_dtype dtype, const int32_t* cand,
                                          const int32_t* parent, const int32_t* depth, int B, int N,
                                          int H, int V, int Dmax, medusa_accept_mode mode,
                                          float temperature, float eps, float delta,
                                          int32_t* accept_len, int32_t* best_node,
                                          int32_t* path_nodes, int32_t* next_tok, void* ws,
                                          size_t ws_bytes, void* stream) {
    if (!hidden_tree || !lm_head || !cand || !parent || !depth || !accept_len || !best_node ||
        !path_nodes || !next_tok)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_project_tree: null pointer");
    if (Dmax < 0) return fail(MEDUSA_ERR_INVALID_ARG, "verify_project_tree: Dmax must be >= 0");
    int rc = check_project_shapes(B, N, H, V);
    if (rc) return rc;
    if (dtype != MEDUSA_BF16)
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_project_tree: only bf16 hidden states and lm_head");
    if (mode != MEDUSA_ACCEPT_GREEDY && mode != MEDUSA_ACCEPT_TYPICAL)
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_project_tree: unknown mode %d", (int)mode);
    if (mode == MEDUSA_ACCEPT_TYPICAL && !(temperature > 0.f))
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_project_tree: temperature must be > 0");
    if (!aligned16(hidden_tree) || !aligned16(lm_head))
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_project_tree: hidden_tree and lm_head must be 16-byte aligned");
    const ProjPlan p = plan_project(B, N, H, V);
    if (!ws || ws_bytes < p.ws_bytes)
        return fail(MEDUSA_ERR_WORKSPACE, "verify_project_tree: workspace of %zu bytes needed, %zu given",
                    p.ws_bytes, ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(MEDUSA_ERR_INVALID_ARG, "verify_project_tree: ws must be 16-byte aligned");
    if (kPSmem > max_smem_optin())
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_project_tree: %d bytes of shared memory needed", kPSmem);
    CUtensorMap tma, tmb;
    rc = rows_tensor_map(&tma, hidden_tree, H, p.rows, kPM);
    if (rc) return rc;
    rc = rows_tensor_map(&tmb, lm_head, H, V, p.tn);
    if (rc) return rc;
    char* w = static_cast<char*>(ws);
    ProjArgs pa{};
    pa.rows = p.rows;
    pa.V = V;
    pa.nkb = p.nkb;
    pa.tn = p.tn;
    pa.tiles = p.tiles;
    pa.splits = p.splits;
    pa.inv_t = mode == MEDUSA_ACCEPT_TYPICAL ? 1.f / temperature : 1.f;
    pa.stats = reinterpret_cast<RowStat*>(w);
    pa.status = reinterpret_cast<int*>(w + p.off_status);
    cudaStream_t st = as_stream(stream);
    auto k = mode == MEDUSA_ACCEPT_TYPICAL ? project_stats_kernel<true> : project_stats_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    cudaError_t e = launch(k, dim3(p.splits, p.nblocks), dim3(kPThreads), (size_t)kPSmem, st, tma, tmb, pa);
    if (e != cudaSuccess)
        return fail(MEDUSA_ERR_CUDA, "verify_project_tree: launch failed: %s", cudaGetErrorString(e));
    RowStat* final_stats = reinterpret_cast<RowStat*>(w + p.off_final);
    float* child_logit = reinterpret_cast<float*>(w + p.off_cl);
    rc = launch_row_finish(mode == MEDUSA_ACCEPT_TYPICAL, pa.stats, p.splits, p.rows, N, V, H,
                           static_cast<const uint16_t*>(hidden_tree), static_cast<const uint16_t*>(lm_head),
                           cand, parent, final_stats, child_logit, st);
    if (rc) return rc;
    AcceptArgs aa{};
    aa.logits = nullptr;
    aa.child_logit = child_logit;
    aa.cand = cand;
    aa.parent = parent;
    aa.depth = depth;
    aa.B = B;
    aa.N = N;
    aa.V = V;
    aa.Dmax = Dmax;
    aa.nchunk = 1;
    aa.inv_t = pa.inv_t;
    aa.eps = eps;
    aa.delta = delta;
    aa.stats = final_stats;
    aa.status = pa.status;
    aa.nstatus = p.nblocks * p.splits;
    aa.accept_len = accept_len;
    aa.best_node = best_node;
    aa.path_nodes = path_nodes;
    aa.next_tok = next_tok;
    return launch_accept_tree(mode == MEDUSA_ACCEPT_TYPICAL, aa, st);
}
