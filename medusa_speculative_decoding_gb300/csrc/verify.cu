// verify.cu -- acceptance of candidates.
//
// Tree ("Medusa Heads" glossary page, "Tree attention and acceptance"): greedy
// decoding accepts a candidate that equals the model's top choice; typical
// acceptance keeps a candidate whose base-model probability clears a threshold
// tied to the entropy of the distribution; the longest accepted branch is kept.
//   row_stats_kernel   : one pass over each verifier-logits chunk (HBM-bound):
//                        argmax, and for typical acceptance the running
//                        (max, sum exp, sum exp * x) of x = logit / T
//   tree_race_kernel, tree_race_finish_kernel : (sampled next token) the
//                        exponential race over the best node's softmax
//   accept_tree_kernel : per sequence: merge chunk stats, test each candidate
//                        against its parent's row, AND along ancestors, pick the
//                        deepest accepted node (lowest index on ties); also the
//                        second kernel of the fused verification projection
//                        (project.cu)
//
// Chain (speculative-decoding e-book page, "Faster without changing the
// result"; "Why a round always yields exactly k + 1 tokens"): accept draft x
// with probability min(1, p(x)/q(x)); at the first rejection draw from
// max(0, p - q) normalised; if all are accepted draw a bonus token from the
// next p.
//   chain_first_kernel  : one warp per sequence: the first rejection and the
//                         key of the row to draw from
//   chain_scan_kernel   : the exponential race over one vocab chunk of that row
//   chain_finish_kernel : merges the chunk winners and writes the k + 1 tokens
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "verify_common.cuh"

namespace medusa {
namespace {

// 2^x on the special-function unit (approximate, flush-to-zero)
__device__ __forceinline__ float exp2_sfu(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kChunk = 4096;     // vocab entries per stats CTA
constexpr int kStatThreads = 256;

template <bool TYPICAL>
__global__ void __launch_bounds__(kStatThreads) row_stats_kernel(const float* __restrict__ logits,
                                                                 int V, int nchunk, float inv_t,
                                                                 RowStat* __restrict__ stats) {
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, row = blockIdx.y;
    const float* x = logits + (size_t)row * V;
    const int v0 = c * kChunk, v1 = min(V, v0 + kChunk);
    float bv = -INFINITY;
    int bi = INT_MAX;
    float m = -INFINITY, s = 0.f, a = 0.f;
    auto take = [&](float l, int v) {
        if (better(l, v, bv, bi)) { bv = l; bi = v; }
        if (TYPICAL) take_msa(m, s, a, l * inv_t);
    };
    // vectorised body when the row start is 16-byte aligned: the thread's
    // share of the chunk (kPer 16-byte words) is loaded at once; for typical
    // acceptance its softmax state is formed in two passes over registers (the
    // maximum, then sum e^(x-m) and sum e^(x-m)(x-m) as independent terms)
    // instead of an online update per entry, which chains every entry on the
    // previous one
    const bool vec = ((reinterpret_cast<uintptr_t>(x + v0) & 15u) == 0);
    int v = v0;
    if (vec) {
        constexpr int kPer = kChunk / (4 * kStatThreads);
        const int nv = (v1 - v0) / 4;
        const float4* x4 = reinterpret_cast<const float4*>(x + v0);
        float e[4 * kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = threadIdx.x + kStatThreads * k;
            const uint4 r = i < nv ? ld_stream16(x4 + i) : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
            e[4 * k] = __uint_as_float(r.x);
            e[4 * k + 1] = __uint_as_float(r.y);
            e[4 * k + 2] = __uint_as_float(r.z);
            e[4 * k + 3] = __uint_as_float(r.w);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = threadIdx.x + kStatThreads * k;
            if (i < nv) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (better(e[4 * k + j], v0 + 4 * i + j, bv, bi)) { bv = e[4 * k + j]; bi = v0 + 4 * i + j; }
            }
        }
        if (TYPICAL) {
            // x = logit / T and its maximum exactly as the acceptance kernel
            // forms them; each weight e^(x - max) on the special-function unit
            // as 2^((x - max) log2 e).  Entries past the chunk were loaded as
            // -inf: no probability mass.
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4 * kPer; ++j) {
                e[j] *= inv_t;
                mx = fmaxf(mx, e[j]);
            }
            if (mx > -INFINITY) {
                float ss = 0.f, sa = 0.f;
#pragma unroll
                for (int j = 0; j < 4 * kPer; ++j) {
                    const float d = e[j] - mx;  // -inf (empty entries) or NaN: weight 0
                    const float w = d > -INFINITY ? exp2_sfu(d * 1.4426950408889634f) : 0.f;
                    ss += w;
                    sa = w > 0.f ? fmaf(w, d, sa) : sa;
                }
                m = mx;
                s = ss;
                a = sa;
            }
        }
        v = v0 + 4 * nv;
    }
    for (int i = v + threadIdx.x; i < v1; i += kStatThreads) take(x[i], i);
    // block reduction
    __shared__ float sv[kStatThreads / 32], sm_[kStatThreads / 32], ss[kStatThreads / 32],
        sa[kStatThreads / 32];
    __shared__ int si[kStatThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        if (TYPICAL) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const float os = __shfl_xor_sync(0xffffffffu, s, o);
            const float oa = __shfl_xor_sync(0xffffffffu, a, o);
            merge_msa(m, s, a, om, os, oa);
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; sm_[warp] = m; ss[warp] = s; sa[warp] = a; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kStatThreads / 32; ++w) {
            if (better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
            if (TYPICAL) merge_msa(m, s, a, sm_[w], ss[w], sa[w]);
        }
        RowStat r;
        r.maxv = bv; r.arg = bi; r.m = m; r.s = s; r.a = a;
        r.pad[0] = r.pad[1] = r.pad[2] = 0.f;
        stats[(size_t)row * nchunk + c] = r;
    }
}

// One CTA per sequence.  When the statistics kernel flagged a failure (a
// nonzero a.status entry), every output of the sequence is -1.
template <bool TYPICAL>
__global__ void __launch_bounds__(kAcceptThreads) accept_tree_kernel(const AcceptArgs a) {
    __shared__ int s_arg[kAcceptThreads];
    __shared__ float s_m[kAcceptThreads], s_s[kAcceptThreads], s_tau[kAcceptThreads];
    __shared__ unsigned char s_pass[kAcceptThreads];
    __shared__ int s_best;
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, N = a.N, V = a.V, Dmax = a.Dmax;
    const int32_t* parent = a.parent;
    const int32_t* depth = a.depth;
    const int u = threadIdx.x;
    int bad = 0;
    for (int i = u; i < a.nstatus; i += blockDim.x) bad |= a.status[i];
    if (__syncthreads_or(bad)) {
        if (u == 0) {
            a.accept_len[b] = -1;
            a.best_node[b] = -1;
            a.next_tok[b] = -1;
        }
        for (int e = u; e <= Dmax; e += blockDim.x) a.path_nodes[(size_t)b * (Dmax + 1) + e] = -1;
        return;
    }
    if (u < N) {
        const RowStat* st = a.stats + ((size_t)b * N + u) * a.nchunk;
        float bv = -INFINITY, m = -INFINITY, s = 0.f, sa = 0.f;
        int bi = INT_MAX;
        // the chunk records are loaded eight at a time before they are merged,
        // so their load latencies overlap instead of chaining
        constexpr int kBatch = 8;
        for (int c0 = 0; c0 < a.nchunk; c0 += kBatch) {
            RowStat rs[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
                if (c0 + k < a.nchunk) rs[k] = st[c0 + k];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (c0 + k < a.nchunk) {
                    if (better(rs[k].maxv, rs[k].arg, bv, bi)) { bv = rs[k].maxv; bi = rs[k].arg; }
                    if (TYPICAL) merge_msa(m, s, sa, rs[k].m, rs[k].s, rs[k].a);
                }
            }
        }
        s_arg[u] = bi;
        if (TYPICAL) {
            // H = -sum P ln P = ln s - a / s  (x relative to m);  tau = min(eps, delta e^-H)
            const float H = logf(s) - sa / s;
            s_m[u] = m;
            s_s[u] = s;
            s_tau[u] = fminf(a.eps, a.delta * expf(-H));
        }
    }
    if (threadIdx.x == 0) s_best = 1023;  // node 0 (the root) unless a deeper node wins
    __syncthreads();
    // candidate tests against the parent's row
    if (u < N) {
        bool pass = true;
        if (u > 0) {
            const int pu = parent[u];
            const int tok = a.cand[(size_t)b * N + u];
            if (pu < 0 || pu >= u || tok < 0 || tok >= V) {
                pass = false;
            } else if (TYPICAL) {
                const float l = a.logits ? a.logits[((size_t)b * N + pu) * V + tok] : a.child_logit[(size_t)b * N + u];
                const float P = expf(l * a.inv_t - s_m[pu]) / s_s[pu];
                pass = P > s_tau[pu];
            } else {
                pass = tok == s_arg[pu];
            }
        }
        s_pass[u] = pass;
    }
    __syncthreads();
    // accepted iff every node on the path to the root passes; the key orders
    // nodes by (depth, -index)
    if (u < N) {
        // a node that passes has a valid parent index below its own, so the walk
        // strictly descends and ends at the root
        bool acc = true;
        int a_ = u;
        while (a_ > 0) {
            if (!s_pass[a_]) { acc = false; break; }
            a_ = parent[a_];
        }
        if (acc) atomicMax(&s_best, min(max(depth[u], 0), 1 << 20) * 1024 + (1023 - u));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int best = 1023 - (s_best & 1023);
        const int d = depth[best];
        a.accept_len[b] = d;
        a.best_node[b] = best;
        a.next_tok[b] = s_arg[best];
        int32_t* path = a.path_nodes + (size_t)b * (Dmax + 1);
        for (int e = 0; e <= Dmax; ++e) path[e] = -1;
        int a_ = best;  // every node on this path passed, so its parents are valid
        while (a_ >= 0) {
            const int da = depth[a_];
            if (da >= 0 && da <= Dmax) path[da] = a_;
            a_ = a_ > 0 ? parent[a_] : -1;
        }
    }
}

// ---------------------------------------------------------------------------
// SplitMix64 (Steele, Lea and Flood, 2014)
// ---------------------------------------------------------------------------
constexpr uint64_t kSmGamma = 0x9E3779B97F4A7C15ull;
// the output function applied to the advanced state
__device__ __forceinline__ uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
// n-th output from state: the state advanced n times by the constant, mixed
__device__ __forceinline__ uint64_t sm64(uint64_t state, uint64_t n) { return sm_mix(state + n * kSmGamma); }
__device__ __forceinline__ uint64_t row_key(uint64_t seed, uint64_t stream, uint64_t b,
                                            uint64_t round, uint64_t pos) {
    uint64_t x = sm64(seed, 1);
    x = sm64(x ^ stream, 1);
    x = sm64(x ^ b, 1);
    x = sm64(x ^ round, 1);
    return sm64(x ^ pos, 1);
}
__device__ __forceinline__ float u24(uint64_t h) { return (float)(h >> 40) * (1.0f / 16777216.0f); }
// The race's uniforms: one generator output h_m = next(key, m + 1) serves the
// vocab entries 2m (bits 40..63) and 2m + 1 (bits 16..39); U+ = (bits + 1) / 2^24.
__device__ __forceinline__ float race_u_even(uint64_t h) {
    return (float)((uint32_t)(h >> 40) + 1u) * (1.0f / 16777216.0f);
}
__device__ __forceinline__ float race_u_odd(uint64_t h) {
    return (float)(((uint32_t)(h >> 16) & 0xFFFFFFu) + 1u) * (1.0f / 16777216.0f);
}
__device__ __forceinline__ float race_u(uint64_t key, int v) {
    const uint64_t h = sm_mix(key + (uint64_t)((v >> 1) + 1) * kSmGamma);
    return (v & 1) ? race_u_odd(h) : race_u_even(h);
}

constexpr int kChainThreads = 256;
constexpr int kChainChunk = 4096;

struct ChainPart {  // per (sequence, chunk)
    float key;      // best race key
    int tok;        // its token
    float pmax;     // fallback: best p and its token
    int pidx;
};

// One warp per sequence: the first rejected position (1-based; gamma + 1 if
// every draft is accepted) and the key of the row the draw reads.  Done once
// here so the scan CTAs can start their row loads right after the wait.
__global__ void __launch_bounds__(256) chain_first_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                          const int32_t* __restrict__ draft, int B, int gamma, int V,
                                                          uint64_t seed, uint64_t round, int* __restrict__ firsts,
                                                          uint64_t* __restrict__ keys) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (b >= B) return;
    int first = gamma + 1;
    for (int i = lane; i < gamma; i += 32) {
        const int x = draft[(size_t)b * gamma + i];
        bool accept = false;
        if (x >= 0 && x < V) {
            const float qi = q[((size_t)b * gamma + i) * V + x];
            const float pi = p[((size_t)b * (gamma + 1) + i) * V + x];
            const float u = u24(sm64(row_key(seed, 1, b, round, i + 1), 1));
            // sign of u*q - p with one rounding: equals the sign of the exact value
            accept = fmaf(u, qi, -pi) < 0.f;
        }
        if (!accept) first = min(first, i + 1);
    }
    first = __reduce_min_sync(0xffffffffu, first);
    if (lane == 0) {
        const bool bonus = first > gamma;
        firsts[b] = first;
        keys[b] = row_key(seed, bonus ? 3 : 2, b, round, bonus ? gamma + 1 : first);
    }
}

__global__ void __launch_bounds__(kChainThreads) chain_scan_kernel(
    const float* __restrict__ p, const float* __restrict__ q,
    int gamma, int V, int nchunk, ChainPart* __restrict__ parts, const int* __restrict__ firsts,
    const uint64_t* __restrict__ keys) {
    pdl_wait();  // the first rejections and draw keys come from chain_first_kernel
    pdl_trigger();
    const int c = blockIdx.x, b = blockIdx.y;
    const int first = firsts[b];
    const bool bonus = first > gamma;
    const int pos = bonus ? gamma + 1 : first;          // 1-based position drawn at
    const float* pr = p + ((size_t)b * (gamma + 1) + (pos - 1)) * V;
    const float* qr = bonus ? nullptr : q + ((size_t)b * gamma + (pos - 1)) * V;
    const uint64_t key = keys[b];
    const int v0 = c * kChainChunk, v1 = min(V, v0 + kChainChunk);
    // The thread's best race key is kept as the fraction be / bw (E = -ln U+,
    // w the weight) and compared by cross-multiplication (one division per
    // thread, not per element).  On the 16-byte path the largest p is not
    // tracked: it is found by a second read of the chunk, only when no weight
    // of the chunk is positive (the scalar path tracks it, without its index).
    //
    // Pruning: once the CTA has seen keys, kb bounds its best key from above.
    // Since -ln U >= 1 - U, an element with (1 - U) > kb * w * (1 + 2^-10) has a
    // key more than 2^-11 (relative) above a key already seen: it can neither
    // win nor tie, so its logarithm and comparison are skipped (by the whole
    // warp when no lane needs them).  The margin is far above the float32
    // rounding of logf, the products and kb itself.  On the 16-byte path the
    // test reads 2^24 (1 - U) = 2^24 - 1 - bits exactly as an integer, a warp
    // votes once per group of four entries, and every lane runs every group
    // (groups past the chunk are zeros and need nothing).
    float be = INFINITY, bw = 1.f, pm = -INFINITY;
    int bt = INT_MAX;
    float kb = INFINITY;
    constexpr float kPruneMargin = 1.f + 1.f / 1024.f;
    auto take = [&](float pv, float qv, int v, float u) {
        pm = fmaxf(pm, pv);
        const float w = bonus ? pv : pv - qv;
        const bool need = w > 0.f && !(1.f - u > kb * w * kPruneMargin);
        if (__any_sync(__activemask(), need)) {
            if (need) {
                const float e = -logf(u);
                const float lhs = e * bw, rhs = be * w;
                if (lhs < rhs || (lhs == rhs && v < bt)) { be = e; bw = w; bt = v; }
            }
        }
    };
    __shared__ unsigned s_kb;
    // the CTA's best key so far (keys are >= 0: their bit patterns order as
    // unsigned integers); called by every thread
    auto refresh_bound = [&]() {
        float k = bt == INT_MAX ? INFINITY : be / bw;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) k = fminf(k, __shfl_xor_sync(0xffffffffu, k, o));
        if ((threadIdx.x & 31) == 0) atomicMin(&s_kb, __float_as_uint(k));
        __syncthreads();
        kb = __uint_as_float(s_kb);
    };
    if (threadIdx.x == 0) s_kb = __float_as_uint(INFINITY);
    __syncthreads();
    const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0 &&
                     (bonus || (reinterpret_cast<uintptr_t>(q) & 15u) == 0);
    if (vec) {
        // every 16-byte load of the chunk is issued before any element is used
        constexpr int kPer = kChainChunk / (4 * kChainThreads);
        uint4 pw[kPer], qw[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int v = v0 + 4 * (threadIdx.x + kChainThreads * k);
            pw[k] = v < v1 ? ld_stream16(pr + v) : make_uint4(0, 0, 0, 0);
            qw[k] = (v < v1 && !bonus) ? ld_stream16(qr + v) : make_uint4(0, 0, 0, 0);
        }
        // entries v..v+3 (v a multiple of 4) use the outputs m = v/2 + 1 and
        // v/2 + 2; the generator state is advanced by additions
        const uint64_t zstep = (uint64_t)(2 * kChainThreads) * kSmGamma;
        uint64_t z = key + (uint64_t)((v0 >> 1) + 2 * threadIdx.x + 1) * kSmGamma;
        float thr = INFINITY;  // 2^24 kb (1 + 2^-10)
#pragma unroll
        for (int k = 0; k < kPer; ++k, z += zstep) {
            const int v = v0 + 4 * (threadIdx.x + kChainThreads * k);
            const bool in = v < v1;
            const uint64_t h0 = sm_mix(z), h1 = sm_mix(z + kSmGamma);
            const uint32_t bits[4] = {(uint32_t)(h0 >> 40), (uint32_t)(h0 >> 16) & 0xFFFFFFu,
                                      (uint32_t)(h1 >> 40), (uint32_t)(h1 >> 16) & 0xFFFFFFu};
            const float pv[4] = {__uint_as_float(pw[k].x), __uint_as_float(pw[k].y), __uint_as_float(pw[k].z),
                                 __uint_as_float(pw[k].w)};
            const float qv[4] = {__uint_as_float(qw[k].x), __uint_as_float(qw[k].y), __uint_as_float(qw[k].z),
                                 __uint_as_float(qw[k].w)};
            float w[4];
            bool need[4], any = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[i] = bonus ? pv[i] : pv[i] - qv[i];
                need[i] = in && w[i] > 0.f && !((float)(0xFFFFFFu - bits[i]) > thr * w[i]);
                any |= need[i];
            }
            if (__any_sync(0xffffffffu, any)) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (need[i]) {
                        const float e = -logf((float)(bits[i] + 1u) * (1.0f / 16777216.0f));
                        const float lhs = e * bw, rhs = be * w[i];
                        if (lhs < rhs || (lhs == rhs && v + i < bt)) { be = e; bw = w[i]; bt = v + i; }
                    }
                }
            }
            if (k == 0) {
                refresh_bound();
                thr = kb * (16777216.f * (1.f + 1.f / 1024.f));
            }
        }
    } else {
        for (int v = v0 + threadIdx.x; v < v1; v += kChainThreads)
            take(pr[v], bonus ? 0.f : qr[v], v, race_u(key, v));
    }
    float bk = bt == INT_MAX ? INFINITY : be / bw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int ot = __shfl_xor_sync(0xffffffffu, bt, o);
        if (ok < bk || (ok == bk && ot < bt)) { bk = ok; bt = ot; }
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
    }
    __shared__ ChainPart sp[kChainThreads / 32];
    __shared__ ChainPart s_r;
    __shared__ int s_pidx;
    __shared__ float s_pm;
    if (threadIdx.x == 0) s_pm = -INFINITY;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sp[warp] = ChainPart{bk, bt, pm, INT_MAX};
    if (threadIdx.x == 0) s_pidx = INT_MAX;
    __syncthreads();
    if (threadIdx.x == 0) {
        ChainPart r = sp[0];
        for (int w = 1; w < kChainThreads / 32; ++w) {
            const ChainPart o = sp[w];
            if (o.key < r.key || (o.key == r.key && o.tok < r.tok)) { r.key = o.key; r.tok = o.tok; }
            r.pmax = fmaxf(r.pmax, o.pmax);
        }
        s_r = r;
    }
    __syncthreads();
    ChainPart r = s_r;
    if (r.tok == INT_MAX && vec) {
        // (lean path) the chunk's largest p was not tracked: find it now
        float m2 = -INFINITY;
        for (int v = v0 + threadIdx.x; v < v1; v += kChainThreads) m2 = fmaxf(m2, pr[v]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
        if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int*>(&s_pm), __float_as_int(m2));
        __syncthreads();
        r.pmax = s_pm;
    }
    if (r.tok == INT_MAX) {
        // no positive weight in this chunk: the lowest token holding its largest
        // p, for the fallback (rare; the chunk is read again)
        for (int v = v0 + threadIdx.x; v < v1; v += kChainThreads)
            if (pr[v] == r.pmax) { atomicMin(&s_pidx, v); break; }
        __syncthreads();
        r.pidx = s_pidx;
    }
    if (threadIdx.x == 0) parts[(size_t)b * nchunk + c] = r;
}

__global__ void __launch_bounds__(32) chain_finish_kernel(const ChainPart* __restrict__ parts,
                                                          const int* __restrict__ firsts,
                                                          const int32_t* __restrict__ draft,
                                                          int gamma, int nchunk,
                                                          int32_t* __restrict__ n_acc,
                                                          int32_t* __restrict__ out_tok) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, lane = threadIdx.x;
    float bk = INFINITY, pm = -INFINITY;
    int bt = INT_MAX, pi = INT_MAX;
    for (int c = lane; c < nchunk; c += 32) {
        const ChainPart r = parts[(size_t)b * nchunk + c];
        if (r.key < bk || (r.key == bk && r.tok < bt)) { bk = r.key; bt = r.tok; }
        if (better(r.pmax, r.pidx, pm, pi)) { pm = r.pmax; pi = r.pidx; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int ot = __shfl_xor_sync(0xffffffffu, bt, o);
        if (ok < bk || (ok == bk && ot < bt)) { bk = ok; bt = ot; }
        const float op = __shfl_xor_sync(0xffffffffu, pm, o);
        const int oi = __shfl_xor_sync(0xffffffffu, pi, o);
        if (better(op, oi, pm, pi)) { pm = op; pi = oi; }
    }
    const int k = firsts[b] - 1;  // accepted drafts
    const int tok = bt != INT_MAX ? bt : pi;
    for (int e = lane; e <= gamma; e += 32)
        out_tok[(size_t)b * (gamma + 1) + e] = e < k ? draft[(size_t)b * gamma + e] : (e == k ? tok : -1);
    if (lane == 0) n_acc[b] = k;
}

struct ChainPlan {
    int nchunk;
    size_t off_parts, off_first, off_keys, ws_bytes;
};
ChainPlan plan_chain(int B, int V) {
    ChainPlan p{};
    p.nchunk = (V + kChainChunk - 1) / kChainChunk;
    p.off_parts = 0;
    p.off_first = align_up((size_t)B * p.nchunk * sizeof(ChainPart), 256);
    p.off_keys = align_up(p.off_first + (size_t)B * sizeof(int), 256);
    p.ws_bytes = align_up(p.off_keys + (size_t)B * sizeof(uint64_t), 256);
    return p;
}

size_t verify_ws(int B, int N, int V) {
    const int nchunk = (V + kChunk - 1) / kChunk;
    return align_up((size_t)B * N * nchunk * sizeof(RowStat), 256);
}

// ---------------------------------------------------------------------------
// Typical acceptance with a sampled next token: after the acceptance kernel
// has picked the best node, the token after it is drawn from softmax(row / T)
// of that node by the exponential race (weights exp(x - m), x = logit / T, m
// the row maximum from the statistics; SplitMix64 row key stream 4, pos 0).
// ---------------------------------------------------------------------------
constexpr int kRaceChunk = 4096;
constexpr int kRaceThreads = 256;

struct RacePart {
    float key;
    int tok;
};

__global__ void __launch_bounds__(kRaceThreads) tree_race_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ best_node, const RowStat* __restrict__ stats,
    int N, int V, int nchunk_stats, float inv_t, uint64_t seed, uint64_t round, int nchunk,
    RacePart* __restrict__ parts) {
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, b = blockIdx.y;
    const int best = best_node[b];
    float be = INFINITY, bw = 1.f;  // best key as the fraction be / bw
    int bt = INT_MAX;
    if (best >= 0 && best < N) {
        const RowStat* st = stats + ((size_t)b * N + best) * nchunk_stats;
        float m = -INFINITY;
        for (int k = 0; k < nchunk_stats; ++k) m = fmaxf(m, st[k].m);
        const float* row = logits + ((size_t)b * N + best) * V;
        const uint64_t key = row_key(seed, 4, b, round, 0);
        const int v0 = c * kRaceChunk, v1 = min(V, v0 + kRaceChunk);
        for (int v = v0 + threadIdx.x; v < v1; v += kRaceThreads) {
            const float w = expf(row[v] * inv_t - m);
            if (w > 0.f) {
                const float e = -logf(race_u(key, v));
                const float lhs = e * bw, rhs = be * w;
                if (lhs < rhs || (lhs == rhs && v < bt)) { be = e; bw = w; bt = v; }
            }
        }
    }
    float bk = bt == INT_MAX ? INFINITY : be / bw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int ot = __shfl_xor_sync(0xffffffffu, bt, o);
        if (ok < bk || (ok == bk && ot < bt)) { bk = ok; bt = ot; }
    }
    __shared__ RacePart sp[kRaceThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sp[warp] = RacePart{bk, bt};
    __syncthreads();
    if (threadIdx.x == 0) {
        RacePart r = sp[0];
        for (int w = 1; w < kRaceThreads / 32; ++w)
            if (sp[w].key < r.key || (sp[w].key == r.key && sp[w].tok < r.tok)) r = sp[w];
        parts[(size_t)b * nchunk + c] = r;
    }
}

// One warp per sequence: the chunks' winners merged into next_tok (left as the
// argmax the acceptance kernel wrote when no weight is positive).
__global__ void __launch_bounds__(32) tree_race_finish_kernel(const RacePart* __restrict__ parts, int nchunk,
                                                              const int32_t* __restrict__ best_node, int N,
                                                              int32_t* __restrict__ next_tok) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, lane = threadIdx.x;
    float bk = INFINITY;
    int bt = INT_MAX;
    for (int c = lane; c < nchunk; c += 32) {
        const RacePart r = parts[(size_t)b * nchunk + c];
        if (r.key < bk || (r.key == bk && r.tok < bt)) { bk = r.key; bt = r.tok; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int ot = __shfl_xor_sync(0xffffffffu, bt, o);
        if (ok < bk || (ok == bk && ot < bt)) { bk = ok; bt = ot; }
    }
    const int best = best_node[b];
    if (lane == 0 && bt != INT_MAX && best >= 0 && best < N) next_tok[b] = bt;
}

constexpr int kFinishWarps = 8;

// One warp per row: lanes merge the row's split records, then a shuffle tree
// merges the lanes; for typical acceptance the same warp computes the logit of
// the row's own candidate against its parent's hidden state.
template <bool TYPICAL>
__global__ void __launch_bounds__(kFinishWarps * 32) row_finish_kernel(
    const RowStat* __restrict__ stats, int splits, int rows, int N, int V, int H,
    const uint16_t* __restrict__ hidden, const uint16_t* __restrict__ lm,
    const int32_t* __restrict__ cand, const int32_t* __restrict__ parent, RowStat* __restrict__ out,
    float* __restrict__ child_logit) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kFinishWarps + (threadIdx.x >> 5);
    // The dot product runs before the dependency wait: the statistics kernel
    // (the previous one) writes none of hidden, lm_head or cand, and it lets
    // this kernel start only after its own wait on everything before it.
    const int b = row / N, u = row - (row / N) * N;
    const uint4* x = nullptr;
    const uint4* w = nullptr;
    if (TYPICAL && row < rows && u > 0) {
        const int pu = parent[u], tok = cand[row];
        if (pu >= 0 && pu < u && tok >= 0 && tok < V) {
            x = reinterpret_cast<const uint4*>(hidden + ((size_t)b * N + pu) * H);
            w = reinterpret_cast<const uint4*>(lm + (size_t)tok * H);
        }
    }
    float dot = 0.f;
    if (x) {
        constexpr int kU = 4;
        const int h8 = H / 8;
        for (int c0 = lane; c0 < h8; c0 += 32 * kU) {
            uint4 xa[kU], wa[kU];
#pragma unroll
            for (int k = 0; k < kU; ++k) {
                const int c = c0 + 32 * k;
                xa[k] = c < h8 ? __ldg(x + c) : make_uint4(0, 0, 0, 0);
                wa[k] = c < h8 ? __ldg(w + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < kU; ++k) {
                dot = fmaf(bf16_lo(xa[k].x), bf16_lo(wa[k].x), dot);
                dot = fmaf(bf16_hi(xa[k].x), bf16_hi(wa[k].x), dot);
                dot = fmaf(bf16_lo(xa[k].y), bf16_lo(wa[k].y), dot);
                dot = fmaf(bf16_hi(xa[k].y), bf16_hi(wa[k].y), dot);
                dot = fmaf(bf16_lo(xa[k].z), bf16_lo(wa[k].z), dot);
                dot = fmaf(bf16_hi(xa[k].z), bf16_hi(wa[k].z), dot);
                dot = fmaf(bf16_lo(xa[k].w), bf16_lo(wa[k].w), dot);
                dot = fmaf(bf16_hi(xa[k].w), bf16_hi(wa[k].w), dot);
            }
        }
        dot = warp_sum(dot);
    }
    pdl_wait();
    pdl_trigger();
    if (row >= rows) return;
    if (TYPICAL && lane == 0) child_logit[row] = x ? dot : __int_as_float(0x7fc00000);
    float bv = -INFINITY, m = -INFINITY, s = 0.f, sa = 0.f;
    int bi = INT_MAX;
    const RowStat* st = stats + (size_t)row * splits;
#pragma unroll 4
    for (int c = lane; c < splits; c += 32) {
        const RowStat r = st[c];
        if (better(r.maxv, r.arg, bv, bi)) { bv = r.maxv; bi = r.arg; }
        if (TYPICAL) merge_msa(m, s, sa, r.m, r.s, r.a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        if (TYPICAL) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const float os = __shfl_xor_sync(0xffffffffu, s, o);
            const float oa = __shfl_xor_sync(0xffffffffu, sa, o);
            merge_msa(m, s, sa, om, os, oa);
        }
    }
    if (lane == 0) {
        RowStat r;
        r.maxv = bv;
        r.arg = bi;
        r.m = m;
        r.s = s;
        r.a = sa;
        r.pad[0] = r.pad[1] = r.pad[2] = 0.f;
        out[row] = r;
    }
}

}  // namespace

int launch_row_finish(bool typical, const RowStat* stats, int splits, int rows, int N, int V, int H,
                      const uint16_t* hidden, const uint16_t* lm, const int32_t* cand,
                      const int32_t* parent, RowStat* out, float* child_logit, cudaStream_t st) {
    auto k = typical ? row_finish_kernel<true> : row_finish_kernel<false>;
    const int grid = (rows + kFinishWarps - 1) / kFinishWarps;
    cudaError_t e = launch(k, dim3(grid), dim3(kFinishWarps * 32), 0, st, stats, splits, rows, N, V, H,
                           hidden, lm, cand, parent, out, child_logit);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "row_finish: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

int launch_accept_tree(bool typical, const AcceptArgs& a, cudaStream_t st) {
    auto k = typical ? accept_tree_kernel<true> : accept_tree_kernel<false>;
    cudaError_t e = launch(k, dim3(a.B), dim3(kAcceptThreads), 0, st, a);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "accept_tree: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

}  // namespace medusa

using namespace medusa;

extern "C" size_t medusa_verify_accept_workspace(int B, int N, int V) {
    if (B < 1 || N < 1 || V < 1) return 0;
    return verify_ws(B, N, V);
}

extern "C" int medusa_verify_accept_tree(const float* logits, const int32_t* cand,
                                         const int32_t* parent, const int32_t* depth, int B, int N,
                                         int V, int Dmax, medusa_accept_mode mode,
                                         float temperature, float eps, float delta,
                                         int32_t* accept_len, int32_t* best_node,
                                         int32_t* path_nodes, int32_t* next_tok, void* ws,
                                         size_t ws_bytes, void* stream) {
    if (!logits || !cand || !parent || !depth || !accept_len || !best_node || !path_nodes ||
        !next_tok)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree: null pointer");
    if (B < 1 || N < 1 || V < 1 || Dmax < 0)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree: bad sizes");
    if (N > kAcceptThreads || B > 65535)
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_accept_tree: N=%d above %d", N, kAcceptThreads);
    if (mode != MEDUSA_ACCEPT_GREEDY && mode != MEDUSA_ACCEPT_TYPICAL)
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_accept_tree: unknown mode %d", (int)mode);
    if (mode == MEDUSA_ACCEPT_TYPICAL && !(temperature > 0.f))
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree: temperature must be > 0");
    const size_t need = verify_ws(B, N, V);
    if (!ws || ws_bytes < need)
        return fail(MEDUSA_ERR_WORKSPACE, "verify_accept_tree: workspace of %zu bytes needed, %zu given",
                    need, ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree: ws must be 16-byte aligned");
    const int nchunk = (V + kChunk - 1) / kChunk;
    if ((long long)B * N > 65535)
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_accept_tree: B*N above 65535");
    RowStat* stats = static_cast<RowStat*>(ws);
    cudaStream_t st = as_stream(stream);
    const float inv_t = 1.f / temperature;
    dim3 g1(nchunk, B * N);
    cudaError_t e;
    if (mode == MEDUSA_ACCEPT_TYPICAL)
        e = launch(row_stats_kernel<true>, g1, dim3(kStatThreads), 0, st, logits, V, nchunk, inv_t, stats);
    else
        e = launch(row_stats_kernel<false>, g1, dim3(kStatThreads), 0, st, logits, V, nchunk, inv_t, stats);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "row_stats: launch failed: %s", cudaGetErrorString(e));
    AcceptArgs aa{};
    aa.logits = logits;
    aa.cand = cand;
    aa.parent = parent;
    aa.depth = depth;
    aa.B = B;
    aa.N = N;
    aa.V = V;
    aa.Dmax = Dmax;
    aa.nchunk = nchunk;
    aa.inv_t = inv_t;
    aa.eps = eps;
    aa.delta = delta;
    aa.stats = stats;
    aa.accept_len = accept_len;
    aa.best_node = best_node;
    aa.path_nodes = path_nodes;
    aa.next_tok = next_tok;
    return launch_accept_tree(mode == MEDUSA_ACCEPT_TYPICAL, aa, st);
}

extern "C" size_t medusa_verify_sample_workspace(int B, int N, int V) {
    if (B < 1 || N < 1 || V < 1) return 0;
    const int nrace = (V + kRaceChunk - 1) / kRaceChunk;
    return align_up(verify_ws(B, N, V) + (size_t)B * nrace * sizeof(RacePart), 256);
}

extern "C" int medusa_verify_accept_tree_sample(const float* logits, const int32_t* cand,
                                                const int32_t* parent, const int32_t* depth, int B, int N,
                                                int V, int Dmax, float temperature, float eps, float delta,
                                                uint64_t seed, uint64_t round, int32_t* accept_len,
                                                int32_t* best_node, int32_t* path_nodes,
                                                int32_t* next_tok, void* ws, size_t ws_bytes,
                                                void* stream) {
    if (!logits || !cand || !parent || !depth || !accept_len || !best_node || !path_nodes || !next_tok)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree_sample: null pointer");
    if (B < 1 || N < 1 || V < 1 || Dmax < 0)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree_sample: bad sizes");
    if (N > kAcceptThreads || B > 65535 || (long long)B * N > 65535)
        return fail(MEDUSA_ERR_UNSUPPORTED, "verify_accept_tree_sample: N=%d above %d or B*N above 65535", N,
                    kAcceptThreads);
    if (!(temperature > 0.f))
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree_sample: temperature must be > 0");
    const size_t need = medusa_verify_sample_workspace(B, N, V);
    if (!ws || ws_bytes < need)
        return fail(MEDUSA_ERR_WORKSPACE, "verify_accept_tree_sample: workspace of %zu bytes needed, %zu given",
                    need, ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_tree_sample: ws must be 16-byte aligned");
    int rc = medusa_verify_accept_tree(logits, cand, parent, depth, B, N, V, Dmax, MEDUSA_ACCEPT_TYPICAL,
                                       temperature, eps, delta, accept_len, best_node, path_nodes, next_tok, ws,
                                       ws_bytes, stream);
    if (rc) return rc;
    const int nstat = (V + kChunk - 1) / kChunk;
    const int nrace = (V + kRaceChunk - 1) / kRaceChunk;
    RacePart* parts = reinterpret_cast<RacePart*>(static_cast<char*>(ws) + verify_ws(B, N, V));
    cudaStream_t st = as_stream(stream);
    cudaError_t e = launch(tree_race_kernel, dim3(nrace, B), dim3(kRaceThreads), 0, st, logits,
                           (const int32_t*)best_node, (const RowStat*)ws, N, V, nstat, 1.f / temperature, seed,
                           round, nrace, parts);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "tree_race: launch failed: %s", cudaGetErrorString(e));
    e = launch(tree_race_finish_kernel, dim3(B), dim3(32), 0, st, (const RacePart*)parts, nrace,
               (const int32_t*)best_node, N, next_tok);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "tree_race_finish: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}

extern "C" size_t medusa_verify_chain_workspace(int B, int gamma, int V) {
    if (B < 1 || gamma < 0 || V < 1) return 0;
    return plan_chain(B, V).ws_bytes;
}

extern "C" int medusa_verify_accept_chain(const float* p, const float* q, const int32_t* draft,
                                          int B, int gamma, int V, uint64_t seed, uint64_t round,
                                          int32_t* n_acc, int32_t* out_tok, void* ws,
                                          size_t ws_bytes, void* stream) {
    if (!p || (gamma > 0 && (!q || !draft)) || !n_acc || !out_tok)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_chain: null pointer");
    if (B < 1 || gamma < 0 || V < 1 || B > 65535)
        return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_chain: bad sizes");
    ChainPlan plan = plan_chain(B, V);
    if (!ws || ws_bytes < plan.ws_bytes)
        return fail(MEDUSA_ERR_WORKSPACE, "verify_accept_chain: workspace of %zu bytes needed, %zu given",
                    plan.ws_bytes, ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(MEDUSA_ERR_INVALID_ARG, "verify_accept_chain: ws must be 16-byte aligned");
    ChainPart* parts = reinterpret_cast<ChainPart*>(static_cast<char*>(ws) + plan.off_parts);
    int* firsts = reinterpret_cast<int*>(static_cast<char*>(ws) + plan.off_first);
    uint64_t* keys = reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + plan.off_keys);
    cudaStream_t st = as_stream(stream);
    cudaError_t e = launch(chain_first_kernel, dim3((B + 7) / 8), dim3(256), 0, st, p, q, draft, B, gamma, V,
                           seed, round, firsts, keys);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "chain_first: launch failed: %s", cudaGetErrorString(e));
    e = launch(chain_scan_kernel, dim3(plan.nchunk, B), dim3(kChainThreads), 0, st, p, q, gamma, V, plan.nchunk,
               parts, (const int*)firsts, (const uint64_t*)keys);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "chain_scan: launch failed: %s", cudaGetErrorString(e));
    e = launch(chain_finish_kernel, dim3(B), dim3(32), 0, st, (const ChainPart*)parts,
               (const int*)firsts, draft, gamma, plan.nchunk, n_acc, out_tok);
    if (e != cudaSuccess) return fail(MEDUSA_ERR_CUDA, "chain_finish: launch failed: %s", cudaGetErrorString(e));
    return MEDUSA_OK;
}
