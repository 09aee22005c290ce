// topk.cuh -- warp-level top-k selection shared by the heads kernels.
#pragma once

#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace medusa {

// Selects, in `passes` rounds, the best remaining (value, index) pair among
// n entries given by get(j) -> (value, index); one warp.  Writes through put().
template <typename Get, typename Put>
__device__ __forceinline__ void warp_select_topk(int n, int passes, Get get, Put put, int lane) {
    float lastv = INFINITY;
    int lasti = -1;
    for (int t = 0; t < passes; ++t) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int j = lane; j < n; j += 32) {
            float x;
            int xi;
            get(j, x, xi);
            if (better(lastv, lasti, x, xi) && better(x, xi, bv, bi)) { bv = x; bi = xi; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) put(t, bv, bi);
        lastv = bv;
        lasti = bi;
    }
}

// Same result as warp_select_topk (passes <= MAXK), for n entries that live in
// global memory: every entry is read once.  Each lane keeps the best MAXK of
// its own entries in a sorted register list; then `passes` rounds pick the best
// list head across the warp and pop it.  (value, index) pairs must be distinct.
template <int MAXK, typename Get, typename Put>
__device__ __forceinline__ void warp_merge_topk(int n, int passes, Get get, Put put, int lane) {
    float lv[MAXK];
    int li[MAXK];
#pragma unroll
    for (int e = 0; e < MAXK; ++e) { lv[e] = -INFINITY; li[e] = INT_MAX; }
    constexpr int kBatch = 4;
    for (int j0 = lane; j0 < n; j0 += 32 * kBatch) {
        float xv[kBatch];
        int xi[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {  // independent loads first
            const int j = j0 + 32 * u;
            if (j < n) get(j, xv[u], xi[u]);
            else { xv[u] = -INFINITY; xi[u] = INT_MAX; }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float x = xv[u];
            int xx = xi[u];
            // insert (x, xx) into the sorted list, dropping the last
#pragma unroll
            for (int e = 0; e < MAXK; ++e) {
                if (better(x, xx, lv[e], li[e])) {
                    const float tv = lv[e];
                    const int ti = li[e];
                    lv[e] = x;
                    li[e] = xx;
                    x = tv;
                    xx = ti;
                }
            }
        }
    }
    for (int t = 0; t < passes; ++t) {
        float bv = lv[0];
        int bi = li[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) put(t, bv, bi);
        if (lv[0] == bv && li[0] == bi) {  // the winner's lane pops its head
#pragma unroll
            for (int e = 0; e + 1 < MAXK; ++e) { lv[e] = lv[e + 1]; li[e] = li[e + 1]; }
            lv[MAXK - 1] = -INFINITY;
            li[MAXK - 1] = INT_MAX;
        }
    }
}

}  // namespace medusa
