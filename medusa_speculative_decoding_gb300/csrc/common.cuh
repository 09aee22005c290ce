// common.cuh -- shared helpers of libmedusa_gb300 (status handling, device
// properties, bf16 decoding, warp reductions, streaming loads).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "medusa.h"

namespace medusa {

// Records a message for medusa_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
// Checks the launch that was just enqueued; returns MEDUSA_OK or MEDUSA_ERR_CUDA.
int check_launch(const char* what);
// Number of SMs of the current device (cached per device).
int sm_count();
// Unique ID (for the life of the process) of the calling thread's current CUDA
// context, or 0 when no context is current yet.
int current_context_id(unsigned long long* id);
// Opt-in maximum dynamic shared memory per block of the current device.
int max_smem_optin();

// ---------------------------------------------------------------------------
// Bounded device waits.  Every mbarrier wait of the tensor-core kernels gives
// up after a limit (about one second by default).  A kernel whose wait gave up
// first lets its own copies and MMAs in flight complete (those drain waits keep
// the default limit), frees its tensor memory, marks its outputs and sets the
// give-up word of its translation unit; medusa_device_status() reads and
// clears the words.  The limit of the first waits can be lowered through
// medusa_set_wait_limit() (a test hook that makes the waits run out on
// purpose).  Each .cu file with such kernels defines its own words with
// MEDUSA_WAIT_CONTROL() and registers a reader and a setter here.
constexpr long long kDefaultWaitCycles = 1ll << 31;  // ~1 s at 2 GHz
void register_wait_control(int (*read_clear)(int* gave_up, cudaStream_t st), int (*set_limit)(long long cycles));
int wait_controls_read_clear(int* gave_up, cudaStream_t st);
int wait_controls_set_limit(long long cycles);

#define MEDUSA_WAIT_CONTROL()                                                                              \
    __device__ int g_wait_gave_up = 0;                                                                     \
    __device__ long long g_wait_limit = ::medusa::kDefaultWaitCycles;                                      \
    int wait_read_clear(int* gave_up, cudaStream_t st) {                                                   \
        static const int zero = 0;                                                                         \
        int v = 0;                                                                                         \
        cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_wait_gave_up, sizeof v, 0, cudaMemcpyDeviceToHost, st); \
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);                                               \
        if (e == cudaSuccess && v)                                                                         \
            e = cudaMemcpyToSymbolAsync(g_wait_gave_up, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st); \
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);                                               \
        if (e != cudaSuccess) return (int)e;                                                               \
        *gave_up = *gave_up || v != 0;                                                                     \
        return 0;                                                                                          \
    }                                                                                                      \
    int wait_set_limit(long long cycles) {                                                                 \
        const long long v = cycles > 0 ? cycles : ::medusa::kDefaultWaitCycles;                            \
        return (int)cudaMemcpyToSymbol(g_wait_limit, &v, sizeof v);                                        \
    }                                                                                                      \
    const bool g_wait_registered = (::medusa::register_wait_control(wait_read_clear, wait_set_limit), true);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization allowed (see pdl_wait below).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Same, with thread-block clusters of (cluster_x, 1, 1) CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                           unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16-byte load that bypasses L1 (weights and caches are streamed once per step).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization, so it may be scheduled while the previous
// kernel on the stream is still running; it calls pdl_wait() before it touches
// anything an earlier kernel wrote (the wait returns once those grids have
// completed and their writes are visible; without the launch attribute it
// returns at once).  pdl_trigger() lets the next kernel's CTAs be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// L2 prefetch of [p, p + bytes) through the bulk-copy unit (no register or shared
// memory destination).  p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// (value, index) order used by every top-k and argmax here: larger value
// first, lower index first among equal values.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

}  // namespace medusa
