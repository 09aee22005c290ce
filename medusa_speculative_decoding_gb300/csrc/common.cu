// common.cu -- status messages, cached device properties, the tensor-map encoder.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "tmap.cuh"

namespace medusa {

static thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MEDUSA_ERR_CUDA, "%s: kernel launch failed: %s", what, cudaGetErrorString(e));
    return MEDUSA_OK;
}

namespace {
constexpr int kMaxDev = 64;
int g_sms[kMaxDev];
int g_smem[kMaxDev];
std::mutex g_mu;

int current_dev() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return 0;
    return d;
}
}  // namespace

int sm_count() {
    int d = current_dev();
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[d] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0)
            v = 148;
        g_sms[d] = v;
    }
    return g_sms[d];
}

int max_smem_optin() {
    int d = current_dev();
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem[d] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess ||
            v <= 0)
            v = 48 * 1024;
        g_smem[d] = v;
    }
    return g_smem[d];
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

int current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return fail(MEDUSA_ERR_CUDA, "the driver lacks cuCtxGetCurrent or cuCtxGetId");
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return fail(MEDUSA_ERR_CUDA, "cuCtxGetCurrent failed");
    *id = 0;  // no context is current yet
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return fail(MEDUSA_ERR_CUDA, "cuCtxGetId failed");
    return MEDUSA_OK;
}

namespace {
struct WaitControl {
    int (*read_clear)(int*, cudaStream_t);
    int (*set_limit)(long long);
};
std::mutex g_wc_mu;
// function-local statics: registration runs during static initialisation of
// the other translation units, whose order is unspecified
WaitControl* wait_controls() {
    static WaitControl tab[8];
    return tab;
}
int& wait_control_count() {
    static int count = 0;
    return count;
}
}  // namespace

void register_wait_control(int (*read_clear)(int*, cudaStream_t), int (*set_limit)(long long)) {
    std::lock_guard<std::mutex> lk(g_wc_mu);
    int& n = wait_control_count();
    if (n < 8) wait_controls()[n++] = WaitControl{read_clear, set_limit};
}

int wait_controls_read_clear(int* gave_up, cudaStream_t st) {
    std::lock_guard<std::mutex> lk(g_wc_mu);
    const int n = wait_control_count();
    for (int i = 0; i < n; ++i) {
        const int e = wait_controls()[i].read_clear(gave_up, st);
        if (e) return fail(MEDUSA_ERR_CUDA, "device status: %s", cudaGetErrorString((cudaError_t)e));
    }
    return MEDUSA_OK;
}

int wait_controls_set_limit(long long cycles) {
    std::lock_guard<std::mutex> lk(g_wc_mu);
    const int n = wait_control_count();
    for (int i = 0; i < n; ++i) {
        const int e = wait_controls()[i].set_limit(cycles);
        if (e) return fail(MEDUSA_ERR_CUDA, "set_wait_limit: %s", cudaGetErrorString((cudaError_t)e));
    }
    return MEDUSA_OK;
}

}  // namespace medusa

extern "C" int medusa_device_status(void* stream) {
    cudaStream_t st = medusa::as_stream(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return medusa::fail(MEDUSA_ERR_CUDA, "device_status: the stream failed: %s", cudaGetErrorString(e));
    int gave_up = 0;
    int rc = medusa::wait_controls_read_clear(&gave_up, st);
    if (rc) return rc;
    if (gave_up)
        return medusa::fail(MEDUSA_ERR_TIMEOUT,
                            "device_status: a bounded device wait gave up; the outputs of the calls it "
                            "belonged to are marked (NaN or -1)");
    return MEDUSA_OK;
}

extern "C" int medusa_set_wait_limit(long long cycles) { return medusa::wait_controls_set_limit(cycles); }

extern "C" const char* medusa_last_error(void) { return medusa::g_msg; }
extern "C" int medusa_abi_version(void) { return 1; }
