// gemm_no_alloc.cu -- om_gemm_f32_no_alloc: the balanced-schedule product
// (om_gemm_f32_ws) for callers that cannot allocate device memory.
//
// The balanced schedule needs one flag word per SM of scratch. Here that
// scratch is a fixed array in static device memory that every GPU loading the
// library holds until the process exits, so the caller passes only its
// inputs and outputs and nothing is allocated per call.
#include <mutex>

#include "om.h"
#include "om_internal.h"

namespace {

// A workspace's worth of words (4 KiB): the schedule's flags, one per SM,
// and the word a caller workspace keeps its status in (unused here).
constexpr int kNoAllocFlagWords = om::kWorkspaceWords;

static __device__ __align__(256) unsigned g_no_alloc_flags[kNoAllocFlagWords];

// Device address of g_no_alloc_flags, per device and per context. In host
// code the array's name is only a host-side stand-in, so the address is
// looked up with the device current and the kernel is given that address.
// The cache is keyed on the current context as well as the device index: a
// new context on the same device (after cudaDeviceReset, or another context
// made current through the driver) maps the array anew, so its address is
// looked up again.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_flags_addr[kMaxDevices] = {};
void *g_flags_ctx[kMaxDevices] = {};

typedef int (*CtxGetCurrentFn)(void **);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    }
    return fn;
}

int flags_on_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return OM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return OM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    void *ctx = nullptr;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    // Without the driver query every call looks the address up afresh.
    const bool have_ctx = get_ctx != nullptr && get_ctx(&ctx) == 0 && ctx != nullptr;
    if (g_flags_addr[dev] == nullptr || !have_ctx || g_flags_ctx[dev] != ctx) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_no_alloc_flags) != cudaSuccess || addr == nullptr)
            return OM_ERR_CUDA;
        g_flags_addr[dev] = addr;
        g_flags_ctx[dev] = have_ctx ? ctx : nullptr;
    }
    *out = g_flags_addr[dev];
    return OM_OK;
}

}  // namespace

extern "C" int om_gemm_f32_no_alloc(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda,
                                    const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                                    void *stream) {
    // The schedule uses one flag per SM; a device with more SMs than the
    // static array has words is beyond what this entry point supports.
    if (om::num_sms() > om::kMaxScheduleCtas) return OM_ERR_TOO_LARGE;
    void *flags = nullptr;
    const int st = flags_on_current_device(&flags);
    if (st != OM_OK) return st;
    // The kernel launch path clears the flags it uses on stream before the
    // kernel runs (the array keeps whatever the previous call left).
    return om::gemm_with_scratch(m, n, k, A, lda, B, ldb, C, ldc, mode, flags,
                                 sizeof(unsigned) * kNoAllocFlagWords, stream);
}
