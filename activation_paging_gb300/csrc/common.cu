// Status strings, per-thread error messages and device queries.
#include <stdarg.h>
#include <stdio.h>

#include <stdlib.h>
#include <string.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "ap_common.cuh"

namespace ap {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

ap_status fail(ap_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

ap_status cuda_fail(cudaError_t e, const char *what)
{
    set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    return AP_ECUDA;
}

static nvtxDomainHandle_t nvtx_domain()
{
    // created once, on first use; nullptr when AP_NVTX=0
    static const nvtxDomainHandle_t d = [] {
        const char *env = getenv("AP_NVTX");
        if (env && strcmp(env, "0") == 0) return (nvtxDomainHandle_t) nullptr;
        return nvtxDomainCreateA("activation_paging");
    }();
    return d;
}

NvtxRange::NvtxRange(const char *name) : on_(false)
{
    nvtxDomainHandle_t d = nvtx_domain();
    if (!d) return;
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(d, &a);
    on_ = true;
}

NvtxRange::~NvtxRange()
{
    if (on_) nvtxDomainRangePop(nvtx_domain());
}

static std::atomic<uint64_t> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

int resident_grid(const void *kernel, int threads, size_t smem)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    return per_sm * sm_count();
}

} // namespace ap

extern "C" const char *ap_status_str(ap_status s)
{
    switch (s) {
    case AP_OK: return "AP_OK";
    case AP_EINVAL: return "AP_EINVAL";
    case AP_EEMPTY: return "AP_EEMPTY";
    case AP_EQFULL: return "AP_EQFULL";
    case AP_ECUDA: return "AP_ECUDA";
    case AP_ESTREAM: return "AP_ESTREAM";
    case AP_ENOTSUP: return "AP_ENOTSUP";
    default: return "AP_UNKNOWN";
    }
}

extern "C" const char *ap_last_error(void) { return ap::g_err; }

extern "C" const char *ap_version(void) { return "0.1.0"; }

extern "C" uint64_t ap_launch_count(void) { return ap::g_launches.load(std::memory_order_relaxed); }
