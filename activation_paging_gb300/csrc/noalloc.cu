// Dispatch for callers that cannot allocate device memory.
//
// ap_dispatch_permute needs a small device work space (per-block expert
// histograms).  Some callers cannot provide one: code running where every
// byte of the GPU is already reserved by another allocator, real-time or
// replay loops that must not enter cudaMalloc (which can synchronise the
// device and take a global lock), and embedders whose memory budget is fixed
// at start-up.  This entry point uses a fixed work space that lives in the
// library itself instead: a file-scope device array, loaded with the module,
// that each GPU holds until the process exits.
#include <cuda.h>

#include <mutex>

#include "ap_common.cuh"

namespace ap {
namespace {

constexpr int64_t kStaticScratchBytes = AP_DISPATCH_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The shared work space.  Host code must not pass `g_dispatch_scratch` itself
// to a kernel: on the host that name is only a stand-in, not a device address.
static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchBytes / sizeof(int32_t)];

// The driver's context queries, reached through the runtime's entry-point
// query (no link against the driver library).
struct CtxApi {
    CUresult (*current)(CUcontext *) = nullptr;
    CUresult (*id)(CUcontext, unsigned long long *) = nullptr;
};

const CtxApi &ctx_api()
{
    static CtxApi api;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
            r1 == cudaDriverEntryPointSuccess && r2 == cudaDriverEntryPointSuccess && p && q) {
            api.current = reinterpret_cast<CUresult (*)(CUcontext *)>(p);
            api.id = reinterpret_cast<CUresult (*)(CUcontext, unsigned long long *)>(q);
        } else {
            (void)cudaGetLastError();
        }
    });
    return api;
}

// Process-unique id of the calling thread's current context, or 0 when none
// is current or the query is unavailable.
unsigned long long current_context_id()
{
    const CtxApi &api = ctx_api();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!api.current || api.current(&c) != CUDA_SUCCESS || !c || api.id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

std::mutex g_mu;
struct Cached {
    void *addr = nullptr;
    unsigned long long ctx = 0; // the context the address belongs to
};
Cached g_addr[kMaxDevices];

// Device address of the work space on the current device.  It is looked up
// (with that device current) on the first call, and again whenever the
// current context is not the one it was looked up in: after cudaDeviceReset
// the device's module is loaded anew, so an address cached before would be
// dead.
ap_status scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "dispatch_permute_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(AP_ENOTSUP, "dispatch_permute_noalloc: device %d unsupported", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    Cached &c = g_addr[dev];
    const unsigned long long ctx = current_context_id();
    if (!c.addr || ctx == 0 || ctx != c.ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess || !p) {
            c = Cached{};
            return cuda_fail(e, "dispatch_permute_noalloc: cudaGetSymbolAddress");
        }
        c.addr = p;
        c.ctx = current_context_id(); // the lookup made the device's context current
    }
    *out = c.addr;
    return AP_OK;
}

} // namespace
} // namespace ap

extern "C" ap_status ap_dispatch_permute_noalloc(const void *x, int64_t T, int32_t H, const int32_t *idx, int32_t k,
                                                 int32_t E, int32_t capacity, int32_t padded, int32_t out_dtype,
                                                 void *xd, float *xd_scale, int64_t xd_rows, int32_t *counts,
                                                 int32_t *live, int32_t *seg_off, int32_t *dest, int32_t *src_tok,
                                                 uint32_t *d_status, void *stream)
{
    AP_NVTX_RANGE("ap_dispatch_permute_noalloc");
    using namespace ap;
    int64_t need = 0;
    ap_status s = ap_dispatch_scratch_bytes(T, k, E, &need);
    if (s != AP_OK) return s;
    if (need > kStaticScratchBytes)
        return fail(AP_EINVAL,
                    "dispatch_permute_noalloc: needs %lld bytes of work space for T=%lld k=%d E=%d, more than the "
                    "built-in %lld; use ap_dispatch_permute with caller-provided scratch",
                    (long long)need, (long long)T, k, E, (long long)kStaticScratchBytes);
    void *scratch = nullptr;
    s = scratch_address(&scratch);
    if (s != AP_OK) return s;
    // The work space needs no clearing: every entry the kernels read is first
    // written by the same call's count kernel.
    return ap_dispatch_permute(x, T, H, idx, k, E, capacity, padded, out_dtype, xd, xd_scale, xd_rows, counts, live,
                               seg_off, dest, src_tok, scratch, kStaticScratchBytes, d_status, stream);
}
