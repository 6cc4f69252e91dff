// SM partitions for the reload-overlap measurement of bench.py (green
// contexts).  Not part of the library (libap.so) or its ABI: it is built into
// libap_bench.so.
//
// A green context is a partition of the device's primary context that owns a
// set of SMs; kernels launched into one of its streams run only on those SMs,
// and it shares the primary context's memory.  apb_green_split makes two
// disjoint partitions, one of at least n SMs (for the paging stream) and one
// of the SMs left, and a stream in each; the pool's paging stream can be the
// first and the compute the second, so reloads and compute never wait for
// each other's blocks.  The driver's calls are reached through the runtime's
// driver entry-point query (no link against the driver library).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

struct Green {
    int missing = 0; // 1 + index of the first entry point the driver lacks, or 0
    CUresult (*device_get)(CUdevice *, int) = nullptr;
    CUresult (*get_resource)(CUdevice, CUdevResource *, CUdevResourceType) = nullptr;
    CUresult (*split)(CUdevResource *, unsigned int *, const CUdevResource *, CUdevResource *, unsigned int,
                      unsigned int) = nullptr;
    CUresult (*gen_desc)(CUdevResourceDesc *, CUdevResource *, unsigned int) = nullptr;
    CUresult (*ctx_create)(CUgreenCtx *, CUdevResourceDesc, CUdevice, unsigned int) = nullptr;
    CUresult (*ctx_destroy)(CUgreenCtx) = nullptr;
    CUresult (*stream_create)(CUstream *, CUgreenCtx, unsigned int, int) = nullptr;
    CUresult (*stream_destroy)(CUstream) = nullptr;
    bool ok = false;
};

// Entry points at the ABI of the header this file is compiled with.
template <typename F>
bool entry(const char *name, F *fn)
{
    const int version = CUDA_VERSION;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
        (void)cudaGetLastError();
        return false;
    }
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Green &green()
{
    static Green g;
    static std::once_flag once;
    std::call_once(once, [] {
        const bool found[] = {entry("cuDeviceGet", &g.device_get),
                              entry("cuDeviceGetDevResource", &g.get_resource),
                              entry("cuDevSmResourceSplitByCount", &g.split),
                              entry("cuDevResourceGenerateDesc", &g.gen_desc),
                              entry("cuGreenCtxCreate", &g.ctx_create),
                              entry("cuGreenCtxDestroy", &g.ctx_destroy),
                              entry("cuGreenCtxStreamCreate", &g.stream_create),
                              entry("cuStreamDestroy", &g.stream_destroy)};
        g.ok = true;
        for (int i = 0; i < (int)(sizeof(found) / sizeof(found[0])); ++i)
            if (!found[i] && g.ok) {
                g.ok = false;
                g.missing = i + 1;
            }
    });
    return g;
}

} // namespace

// Two disjoint SM partitions of `device` and a stream in each.  n_small: the
// fewest SMs the first partition may have (the driver rounds up to its
// partition granularity).  Outputs: the two streams (cudaStream_t), the SM
// count of each, and the two green contexts (for apb_green_destroy).  The
// first stream gets the device's highest stream priority.  Returns 0, -i when
// the driver lacks the i-th entry point this file uses (1: cuDeviceGet ... 8:
// cuStreamDestroy), or a CUDA driver error code.
extern "C" int apb_green_split(int device, int n_small, void **stream_small, void **stream_rest, int *sm_small,
                               int *sm_rest, void **ctx_small, void **ctx_rest)
{
    const Green &g = green();
    if (!g.ok) return -g.missing;
    if (!stream_small || !stream_rest || !sm_small || !sm_rest || !ctx_small || !ctx_rest || n_small < 1)
        return (int)CUDA_ERROR_INVALID_VALUE;
    *stream_small = *stream_rest = *ctx_small = *ctx_rest = nullptr;
    if (cudaSetDevice(device) != cudaSuccess || cudaFree(nullptr) != cudaSuccess) // primary context current
        return (int)CUDA_ERROR_INVALID_DEVICE;
    CUdevice dev;
    CUresult r = g.device_get(&dev, device);
    if (r != CUDA_SUCCESS) return (int)r;
    CUdevResource all = {}, part = {}, rest = {};
    r = g.get_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM);
    if (r != CUDA_SUCCESS) return (int)r;
    unsigned int ngroups = 1;
    r = g.split(&part, &ngroups, &all, &rest, 0, (unsigned int)n_small);
    if (r != CUDA_SUCCESS) return (int)r;
    if (ngroups != 1 || rest.sm.smCount == 0) return (int)CUDA_ERROR_INVALID_RESOURCE_CONFIGURATION;
    CUdevResourceDesc d_small, d_rest;
    if ((r = g.gen_desc(&d_small, &part, 1)) != CUDA_SUCCESS) return (int)r;
    if ((r = g.gen_desc(&d_rest, &rest, 1)) != CUDA_SUCCESS) return (int)r;
    CUgreenCtx c_small = nullptr, c_rest = nullptr;
    if ((r = g.ctx_create(&c_small, d_small, dev, CU_GREEN_CTX_DEFAULT_STREAM)) != CUDA_SUCCESS) return (int)r;
    if ((r = g.ctx_create(&c_rest, d_rest, dev, CU_GREEN_CTX_DEFAULT_STREAM)) != CUDA_SUCCESS) {
        g.ctx_destroy(c_small);
        return (int)r;
    }
    int lo = 0, hi = 0;
    (void)cudaDeviceGetStreamPriorityRange(&lo, &hi);
    CUstream s_small = nullptr, s_rest = nullptr;
    r = g.stream_create(&s_small, c_small, CU_STREAM_NON_BLOCKING, hi);
    if (r == CUDA_SUCCESS) r = g.stream_create(&s_rest, c_rest, CU_STREAM_NON_BLOCKING, 0);
    if (r != CUDA_SUCCESS) {
        if (s_small) g.stream_destroy(s_small);
        g.ctx_destroy(c_small);
        g.ctx_destroy(c_rest);
        return (int)r;
    }
    *stream_small = s_small;
    *stream_rest = s_rest;
    *sm_small = (int)part.sm.smCount;
    *sm_rest = (int)rest.sm.smCount;
    *ctx_small = c_small;
    *ctx_rest = c_rest;
    return 0;
}

// Destroys what apb_green_split made (after the caller synchronised the
// streams).  Returns 0 or the first driver error.
extern "C" int apb_green_destroy(void *stream_small, void *stream_rest, void *ctx_small, void *ctx_rest)
{
    const Green &g = green();
    if (!g.ok) return -1;
    int rc = 0;
    CUresult r;
    if (stream_small && (r = g.stream_destroy((CUstream)stream_small)) != CUDA_SUCCESS && !rc) rc = (int)r;
    if (stream_rest && (r = g.stream_destroy((CUstream)stream_rest)) != CUDA_SUCCESS && !rc) rc = (int)r;
    if (ctx_small && (r = g.ctx_destroy((CUgreenCtx)ctx_small)) != CUDA_SUCCESS && !rc) rc = (int)r;
    if (ctx_rest && (r = g.ctx_destroy((CUgreenCtx)ctx_rest)) != CUDA_SUCCESS && !rc) rc = (int)r;
    return rc;
}
