// Growable device arena: reserved device addresses whose prefix is backed by
// physical memory on demand (CUDA virtual memory management).
//
// Megatron-LM pull 7342, "Summary": the activation arena's capacity grows
// lazily.  Growing in place keeps every page of a pool at its address, so a
// pool can take more pages while records still hold the old ones, and no page
// is ever copied to a new buffer.
//
// The driver's virtual-memory calls are reached through the runtime's
// driver entry-point query, so the library needs no link against the driver
// library (it still loads on a machine without a GPU).
#include <cuda.h>

#include <mutex>
#include <new>
#include <vector>

#include "ap_common.cuh"

namespace {

using ap::fail;

struct Vmm {
    CUresult (*granularity)(size_t *, const CUmemAllocationProp *, CUmemAllocationGranularity_flags) = nullptr;
    CUresult (*reserve)(CUdeviceptr *, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
    CUresult (*free_range)(CUdeviceptr, size_t) = nullptr;
    CUresult (*create)(CUmemGenericAllocationHandle *, size_t, const CUmemAllocationProp *,
                       unsigned long long) = nullptr;
    CUresult (*release)(CUmemGenericAllocationHandle) = nullptr;
    CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long) = nullptr;
    CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
    CUresult (*access)(CUdeviceptr, size_t, const CUmemAccessDesc *, size_t) = nullptr;
    bool ok = false;
};

template <typename F>
bool entry(const char *name, F *fn)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
        (void)cudaGetLastError();
        return false;
    }
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Vmm &vmm()
{
    static Vmm v;
    static std::once_flag once;
    std::call_once(once, [] {
        v.ok = entry("cuMemGetAllocationGranularity", &v.granularity) && entry("cuMemAddressReserve", &v.reserve) &&
               entry("cuMemAddressFree", &v.free_range) && entry("cuMemCreate", &v.create) &&
               entry("cuMemRelease", &v.release) && entry("cuMemMap", &v.map) && entry("cuMemUnmap", &v.unmap) &&
               entry("cuMemSetAccess", &v.access);
    });
    return v;
}

ap_status drv_fail(CUresult r, const char *what)
{
    return fail(AP_ECUDA, "%s: CUDA driver error %d", what, (int)r);
}

CUmemAllocationProp device_prop(int device)
{
    CUmemAllocationProp prop = {};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = device;
    return prop;
}

} // namespace

struct ap_arena {
    int device = 0;
    CUdeviceptr base = 0;
    size_t reserved = 0, mapped = 0, gran = 0;
    struct Chunk {
        CUmemGenericAllocationHandle handle;
        size_t offset, bytes;
    };
    std::vector<Chunk> chunks; // one mapping per grow, in address order
};

extern "C" ap_status ap_arena_create(ap_arena **out, int64_t max_bytes, int32_t device)
{
    AP_NVTX_RANGE("ap_arena_create");
    if (!out) return fail(AP_EINVAL, "arena_create: out is NULL");
    *out = nullptr;
    if (max_bytes <= 0) return fail(AP_EINVAL, "arena_create: max_bytes must be > 0");
    const Vmm &v = vmm();
    if (!v.ok) return fail(AP_ENOTSUP, "arena_create: the driver offers no virtual memory management");
    cudaError_t e = cudaSetDevice(device);
    if (e == cudaSuccess) e = cudaFree(nullptr); // make the device's primary context current
    if (e != cudaSuccess) return ap::cuda_fail(e, "arena_create: device");
    const CUmemAllocationProp prop = device_prop(device);
    size_t gran = 0;
    CUresult r = v.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED);
    if (r != CUDA_SUCCESS || gran == 0) return drv_fail(r, "arena_create: granularity");
    const size_t reserved = ((size_t)max_bytes + gran - 1) / gran * gran;
    CUdeviceptr base = 0;
    r = v.reserve(&base, reserved, gran, 0, 0);
    if (r != CUDA_SUCCESS) return drv_fail(r, "arena_create: address reservation");
    ap_arena *a = new (std::nothrow) ap_arena();
    if (!a) {
        v.free_range(base, reserved);
        return fail(AP_EINVAL, "arena_create: out of host memory");
    }
    a->device = device;
    a->base = base;
    a->reserved = reserved;
    a->gran = gran;
    *out = a;
    return AP_OK;
}

extern "C" ap_status ap_arena_grow(ap_arena *a, int64_t bytes)
{
    AP_NVTX_RANGE("ap_arena_grow");
    if (!a) return fail(AP_EINVAL, "arena_grow: NULL arena");
    if (bytes < 0 || (size_t)bytes > a->reserved)
        return fail(AP_EINVAL, "arena_grow: %lld bytes outside the %lld reserved", (long long)bytes,
                    (long long)a->reserved);
    const size_t need = ((size_t)bytes + a->gran - 1) / a->gran * a->gran;
    if (need <= a->mapped) return AP_OK;
    const Vmm &v = vmm();
    const size_t add = need - a->mapped;
    const CUmemAllocationProp prop = device_prop(a->device);
    CUmemGenericAllocationHandle h = 0;
    CUresult r = v.create(&h, add, &prop, 0);
    if (r != CUDA_SUCCESS) return drv_fail(r, "arena_grow: physical allocation");
    r = v.map(a->base + a->mapped, add, 0, h, 0);
    if (r != CUDA_SUCCESS) {
        v.release(h);
        return drv_fail(r, "arena_grow: map");
    }
    CUmemAccessDesc acc = {};
    acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc.location.id = a->device;
    acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    r = v.access(a->base + a->mapped, add, &acc, 1);
    if (r != CUDA_SUCCESS) {
        v.unmap(a->base + a->mapped, add);
        v.release(h);
        return drv_fail(r, "arena_grow: access");
    }
    a->chunks.push_back({h, a->mapped, add});
    a->mapped = need;
    return AP_OK;
}

extern "C" ap_status ap_arena_info(const ap_arena *a, void **base, int64_t *mapped_bytes, int64_t *reserved_bytes)
{
    if (!a) return fail(AP_EINVAL, "arena_info: NULL arena");
    if (base) *base = reinterpret_cast<void *>(a->base);
    if (mapped_bytes) *mapped_bytes = (int64_t)a->mapped;
    if (reserved_bytes) *reserved_bytes = (int64_t)a->reserved;
    return AP_OK;
}

extern "C" ap_status ap_arena_destroy(ap_arena *a)
{
    AP_NVTX_RANGE("ap_arena_destroy");
    if (!a) return AP_OK;
    const Vmm &v = vmm();
    ap_status s = AP_OK;
    for (const ap_arena::Chunk &c : a->chunks) {
        if (v.unmap(a->base + c.offset, c.bytes) != CUDA_SUCCESS) s = fail(AP_ECUDA, "arena_destroy: unmap");
        if (v.release(c.handle) != CUDA_SUCCESS) s = fail(AP_ECUDA, "arena_destroy: release");
    }
    if (a->base && v.free_range(a->base, a->reserved) != CUDA_SUCCESS) s = fail(AP_ECUDA, "arena_destroy: free");
    delete a;
    return s;
}
