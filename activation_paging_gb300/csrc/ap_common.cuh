// Shared device and host helpers of the CUDA library (not part of the ABI).
#pragma once

#include <utility>

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ap.h"

namespace ap {

constexpr int kWarp = 32;

// ---- host-side error reporting ------------------------------------------------
void set_error(const char *fmt, ...);
ap_status fail(ap_status s, const char *fmt, ...);
ap_status cuda_fail(cudaError_t e, const char *what);
int sm_count();
// Counts one enqueued kernel (ap_launch_count); every launch site calls it once.
void note_launch();
// Blocks of `kernel` (launched with `threads` threads and `smem` dynamic shared
// bytes) that fit on the whole GPU at once: SMs x resident blocks per SM.
// Grid-stride kernels launched with this grid run in exactly one wave.
int resident_grid(const void *kernel, int threads, size_t smem = 0);

// Dispatch stages shared by the dispatch entry points (dispatch.cu): argument
// checks, then the count/rank and scan launches that produce counts, live,
// seg_off and the in-block ranks the copy kernels turn into dest and src_tok.
ap_status dispatch_check(const char *who, const void *x, int64_t T, int32_t H, const int32_t *idx, int32_t k,
                         int32_t E, int32_t capacity, int32_t padded, const void *xd, int64_t xd_rows,
                         const int32_t *counts, const int32_t *live, const int32_t *seg_off, const int32_t *dest,
                         const void *scratch, int64_t scratch_bytes);
ap_status dispatch_metadata(int64_t T, const int32_t *idx, int32_t k, int32_t E, int32_t capacity, int32_t padded,
                            int32_t *counts, int32_t *live, int32_t *seg_off, int32_t *dest, void *scratch,
                            uint32_t *d_status, cudaStream_t st, const void *x = nullptr, int64_t x_rb = 0);
// The count/rank stage alone (block histograms into scratch, in-block ranks
// into dest), and the number of count/rank blocks; the fused dispatch + stash
// runs its own scan (see dispatch_scan.cuh).  x / x_rb (here, in
// dispatch_metadata and in dispatch_route_count_rank): the input rows the row
// copy after these kernels reads; each count/rank block prefetches its own
// rows into L2 (nullptr: none).
ap_status dispatch_count_rank(int64_t T, const int32_t *idx, int32_t k, int32_t E, void *scratch, int32_t *dest,
                              uint32_t *d_status, cudaStream_t st, const void *x = nullptr, int64_t x_rb = 0);
int dispatch_blocks(int64_t T);
// Route (as ap_route_topk, into idx and w) and count/rank in one launch: the
// same outputs as ap_route_topk followed by dispatch_count_rank.  Arguments
// are checked by the caller.
ap_status dispatch_route_count_rank(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *idx, float *w,
                                    void *scratch, int32_t *dest, cudaStream_t st, const void *x = nullptr,
                                    int64_t x_rb = 0);

// ---- NVTX ranges ---------------------------------------------------------------
// Every entry point that enqueues GPU work or waits on the GPU opens a range
// named after itself (domain "activation_paging") for the length of the host
// call, so a trace of a step attributes each call's launches and waits to
// route, dispatch, push, pop or combine.  AP_NVTX=0 in the environment turns
// the ranges off; without a tool attached a range costs one call into an
// empty stub.
class NvtxRange {
  public:
    explicit NvtxRange(const char *name);
    ~NvtxRange();
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;

  private:
    bool on_;
};
#define AP_NVTX_RANGE(name) ::ap::NvtxRange ap_nvtx_range_(name)

#define AP_CHECK_LAUNCH(what)                                   \
    do {                                                        \
        cudaError_t e_ = cudaGetLastError();                    \
        if (e_ != cudaSuccess) return ::ap::cuda_fail(e_, what); \
        ::ap::note_launch();                                    \
    } while (0)

// ---- programmatic dependent launch -------------------------------------------
// Every kernel of the library begins with pdl_begin() and is launched with
// launch(), i.e. with programmatic stream serialization: the next kernel on
// the stream may start launching once every block of this one has started,
// and its blocks then wait in their own pdl_begin() until this grid has
// finished and its memory is visible.  The chains of small dependent kernels
// (route, count/rank, scan + plan, copy, pop copy, combine) thereby
// overlap each launch with the end of the kernel before it; no kernel touches
// memory before its wait, so results do not change.  After a kernel launched
// without the attribute, or an event, the wait returns at once.
template <typename... KArgs, typename... Args>
inline void launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...); // errors surface in AP_CHECK_LAUNCH
}

__device__ __forceinline__ void pdl_begin()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- device helpers ----------------------------------------------------------
__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Streaming (evict-first) global loads/stores for data touched once.
__device__ __forceinline__ int4 ld_stream(const int4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(int4 *p, int4 v) { __stcs(p, v); }
__device__ __forceinline__ int2 ld_stream(const int2 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(int2 *p, int2 v) { __stcs(p, v); }
__device__ __forceinline__ int ld_stream(const int *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(int *p, int v) { __stcs(p, v); }
__device__ __forceinline__ short ld_stream(const short *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(short *p, short v) { __stcs(p, v); }
__device__ __forceinline__ char ld_stream(const char *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(char *p, char v) { __stcs(p, v); }

// Copy n bytes from src to dst with all threads of the block, vectorised to the
// widest width both pointers share (16, 8, 4, 2 or 1 bytes), with byte-wise
// heads and tails.  Eight loads are issued before their stores so each
// thread keeps 128 bytes in flight, and the last, partial pass goes in
// predicated groups rather than one vector at a time, so ranges that are not
// a multiple of 8 vectors per thread (e.g. 15 rows of 2056 bytes) keep
// several loads in flight too.
template <typename V>
__device__ __forceinline__ void block_copy_vec(uint8_t *dst, const uint8_t *src, int64_t nvec)
{
    const V *s = reinterpret_cast<const V *>(src);
    V *d = reinterpret_cast<V *>(dst);
    const int64_t nt = blockDim.x;
    int64_t i = threadIdx.x;
    constexpr int U = 8;
    for (; i + (U - 1) * nt < nvec; i += U * nt) {
        V r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = ld_stream(s + i + u * nt);
#pragma unroll
        for (int u = 0; u < U; ++u) st_stream(d + i + u * nt, r[u]);
    }
    // the partial pass, in predicated groups of 2 (larger groups spill
    // registers in the copy kernels, and 2 measured faster than 4 on rows of
    // 2056 bytes); narrower vectors (rare, short ranges) one at a time
    constexpr int UT = sizeof(V) >= 8 ? 2 : 1;
    for (; i < nvec; i += UT * nt) {
        V r[UT];
#pragma unroll
        for (int u = 0; u < UT; ++u)
            if (i + u * nt < nvec) r[u] = ld_stream(s + i + u * nt);
#pragma unroll
        for (int u = 0; u < UT; ++u)
            if (i + u * nt < nvec) st_stream(d + i + u * nt, r[u]);
    }
}

__device__ __forceinline__ void block_copy(uint8_t *dst, const uint8_t *src, int64_t n)
{
    if (n <= 0) return;
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(dst) ^ reinterpret_cast<uintptr_t>(src));
    int A = 16;
    while (A > 1 && (mis & (uintptr_t)(A - 1))) A >>= 1;
    int64_t head = (int64_t)((A - (reinterpret_cast<uintptr_t>(dst) & (uintptr_t)(A - 1))) & (uintptr_t)(A - 1));
    if (head > n) head = n;
    for (int64_t i = threadIdx.x; i < head; i += blockDim.x) dst[i] = src[i];
    dst += head;
    src += head;
    n -= head;
    const int64_t nvec = n / A;
    switch (A) {
    case 16: block_copy_vec<int4>(dst, src, nvec); break;
    case 8: block_copy_vec<int2>(dst, src, nvec); break;
    case 4: block_copy_vec<int>(dst, src, nvec); break;
    case 2: block_copy_vec<short>(dst, src, nvec); break;
    default: block_copy_vec<char>(dst, src, nvec); break;
    }
    const int64_t done = nvec * A;
    for (int64_t i = done + threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

} // namespace ap
