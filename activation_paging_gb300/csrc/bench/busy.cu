// Synthetic compute for the reload-overlap measurement of bench.py, and the
// host NUMA query its host-side setup uses.  Not part of the library
// (libap.so) or its ABI: it is built into libap_bench.so.
//
// Each block of k_busy holds one whole SM: 1024 threads and the largest
// dynamic shared-memory allocation a block may take, so no other block (every
// block reserves some shared memory) fits on that SM while it runs.  A grid
// of n blocks therefore keeps n SMs busy with arithmetic and leaves the other
// SMs free for work on other streams; the block spins on a fixed count of
// fused multiply-adds and touches no global memory except one final store.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void __launch_bounds__(1024, 1) k_busy(long long iters, float *sink)
{
    extern __shared__ float smem[];
    float a = 1.0f + threadIdx.x * 1e-6f, b = 0.999999f, c = 1e-7f;
    for (long long i = 0; i < iters; ++i) {
        a = fmaf(a, b, c);
        b = fmaf(b, a, -c);
    }
    smem[threadIdx.x] = a + b;
    __syncthreads();
    if (threadIdx.x == 0) sink[blockIdx.x] = smem[blockIdx.x & 1023];
}

} // namespace

// Largest dynamic shared memory one block may take on the current device.
static int max_block_smem()
{
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
    return v;
}

// Launch nblocks whole-SM blocks that each run `iters` iterations on
// `stream`.  sink: device float[nblocks].  Returns 0, or a CUDA error code.
extern "C" int apb_busy_sms(int nblocks, long long iters, float *sink, void *stream)
{
    if (nblocks < 1 || iters < 0 || !sink) return (int)cudaErrorInvalidValue;
    const int smem = max_block_smem();
    if (smem <= 0) return (int)cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(k_busy, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return (int)e;
    k_busy<<<nblocks, 1024, smem, (cudaStream_t)stream>>>(iters, sink);
    return (int)cudaGetLastError();
}

// The host NUMA node nearest `device` (cudaDevAttrHostNumaId), or -1 when the
// system reports none or the query fails.  The bench runs its host threads
// there, so the pinned buffers it allocates sit next to the GPU.
extern "C" int apb_host_numa_id(int device)
{
    int v = -1;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrHostNumaId, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return v;
}
