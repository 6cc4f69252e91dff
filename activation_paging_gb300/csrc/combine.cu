// Combine / un-permute: out[t] = bf16(sum_j w[t, j] * y[dest[t, j]]).
//
// The dense BF16 [T, H] output of combine with un-permute (OpenPipe/ART pull
// 971, description and review).  One warp per (token, column chunk); each
// lane owns VE consecutive columns per step and gathers the k expert rows of
// its columns, all k loads in flight before the accumulation.  Accumulation is single
// precision with separately rounded multiply and add, j ascending (no FMA),
// then one round-to-nearest-even conversion to BF16.
#include <cuda_bf16.h>

#include "ap_common.cuh"

namespace ap {
namespace {

template <int VE> struct Vec;
template <> struct Vec<8> { using T = int4; };
template <> struct Vec<4> { using T = int2; };
template <> struct Vec<2> { using T = int; };
template <> struct Vec<1> { using T = short; };

__device__ __forceinline__ float lo_bf16(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

template <int VE>
__device__ __forceinline__ void unpack(const typename Vec<VE>::T &v, float *f)
{
    if constexpr (VE == 1) {
        f[0] = __uint_as_float(((uint32_t)(uint16_t)v) << 16);
    } else {
        uint32_t u[VE / 2];
        memcpy(u, &v, sizeof(u));
#pragma unroll
        for (int i = 0; i < VE / 2; ++i) {
            f[2 * i] = lo_bf16(u[i]);
            f[2 * i + 1] = hi_bf16(u[i]);
        }
    }
}

template <int VE>
__device__ __forceinline__ typename Vec<VE>::T pack(const float *f)
{
    typename Vec<VE>::T v;
    uint16_t h[VE];
#pragma unroll
    for (int i = 0; i < VE; ++i) h[i] = __bfloat16_as_ushort(__float2bfloat16_rn(f[i]));
    memcpy(&v, h, sizeof(v));
    return v;
}

// Work item = (token, column chunk of U*32 lane steps); items are strided over
// all resident warps so every warp gets the same share (no partial last wave).
// U column steps are unrolled and KB rows are gathered per batch, so U*KB row
// loads are in flight per lane; each warp reads U*32*16 contiguous bytes of a
// row (1 KB for BF16 rows with U = 2), which a sweep on GB300 found faster
// than narrower pieces or deeper batches with fewer resident warps.
template <int VE, int U, int KB>
__global__ void __launch_bounds__(256, 4) k_combine(const uint16_t *__restrict__ y, int64_t y_rows, int H,
                                                 const int32_t *__restrict__ dest, const float *__restrict__ w,
                                                 int64_t T, int k, uint16_t *__restrict__ out, uint32_t *d_status)
{
    pdl_begin();
    using V = typename Vec<VE>::T;
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    const int nstep = H / VE;
    const int chunks = (nstep + U * kWarp - 1) / (U * kWarp);
    const int64_t items = T * chunks;
    for (int64_t it = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; it < items; it += warps) {
        const int64_t t = it / chunks;
        const int s0 = (int)(it - t * chunks) * U * kWarp;
        int32_t my_d = -1;
        float my_w = 0.f;
        if (lane < k) {
            my_d = dest[t * k + lane];
            my_w = w ? w[t * k + lane] : 1.0f; // no weights: the dispatch backward (unit weights)
            if (my_d >= y_rows) {
                if (d_status && s0 == 0) atomicOr(d_status, AP_FLAG_BAD_INDEX);
                my_d = -1;
            }
        }
        float acc[U][VE];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < VE; ++i) acc[u][i] = 0.f;
        // KB rows per batch: every load of the batch is issued before the first
        // add, then the adds run in j order
        for (int j0 = 0; j0 < k; j0 += KB) {
            int32_t d[KB];
            float wj[KB];
            V v[KB][U];
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
                const int j = j0 + jj;
                d[jj] = __shfl_sync(0xffffffffu, my_d, j & (kWarp - 1));
                wj[jj] = __shfl_sync(0xffffffffu, my_w, j & (kWarp - 1));
                if (j >= k) d[jj] = -1;
                if (d[jj] >= 0) {
                    const V *yrow = reinterpret_cast<const V *>(y + (int64_t)d[jj] * H);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int s = s0 + u * kWarp + lane;
                        if (s < nstep) v[jj][u] = ld_stream(yrow + s);
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
                if (d[jj] < 0) continue;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float f[VE];
                    unpack<VE>(v[jj][u], f);
#pragma unroll
                    for (int i = 0; i < VE; ++i) acc[u][i] = __fadd_rn(acc[u][i], __fmul_rn(wj[jj], f[i]));
                }
            }
        }
        uint16_t *orow = out + t * H;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * kWarp + lane;
            if (s < nstep) st_stream(reinterpret_cast<V *>(orow) + s, pack<VE>(acc[u]));
        }
    }
}

template <int VE, int U>
void launch_combine(const uint16_t *y, int64_t y_rows, int H, const int32_t *dest, const float *w, int64_t T, int k,
                    uint16_t *out, uint32_t *d_status, cudaStream_t st)
{
    constexpr int KB = 2;
    static const int resident = resident_grid((const void *)k_combine<VE, U, KB>, 256);
    const int nstep = H / VE;
    const int64_t items = T * ((nstep + U * kWarp - 1) / (U * kWarp));
    const int64_t want = (items + 7) / 8;
    const int grid = (int)(want < resident ? want : resident);
    launch(k_combine<VE, U, KB>, grid, 256, 0, st, y, y_rows, H, dest, w, T, k, out, d_status);
}

// Backward of combine, one warp per token (a deterministic dot product):
//   dy[dest(t,j)] = bf16(w[t,j] * dout[t]),  dw[t,j] = <dout[t], y[dest(t,j)]>.
// Each lane accumulates its columns in order, then a fixed butterfly sums the
// lanes.  dout[t] is re-read for every j from L1.
template <int VE>
__global__ void __launch_bounds__(256) k_combine_bwd(const uint16_t *__restrict__ dout,
                                                     const uint16_t *__restrict__ y, int64_t y_rows, int H,
                                                     const int32_t *__restrict__ dest, const float *__restrict__ w,
                                                     int64_t T, int k, uint16_t *__restrict__ dy,
                                                     float *__restrict__ dw, uint32_t *d_status)
{
    pdl_begin();
    using V = typename Vec<VE>::T;
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    const int nstep = H / VE;
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        int32_t my_d = -1;
        float my_w = 0.f;
        if (lane < k) {
            my_d = dest[t * k + lane];
            my_w = w[t * k + lane];
            if (my_d >= y_rows) {
                if (d_status) atomicOr(d_status, AP_FLAG_BAD_INDEX);
                my_d = -1;
            }
        }
        const V *grow = reinterpret_cast<const V *>(dout + t * H);
        for (int j = 0; j < k; ++j) {
            const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
            const float wj = __shfl_sync(0xffffffffu, my_w, j);
            if (d < 0) {
                if (lane == 0) dw[t * k + j] = 0.f;
                continue;
            }
            const V *yrow = reinterpret_cast<const V *>(y + (int64_t)d * H);
            V *dyrow = reinterpret_cast<V *>(dy + (int64_t)d * H);
            float dot = 0.f;
            for (int s = lane; s < nstep; s += kWarp) {
                float g[VE], yv[VE], o[VE];
                unpack<VE>(grow[s], g);
                unpack<VE>(ld_stream(yrow + s), yv);
#pragma unroll
                for (int i = 0; i < VE; ++i) {
                    o[i] = __fmul_rn(wj, g[i]);
                    dot = fmaf(g[i], yv[i], dot);
                }
                st_stream(dyrow + s, pack<VE>(o));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            if (lane == 0) dw[t * k + j] = dot;
        }
    }
}

// Combine backward for BF16 rows in 16-byte vectors, split by columns: each
// block takes two tokens at a time and gives each token four warps; warp q of
// a token owns column pieces q, q + 4, ... of U * 32 vectors (512 bytes of a
// row for U = 1).  For every pair j (KB rows per batch, all loads of a batch
// in flight before the first use) a warp writes its pieces of dy and sums its
// part of the dot product (columns ascending within a lane, then a butterfly);
// the four parts of dw[t, j] are added in warp order through shared memory,
// so dw is deterministic.  More warps in flight per token than one warp per
// token, with few registers per lane.  A sweep on GB300 over (U, KB) in
// {1, 2, 4} x {2, 4, 8} chose U = 1, KB = 4 (0.93 of the copy rate at the
// Qwen3-like chunk; one warp per token reached 0.44).
constexpr int kBwdWarpsPerTok = 4;

template <int U, int KB>
__global__ void __launch_bounds__(256, 4) k_combine_bwd_pieces(const uint16_t *__restrict__ dout,
                                                              const uint16_t *__restrict__ y, int64_t y_rows, int H,
                                                              const int32_t *__restrict__ dest,
                                                              const float *__restrict__ w, int64_t T, int k,
                                                              uint16_t *__restrict__ dy, float *__restrict__ dw,
                                                              uint32_t *d_status)
{
    pdl_begin();
    using V = int4;
    constexpr int kTokPerIter = 8 / kBwdWarpsPerTok; // tokens a 256-thread block takes at a time
    __shared__ float s_part[kTokPerIter][kWarp][kBwdWarpsPerTok];
    const int lane = (int)lane_id(), wid = threadIdx.x / kWarp;
    const int tb = wid / kBwdWarpsPerTok, q = wid % kBwdWarpsPerTok;
    const int nstep = H / 8;
    const int pieces = (nstep + U * kWarp - 1) / (U * kWarp);
    for (int64_t t0 = (int64_t)blockIdx.x * kTokPerIter; t0 < T; t0 += (int64_t)gridDim.x * kTokPerIter) {
        const int64_t t = t0 + tb;
        const bool tv = t < T; // warp-uniform
        int32_t my_d = -1;
        float my_w = 0.f;
        if (tv && lane < k) {
            my_d = dest[t * k + lane];
            my_w = w[t * k + lane];
            if (my_d >= y_rows) {
                if (d_status && q == 0) atomicOr(d_status, AP_FLAG_BAD_INDEX);
                my_d = -1;
            }
        }
        const V *grow = reinterpret_cast<const V *>(dout + (tv ? t : 0) * H);
        for (int j0 = 0; j0 < k; j0 += KB) {
            int32_t d[KB];
            float wj[KB];
            float dot[KB];
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
                d[jj] = __shfl_sync(0xffffffffu, my_d, (j0 + jj) & (kWarp - 1));
                wj[jj] = __shfl_sync(0xffffffffu, my_w, (j0 + jj) & (kWarp - 1));
                if (j0 + jj >= k || !tv) d[jj] = -1;
                dot[jj] = 0.f;
            }
            for (int pc = q; pc < pieces; pc += kBwdWarpsPerTok) {
                const int s0 = pc * U * kWarp;
                V yv[KB][U];
#pragma unroll
                for (int jj = 0; jj < KB; ++jj) {
                    if (d[jj] < 0) continue;
                    const V *yrow = reinterpret_cast<const V *>(y + (int64_t)d[jj] * H);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int s = s0 + u * kWarp + lane;
                        if (s < nstep) yv[jj][u] = ld_stream(yrow + s);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int s = s0 + u * kWarp + lane;
                    if (s >= nstep) continue;
                    float g[8];
                    unpack<8>(grow[s], g);
#pragma unroll
                    for (int jj = 0; jj < KB; ++jj) {
                        if (d[jj] < 0) continue;
                        float yf[8], o[8];
                        unpack<8>(yv[jj][u], yf);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o[i] = __fmul_rn(wj[jj], g[i]);
                            dot[jj] = fmaf(g[i], yf[i], dot[jj]);
                        }
                        st_stream(reinterpret_cast<V *>(dy + (int64_t)d[jj] * H) + s, pack<8>(o));
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) dot[jj] += __shfl_xor_sync(0xffffffffu, dot[jj], off);
                if (lane == 0 && j0 + jj < k) s_part[tb][j0 + jj][q] = dot[jj];
            }
        }
        __syncthreads();
        // dw[t, j]: the four warps' parts in warp order (a dropped pair gives 0)
        if (threadIdx.x < kTokPerIter * kWarp) {
            const int tt = threadIdx.x / kWarp, j = threadIdx.x % kWarp;
            const int64_t t2 = t0 + tt;
            if (t2 < T && j < k) {
                float sum = 0.f;
#pragma unroll
                for (int qq = 0; qq < kBwdWarpsPerTok; ++qq) sum += s_part[tt][j][qq];
                const int32_t dd = dest[t2 * k + j];
                dw[t2 * k + j] = (dd >= 0 && dd < y_rows) ? sum : 0.f;
            }
        }
        __syncthreads();
    }
}

template <int U, int KB>
void launch_combine_bwd_pieces(const uint16_t *dout, const uint16_t *y, int64_t y_rows, int H, const int32_t *dest,
                               const float *w, int64_t T, int k, uint16_t *dy, float *dw, uint32_t *d_status,
                               cudaStream_t st)
{
    static const int resident = resident_grid((const void *)k_combine_bwd_pieces<U, KB>, 256);
    const int64_t want = (T + 1) / 2;
    launch(k_combine_bwd_pieces<U, KB>, (int)(want < resident ? want : resident), 256, 0, st, dout, y, y_rows, H,
           dest, w, T, k, dy, dw, d_status);
}

template <int VE>
void launch_combine_bwd(const uint16_t *dout, const uint16_t *y, int64_t y_rows, int H, const int32_t *dest,
                        const float *w, int64_t T, int k, uint16_t *dy, float *dw, uint32_t *d_status,
                        cudaStream_t st)
{
    static const int resident = resident_grid((const void *)k_combine_bwd<VE>, 256);
    const int64_t want = (T + 7) / 8;
    launch(k_combine_bwd<VE>, (int)(want < resident ? want : resident), 256, 0, st, dout, y, y_rows, H, dest, w, T, k,
                                                                              dy, dw, d_status);
}

} // namespace
} // namespace ap

extern "C" ap_status ap_combine_backward(const void *dout, const void *y, int64_t y_rows, int32_t H,
                                         const int32_t *dest, const float *w, int64_t T, int32_t k, void *dy,
                                         float *dw, uint32_t *d_status, void *stream)
{
    AP_NVTX_RANGE("ap_combine_backward");
    using namespace ap;
    if (T < 0 || H < 1 || k < 1 || k > 32 || y_rows < 0)
        return fail(AP_EINVAL, "combine_backward: bad sizes T=%lld H=%d k=%d", (long long)T, H, k);
    if (T == 0) return AP_OK;
    if (!dout || !dest || !w || !dw || (y_rows > 0 && (!y || !dy)))
        return fail(AP_EINVAL, "combine_backward: NULL pointer");
    cudaStream_t st = (cudaStream_t)stream;
    const uintptr_t al = reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(y) |
                         reinterpret_cast<uintptr_t>(dy);
    const uint16_t *g = static_cast<const uint16_t *>(dout);
    const uint16_t *yy = static_cast<const uint16_t *>(y);
    uint16_t *d = static_cast<uint16_t *>(dy);
    if (H % 8 == 0 && (al & 15) == 0)
        launch_combine_bwd_pieces<1, 4>(g, yy, y_rows, H, dest, w, T, k, d, dw, d_status, st);
    else
        launch_combine_bwd<1>(g, yy, y_rows, H, dest, w, T, k, d, dw, d_status, st);
    AP_CHECK_LAUNCH("combine_backward launch");
    return AP_OK;
}

extern "C" ap_status ap_dispatch_backward(const void *dxd, int64_t rows, int32_t H, const int32_t *dest, int64_t T,
                                          int32_t k, void *dx, uint32_t *d_status, void *stream)
{
    AP_NVTX_RANGE("ap_dispatch_backward");
    using namespace ap;
    if (T < 0 || H < 1 || k < 1 || k > 32 || rows < 0)
        return fail(AP_EINVAL, "dispatch_backward: bad sizes T=%lld H=%d k=%d", (long long)T, H, k);
    if (T == 0) return AP_OK;
    if (!dest || !dx || (!dxd && rows > 0)) return fail(AP_EINVAL, "dispatch_backward: NULL pointer");
    cudaStream_t st = (cudaStream_t)stream;
    const uint16_t *yy = static_cast<const uint16_t *>(dxd);
    uint16_t *oo = static_cast<uint16_t *>(dx);
    const uintptr_t al = reinterpret_cast<uintptr_t>(dxd) | reinterpret_cast<uintptr_t>(dx);
    if (H % 8 == 0 && (al & 15) == 0)
        launch_combine<8, 2>(yy, rows, H, dest, nullptr, T, k, oo, d_status, st);
    else if (H % 4 == 0 && (al & 7) == 0)
        launch_combine<4, 4>(yy, rows, H, dest, nullptr, T, k, oo, d_status, st);
    else if (H % 2 == 0 && (al & 3) == 0)
        launch_combine<2, 4>(yy, rows, H, dest, nullptr, T, k, oo, d_status, st);
    else
        launch_combine<1, 4>(yy, rows, H, dest, nullptr, T, k, oo, d_status, st);
    AP_CHECK_LAUNCH("dispatch_backward launch");
    return AP_OK;
}

extern "C" ap_status ap_combine_unpermute(const void *y, int64_t y_rows, int32_t H, const int32_t *dest, const float *w,
                                          int64_t T, int32_t k, void *out, uint32_t *d_status, void *stream)
{
    AP_NVTX_RANGE("ap_combine_unpermute");
    using namespace ap;
    if (T < 0 || H < 1 || k < 1 || k > 32 || y_rows < 0)
        return fail(AP_EINVAL, "combine_unpermute: bad sizes T=%lld H=%d k=%d", (long long)T, H, k);
    if (T == 0) return AP_OK;
    if (!dest || !w || !out || (!y && y_rows > 0)) return fail(AP_EINVAL, "combine_unpermute: NULL pointer");
    cudaStream_t st = (cudaStream_t)stream;
    const uint16_t *yy = static_cast<const uint16_t *>(y);
    uint16_t *oo = static_cast<uint16_t *>(out);
    const uintptr_t al = reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(out);
    if (H % 8 == 0 && (al & 15) == 0)
        launch_combine<8, 2>(yy, y_rows, H, dest, w, T, k, oo, d_status, st);
    else if (H % 4 == 0 && (al & 7) == 0)
        launch_combine<4, 4>(yy, y_rows, H, dest, w, T, k, oo, d_status, st);
    else if (H % 2 == 0 && (al & 3) == 0)
        launch_combine<2, 4>(yy, y_rows, H, dest, w, T, k, oo, d_status, st);
    else
        launch_combine<1, 4>(yy, y_rows, H, dest, w, T, k, oo, d_status, st);
    AP_CHECK_LAUNCH("combine launch");
    return AP_OK;
}
