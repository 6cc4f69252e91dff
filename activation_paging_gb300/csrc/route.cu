// Router: softmax -> top-k -> renormalised weights, one warp per token.
//
// Top-k routing over the experts (Megatron-LM pull 7342, "Validation and
// performance": top-k 8).  Selection compares the raw logits (an equal logit
// goes to the lower expert id) in k rounds of a warp arg-max; lane j keeps the
// j-th winner.  Because the softmax denominator cancels in the
// renormalisation, w_j = exp(l_j - m) / sum_sel exp(l_i - m), with m the row
// maximum (= the first winner), so only k exponentials are evaluated.
#include <float.h>

#include "ap_common.cuh"

namespace ap {
namespace {

// (v, e) beats (bv, be) when its logit is larger, or equal with a lower id.
__device__ __forceinline__ bool better(float v, int e, float bv, int be)
{
    return (v > bv) || (v == bv && e < be);
}

template <int NV>
__global__ void __launch_bounds__(256) k_route_topk(const float *__restrict__ logits, int64_t T, int E, int k,
                                                     int32_t *__restrict__ idx, float *__restrict__ w)
{
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        const float *row = logits + t * E;
        float v[NV];
        unsigned avail = 0; // bit i: value i of this lane is a real, unselected expert
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + kWarp * i;
            v[i] = (e < E) ? __ldcs(row + e) : -FLT_MAX;
            if (e < E) avail |= 1u << i;
        }
        float my_v = 0.f;
        int my_e = 0;
        for (int j = 0; j < k; ++j) {
            // best remaining value of this lane
            float bv = -FLT_MAX;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int e = lane + kWarp * i;
                if ((avail >> i) & 1u) {
                    if (be == 0x7fffffff || better(v[i], e, bv, be)) {
                        bv = v[i];
                        be = e;
                    }
                }
            }
            // warp arg-max (butterfly: every lane ends with the winner)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (oe != 0x7fffffff && (be == 0x7fffffff || better(ov, oe, bv, be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & (kWarp - 1)) == lane) avail &= ~(1u << (be / kWarp));
            if (lane == j) {
                my_v = bv;
                my_e = be;
            }
        }
        const float m = __shfl_sync(0xffffffffu, my_v, 0); // the largest logit
        const float z = (lane < k) ? expf(my_v - m) : 0.f;
        float s = z;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane < k) {
            idx[t * k + lane] = my_e;
            w[t * k + lane] = __fdiv_rn(z, s);
        }
    }
}

} // namespace
} // namespace ap

extern "C" ap_status ap_route_topk(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *idx, float *w,
                                   void *stream)
{
    using namespace ap;
    if (T < 0 || T >= (int64_t(1) << 31) || E < 1 || E > 1024 || k < 1 || k > E || k > 32)
        return fail(AP_EINVAL, "route_topk: bad sizes T=%lld E=%d k=%d", (long long)T, E, k);
    if (T == 0) return AP_OK;
    if (!logits || !idx || !w) return fail(AP_EINVAL, "route_topk: NULL pointer");
    cudaStream_t st = (cudaStream_t)stream;
    const int threads = 256;
    const int64_t want = (T + 7) / 8;
    const int grid = (int)(want < (int64_t)sm_count() * 16 ? want : (int64_t)sm_count() * 16);
    if (E <= 32)
        k_route_topk<1><<<grid, threads, 0, st>>>(logits, T, E, k, idx, w);
    else if (E <= 64)
        k_route_topk<2><<<grid, threads, 0, st>>>(logits, T, E, k, idx, w);
    else if (E <= 128)
        k_route_topk<4><<<grid, threads, 0, st>>>(logits, T, E, k, idx, w);
    else if (E <= 256)
        k_route_topk<8><<<grid, threads, 0, st>>>(logits, T, E, k, idx, w);
    else if (E <= 512)
        k_route_topk<16><<<grid, threads, 0, st>>>(logits, T, E, k, idx, w);
    else
        k_route_topk<32><<<grid, threads, 0, st>>>(logits, T, E, k, idx, w);
    AP_CHECK_LAUNCH("route_topk launch");
    return AP_OK;
}
