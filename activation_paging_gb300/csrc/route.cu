// Router: softmax -> top-k -> renormalised weights, one warp per token.
//
// Top-k routing over the experts (Megatron-LM pull 7342, "Validation and
// performance": top-k 8).  Selection compares the raw logits (an equal logit
// goes to the lower expert id) in k rounds of a warp arg-max built from two
// redux.sync reductions; lane j keeps the j-th winner.  Because the softmax
// denominator cancels in the renormalisation,
// w_j = exp(l_j - m) / sum_sel exp(l_i - m), with m the row maximum (= the
// first winner), so only k exponentials are evaluated.
#include <float.h>

#include "ap_common.cuh"

namespace ap {
namespace {

// Order-preserving map of a finite float to uint32 (larger float -> larger
// key); -0 is first turned into +0 so that the two compare equal, as floats do.
__device__ __forceinline__ uint32_t order_key(float v)
{
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (ka, ea) before (kb, eb): larger key first, then the lower expert id.
__device__ __forceinline__ bool before(uint32_t ka, int ea, uint32_t kb, int eb)
{
    return ka > kb || (ka == kb && ea < eb);
}

// Each lane sorts its NV candidates (odd-even transposition, constant
// indices), then k rounds each take the warp-wide best head with two
// redux.sync reductions (max key, then min id among equal keys); the winning
// lane shifts its list.  Lane j keeps the j-th winner.
template <int NV>
__global__ void __launch_bounds__(256) k_route_topk(const float *__restrict__ logits, int64_t T, int E, int k,
                                                     int32_t *__restrict__ idx, float *__restrict__ w)
{
    pdl_begin();
    constexpr int kNone = 0x7fffffff;
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        const float *row = logits + t * E;
        uint32_t key[NV];
        int ex[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + kWarp * i;
            const bool ok = e < E;
            key[i] = ok ? order_key(__ldcs(row + e)) : 0u; // 0 sorts below every finite logit
            ex[i] = ok ? e : kNone;
        }
#pragma unroll
        for (int r = 0; r < NV; ++r) {
#pragma unroll
            for (int i = r & 1; i + 1 < NV; i += 2) {
                if (before(key[i + 1], ex[i + 1], key[i], ex[i])) {
                    const uint32_t tk = key[i];
                    key[i] = key[i + 1];
                    key[i + 1] = tk;
                    const int te = ex[i];
                    ex[i] = ex[i + 1];
                    ex[i + 1] = te;
                }
            }
        }
        uint32_t my_key = 0;
        int my_e = 0;
        for (int j = 0; j < k; ++j) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
            const int emin = __reduce_min_sync(0xffffffffu, key[0] == m ? ex[0] : kNone);
            if (key[0] == m && ex[0] == emin) {
#pragma unroll
                for (int i = 0; i + 1 < NV; ++i) {
                    key[i] = key[i + 1];
                    ex[i] = ex[i + 1];
                }
                key[NV - 1] = 0u;
                ex[NV - 1] = kNone;
            }
            if (lane == j) {
                my_key = m;
                my_e = emin;
            }
        }
        const float mv = key_value(__shfl_sync(0xffffffffu, my_key, 0)); // the largest logit
        const float z = (lane < k) ? expf(key_value(my_key) - mv) : 0.f;
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
        launch(k_route_topk<1>, grid, threads, 0, st, logits, T, E, k, idx, w);
    else if (E <= 64)
        launch(k_route_topk<2>, grid, threads, 0, st, logits, T, E, k, idx, w);
    else if (E <= 128)
        launch(k_route_topk<4>, grid, threads, 0, st, logits, T, E, k, idx, w);
    else if (E <= 256)
        launch(k_route_topk<8>, grid, threads, 0, st, logits, T, E, k, idx, w);
    else if (E <= 512)
        launch(k_route_topk<16>, grid, threads, 0, st, logits, T, E, k, idx, w);
    else
        launch(k_route_topk<32>, grid, threads, 0, st, logits, T, E, k, idx, w);
    AP_CHECK_LAUNCH("route_topk launch");
    return AP_OK;
}
