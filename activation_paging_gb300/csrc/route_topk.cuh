// Top-k routing of one token by one warp, shared by the router and the fused
// route + count/rank kernel.
//
// Top-k routing over the experts (Megatron-LM pull 7342, "Validation and
// performance": top-k 8).  Selection compares the raw logits (an equal logit
// goes to the lower expert id) in k rounds of a warp arg-max built from two
// redux.sync reductions; lane j keeps the j-th winner.  Because the softmax
// denominator cancels in the renormalisation,
// w_j = exp(l_j - m) / sum_sel exp(l_i - m), with m the row maximum (= the
// first winner), so only k exponentials are evaluated.
#pragma once

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
// lane shifts its list.  All 32 lanes call it; lane j < k receives the j-th
// expert in *e and its renormalised weight in *wt.
template <int NV>
__device__ __forceinline__ void route_token(const float *__restrict__ row, int E, int k, int lane, int *e, float *wt)
{
    constexpr int kNone = 0x7fffffff;
    uint32_t key[NV];
    int ex[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int ei = lane + kWarp * i;
        const bool ok = ei < E;
        key[i] = ok ? order_key(__ldcs(row + ei)) : 0u; // 0 sorts below every finite logit
        ex[i] = ok ? ei : kNone;
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
    *e = my_e;
    *wt = __fdiv_rn(z, s);
}

} // namespace
} // namespace ap
