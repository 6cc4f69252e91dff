// Router: softmax -> top-k -> renormalised weights, one warp per token.
//
// Top-k routing over the experts (Megatron-LM pull 7342, "Validation and
// performance": top-k 8).  Selection compares the raw logits (an equal logit
// goes to the lower expert id) in k rounds of a warp arg-max built from two
// redux.sync reductions; lane j keeps the j-th winner.  Because the softmax
// denominator cancels in the renormalisation,
// w_j = exp(l_j - m) / sum_sel exp(l_i - m), with m the row maximum (= the
// first winner), so only k exponentials are evaluated.
#include "route_topk.cuh"

namespace ap {
namespace {

// One warp per token (route_topk.cuh).
template <int NV>
__global__ void __launch_bounds__(256) k_route_topk(const float *__restrict__ logits, int64_t T, int E, int k,
                                                     int32_t *__restrict__ idx, float *__restrict__ w)
{
    pdl_begin();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        int e;
        float wt;
        route_token<NV>(logits + t * E, E, k, lane, &e, &wt);
        if (lane < k) {
            idx[t * k + lane] = e;
            w[t * k + lane] = wt;
        }
    }
}

} // namespace
} // namespace ap

extern "C" ap_status ap_route_topk(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *idx, float *w,
                                   void *stream)
{
    AP_NVTX_RANGE("ap_route_topk");
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
