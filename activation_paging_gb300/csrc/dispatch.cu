// Dispatch: expert counts, stable capacity-bounded ranks and the row permute.
//
// Expert-major, capacity-shaped dispatch buffers (Megatron-LM pull 7342,
// "Summary"; torchtitan pull 5541, "AI-Generated Details": the capacity shape
// that reload restores).  Three launches on the caller's stream:
//   1. k_count_rank - per block of kTokPerBlk tokens: the expert histogram
//                 -> blk[b][e], and each pair's stable rank inside the block
//                 (warp match_any + popc over 32 pairs at a time, pairs in
//                 t-then-j order) -> dest (temporarily);
//   2. k_scan   - one CTA: exclusive scan of blk over b per expert (block base
//                 offsets), counts, live = min(count, C), segment offsets;
//   3. k_copy_* - one warp per token: lanes j < k finish their pair's row
//                 (block base + in-block rank, capacity test) -> dest, src_tok;
//                 the row is read once and written to its k destinations with
//                 16-byte vectors (BF16), or quantised once to E4M3 with a
//                 per-row scale and written k times.
// The ranks are deterministic: no global atomics decide any order.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dispatch_scan.cuh"
#include "route_topk.cuh"

namespace ap {
namespace {

constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / kWarp;

// One CTA of 1024 threads: the expert scan (dispatch_scan.cuh).
__global__ void __launch_bounds__(1024) k_scan(int32_t *__restrict__ blk, int nblk, int E, int capacity,
                                                int padded, int32_t *__restrict__ counts,
                                                int32_t *__restrict__ live, int32_t *__restrict__ seg_off)
{
    pdl_begin();
    int32_t my_live, my_off;
    scan_body(blk, nblk, E, capacity, padded, counts, live, seg_off, my_live, my_off);
}

// Block histogram and stable in-block ranks of the pairs [p0, p1) of one
// count/rank block (pair p = t*k + j), read from pidx[p - p0] (global or
// shared memory) by W warps.  The pairs are split into W contiguous ranges;
// each warp counts its range into cnt[w][e] (shared), a per-expert scan over
// warps gives each warp's base inside the block (the block totals go to
// blk_row[e]), then each warp walks its range 32 pairs at a time in order
// (match_any + popc).  dest[p] temporarily holds the pair's rank inside its
// block (-1 for an invalid id); the copy kernels add the block's base from the
// scan and write the final row.  The ranks do not depend on W.  Returns true
// if an id was out of range.
template <int W>
__device__ __forceinline__ bool block_count_rank(const int32_t *pidx, int64_t p0, int64_t p1, int E, int32_t *cnt,
                                                 int32_t *__restrict__ blk_row, int32_t *__restrict__ dest)
{
    const int lane = (int)lane_id(), wid = threadIdx.x / kWarp;
    for (int i = threadIdx.x; i < W * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int64_t per_warp = ((p1 - p0) + W - 1) / W;
    const int64_t w0 = p0 + wid * per_warp;
    const int64_t w1 = (w0 + per_warp < p1) ? w0 + per_warp : p1;
    int32_t *my = cnt + wid * E;
    bool bad = false;
    // phase 1: count per warp
    for (int64_t p = w0 + lane; p < w1; p += kWarp) {
        const int e = pidx[p - p0];
        if (e >= 0 && e < E) atomicAdd(&my[e], 1);
        else bad = true;
    }
    __syncthreads();
    // phase 2: per expert, exclusive scan over warps; the block total is the block's count
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = 0;
#pragma unroll
        for (int w2 = 0; w2 < W; ++w2) {
            const int32_t c = cnt[w2 * E + e];
            cnt[w2 * E + e] = run;
            run += c;
        }
        blk_row[e] = run;
    }
    __syncthreads();
    // phase 3: ordered walk, 32 pairs per step
    for (int64_t pb = w0; pb < w1; pb += kWarp) {
        const int64_t p = pb + lane;
        const bool in = p < w1;
        int e = in ? pidx[p - p0] : -1;
        const bool valid = in && e >= 0 && e < E;
        if (!valid) e = -1 - (int)(in ? 0 : 1); // -1: bad id, -2: past the end
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (valid) dest[p] = my[e] + __popc(peers & lanemask_lt());
        else if (in) dest[p] = -1;
        __syncwarp();
        if (valid && (peers & lanemask_lt()) == 0) my[e] += __popc(peers);
        __syncwarp();
    }
    return bad;
}

// Input rows a later kernel of the call reads, brought into L2 ahead of it.
// The metadata kernels that run before a row copy leave HBM idle; a bulk
// prefetch of their block's rows [t0, t0 + ntok) then lets the copy read its
// input from L2 while it streams its writes.  A hint only: nothing waits on
// it and no result depends on it, and L2 is where global memory is coherent,
// so the kernels issue it before their dependency wait, overlapping the tail
// of the kernel before them.  x and rb are 16-byte multiples (the caller
// passes x = nullptr otherwise).
struct RowPrefetch {
    const uint8_t *x;
    int64_t rb;
};

__device__ __forceinline__ void prefetch_rows_l2(RowPrefetch pf, int64_t t0, int64_t ntok)
{
    if (!pf.x || ntok <= 0) return;
    constexpr int64_t kPiece = 64 << 10;
    const int64_t begin = t0 * pf.rb, bytes = ntok * pf.rb;
    for (int64_t i = threadIdx.x; i * kPiece < bytes; i += blockDim.x) {
        const int64_t off = i * kPiece;
        const uint32_t n = (uint32_t)(bytes - off < kPiece ? bytes - off : kPiece);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(pf.x + begin + off), "r"(n) : "memory");
    }
}

// Count/rank blocks of kTokPerBlk tokens reading idx from global memory.
__global__ void __launch_bounds__(kRankThreads) k_count_rank(const int32_t *__restrict__ idx, int64_t T, int k, int E,
                                                             int32_t *__restrict__ blk, int32_t *__restrict__ dest,
                                                             uint32_t *d_status, RowPrefetch pf)
{
    { // a hint that changes no value: issued before the wait, so it overlaps the previous kernel's tail
        const int64_t t0 = (int64_t)blockIdx.x * kTokPerBlk;
        prefetch_rows_l2(pf, t0, (T - t0 < kTokPerBlk) ? T - t0 : kTokPerBlk);
    }
    pdl_begin();
    extern __shared__ int32_t cnt[]; // [kRankWarps][E]
    const int64_t p0 = (int64_t)blockIdx.x * kTokPerBlk * k;
    const int64_t p1 = (p0 + (int64_t)kTokPerBlk * k < T * k) ? p0 + (int64_t)kTokPerBlk * k : T * k;
    const bool bad = block_count_rank<kRankWarps>(idx + p0, p0, p1, E, cnt, blk + (int64_t)blockIdx.x * E, dest);
    if (bad && d_status) atomicOr(d_status, AP_FLAG_BAD_INDEX);
}

// Route + count/rank: one block of 32 warps routes its kTokPerBlk tokens
// (route_topk.cuh; warp w takes tokens w and w + 32), writes idx and w, keeps
// the block's ids in shared memory and ranks them there (block_count_rank), so
// the ids are never read back from global memory.  Same idx, w, block counts
// and ranks as k_route_topk followed by k_count_rank.
constexpr int kRouteRankWarps = 32;

template <int NV>
__global__ void __launch_bounds__(kRouteRankWarps * kWarp) k_route_count_rank(
    const float *__restrict__ logits, int64_t T, int E, int k, int32_t *__restrict__ idx, float *__restrict__ w,
    int32_t *__restrict__ blk, int32_t *__restrict__ dest, RowPrefetch pf)
{
    {
        const int64_t t0 = (int64_t)blockIdx.x * kTokPerBlk;
        prefetch_rows_l2(pf, t0, (T - t0 < kTokPerBlk) ? T - t0 : kTokPerBlk); // before the wait, as k_count_rank
    }
    pdl_begin();
    extern __shared__ int32_t smem[]; // cnt [32][E], then the block's ids [kTokPerBlk * k]
    int32_t *cnt = smem;
    int32_t *sidx = smem + kRouteRankWarps * E;
    const int lane = (int)lane_id(), wid = threadIdx.x / kWarp;
    const int64_t t0 = (int64_t)blockIdx.x * kTokPerBlk;
    const int ntok = (int)((T - t0 < kTokPerBlk) ? T - t0 : kTokPerBlk);
    for (int tt = wid; tt < ntok; tt += kRouteRankWarps) {
        int e;
        float wt;
        route_token<NV>(logits + (t0 + tt) * E, E, k, lane, &e, &wt);
        if (lane < k) {
            const int64_t p = (t0 + tt) * k + lane;
            idx[p] = e;
            w[p] = wt;
            sidx[tt * k + lane] = e;
        }
    }
    // block_count_rank starts with a barrier after clearing cnt: sidx is complete by then
    (void)block_count_rank<kRouteRankWarps>(sidx, t0 * k, (t0 + ntok) * k, E, cnt, blk + (int64_t)blockIdx.x * E,
                                            dest); // routed ids are always in range
}

// ---- BF16 row copy: one warp per token, row read once, written k times ------
template <typename V>
__global__ void __launch_bounds__(256) k_copy_rows(const uint8_t *__restrict__ x, int64_t T, int64_t rb,
                                                   const int32_t *__restrict__ idx, int32_t *__restrict__ dest,
                                                   int k, int E, int capacity, const int32_t *__restrict__ blk,
                                                   const int32_t *__restrict__ seg_off,
                                                   int32_t *__restrict__ src_tok, uint8_t *__restrict__ xd)
{
    pdl_begin();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    const int64_t nvec = rb / (int64_t)sizeof(V);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        const int32_t my_d =
            (lane < k) ? finalize_dest(idx, dest, src_tok, blk, seg_off, t, lane, k, E, capacity) : -1;
        const V *src = reinterpret_cast<const V *>(x + t * rb);
        constexpr int U = 4;
        // warp-uniform loop: every lane reaches the shuffles below
        for (int64_t base = 0; base < nvec; base += U * kWarp) {
            V r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = base + u * kWarp + lane;
                if (v < nvec) r[u] = ld_stream(src + v);
            }
            for (int j = 0; j < k; ++j) {
                const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
                if (d < 0) continue;
                V *dst = reinterpret_cast<V *>(xd + (int64_t)d * rb);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = base + u * kWarp + lane;
                    if (v < nvec) dst[v] = r[u];
                }
            }
        }
    }
}

// ---- E4M3 quantise + copy: one warp per token -------------------------------

// VE bf16 elements per lane step: 8 (16-byte loads, 8-byte stores), 4, 2 or 1.
template <int VE>
__global__ void __launch_bounds__(256) k_copy_rows_e4m3(const uint16_t *__restrict__ x, int64_t T, int H,
                                                        const int32_t *__restrict__ idx, int32_t *__restrict__ dest,
                                                        int k, int E, int capacity, const int32_t *__restrict__ blk,
                                                        const int32_t *__restrict__ seg_off,
                                                        int32_t *__restrict__ src_tok, uint8_t *__restrict__ xd,
                                                        float *__restrict__ xd_scale)
{
    pdl_begin();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    const int nstep = H / VE;
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        const int32_t my_d =
            (lane < k) ? finalize_dest(idx, dest, src_tok, blk, seg_off, t, lane, k, E, capacity) : -1;
        const uint16_t *row = x + t * H;
        // pass 1: amax
        float amax = 0.f;
        for (int s = lane; s < nstep; s += kWarp) {
            uint16_t e[VE];
            if constexpr (VE == 8) {
                const int4 v = *reinterpret_cast<const int4 *>(row + s * 8);
                memcpy(e, &v, 16);
            } else if constexpr (VE == 4) {
                const int2 v = *reinterpret_cast<const int2 *>(row + s * 4);
                memcpy(e, &v, 8);
            } else if constexpr (VE == 2) {
                const int v = *reinterpret_cast<const int *>(row + s * 2);
                memcpy(e, &v, 4);
            } else {
                e[0] = row[s];
            }
#pragma unroll
            for (int i = 0; i < VE; ++i) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(e[i])));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
        const float inv = (amax == 0.f) ? 1.f : __fdiv_rn(448.f, amax);
        if (lane < k && my_d >= 0) xd_scale[my_d] = scale;
        // pass 2: quantise once, store to every destination (warp-uniform loop)
        for (int s0 = 0; s0 < nstep; s0 += kWarp) {
            const int s = s0 + lane;
            const bool on = s < nstep;
            uint16_t e[VE];
#pragma unroll
            for (int i = 0; i < VE; ++i) e[i] = 0;
            if (on) {
            if constexpr (VE == 8) {
                const int4 v = *reinterpret_cast<const int4 *>(row + s * 8);
                memcpy(e, &v, 16);
            } else if constexpr (VE == 4) {
                const int2 v = *reinterpret_cast<const int2 *>(row + s * 4);
                memcpy(e, &v, 8);
            } else if constexpr (VE == 2) {
                const int v = *reinterpret_cast<const int *>(row + s * 2);
                memcpy(e, &v, 4);
            } else {
                e[0] = row[s];
            }
            }
            uint8_t q[VE];
#pragma unroll
            for (int i = 0; i < VE; ++i) q[i] = to_e4m3(__fmul_rn(bf16_bits_to_f32(e[i]), inv));
            for (int j = 0; j < k; ++j) {
                const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
                if (d < 0 || !on) continue;
                uint8_t *dst = xd + (int64_t)d * H + (int64_t)s * VE;
                if constexpr (VE == 8) {
                    int2 o;
                    memcpy(&o, q, 8);
                    *reinterpret_cast<int2 *>(dst) = o;
                } else if constexpr (VE == 4) {
                    int o;
                    memcpy(&o, q, 4);
                    *reinterpret_cast<int *>(dst) = o;
                } else if constexpr (VE == 2) {
                    short o;
                    memcpy(&o, q, 2);
                    *reinterpret_cast<short *>(dst) = o;
                } else {
                    dst[0] = q[0];
                }
            }
        }
    }
}

// E4M3 with the whole row held in registers (VE = 8 bf16 per 16-byte vector,
// at most NR vectors per lane, i.e. H <= 256 * NR): one read of the row, amax
// from registers, quantise once, store to every destination.  Same arithmetic
// as k_copy_rows_e4m3.
template <int NR>
__global__ void __launch_bounds__(256) k_copy_rows_e4m3_reg(const uint16_t *__restrict__ x, int64_t T, int H,
                                                            const int32_t *__restrict__ idx,
                                                            int32_t *__restrict__ dest, int k, int E, int capacity,
                                                            const int32_t *__restrict__ blk,
                                                            const int32_t *__restrict__ seg_off,
                                                            int32_t *__restrict__ src_tok, uint8_t *__restrict__ xd,
                                                            float *__restrict__ xd_scale)
{
    pdl_begin();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    const int nstep = H / 8;
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        const int32_t my_d =
            (lane < k) ? finalize_dest(idx, dest, src_tok, blk, seg_off, t, lane, k, E, capacity) : -1;
        const int4 *row = reinterpret_cast<const int4 *>(x + t * H);
        int4 v[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int s = lane + i * kWarp;
            v[i] = (s < nstep) ? ld_stream(row + s) : make_int4(0, 0, 0, 0);
        }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            m = absmax_bf16x2(m, (uint32_t)v[i].x);
            m = absmax_bf16x2(m, (uint32_t)v[i].y);
            m = absmax_bf16x2(m, (uint32_t)v[i].z);
            m = absmax_bf16x2(m, (uint32_t)v[i].w);
        }
        float scale, inv;
        e4m3_scales(__reduce_max_sync(0xffffffffu, absmax_bits(m)), scale, inv);
        if (lane < k && my_d >= 0) xd_scale[my_d] = scale;
        // codes replace the values in place (8 code bytes in the vector's first half)
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int2 c = quantize8_e4m3(v[i], inv);
            v[i].x = c.x;
            v[i].y = c.y;
        }
        for (int j = 0; j < k; ++j) {
            const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
            if (d < 0) continue;
            uint8_t *drow = xd + (int64_t)d * H;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const int s = lane + i * kWarp;
                if (s < nstep) *reinterpret_cast<int2 *>(drow + (int64_t)s * 8) = make_int2(v[i].x, v[i].y);
            }
        }
    }
}

// Pairs of values per conversion instruction, as the dispatch kernels convert.
__global__ void k_cast_e4m3(const float *__restrict__ in, uint8_t *__restrict__ out, int64_t n)
{
    pdl_begin();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; 2 * i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (2 * i + 1 < n) {
            const uint16_t q = __nv_cvt_float2_to_fp8x2(make_float2(in[2 * i], in[2 * i + 1]), __NV_SATFINITE,
                                                        __NV_E4M3);
            out[2 * i] = (uint8_t)(q & 0xffu);
            out[2 * i + 1] = (uint8_t)(q >> 8);
        } else {
            out[2 * i] = to_e4m3(in[2 * i]);
        }
    }
}

int64_t nblocks(int64_t T) { return (T + kTokPerBlk - 1) / kTokPerBlk; }

// Arguments every copy kernel needs to finish the pairs' rows (finalize_dest).
struct Ranks {
    const int32_t *idx;
    int32_t *dest;
    int k, E, capacity;
    const int32_t *blk, *seg_off;
    int32_t *src_tok;
};

template <typename V>
void launch_copy(const uint8_t *x, int64_t T, int64_t rb, const Ranks &r, uint8_t *xd, cudaStream_t st)
{
    // one warp per token; blocks beyond the resident ones start as others retire
    const int64_t want = (T + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 16;
    launch(k_copy_rows<V>, (int)(want < cap ? want : cap), 256, 0, st, x, T, rb, r.idx, r.dest, r.k, r.E, r.capacity,
                                                                   r.blk, r.seg_off, r.src_tok, xd);
}

template <int NR>
void launch_e4m3_reg(const uint16_t *x, int64_t T, int H, const Ranks &r, uint8_t *xd, float *xd_scale,
                     cudaStream_t st)
{
    const int64_t want = (T + 7) / 8; // one warp per token
    const int64_t cap = (int64_t)sm_count() * 16;
    launch(k_copy_rows_e4m3_reg<NR>, (int)(want < cap ? want : cap), 256, 0, st, 
        x, T, H, r.idx, r.dest, r.k, r.E, r.capacity, r.blk, r.seg_off, r.src_tok, xd, xd_scale);
}

template <int VE>
void launch_e4m3(const uint16_t *x, int64_t T, int H, const Ranks &r, uint8_t *xd, float *xd_scale, cudaStream_t st)
{
    static const int resident = resident_grid((const void *)k_copy_rows_e4m3<VE>, 256);
    const int64_t want = (T + 7) / 8; // one warp per token
    launch(k_copy_rows_e4m3<VE>, (int)(want < resident ? want : resident), 256, 0, st, 
        x, T, H, r.idx, r.dest, r.k, r.E, r.capacity, r.blk, r.seg_off, r.src_tok, xd, xd_scale);
}

} // namespace
} // namespace ap

extern "C" ap_status ap_dispatch_scratch_bytes(int64_t T, int32_t k, int32_t E, int64_t *bytes)
{
    using namespace ap;
    if (!bytes || T < 0 || k < 1 || E < 1) return fail(AP_EINVAL, "dispatch_scratch_bytes: bad arguments");
    *bytes = (nblocks(T) * E * (int64_t)sizeof(int32_t) + 255) / 256 * 256;
    if (*bytes == 0) *bytes = 256;
    return AP_OK;
}

namespace ap {

ap_status dispatch_check(const char *who, const void *x, int64_t T, int32_t H, const int32_t *idx, int32_t k,
                         int32_t E, int32_t capacity, int32_t padded, const void *xd, int64_t xd_rows,
                         const int32_t *counts, const int32_t *live, const int32_t *seg_off, const int32_t *dest,
                         const void *scratch, int64_t scratch_bytes)
{
    if (T < 0 || H < 1 || k < 1 || k > 32 || E < 1 || E > 1024 || T * (int64_t)k >= (int64_t(1) << 31))
        return fail(AP_EINVAL, "%s: bad sizes T=%lld H=%d k=%d E=%d", who, (long long)T, H, k, E);
    if (padded && capacity <= 0) return fail(AP_EINVAL, "%s: padded layout needs capacity > 0", who);
    const int64_t need_rows = padded ? (int64_t)E * capacity : T * (int64_t)k;
    if (xd_rows < need_rows)
        return fail(AP_EINVAL, "%s: xd_rows %lld < %lld", who, (long long)xd_rows, (long long)need_rows);
    int64_t need_scratch = 0;
    ap_dispatch_scratch_bytes(T, k, E, &need_scratch);
    if (scratch_bytes < need_scratch)
        return fail(AP_EINVAL, "%s: scratch %lld < %lld bytes", who, (long long)scratch_bytes,
                    (long long)need_scratch);
    if (!counts || !live || !seg_off || !scratch || (T > 0 && (!x || !idx || !dest || !xd)))
        return fail(AP_EINVAL, "%s: NULL pointer", who);
    return AP_OK;
}

// The row prefetch of the copy that follows: only for 16-byte aligned rows.
static RowPrefetch row_prefetch(const void *x, int64_t x_rb)
{
    const bool ok = x && ((reinterpret_cast<uintptr_t>(x) | (uintptr_t)x_rb) & 15) == 0;
    return RowPrefetch{ok ? static_cast<const uint8_t *>(x) : nullptr, x_rb};
}

ap_status dispatch_count_rank(int64_t T, const int32_t *idx, int32_t k, int32_t E, void *scratch, int32_t *dest,
                              uint32_t *d_status, cudaStream_t st, const void *x, int64_t x_rb)
{
    const int64_t nb = nblocks(T);
    if (nb == 0) return AP_OK;
    const size_t smem = (size_t)kRankWarps * E * sizeof(int32_t);
    launch(k_count_rank, (unsigned)nb, kRankThreads, smem, st, idx, T, k, E, static_cast<int32_t *>(scratch), dest,
           d_status, row_prefetch(x, x_rb));
    AP_CHECK_LAUNCH("dispatch count/rank launch");
    return AP_OK;
}

int dispatch_blocks(int64_t T) { return (int)nblocks(T); }

template <int NV>
ap_status launch_route_count_rank(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *idx, float *w,
                                  int32_t *blk, int32_t *dest, cudaStream_t st, RowPrefetch pf)
{
    const size_t smem = ((size_t)kRouteRankWarps * E + (size_t)kTokPerBlk * k) * sizeof(int32_t);
    static const cudaError_t attr = cudaFuncSetAttribute((const void *)k_route_count_rank<NV>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)((kRouteRankWarps * 1024 + kTokPerBlk * 32) *
                                                               sizeof(int32_t)));
    if (attr != cudaSuccess) return cuda_fail(attr, "route + count/rank: shared memory limit");
    launch(k_route_count_rank<NV>, (unsigned)nblocks(T), kRouteRankWarps * kWarp, smem, st, logits, T, E, k, idx, w,
           blk, dest, pf);
    AP_CHECK_LAUNCH("route + count/rank launch");
    return AP_OK;
}

ap_status dispatch_route_count_rank(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *idx, float *w,
                                    void *scratch, int32_t *dest, cudaStream_t st, const void *x, int64_t x_rb)
{
    if (nblocks(T) == 0) return AP_OK;
    int32_t *blk = static_cast<int32_t *>(scratch);
    const RowPrefetch pf = row_prefetch(x, x_rb);
    if (E <= 32) return launch_route_count_rank<1>(logits, T, E, k, idx, w, blk, dest, st, pf);
    if (E <= 64) return launch_route_count_rank<2>(logits, T, E, k, idx, w, blk, dest, st, pf);
    if (E <= 128) return launch_route_count_rank<4>(logits, T, E, k, idx, w, blk, dest, st, pf);
    if (E <= 256) return launch_route_count_rank<8>(logits, T, E, k, idx, w, blk, dest, st, pf);
    // more than 8 candidates per lane do not fit a 1024-thread block's
    // registers: route and count/rank as two launches
    ap_status s = ap_route_topk(logits, T, E, k, idx, w, st);
    if (s != AP_OK) return s;
    return dispatch_count_rank(T, idx, k, E, scratch, dest, nullptr, st, x, x_rb);
}

ap_status dispatch_metadata(int64_t T, const int32_t *idx, int32_t k, int32_t E, int32_t capacity, int32_t padded,
                            int32_t *counts, int32_t *live, int32_t *seg_off, int32_t *dest, void *scratch,
                            uint32_t *d_status, cudaStream_t st, const void *x, int64_t x_rb)
{
    ap_status s = dispatch_count_rank(T, idx, k, E, scratch, dest, d_status, st, x, x_rb);
    if (s != AP_OK) return s;
    launch(k_scan, 1, 1024, 0, st, static_cast<int32_t *>(scratch), (int)nblocks(T), E, capacity, padded, counts, live,
                               seg_off);
    AP_CHECK_LAUNCH("dispatch scan launch");
    return AP_OK;
}

} // namespace ap

extern "C" ap_status ap_dispatch_permute(const void *x, int64_t T, int32_t H, const int32_t *idx, int32_t k,
                                         int32_t E, int32_t capacity, int32_t padded, int32_t out_dtype, void *xd,
                                         float *xd_scale, int64_t xd_rows, int32_t *counts, int32_t *live,
                                         int32_t *seg_off, int32_t *dest, int32_t *src_tok, void *scratch,
                                         int64_t scratch_bytes, uint32_t *d_status, void *stream)
{
    AP_NVTX_RANGE("ap_dispatch_permute");
    using namespace ap;
    if (out_dtype != AP_DTYPE_BF16 && out_dtype != AP_DTYPE_E4M3)
        return fail(AP_EINVAL, "dispatch_permute: unknown out_dtype %d", out_dtype);
    ap_status s = dispatch_check("dispatch_permute", x, T, H, idx, k, E, capacity, padded, xd, xd_rows, counts, live,
                                 seg_off, dest, scratch, scratch_bytes);
    if (s != AP_OK) return s;
    if (out_dtype == AP_DTYPE_E4M3 && T > 0 && !xd_scale)
        return fail(AP_EINVAL, "dispatch_permute: E4M3 needs xd_scale");
    cudaStream_t st = (cudaStream_t)stream;
    s = dispatch_metadata(T, idx, k, E, capacity, padded, counts, live, seg_off, dest, scratch, d_status, st, x,
                          (int64_t)H * 2);
    if (s != AP_OK || T == 0) return s;
    const Ranks ranks{idx, dest, k, E, capacity, static_cast<const int32_t *>(scratch), seg_off, src_tok};
    if (out_dtype == AP_DTYPE_BF16) {
        const int64_t rb = (int64_t)H * 2;
        const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xd) | (uintptr_t)rb;
        const uint8_t *xs = static_cast<const uint8_t *>(x);
        uint8_t *xo = static_cast<uint8_t *>(xd);
        if ((al & 15) == 0)
            launch_copy<int4>(xs, T, rb, ranks, xo, st);
        else if ((al & 7) == 0)
            launch_copy<int2>(xs, T, rb, ranks, xo, st);
        else if ((al & 3) == 0)
            launch_copy<int>(xs, T, rb, ranks, xo, st);
        else
            launch_copy<short>(xs, T, rb, ranks, xo, st);
    } else {
        const uint16_t *xs = static_cast<const uint16_t *>(x);
        uint8_t *xo = static_cast<uint8_t *>(xd);
        const uintptr_t ax = reinterpret_cast<uintptr_t>(x), ao = reinterpret_cast<uintptr_t>(xd);
        if (H % 8 == 0 && (ax & 15) == 0 && (ao & 7) == 0 && H <= 256 * 4)
            launch_e4m3_reg<4>(xs, T, H, ranks, xo, xd_scale, st);
        else if (H % 8 == 0 && (ax & 15) == 0 && (ao & 7) == 0 && H <= 256 * 8)
            launch_e4m3_reg<8>(xs, T, H, ranks, xo, xd_scale, st);
        else if (H % 8 == 0 && (ax & 15) == 0 && (ao & 7) == 0 && H <= 256 * 9)
            launch_e4m3_reg<9>(xs, T, H, ranks, xo, xd_scale, st);
        else if (H % 8 == 0 && (ax & 15) == 0 && (ao & 7) == 0)
            launch_e4m3<8>(xs, T, H, ranks, xo, xd_scale, st);
        else if (H % 4 == 0 && (ax & 7) == 0 && (ao & 3) == 0)
            launch_e4m3<4>(xs, T, H, ranks, xo, xd_scale, st);
        else if (H % 2 == 0 && (ax & 3) == 0 && (ao & 1) == 0)
            launch_e4m3<2>(xs, T, H, ranks, xo, xd_scale, st);
        else
            launch_e4m3<1>(xs, T, H, ranks, xo, xd_scale, st);
    }
    AP_CHECK_LAUNCH("dispatch copy launch");
    return AP_OK;
}

extern "C" ap_status ap_count_rank(const float *logits, float *w, int32_t *idx, int64_t T, int32_t k, int32_t E,
                                   const void *x, int64_t row_bytes, int32_t *dest, void *scratch,
                                   int64_t scratch_bytes, int32_t capacity, int32_t padded, int32_t *counts,
                                   int32_t *live, int32_t *seg_off, uint32_t *d_status, void *stream)
{
    AP_NVTX_RANGE("ap_count_rank");
    using namespace ap;
    if (T < 0 || k < 1 || k > 32 || E < 1 || E > 1024 || T * (int64_t)k >= (int64_t(1) << 31))
        return fail(AP_EINVAL, "count_rank: bad sizes T=%lld k=%d E=%d", (long long)T, k, E);
    if (logits && k > E) return fail(AP_EINVAL, "count_rank: k=%d > E=%d", k, E);
    int64_t need = 0;
    ap_dispatch_scratch_bytes(T, k, E, &need);
    if (scratch_bytes < need)
        return fail(AP_EINVAL, "count_rank: scratch %lld < %lld bytes", (long long)scratch_bytes, (long long)need);
    if (!scratch || (T > 0 && (!idx || !dest || (logits && !w)))) return fail(AP_EINVAL, "count_rank: NULL pointer");
    if (row_bytes < 0) return fail(AP_EINVAL, "count_rank: row_bytes %lld < 0", (long long)row_bytes);
    const bool scan = counts || live || seg_off;
    if (scan && (!counts || !live || !seg_off)) return fail(AP_EINVAL, "count_rank: counts, live, seg_off: all or none");
    if (scan && padded && capacity <= 0) return fail(AP_EINVAL, "count_rank: padded layout needs capacity > 0");
    cudaStream_t st = (cudaStream_t)stream;
    ap_status s = logits ? dispatch_route_count_rank(logits, T, E, k, idx, w, scratch, dest, st, x, row_bytes)
                         : dispatch_count_rank(T, idx, k, E, scratch, dest, d_status, st, x, row_bytes);
    if (s != AP_OK || !scan) return s;
    // the dispatch's expert scan: block bases in place of the histograms, counts, live, seg_off
    // the fewest threads the scan takes (at least E): a small block finds room beside running copies sooner
    const int threads = E <= 256 ? 256 : (E <= 512 ? 512 : 1024);
    launch(k_scan, 1, threads, 0, st, static_cast<int32_t *>(scratch), (int)nblocks(T), E, capacity, padded, counts,
           live, seg_off);
    AP_CHECK_LAUNCH("count_rank scan launch");
    return AP_OK;
}

extern "C" ap_status ap_cast_e4m3(const float *in, uint8_t *out, int64_t n, void *stream)
{
    AP_NVTX_RANGE("ap_cast_e4m3");
    using namespace ap;
    if (n < 0) return fail(AP_EINVAL, "cast_e4m3: n < 0");
    if (n == 0) return AP_OK;
    if (!in || !out) return fail(AP_EINVAL, "cast_e4m3: NULL pointer");
    const int64_t want = (n + 255) / 256;
    const int grid = (int)(want < (int64_t)sm_count() * 8 ? want : (int64_t)sm_count() * 8);
    launch(k_cast_e4m3, grid, 256, 0, (cudaStream_t)stream, in, out, n);
    AP_CHECK_LAUNCH("cast_e4m3 launch");
    return AP_OK;
}
