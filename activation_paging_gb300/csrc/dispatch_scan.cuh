// Expert scan of the dispatch, shared by the dispatch kernels (dispatch.cu)
// and the fused scan + stash plan kernel (stash.cu).
#pragma once

#include <cuda_fp8.h>

#include "ap_common.cuh"

namespace ap {
namespace {

constexpr int kTokPerBlk = 64; // tokens per count/rank block

// One CTA of 1024 threads.  blk[b][e] -> exclusive base over b (in place).
// Thread (e, part) owns expert e over a contiguous range of blocks: it sums
// its range, adds the sums of the earlier parts, then rewrites its range as
// running bases.  Then counts, live = min(count, C) and segment offsets.
// my_live / my_off: thread tid < E also returns expert tid's live count and
// segment offset in registers (for a page plan run by the same CTA).
__device__ __forceinline__ void scan_body(int32_t *__restrict__ blk, int nblk, int E, int capacity, int padded,
                                          int32_t *__restrict__ counts, int32_t *__restrict__ live,
                                          int32_t *__restrict__ seg_off, int32_t &my_live, int32_t &my_off)
{
    __shared__ int32_t s_tot[1024];
    __shared__ int32_t s_warp[32];
    const int tid = threadIdx.x;
    const int parts = blockDim.x / E; // >= 1 since E <= 1024
    const int e = tid % E, part = tid / E;
    const bool active = part < parts;
    const int per = (nblk + parts - 1) / parts;
    const int b0 = part * per;
    const int b1 = (b0 + per < nblk) ? b0 + per : nblk;
    // short ranges stay in registers between the two passes (one round trip)
    constexpr int kReg = 16;
    const bool in_reg = per <= kReg;
    int32_t cr[kReg];
    int32_t sum = 0;
    if (active && in_reg) {
#pragma unroll
        for (int u = 0; u < kReg; ++u) cr[u] = (b0 + u < b1) ? blk[(int64_t)(b0 + u) * E + e] : 0;
#pragma unroll
        for (int u = 0; u < kReg; ++u) sum += cr[u];
    } else if (active) {
        int b = b0;
        for (; b + 8 <= b1; b += 8) {
            int32_t c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = blk[(int64_t)(b + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) sum += c[u];
        }
        for (; b < b1; ++b) sum += blk[(int64_t)b * E + e];
    }
    s_tot[tid] = active ? sum : 0;
    __syncthreads();
    int32_t total = 0;
    if (active) {
        int32_t run = 0;
        for (int p = 0; p < parts; ++p) {
            if (p == part) run = total;
            total += s_tot[p * E + e];
        }
        if (in_reg) {
#pragma unroll
            for (int u = 0; u < kReg; ++u) {
                if (b0 + u < b1) blk[(int64_t)(b0 + u) * E + e] = run;
                run += cr[u];
            }
        } else {
            int b = b0;
            for (; b + 8 <= b1; b += 8) {
                int32_t c[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) c[u] = blk[(int64_t)(b + u) * E + e];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    blk[(int64_t)(b + u) * E + e] = run;
                    run += c[u];
                }
            }
            for (; b < b1; ++b) {
                const int32_t c = blk[(int64_t)b * E + e];
                blk[(int64_t)b * E + e] = run;
                run += c;
            }
        }
    }
    // threads tid < E (part 0) own expert tid's totals
    const int32_t l = (tid < E) ? ((capacity > 0 && total > capacity) ? capacity : total) : 0;
    if (tid < E) {
        counts[tid] = total;
        live[tid] = l;
    }
    // exclusive scan of live over experts (compact layout)
    int32_t x = l;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int32_t v = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += y;
        }
        s_warp[lane] = v;
    }
    __syncthreads();
    const int32_t incl = x + (wid > 0 ? s_warp[wid - 1] : 0);
    my_live = l;
    my_off = padded ? tid * capacity : incl - l;
    if (tid < E) seg_off[tid] = my_off;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// E4M3 code of a float: round to nearest even, finite overflow saturates.
__device__ __forceinline__ uint8_t to_e4m3(float v)
{
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Row amax of the E4M3 quantisation on packed BF16 (two values per 32-bit
// word).  |x| clears the sign bits; NaN halves (above 0x7F80) become 0, so a
// NaN never wins, as in a float max; the halves are then maxed as unsigned
// 16-bit integers, whose order is the order of non-negative values.  Exactly
// max |x| over the non-NaN values, two values per instruction.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t w)
{
    const uint32_t a = w & 0x7fff7fffu;
    return __vmaxu2(m, a & ~__vcmpgtu2(a, 0x7f807f80u));
}

// The larger half of a packed absmax as the bits of a non-negative float
// (unsigned order = value order, so a warp reduces it with one redux.sync).
__device__ __forceinline__ uint32_t absmax_bits(uint32_t m)
{
    const uint32_t lo = m & 0xffffu, hi = m >> 16;
    return (lo > hi ? lo : hi) << 16;
}

// E4M3 codes of the eight BF16 values of v times inv, in element order: each
// product is rounded to float, then converted with round-to-nearest-even and
// finite saturation, two values per conversion instruction.
__device__ __forceinline__ int2 quantize8_e4m3(const int4 &v, float inv)
{
    const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __fmul_rn(__uint_as_float(w[i] << 16), inv);
        const float hi = __fmul_rn(__uint_as_float(w[i] & 0xffff0000u), inv);
        q[i] = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    }
    return make_int2((int)(q[0] | (q[1] << 16)), (int)(q[2] | (q[3] << 16)));
}

// Scale and inverse scale of a row from its amax bits (amax 0: both 1).
__device__ __forceinline__ void e4m3_scales(uint32_t amax_bits, float &scale, float &inv)
{
    const float amax = __uint_as_float(amax_bits);
    scale = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
    inv = (amax == 0.f) ? 1.f : __fdiv_rn(448.f, amax);
}

// Row of pair (t, j) from its in-block rank (left in dest by k_count_rank) and
// the block bases (left in blk by the scan): rank = base[b][e] + in-block
// rank; kept iff capacity <= 0 or rank < capacity.  Writes the final dest and,
// for a kept pair, src_tok; returns the row or -1.  Called once per pair.
__device__ __forceinline__ int32_t finalize_dest(const int32_t *__restrict__ idx, int32_t *__restrict__ dest,
                                                 int32_t *__restrict__ src_tok, const int32_t *__restrict__ blk,
                                                 const int32_t *__restrict__ seg_off, int64_t t, int j, int k, int E,
                                                 int capacity)
{
    const int64_t p = t * k + j;
    const int32_t lr = dest[p];
    if (lr < 0) return -1; // invalid expert id: already -1
    const int e = idx[p];
    const int32_t r = blk[(t / kTokPerBlk) * E + e] + lr;
    int32_t d = -1;
    if (capacity <= 0 || r < capacity) {
        d = seg_off[e] + r;
        if (src_tok) src_tok[d] = (int32_t)t;
    }
    dest[p] = d;
    return d;
}

} // namespace
} // namespace ap
