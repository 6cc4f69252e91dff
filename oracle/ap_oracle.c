/*
 * CPU oracle for the MoE token-movement path with a paged activation stash.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load this file's
 * library: only the tests, the smoke check of the build entry point and the
 * CPU-baseline / reference arm of the benchmark call it.  It shares no source,
 * header, table or helper with the CUDA library; both sides receive the same
 * seeded input bytes and nothing else.
 *
 * Plain, single-threaded C99, compiled with -ffp-contract=off so that every
 * float expression below is one IEEE operation rounded to nearest-even (no
 * fused multiply-add).  Each function follows the plain definition of its
 * step, in the order the sources state it, and cites the passage it follows.
 * Sources (web pages):
 *   [TT5541]  torchtitan pull 5541, HybridEP eager scheduling with a paged
 *             activation stash, section "AI-Generated Details".
 *   [TT5542]  torchtitan pull 5542, "[graph_trainer] Overlap HybridEP and
 *             paging across combined PP graphs".
 *   [MG7342]  Megatron-LM pull 7342, token-wise ChunkedEP for Qwen3 MoE
 *             ("Summary", "Validation and performance").
 *   [ART971]  OpenPipe/ART pull 971, "Price HybridEP recompute outputs at the
 *             live communication extent".
 * Where the sources are silent the oracle takes one stated reading; the
 * readings are listed beside each function.
 *
 * Parity status: each function is pinned by CPU tests that do not re-run its
 * own arithmetic (tests/test_oracle_*.py):
 *   or_route_topk           closed forms, numpy's stable sort and scipy's
 *                           softmax, ties, shift invariance, k = E and
 *                           E = k = 1 (test_oracle_route.py);
 *   or_dispatch_plan        brute-force counting, stable ranks, capacity and
 *                           both layouts, sum rules (test_oracle_dispatch.py);
 *   or_permute_rows         rows at dest, canary rows untouched
 *                           (test_oracle_dispatch.py);
 *   or_e4m3_encode(_n),
 *   or_e4m3_decode          an independent OCP E4M3 decoder: every code,
 *                           every midpoint, nearest on a grid, saturation
 *                           (test_oracle_fp8.py);
 *   or_quantize_rows_e4m3   scale = amax/448 in single precision, the largest
 *                           element at +-448, dequantisation error within
 *                           half a step (test_oracle_fp8.py);
 *   or_permute_rows_fp8     a numpy restatement of the row and scale
 *                           placement on hand-built dest maps with drops,
 *                           and the padded FP8 dispatch (test_oracle_fp8.py);
 *   or_combine, or_f32_to_bf16  exact double sums within the FP32 bound,
 *                           k = 1, all-dropped tokens, identity experts
 *                           (test_oracle_combine.py);
 *   or_combine_backward,
 *   or_dispatch_backward    exact gradients in rationals, unit weights,
 *                           dropped pairs, bad rows (test_oracle_backward.py);
 *   or_pool_*               FIFO order, byte survival, page conservation,
 *                           wrap-around, spill and loss, sticky flags, P = 1
 *                           (test_oracle_pool.py); calibration demand and
 *                           growth (test_oracle_calibrate.py).
 * None is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL -1
#define OR_EEMPTY -2
#define OR_EQFULL -3

/* Sticky flag bits of the pool (same meaning as the library's; the values are
 * an interface both sides must agree on, like a file format). */
#define OR_FLAG_POOL_OVERFLOW 0x1u   /* device pool exhausted, excess spilled  */
#define OR_FLAG_SPILL_OVERFLOW 0x2u  /* spill exhausted too, pages lost       */
#define OR_FLAG_RECORD_OVERFLOW 0x4u /* record needed more page-table entries */
#define OR_FLAG_BAD_COUNT 0x8u       /* live/offset outside the given buffer  */
#define OR_FLAG_BAD_INDEX 0x10u      /* expert or row index out of range      */

/* ------------------------------------------------------------------------- */
/* BF16 helpers.  BF16 is the top half of an IEEE single.                     */
/* ------------------------------------------------------------------------- */
static float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round an IEEE single to BF16 with round-to-nearest-even, written from the
 * definition: keep the high 16 bits, and add one unit in the last kept place
 * when the dropped half is above one half, or exactly one half with an odd
 * kept part.  NaN never reaches this in the method (finite inputs only). */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------------- */
/* (1) Router: softmax, top-k, renormalised weights.                          */
/*   [MG7342] "Validation and performance": top-k 8 routing over the experts. */
/*   Reading (sources silent): softmax in double over all E logits; the k     */
/*   largest logits are taken, an equal logit going to the lower expert id,   */
/*   in descending order (j = 0 is the top choice); w_j = p_j / sum_sel p,    */
/*   computed in double and rounded once to single.  Selection compares the  */
/*   raw single-precision logits, so the indices do not depend on exp().      */
/* ------------------------------------------------------------------------- */
int or_route_topk(const float *logits, int64_t T, int32_t E, int32_t k,
                  int32_t *idx, float *w)
{
    if (T < 0 || E < 1 || k < 1 || k > E)
        return OR_EINVAL;
    double *p = (double *)malloc((size_t)E * sizeof(double));
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!p || !taken) {
        free(p);
        free(taken);
        return OR_EINVAL;
    }
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        /* softmax over all experts */
        double m = (double)l[0];
        for (int32_t e = 1; e < E; ++e)
            if ((double)l[e] > m)
                m = (double)l[e];
        double Z = 0.0;
        for (int32_t e = 0; e < E; ++e) {
            p[e] = exp((double)l[e] - m);
            Z += p[e];
        }
        for (int32_t e = 0; e < E; ++e)
            p[e] = p[e] / Z;
        /* top-k by repeated selection of the best remaining logit */
        memset(taken, 0, (size_t)E);
        double S = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best]) /* strict: ties keep lower e */
                    best = e;
            }
            taken[best] = 1;
            idx[t * k + j] = best;
            S += p[best];
        }
        /* renormalise over the selected experts */
        for (int32_t j = 0; j < k; ++j)
            w[t * k + j] = (float)(p[idx[t * k + j]] / S);
    }
    free(p);
    free(taken);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* (2) Expert counts, capacity, stable rank, destination rows.                */
/*   [TT5541] "AI-Generated Details": reload restores the original capacity   */
/*   shape; [TT5542]: capacity division; [MG7342] "Summary": dispatch into    */
/*   expert buffers.                                                          */
/*   Readings: pairs (t, j) are visited t ascending then j ascending and each */
/*   expert keeps a running count, so a pair's rank is the number of earlier  */
/*   pairs routed to the same expert; a pair is kept iff capacity <= 0        */
/*   (dropless) or rank < capacity (first arrivals win).  live[e] = number of */
/*   kept rows.  Padded layout: seg_off[e] = e * capacity.  Compact layout:   */
/*   seg_off = exclusive prefix sum of live.  Dropped pairs get dest = -1.    */
/*   An expert id outside [0, E) is skipped (dest = -1) and flagged.          */
/* ------------------------------------------------------------------------- */
int or_dispatch_plan(const int32_t *idx, int64_t T, int32_t k, int32_t E,
                     int32_t capacity, int32_t padded, int32_t *counts,
                     int32_t *live, int32_t *seg_off, int32_t *dest,
                     int32_t *src_tok, int64_t src_tok_len, uint32_t *status)
{
    if (T < 0 || k < 1 || E < 1 || (padded && capacity <= 0))
        return OR_EINVAL;
    int32_t *rank = (int32_t *)malloc((size_t)(T * k + 1) * sizeof(int32_t));
    if (!rank)
        return OR_EINVAL;
    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = idx[t * k + j];
            if (e < 0 || e >= E) {
                rank[t * k + j] = -1;
                if (status)
                    *status |= OR_FLAG_BAD_INDEX;
                continue;
            }
            rank[t * k + j] = counts[e];
            counts[e] += 1;
        }
    }
    for (int32_t e = 0; e < E; ++e)
        live[e] = (capacity <= 0 || counts[e] < capacity) ? counts[e] : capacity;
    if (padded) {
        for (int32_t e = 0; e < E; ++e)
            seg_off[e] = e * capacity;
    } else {
        int32_t run = 0;
        for (int32_t e = 0; e < E; ++e) {
            seg_off[e] = run;
            run += live[e];
        }
    }
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t r = rank[t * k + j];
            int32_t e = idx[t * k + j];
            if (r < 0 || (capacity > 0 && r >= capacity)) {
                dest[t * k + j] = -1;
                continue;
            }
            int32_t row = seg_off[e] + r;
            dest[t * k + j] = row;
            if (src_tok && row < src_tok_len)
                src_tok[row] = (int32_t)t;
        }
    }
    free(rank);
    return OR_OK;
}

/* (3a) BF16 (or any opaque) payload: row dest(t, j) of xd is a byte copy of
 * row t of x, for every kept pair.  Rows never written keep their content.
 * [MG7342] "Summary" (dispatch to expert buffers). */
void or_permute_rows(const uint8_t *x, int64_t T, int64_t row_bytes,
                     const int32_t *dest, int32_t k, uint8_t *xd)
{
    for (int64_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t r = dest[t * k + j];
            if (r >= 0)
                memcpy(xd + (int64_t)r * row_bytes, x + t * row_bytes, (size_t)row_bytes);
        }
}

/* ------------------------------------------------------------------------- */
/* (3b) FP8 E4M3 payload with a per-row FP32 scale.                           */
/*   [TT5541] "Verification": the stash carries BF16 and FP8 payloads.        */
/*   Reading (sources silent on the recipe): E4M3 as in the OCP 8-bit         */
/*   floating point specification — 1 sign bit, 4 exponent bits with bias 7,  */
/*   3 mantissa bits, subnormals at exponent field 0, no infinity, the code   */
/*   S.1111.111 is NaN, largest finite magnitude 448.  Conversion rounds to   */
/*   nearest with ties to the even code and saturates finite overflow to      */
/*   +-448.  Per row: amax = max |x|; scale = amax / 448 and                  */
/*   inv = 448 / amax (single-precision divisions; both 1 when amax == 0);    */
/*   q = e4m3(x * inv) with a single-precision multiply; dequantised value is */
/*   q * scale.                                                               */
/* ------------------------------------------------------------------------- */

/* Value of a non-negative code 0x00..0x7E (0x7F is NaN). */
static double or_e4m3_magnitude(int code)
{
    int ef = (code >> 3) & 15;
    int mf = code & 7;
    if (ef == 0)
        return ldexp((double)mf, -9); /* subnormal: m/8 * 2^(1-7) */
    return ldexp((double)(8 + mf), ef - 10); /* (1 + m/8) * 2^(e-7) */
}

uint8_t or_e4m3_encode(float v)
{
    if (v != v)
        return 0x7Fu;
    uint8_t sign = signbit(v) ? 0x80u : 0x00u;
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7Eu); /* saturate finite overflow */
    /* largest code whose magnitude is <= a (codes are increasing) */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (or_e4m3_magnitude(mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int code = lo;
    if (or_e4m3_magnitude(code) != a) {
        double below = or_e4m3_magnitude(code);
        double above = or_e4m3_magnitude(code + 1);
        double half = (below + above) / 2.0; /* exact in double */
        if (a > half || (a == half && (code & 1)))
            code += 1;
    }
    return (uint8_t)(sign | (uint8_t)code);
}

double or_e4m3_decode(uint8_t c)
{
    if ((c & 0x7F) == 0x7F)
        return NAN;
    double m = or_e4m3_magnitude(c & 0x7F);
    return (c & 0x80) ? -m : m;
}

void or_e4m3_encode_n(const float *in, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_e4m3_encode(in[i]);
}

/* Quantise each BF16 row of x [T, H] to E4M3 codes q [T, H] and scale [T]. */
void or_quantize_rows_e4m3(const uint16_t *x, int64_t T, int32_t H,
                           uint8_t *q, float *scale)
{
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *row = x + t * H;
        float amax = 0.0f;
        for (int32_t h = 0; h < H; ++h) {
            float a = fabsf(or_bf16_to_f32(row[h]));
            if (a > amax)
                amax = a;
        }
        float s, inv;
        if (amax == 0.0f) {
            s = 1.0f;
            inv = 1.0f;
        } else {
            s = amax / 448.0f;
            inv = 448.0f / amax;
        }
        scale[t] = s;
        for (int32_t h = 0; h < H; ++h) {
            float v = or_bf16_to_f32(row[h]) * inv;
            q[t * H + h] = or_e4m3_encode(v);
        }
    }
}

/* FP8 dispatch: the quantised row t (H code bytes) and its scale are copied to
 * every kept destination row. */
void or_permute_rows_fp8(const uint8_t *q, const float *scale, int64_t T,
                         int32_t H, const int32_t *dest, int32_t k,
                         uint8_t *xd, float *xd_scale)
{
    for (int64_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t r = dest[t * k + j];
            if (r >= 0) {
                memcpy(xd + (int64_t)r * H, q + t * H, (size_t)H);
                xd_scale[r] = scale[t];
            }
        }
}

/* ------------------------------------------------------------------------- */
/* (6) Combine / un-permute.                                                  */
/*   [ART971] description and review: combine with un-permute writes a fresh  */
/*   dense BF16 output.  Reading (sources silent on the arithmetic): for each */
/*   token, acc = 0 in single precision; for j = 0..k-1 with a kept row,      */
/*   acc = acc + (w[t, j] * y[row]) as two separately rounded single          */
/*   operations; out = BF16(acc) rounded to nearest-even.  A token whose      */
/*   rows were all dropped gives +0.  A row index >= y_rows is skipped and    */
/*   flagged.                                                                 */
/* ------------------------------------------------------------------------- */
void or_combine(const uint16_t *y, int64_t y_rows, int32_t H,
                const int32_t *dest, const float *w, int64_t T, int32_t k,
                uint16_t *out, uint32_t *status)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                int32_t r = dest[t * k + j];
                if (r < 0)
                    continue;
                if (r >= y_rows) {
                    if (status)
                        *status |= OR_FLAG_BAD_INDEX;
                    continue;
                }
                float prod = w[t * k + j] * or_bf16_to_f32(y[(int64_t)r * H + h]);
                acc = acc + prod;
            }
            out[t * H + h] = or_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* (7) Backward of combine and of dispatch.                                   */
/*   [MG7342] "Summary": forward, backward and fused forward/backward         */
/*   primitives of the token movement.  The pages give no formulas; these are */
/*   the derivatives of the forward definitions above:                        */
/*     out[t] = sum_j w[t,j] * y[dest(t,j)]   and   xd[dest(t,j)] = x[t].     */
/*   Combine backward: dy[dest(t,j)] = BF16(w[t,j] * dout[t]) (one single     */
/*   multiply, nearest-even), dw[t,j] = <dout[t], y[dest(t,j)]> summed in     */
/*   double and rounded once to single; a dropped pair gets dw = 0 and        */
/*   writes no row.  Dispatch backward: dx[t] = BF16(sum_j dxd[dest(t,j)])    */
/*   with a single-precision accumulator, j ascending (the combine with unit  */
/*   weights).                                                                */
/* ------------------------------------------------------------------------- */
void or_combine_backward(const uint16_t *dout, const uint16_t *y, int64_t y_rows,
                         int32_t H, const int32_t *dest, const float *w,
                         int64_t T, int32_t k, uint16_t *dy, float *dw,
                         uint32_t *status)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t r = dest[t * k + j];
            dw[t * k + j] = 0.0f;
            if (r < 0)
                continue;
            if (r >= y_rows) {
                if (status)
                    *status |= OR_FLAG_BAD_INDEX;
                continue;
            }
            double dot = 0.0;
            for (int32_t h = 0; h < H; ++h) {
                float g = or_bf16_to_f32(dout[t * H + h]);
                float prod = w[t * k + j] * g;
                dy[(int64_t)r * H + h] = or_f32_to_bf16(prod);
                dot += (double)g * (double)or_bf16_to_f32(y[(int64_t)r * H + h]);
            }
            dw[t * k + j] = (float)dot;
        }
    }
}

void or_dispatch_backward(const uint16_t *dxd, int64_t rows, int32_t H,
                          const int32_t *dest, int64_t T, int32_t k, uint16_t *dx,
                          uint32_t *status)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                int32_t r = dest[t * k + j];
                if (r < 0)
                    continue;
                if (r >= rows) {
                    if (status)
                        *status |= OR_FLAG_BAD_INDEX;
                    continue;
                }
                acc = acc + or_bf16_to_f32(dxd[(int64_t)r * H + h]);
            }
            dx[t * H + h] = or_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* (4)-(5) Paged stash: fixed page pool, free list, spill, per-slot FIFO.     */
/*   [TT5541] "AI-Generated Details": one high-priority paging stream         */
/*   serialises free-list changes; per-slot records stay FIFO; copy loops in  */
/*   page-aligned multi-token tiles with live-prefix and page-tail masks and  */
/*   64-bit addressing; CUDA allocation, host spill and a sticky overflow     */
/*   flag; reload restores the original capacity shape.                       */
/*   [TT5541] "Verification": wrapped allocation and recycling, host spill,   */
/*   overflow.                                                                */
/* Readings (sources silent):                                                 */
/*   - the free list is a ring of N page ids, initially 0..N-1, pages taken   */
/*     from its head and returned to its tail; the spill list likewise over   */
/*     the spill pages;                                                       */
/*   - a push visits segments in order and, inside a segment, its            */
/*     ceil(live/P) pages in order; each page takes the next free device      */
/*     page, else the next free spill page (the excess spills), else it is    */
/*     lost (not copied);                                                     */
/*   - page-table entries: device page p -> p, spill page s -> NMAX + s,     */
/*     lost -> -1 (NMAX, the most device pages the pool may grow to, is N     */
/*     for a pool that never grows);                                          */
/*   - calibration ([TT5541] "AI-Generated Details": calibration parks live   */
/*     prefixes before the buffers exist): a pool may start with N = 0 device */
/*     pages, so every page of a push goes to the spill pages (or is lost);   */
/*     the pages held by queued records and their high-water mark measure the */
/*     device pages the schedule needs, and or_pool_grow adds them;           */
/*   - rows inside a page are dense: plane 0 at r*rb0, plane 1 at            */
/*     roundup16(P*rb0) + r*rb1; bytes of a page past its live rows are left  */
/*     untouched (page-tail mask); rows >= live are never copied (live-prefix */
/*     mask), and pop does not zero-fill them;                                */
/*   - "exactly full" is not an overflow; flags stay set until reset;         */
/*   - pop takes the slot's oldest record, copies every page back to the      */
/*     same rows, and returns pages in page-table order;                      */
/*   - a segment whose offset/live lie outside the source (push) or           */
/*     destination (pop) rows is not copied and sets BAD_COUNT; a record that */
/*     needs more than max_pages_per_record pages keeps the first ones and    */
/*     sets RECORD_OVERFLOW.                                                  */
/* ------------------------------------------------------------------------- */
typedef struct {
    uint64_t id;
    int32_t nplanes;
    int64_t rb[2];
    int32_t nseg;
    int32_t *seg_off; /* snapshot at push */
    int32_t *live;    /* snapshot at push, after validation */
    int64_t npages;
    int64_t ndev, nspill, nlost;
    int32_t *page_table; /* [npages] */
    int64_t *row0;       /* [npages] first source row of the page */
    int32_t *nrows;      /* [npages] rows held by the page */
} or_record;

typedef struct {
    int32_t P;
    int64_t page_bytes, N, SP;
    int64_t NMAX; /* most device pages the pool may grow to; spill ids start here */
    int32_t S, R, max_segs;
    int64_t max_pages;
    int32_t *ring, *spill_ring;
    uint64_t head, tail, spill_head, spill_tail;
    uint32_t flags;
    int64_t high_water, spill_high_water;
    int64_t held, held_high_water; /* pages (device + spill + lost) of queued records */
    uint8_t *pool;  /* N * page_bytes, or NULL (metadata only) */
    uint8_t *spill; /* SP * page_bytes, or NULL */
    or_record *q;   /* [S * R] */
    int32_t *q_head, *q_count;
    uint64_t next_id;
} or_pool;

static void or_record_free(or_record *r)
{
    free(r->seg_off);
    free(r->live);
    free(r->page_table);
    free(r->row0);
    free(r->nrows);
    memset(r, 0, sizeof(*r));
}

static int64_t or_roundup16(int64_t v) { return (v + 15) / 16 * 16; }

/* NMAX: the most device pages the pool may grow to (or_pool_grow); 0 means N.
 * N may be 0 (no device pages yet) when NMAX >= 1. */
or_pool *or_pool_new(int32_t P, int64_t page_bytes, int64_t N, int32_t S,
                     int32_t R, int32_t max_segs, int64_t max_pages,
                     int64_t SP, int32_t keep_bytes, uint8_t fill, int64_t NMAX)
{
    if (NMAX == 0)
        NMAX = N;
    if (P < 1 || page_bytes < 1 || N < 0 || NMAX < 1 || N > NMAX || S < 1 || R < 1 ||
        max_segs < 1 || max_pages < 1 || SP < 0)
        return NULL;
    or_pool *p = (or_pool *)calloc(1, sizeof(or_pool));
    p->P = P;
    p->page_bytes = page_bytes;
    p->N = N;
    p->NMAX = NMAX;
    p->SP = SP;
    p->S = S;
    p->R = R;
    p->max_segs = max_segs;
    p->max_pages = max_pages;
    p->ring = (int32_t *)malloc((size_t)NMAX * sizeof(int32_t));
    p->spill_ring = (int32_t *)malloc((size_t)(SP + 1) * sizeof(int32_t));
    p->q = (or_record *)calloc((size_t)S * R, sizeof(or_record));
    p->q_head = (int32_t *)calloc((size_t)S, sizeof(int32_t));
    p->q_count = (int32_t *)calloc((size_t)S, sizeof(int32_t));
    if (keep_bytes) {
        /* room for every page the pool may grow to; pages join with the fill */
        p->pool = (uint8_t *)malloc((size_t)(NMAX * page_bytes));
        memset(p->pool, fill, (size_t)(NMAX * page_bytes));
        if (SP > 0) {
            p->spill = (uint8_t *)malloc((size_t)(SP * page_bytes));
            memset(p->spill, fill, (size_t)(SP * page_bytes));
        }
    }
    /* every slot of the ring, also those a grow brings into use later */
    for (int64_t i = 0; i < NMAX; ++i)
        p->ring[i] = (int32_t)i;
    for (int64_t i = 0; i < SP; ++i)
        p->spill_ring[i] = (int32_t)i;
    p->head = 0;
    p->tail = (uint64_t)N;
    p->spill_head = 0;
    p->spill_tail = (uint64_t)SP;
    p->next_id = 1;
    return p;
}

void or_pool_free(or_pool *p)
{
    if (!p)
        return;
    for (int64_t i = 0; i < (int64_t)p->S * p->R; ++i)
        or_record_free(&p->q[i]);
    free(p->ring);
    free(p->spill_ring);
    free(p->q);
    free(p->q_head);
    free(p->q_count);
    free(p->pool);
    free(p->spill);
    free(p);
}

/* Reset: every page free in id order, flags and statistics cleared, queues
 * emptied.  Pool bytes are not touched. */
void or_pool_reset(or_pool *p)
{
    for (int64_t i = 0; i < (int64_t)p->S * p->R; ++i)
        or_record_free(&p->q[i]);
    for (int32_t s = 0; s < p->S; ++s) {
        p->q_head[s] = 0;
        p->q_count[s] = 0;
    }
    for (int64_t i = 0; i < p->NMAX; ++i)
        p->ring[i] = (int32_t)i;
    for (int64_t i = 0; i < p->SP; ++i)
        p->spill_ring[i] = (int32_t)i;
    p->head = 0;
    p->tail = (uint64_t)p->N;
    p->spill_head = 0;
    p->spill_tail = (uint64_t)p->SP;
    p->flags = 0;
    p->high_water = 0;
    p->spill_high_water = 0;
    p->held = 0;
    p->held_high_water = 0;
}

/* Lazy sizing ([MG7342] "Summary": the activation arena's capacity grows
 * lazily).  Reading: the pool gains device pages N .. new_N-1 while records
 * stay queued.  The free ring is rewritten from position 0 as the free pages
 * in the order they would have been taken, followed by the new pages in id
 * order (head = 0, tail = free + new); pages in use, page tables and spill
 * ids (which start at NMAX) do not change. */
int or_pool_grow(or_pool *p, int64_t new_N)
{
    if (new_N < p->N || new_N > p->NMAX)
        return OR_EINVAL;
    uint64_t avail = p->tail - p->head;
    int32_t *tmp = (int32_t *)malloc((size_t)(avail + 1) * sizeof(int32_t));
    for (uint64_t i = 0; i < avail; ++i)
        tmp[i] = p->ring[(p->head + i) % (uint64_t)p->N];
    for (uint64_t i = 0; i < avail; ++i)
        p->ring[i] = tmp[i];
    for (int64_t j = 0; j < new_N - p->N; ++j)
        p->ring[avail + (uint64_t)j] = (int32_t)(p->N + j);
    free(tmp);
    p->head = 0;
    p->tail = avail + (uint64_t)(new_N - p->N);
    p->N = new_N;
    return OR_OK;
}

static int or_layout_ok(const or_pool *p, int32_t nplanes, const int64_t *rb)
{
    if (nplanes < 1 || nplanes > 2)
        return 0;
    if (rb[0] < 1 || (nplanes == 2 && rb[1] < 1))
        return 0;
    int64_t need = (int64_t)p->P * rb[0];
    if (nplanes == 2)
        need = or_roundup16(need) + (int64_t)p->P * rb[1];
    return need <= p->page_bytes;
}

static uint8_t *or_page_addr(or_pool *p, int32_t id)
{
    if (id < 0)
        return NULL;
    if (id < p->N)
        return p->pool ? p->pool + (int64_t)id * p->page_bytes : NULL;
    return p->spill ? p->spill + (int64_t)(id - p->NMAX) * p->page_bytes : NULL;
}

int or_pool_push(or_pool *p, int32_t slot, int32_t nplanes,
                 const uint8_t *const *src, const int64_t *rb, int64_t src_rows,
                 int32_t nseg, const int32_t *seg_off, const int32_t *live,
                 uint64_t *record_id)
{
    if (slot < 0 || slot >= p->S || nseg < 0 || nseg > p->max_segs ||
        src_rows < 0 || !or_layout_ok(p, nplanes, rb))
        return OR_EINVAL;
    if (p->q_count[slot] >= p->R)
        return OR_EQFULL;
    int32_t pos = (p->q_head[slot] + p->q_count[slot]) % p->R;
    or_record *rec = &p->q[(int64_t)slot * p->R + pos];
    or_record_free(rec);
    rec->id = p->next_id++;
    rec->nplanes = nplanes;
    rec->rb[0] = rb[0];
    rec->rb[1] = nplanes == 2 ? rb[1] : 0;
    rec->nseg = nseg;
    rec->seg_off = (int32_t *)malloc((size_t)(nseg + 1) * sizeof(int32_t));
    rec->live = (int32_t *)malloc((size_t)(nseg + 1) * sizeof(int32_t));
    rec->page_table = (int32_t *)malloc((size_t)p->max_pages * sizeof(int32_t));
    rec->row0 = (int64_t *)malloc((size_t)p->max_pages * sizeof(int64_t));
    rec->nrows = (int32_t *)malloc((size_t)p->max_pages * sizeof(int32_t));

    /* live prefix of each segment, checked against the source rows */
    for (int32_t s = 0; s < nseg; ++s) {
        int32_t o = seg_off[s], l = live[s];
        rec->seg_off[s] = o;
        if (l < 0 || o < 0 || (int64_t)o + (int64_t)l > src_rows) {
            p->flags |= OR_FLAG_BAD_COUNT;
            l = 0;
        }
        rec->live[s] = l;
    }

    /* take pages one at a time: segment order, then page order */
    int64_t n = 0;
    for (int32_t s = 0; s < nseg; ++s) {
        int64_t pages = ((int64_t)rec->live[s] + p->P - 1) / p->P;
        for (int64_t pg = 0; pg < pages; ++pg) {
            if (n >= p->max_pages) {
                p->flags |= OR_FLAG_RECORD_OVERFLOW;
                break;
            }
            int32_t id;
            if (p->tail - p->head > 0) {
                id = p->ring[p->head % (uint64_t)p->N];
                p->head += 1;
                rec->ndev += 1;
            } else {
                p->flags |= OR_FLAG_POOL_OVERFLOW;
                if (p->spill_tail - p->spill_head > 0) {
                    id = (int32_t)(p->NMAX + p->spill_ring[p->spill_head % (uint64_t)p->SP]);
                    p->spill_head += 1;
                    rec->nspill += 1;
                } else {
                    p->flags |= OR_FLAG_SPILL_OVERFLOW;
                    id = -1;
                    rec->nlost += 1;
                }
            }
            int64_t r0 = pg * p->P;
            int64_t rows = rec->live[s] - r0;
            if (rows > p->P)
                rows = p->P;
            rec->page_table[n] = id;
            rec->row0[n] = (int64_t)rec->seg_off[s] + r0;
            rec->nrows[n] = (int32_t)rows;
            /* copy the live rows of this page, plane by plane */
            uint8_t *page = or_page_addr(p, id);
            if (page) {
                int64_t plane_off = 0;
                for (int32_t pl = 0; pl < nplanes; ++pl) {
                    memcpy(page + plane_off, src[pl] + rec->row0[n] * rb[pl],
                           (size_t)(rows * rb[pl]));
                    plane_off = or_roundup16((int64_t)p->P * rb[0]);
                }
            }
            n += 1;
        }
    }
    rec->npages = n;
    p->held += n;
    if (p->held > p->held_high_water)
        p->held_high_water = p->held;

    int64_t in_use = p->N - (int64_t)(p->tail - p->head);
    if (in_use > p->high_water)
        p->high_water = in_use;
    int64_t spill_use = p->SP - (int64_t)(p->spill_tail - p->spill_head);
    if (spill_use > p->spill_high_water)
        p->spill_high_water = spill_use;

    p->q_count[slot] += 1;
    if (record_id)
        *record_id = rec->id;
    return OR_OK;
}

int or_pool_pop(or_pool *p, int32_t slot, int32_t nplanes, uint8_t *const *dst,
                int64_t dst_rows, uint64_t *record_id)
{
    if (slot < 0 || slot >= p->S)
        return OR_EINVAL;
    if (p->q_count[slot] == 0)
        return OR_EEMPTY;
    or_record *rec = &p->q[(int64_t)slot * p->R + p->q_head[slot]];
    if (nplanes != rec->nplanes || dst_rows < 0)
        return OR_EINVAL;
    for (int64_t n = 0; n < rec->npages; ++n) {
        int32_t id = rec->page_table[n];
        const uint8_t *page = or_page_addr(p, id);
        if (page && dst) {
            if (rec->row0[n] + rec->nrows[n] > dst_rows) {
                p->flags |= OR_FLAG_BAD_COUNT;
            } else {
                int64_t plane_off = 0;
                for (int32_t pl = 0; pl < nplanes; ++pl) {
                    memcpy(dst[pl] + rec->row0[n] * rec->rb[pl], page + plane_off,
                           (size_t)(rec->nrows[n] * rec->rb[pl]));
                    plane_off = or_roundup16((int64_t)p->P * rec->rb[0]);
                }
            }
        } else if (id >= 0 && rec->row0[n] + rec->nrows[n] > dst_rows) {
            p->flags |= OR_FLAG_BAD_COUNT;
        }
        /* recycle the page */
        if (id >= 0 && id < p->N) {
            p->ring[p->tail % (uint64_t)p->N] = id;
            p->tail += 1;
        } else if (id >= p->NMAX) {
            p->spill_ring[p->spill_tail % (uint64_t)p->SP] = (int32_t)(id - p->NMAX);
            p->spill_tail += 1;
        }
    }
    p->held -= rec->npages;
    if (record_id)
        *record_id = rec->id;
    or_record_free(rec);
    p->q_head[slot] = (p->q_head[slot] + 1) % p->R;
    p->q_count[slot] -= 1;
    return OR_OK;
}

/* ---- state read-out for the tests ---- */
/* hw5: device high water, spill high water, pages held by queued records,
 * their high water, current device pages N. */
void or_pool_state(const or_pool *p, uint64_t *ctr4, uint32_t *flags,
                   int64_t *hw5)
{
    ctr4[0] = p->head;
    ctr4[1] = p->tail;
    ctr4[2] = p->spill_head;
    ctr4[3] = p->spill_tail;
    *flags = p->flags;
    hw5[0] = p->high_water;
    hw5[1] = p->spill_high_water;
    hw5[2] = p->held;
    hw5[3] = p->held_high_water;
    hw5[4] = p->N;
}

void or_pool_rings(const or_pool *p, int32_t *ring, int32_t *spill_ring)
{
    memcpy(ring, p->ring, (size_t)p->N * sizeof(int32_t));
    if (p->SP > 0)
        memcpy(spill_ring, p->spill_ring, (size_t)p->SP * sizeof(int32_t));
}

int32_t or_pool_queue_len(const or_pool *p, int32_t slot)
{
    return (slot < 0 || slot >= p->S) ? -1 : p->q_count[slot];
}

/* Record at queue position `qpos` of a slot (0 = oldest).  Writes
 * info[0..5] = {id, npages, ndev, nspill, nlost, nseg} and the page table,
 * page start rows and row counts (up to cap entries). */
int or_pool_record(const or_pool *p, int32_t slot, int32_t qpos, int64_t *info,
                   int32_t *page_table, int64_t *row0, int32_t *nrows,
                   int64_t cap)
{
    if (slot < 0 || slot >= p->S || qpos < 0 || qpos >= p->q_count[slot])
        return OR_EINVAL;
    const or_record *rec = &p->q[(int64_t)slot * p->R + (p->q_head[slot] + qpos) % p->R];
    info[0] = (int64_t)rec->id;
    info[1] = rec->npages;
    info[2] = rec->ndev;
    info[3] = rec->nspill;
    info[4] = rec->nlost;
    info[5] = rec->nseg;
    int64_t n = rec->npages < cap ? rec->npages : cap;
    for (int64_t i = 0; i < n; ++i) {
        if (page_table)
            page_table[i] = rec->page_table[i];
        if (row0)
            row0[i] = rec->row0[i];
        if (nrows)
            nrows[i] = rec->nrows[i];
    }
    return OR_OK;
}

uint8_t *or_pool_bytes(or_pool *p) { return p->pool; }
uint8_t *or_pool_spill_bytes(or_pool *p) { return p->spill; }
