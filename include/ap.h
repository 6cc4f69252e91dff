/*
 * ap.h - C ABI of the GB300 token-movement library for a top-k MoE layer with
 * a paged activation stash (libap.so).
 *
 * The path: route_topk -> dispatch_permute -> stash_push ... stash_pop ->
 * combine_unpermute, all on one GPU.  Every call is asynchronous on the CUDA
 * stream it is given (passed as `void *`, a cudaStream_t; NULL = legacy
 * default stream) and launches only this library's kernels.  No call
 * allocates device memory: the caller owns every buffer (device pointers
 * unless marked "host").  No call synchronises the host except the explicit
 * read-out calls at the end of this header.
 *
 * Errors: every call returns an ap_status.  Argument and queue errors are
 * detected on the host and returned before anything is launched.  Conditions
 * only the GPU can see (pool overflow, lost spill pages, out-of-range counts
 * or indices) never fault and never stop the stream: the kernel skips the
 * offending copy and ORs a bit into a sticky device status word, read later
 * (the deferred overflow handling of torchtitan pull 5541, AI-Generated
 * Details, last paragraph).
 *
 * Sources (web pages) cited below:
 *   torchtitan pull 5541 - HybridEP eager scheduling with a paged activation
 *     stash, "AI-Generated Details" and "Verification";
 *   torchtitan pull 5542 - "[graph_trainer] Overlap HybridEP and paging
 *     across combined PP graphs";
 *   Megatron-LM pull 7342 - token-wise ChunkedEP for Qwen3 MoE, "Summary",
 *     "Validation and performance";
 *   OpenPipe/ART pull 971 - "Price HybridEP recompute outputs at the live
 *     communication extent".
 */
#ifndef AP_H_
#define AP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------- */
typedef int32_t ap_status;
#define AP_OK 0
#define AP_EINVAL (-1)     /* bad argument (size, pointer, layout)             */
#define AP_EEMPTY (-2)     /* stash_pop on a slot with no record               */
#define AP_EQFULL (-3)     /* stash_push on a slot whose record queue is full  */
#define AP_ECUDA (-4)      /* a CUDA runtime call failed (see ap_last_error)   */
#define AP_ESTREAM (-5)    /* pool call on a stream other than the paging one  */
#define AP_ENOTSUP (-6)    /* configuration not supported by this build        */

/* ---- sticky device status bits --------------------------------------------- */
#define AP_FLAG_POOL_OVERFLOW 0x1u   /* device pages ran out; the excess spilled */
#define AP_FLAG_SPILL_OVERFLOW 0x2u  /* spill pages ran out too; pages lost      */
#define AP_FLAG_RECORD_OVERFLOW 0x4u /* a record needed > max_pages_per_record   */
#define AP_FLAG_BAD_COUNT 0x8u       /* a segment lay outside the given rows     */
#define AP_FLAG_BAD_INDEX 0x10u      /* an expert id or row index out of range   */
#define AP_FLAG_CORRUPT 0x20u        /* a page id read back out of range         */

/* payload types of dispatch_permute */
#define AP_DTYPE_BF16 0
#define AP_DTYPE_E4M3 1

/* Human-readable name of a status code (static string). */
const char *ap_status_str(ap_status s);
/* Last error message of the calling thread (static per thread, never NULL). */
const char *ap_last_error(void);
/* Library version, e.g. "0.1.0". */
const char *ap_version(void);

/* Number of kernels this library has enqueued in this process (launched on a
 * stream, or recorded into a CUDA graph under stream capture; a graph replay
 * does not count again).  Every call that enqueues work adds its launches here
 * after the launch succeeded.  Thread-safe; never fails. */
uint64_t ap_launch_count(void);

/* ============================================================================
 * route_topk
 *
 * Router of a top-k MoE layer: per token, p = softmax(logits) over the E
 * experts, the k largest logits are selected in descending order (an equal
 * logit goes to the lower expert id; j = 0 is the top choice), and the
 * selected probabilities are renormalised, w_j = p_j / sum_sel p.  Since the
 * softmax denominator cancels, w_j = exp(l_j - m) / sum_sel exp(l_i - m) with
 * m the row maximum, computed in single precision.  Top-k routing with k = 8:
 * Megatron-LM pull 7342, "Validation and performance".
 *
 *   logits  [T, E] float32, row-major (device, read)
 *   idx     [T, k] int32 (device, written): expert ids
 *   w       [T, k] float32 (device, written): renormalised weights
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), 0 <= T < 2^31.  Logits must
 * be finite.  Returns AP_EINVAL on a bad size or NULL pointer with T > 0.
 * ========================================================================== */
ap_status ap_route_topk(const float *logits, int64_t T, int32_t E, int32_t k,
                        int32_t *idx, float *w, void *stream);

/* ============================================================================
 * dispatch_permute
 *
 * Expert-major, capacity-bounded permutation of token rows (dispatch into
 * expert buffers, Megatron-LM pull 7342 "Summary"; capacity-shaped buffers,
 * torchtitan pull 5541 "AI-Generated Details" and pull 5542).
 *
 * Pairs (t, j) are ranked in t-then-j order within their expert: the rank of
 * a pair is the number of earlier pairs routed to the same expert.  A pair is
 * kept iff capacity <= 0 (dropless) or rank < capacity; dropped pairs get
 * dest = -1.  live[e] = kept rows of expert e.  Layout: padded (padded = 1,
 * needs capacity > 0): seg_off[e] = e * capacity, xd has E*capacity rows;
 * compact: seg_off = exclusive prefix sum of live, xd has sum(live) <= T*k
 * rows.  Row dest(t, j) of xd receives row t of x:
 *   AP_DTYPE_BF16: the H BF16 values, byte for byte;
 *   AP_DTYPE_E4M3: per token amax = max|x[t]|, scale = amax/448,
 *     q = e4m3_rn_satfinite(x * (448/amax)) (scale = 1 and q = e4m3(x) when
 *     amax = 0); xd row = H code bytes, xd_scale[row] = scale.
 * Rows of xd not written (padding, drops) keep their previous contents.
 *
 *   x        [T, H] bf16 (device, read)
 *   idx      [T, k] int32 expert ids (device, read); ids outside [0, E) are
 *            skipped (dest -1) and set AP_FLAG_BAD_INDEX in *d_status
 *   xd       [xd_rows, H] bf16 or uint8 (device, written)
 *   xd_scale [xd_rows] float32 (device, written; E4M3 only, else NULL)
 *   counts, live, seg_off  [E] int32 (device, written)
 *   dest     [T, k] int32 (device, written)
 *   src_tok  [xd_rows] int32 (device, written for kept rows only; may be NULL)
 *   scratch  device work space of ap_dispatch_scratch_bytes() bytes, 16-byte
 *            aligned; its contents need no initialisation
 *   d_status device uint32 word, bits ORed in (may be NULL)
 * xd_rows must be >= E*capacity (padded) or >= T*k (compact), so no write can
 * leave the buffer.  Limits: 1 <= E <= 1024, 1 <= k <= 32, H >= 1,
 * T*k < 2^31.
 * ========================================================================== */
ap_status ap_dispatch_scratch_bytes(int64_t T, int32_t k, int32_t E,
                                    int64_t *bytes);
ap_status ap_dispatch_permute(const void *x, int64_t T, int32_t H,
                              const int32_t *idx, int32_t k, int32_t E,
                              int32_t capacity, int32_t padded,
                              int32_t out_dtype, void *xd, float *xd_scale,
                              int64_t xd_rows, int32_t *counts, int32_t *live,
                              int32_t *seg_off, int32_t *dest,
                              int32_t *src_tok, void *scratch,
                              int64_t scratch_bytes, uint32_t *d_status,
                              void *stream);

/* ============================================================================
 * dispatch_permute_noalloc
 *
 * No counterpart on the pages: a convenience for callers that cannot allocate
 * device memory.  Such callers include code running where another allocator
 * already holds every byte of the GPU, replay or real-time loops that must not
 * enter cudaMalloc (it can synchronise the device and takes a global lock),
 * and embedders with a memory budget fixed at start-up.
 *
 * Same arguments, results and errors as ap_dispatch_permute, without the
 * scratch arguments: the work space is a fixed array of
 * AP_DISPATCH_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU
 * that loads the library holds until the process exits.  Sizes whose work
 * space (ap_dispatch_scratch_bytes) exceeds it are rejected with AP_EINVAL
 * before anything is launched.  The call allocates nothing.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture.  The cached address belongs to the device's context: after
 * cudaDeviceReset the next call looks it up again in the new context (make
 * that call, too, before any capture).  All calls share the one array, so calls that overlap on the GPU
 * (on different streams without ordering between them) race: order them on
 * one stream or with events.  Contents left by a previous call do not matter;
 * every entry a call reads is first written by that call.
 * ========================================================================== */
#define AP_DISPATCH_NOALLOC_SCRATCH_BYTES (1 << 20)
ap_status ap_dispatch_permute_noalloc(const void *x, int64_t T, int32_t H,
                                      const int32_t *idx, int32_t k, int32_t E,
                                      int32_t capacity, int32_t padded,
                                      int32_t out_dtype, void *xd,
                                      float *xd_scale, int64_t xd_rows,
                                      int32_t *counts, int32_t *live,
                                      int32_t *seg_off, int32_t *dest,
                                      int32_t *src_tok, uint32_t *d_status,
                                      void *stream);

/* ============================================================================
 * combine_unpermute
 *
 * Top-k weighted un-permute back to a dense BF16 [T, H] output (combine with
 * un-permute writing a fresh dense BF16 output: OpenPipe/ART pull 971,
 * description and review).  Per token and column:
 *   acc = 0 (float32); for j = 0..k-1 with dest[t, j] >= 0:
 *     acc = acc + w[t, j] * y[dest[t, j]]   (separately rounded mul and add)
 *   out[t] = bf16_round_nearest_even(acc)
 * A token whose rows were all dropped gets +0.  A row index >= y_rows is
 * skipped and sets AP_FLAG_BAD_INDEX in *d_status (may be NULL).
 *
 *   y     [y_rows, H] bf16 (device, read)
 *   dest  [T, k] int32, w [T, k] float32 (device, read)
 *   out   [T, H] bf16 (device, written; exactly T rows)
 * Limits: H >= 1, 1 <= k <= 32.
 * ========================================================================== */
ap_status ap_combine_unpermute(const void *y, int64_t y_rows, int32_t H,
                               const int32_t *dest, const float *w, int64_t T,
                               int32_t k, void *out, uint32_t *d_status,
                               void *stream);

/* ============================================================================
 * Backward of combine and of dispatch (the backward primitives of the token
 * movement: Megatron-LM pull 7342, "Summary").  The pages give no formulas;
 * these are the derivatives of the forward definitions above.
 *
 * ap_combine_backward: for every kept pair (t, j) with row r = dest[t, j]:
 *   dy[r]   = bf16_round_nearest_even(w[t, j] * dout[t])  (one float multiply)
 *   dw[t,j] = sum_h dout[t, h] * y[r, h]   (float32; per-lane partial sums in
 *             column order, then a fixed butterfly over the 32 lanes)
 * A dropped pair gets dw = 0.  Rows of dy that no pair maps to are not
 * written.  A row index >= y_rows is skipped (dw = 0) and sets
 * AP_FLAG_BAD_INDEX in *d_status (may be NULL).
 *   dout [T, H] bf16, y [y_rows, H] bf16, dest/w [T, k] (device, read)
 *   dy [y_rows, H] bf16, dw [T, k] float32 (device, written)
 *
 * ap_dispatch_backward: dx[t] = bf16(sum_j dxd[dest[t, j]]) with a float32
 * accumulator, j ascending, dropped pairs skipped (the combine with unit
 * weights).  dxd [rows, H] bf16, dest [T, k], dx [T, H] bf16 (device).
 * Limits of both: H >= 1, 1 <= k <= 32.
 * ========================================================================== */
ap_status ap_combine_backward(const void *dout, const void *y, int64_t y_rows,
                              int32_t H, const int32_t *dest, const float *w,
                              int64_t T, int32_t k, void *dy, float *dw,
                              uint32_t *d_status, void *stream);
ap_status ap_dispatch_backward(const void *dxd, int64_t rows, int32_t H,
                               const int32_t *dest, int64_t T, int32_t k,
                               void *dx, uint32_t *d_status, void *stream);

/* ============================================================================
 * Paged activation stash (torchtitan pull 5541, "AI-Generated Details":
 * binding live counts to sources, one high-priority paging stream that
 * serialises free-list changes, FIFO records per slot, page-aligned
 * multi-token copy tiles with one page resolved per tile and only the page's
 * first tile recording or recycling it, live-prefix and page-tail masks,
 * 64-bit addressing, host spill, sticky overflow, a grid bound that changes
 * neither capacity nor the rows copied; "Verification": wrapped allocation
 * and recycling, changing device counts, BF16/FP8 payloads, host spill).
 *
 * A pool is N pages of page_bytes bytes of device memory plus spill_pages
 * pages of mapped pinned host memory.  Free pages form a ring: pages are
 * taken from its head and returned to its tail.  A push copies the live
 * prefix of each of nseg segments (rows seg_off[s] .. seg_off[s]+live[s]-1
 * of every plane; live and seg_off are read on the device, so they may
 * change between CUDA-graph replays) into ceil(live[s]/P) pages, segment by
 * segment; each page takes the next free device page, else the next free
 * spill page (AP_FLAG_POOL_OVERFLOW), else it is lost and not copied
 * (AP_FLAG_SPILL_OVERFLOW).  Inside a page, plane 0 rows are dense at
 * r * row_bytes[0]; plane 1 (e.g. FP8 scales) starts at
 * roundup16(P * row_bytes[0]).  Bytes past a page's live rows are untouched.
 * A pop takes the slot's oldest record, copies every page back to the same
 * rows of the destination planes (rows outside the live prefixes are not
 * touched) and returns the pages to the free ring in page order.
 * A pool filled exactly to its last page has not overflowed.  Flags stay set
 * until ap_pool_reset.
 * ========================================================================== */
typedef struct ap_pool ap_pool; /* opaque host object */

typedef struct {
    int32_t page_tokens;          /* P: rows per page, >= 1                    */
    int32_t num_slots;            /* S: independent FIFO record queues         */
    int64_t page_bytes;           /* bytes per page, multiple of 16            */
    int64_t num_pages;            /* N: device pages now, 0 .. max_num_pages   */
    int64_t spill_pages;          /* host spill pages, >= 0                    */
    int32_t max_records_per_slot; /* queue depth of each slot                  */
    int32_t max_segments;         /* largest nseg of a push                    */
    int64_t max_pages_per_record; /* page-table entries per record             */
    int32_t max_ctas;             /* copy grid bound; 0: environment variable
                                     AP_STASH_MAX_CTAS if set, else 2048       */
    int32_t reserved;             /* must be 0                                 */
    int64_t max_num_pages;        /* most device pages ap_pool_grow may reach;
                                     0: num_pages (the pool never grows).  Spill
                                     page ids start here.  num_pages may be 0
                                     when this is >= 1 (calibration: no device
                                     pages yet)                                */
} ap_pool_config;

/* Device state block at the start of the metadata buffer (read-only for
 * users; counters grow monotonically between grows, ring positions are
 * counter mod the current number of pages; ap_pool_grow re-bases the device
 * ring to head = 0). */
typedef struct {
    uint64_t head, tail;             /* free device ring: free = tail - head   */
    uint64_t spill_head, spill_tail; /* free spill ring                        */
    uint32_t flags;                  /* sticky AP_FLAG_* bits                  */
    uint32_t copy_done;              /* blocks of the running fused copy that
                                        have read the rings (its last block
                                        moves the state on and sets it back
                                        to 0); 0 between calls                */
    int64_t high_water;              /* most device pages ever in use          */
    int64_t spill_high_water;        /* most spill pages ever in use           */
    int64_t held;                    /* pages (device + spill + lost) of the
                                        queued records                         */
    int64_t held_high_water;         /* most pages ever held by queued records:
                                        the device pages at which no push of
                                        the same schedule spills (calibration) */
    int64_t num_pages;               /* device pages now                       */
    int64_t pad[6];
} ap_pool_state;

/* Per-record summary returned by ap_pool_read_record. */
typedef struct {
    uint64_t record_id;
    int32_t slot, nseg;
    int64_t npages, ndev, nspill, nlost;
} ap_record_info;

/* Sizes the caller must provide: device pool bytes (N * page_bytes; a pool
 * that will grow needs max_num_pages * page_bytes of address range by then),
 * device metadata bytes, and host spill bytes (spill_pages * page_bytes). */
ap_status ap_pool_required_bytes(const ap_pool_config *cfg,
                                 int64_t *dev_pool_bytes,
                                 int64_t *dev_meta_bytes,
                                 int64_t *host_spill_bytes);

/* Create a pool over caller-owned memory.  dev_pool: device, 256-byte aligned,
 * dev_pool_bytes (may be NULL when num_pages == 0: its first grow gives it).
 * dev_meta: device, 256-byte aligned, dev_meta_bytes.
 * host_spill: pinned host memory (cudaHostAlloc / torch pin_memory) of
 * host_spill_bytes, mapped into the device address space; NULL iff
 * spill_pages == 0.  paging_stream: the one stream every later push, pop and
 * reset of this pool must use (create it with high priority).  Enqueues the
 * reset of the metadata on that stream; allocates only the host object and a
 * few bytes of pinned host memory for read-outs. */
ap_status ap_pool_init(ap_pool **out, const ap_pool_config *cfg,
                       void *dev_pool, void *dev_meta, void *host_spill,
                       void *paging_stream);
/* Asynchronously return every page, clear flags and statistics, and empty
 * the record queues.  Pool bytes are not touched. */
ap_status ap_pool_reset(ap_pool *pool, void *stream);
/* Lazy sizing (Megatron-LM pull 7342, "Summary": the activation arena's
 * capacity grows lazily; torchtitan pull 5541, "AI-Generated Details":
 * calibration before the paged buffers exist).  Grow the device pool to
 * num_pages (num_pages .. max_num_pages) on the paging stream, with records
 * still queued: pages N .. num_pages-1 join the free ring after the pages
 * already free (the ring is rewritten from position 0 in the order the free
 * pages would have been taken: head = 0, tail = free + new).  Pages in use,
 * page tables, spill pages and flags do not change.  dev_pool: the pool
 * memory, now at least num_pages * page_bytes bytes; it must be the address
 * given before (grow the mapping in place, e.g. with ap_arena_grow) unless
 * the pool had no device pages, in which case it is the first pool address.
 * Kernels take the page count by value: a CUDA graph captured before a grow
 * must be captured again.  A typical use: run one step on a pool created
 * with num_pages = 0 and spill pages for its records (the live prefixes are
 * parked in pinned host memory and reload restores them), read
 * held_high_water, grow to it, reset, and run. */
ap_status ap_pool_grow(ap_pool *pool, int64_t num_pages, void *dev_pool, void *stream);
/* Free the host object (not the caller's buffers). */
ap_status ap_pool_destroy(ap_pool *pool);
/* Resolved copy-grid bound of the pool (max_ctas after the environment). */
ap_status ap_pool_max_ctas(const ap_pool *pool, int32_t *max_ctas);
/* Change the copy-grid bound for later pushes and pops (>= 1; 0 re-reads the
 * environment / default).  Like the bound itself, it changes neither the
 * capacity nor the rows copied, only how many CTAs the copy kernels occupy,
 * and so how much of the GPU stays free for concurrent compute. */
ap_status ap_pool_set_max_ctas(ap_pool *pool, int32_t max_ctas);

/* Push one record into `slot`.
 *   nplanes      1 or 2
 *   src_planes   host array of nplanes device pointers, each [src_rows, rb]
 *   row_bytes    host array of nplanes row sizes in bytes
 *   src_rows     rows of every source plane (bounds every copy)
 *   nseg         segments, 0 .. max_segments
 *   d_seg_off, d_live  [nseg] int32 (device, read at execution time and
 *                snapshotted into the record); a segment with live < 0,
 *                seg_off < 0 or seg_off + live > src_rows is not copied and
 *                sets AP_FLAG_BAD_COUNT
 *   record_id    (host, written) monotonically increasing id, first is 1
 * Returns AP_EQFULL when the slot queue is full, AP_ESTREAM when `stream` is
 * not the paging stream, AP_EINVAL when the planes do not fit a page. */
ap_status ap_stash_push(ap_pool *pool, int32_t slot, int32_t nplanes,
                        const void *const *src_planes,
                        const int64_t *row_bytes, int64_t src_rows,
                        int32_t nseg, const int32_t *d_seg_off,
                        const int32_t *d_live, uint64_t *record_id,
                        void *stream);

/* Fused dispatch + push (the stash commit made by the producer of the rows:
 * torchtitan pull 5541, "AI-Generated Details", first paragraph).  Exactly
 * the results of ap_dispatch_permute(..., out_dtype, ...) followed by
 * ap_stash_push(pool, slot, planes, ..., xd_rows, E, seg_off, live, ...)
 * with planes = {xd} (BF16 rows of 2H bytes) or {xd, xd_scale} (E4M3 rows of
 * H bytes + 4-byte scales): the same dispatch outputs, record, page table,
 * pool bytes and flags; but each token row is read once and written to its
 * dispatch rows and its pages in the same pass, so the push does not read xd
 * back.  Runs on the paging stream.  BF16 rows must be 8-byte aligned
 * (H % 4 == 0, 8-aligned buffers); E4M3 needs H % 8 == 0, H <= 4096, x
 * 16-aligned and xd 8-aligned; otherwise AP_ENOTSUP.  E must not exceed
 * max_segments. */
ap_status ap_dispatch_stash(ap_pool *pool, int32_t slot, const void *x,
                            int64_t T, int32_t H, const int32_t *idx,
                            int32_t k, int32_t E, int32_t capacity,
                            int32_t padded, int32_t out_dtype, void *xd,
                            float *xd_scale, int64_t xd_rows,
                            int32_t *counts, int32_t *live, int32_t *seg_off,
                            int32_t *dest, int32_t *src_tok, void *scratch,
                            int64_t scratch_bytes, uint32_t *d_status,
                            uint64_t *record_id, void *stream);

/* Route + fused dispatch + push: ap_route_topk(logits, T, E, k, idx, w)
 * followed by ap_dispatch_stash(pool, slot, x, T, H, idx, k, E, ...), with the
 * same results (idx, w, every dispatch output, the record, pool bytes and
 * flags), but the routing runs inside the count/rank launch: each block of
 * 64 tokens routes them (one warp per token) and ranks their pairs from
 * shared memory, so the ids are not read back and one launch is saved (for
 * E <= 256; wider routers take the two launches).  logits: device f32 [T, E];
 * idx (int32) and w (f32): device outputs [T, k].  Other arguments, streams
 * and errors as ap_dispatch_stash, plus AP_EINVAL for k > E or NULL
 * logits / w with T > 0. */
ap_status ap_route_dispatch_stash(ap_pool *pool, int32_t slot, const float *logits, float *w, const void *x,
                                  int64_t T, int32_t H, int32_t *idx, int32_t k, int32_t E, int32_t capacity,
                                  int32_t padded, int32_t out_dtype, void *xd, float *xd_scale, int64_t xd_rows,
                                  int32_t *counts, int32_t *live, int32_t *seg_off, int32_t *dest,
                                  int32_t *src_tok, void *scratch, int64_t scratch_bytes, uint32_t *d_status,
                                  uint64_t *record_id, void *stream);

/* Count/rank alone, on any stream: the first launch of ap_dispatch_stash
 * (and, with logits != NULL, of ap_route_dispatch_stash, routing into idx
 * and w first), for callers that overlap it with other work and then call
 * ap_dispatch_stash_ranked on the paging stream.  The ranking of pairs is the
 * one ap_dispatch_permute documents (t-then-j order within each expert; the
 * capacity-shaped, expert-major dispatch of Megatron-LM pull 7342, "Summary",
 * and torchtitan pull 5541, "AI-Generated Details").  Overlapping it with the
 * previous pool call is the early-launch, late-wait scheduling of torchtitan
 * pull 5542 (body) applied to the dispatch's metadata work.
 *
 *   logits   [T, E] f32 (device, read) or NULL: idx is then an input
 *   w        [T, k] f32 (device, written when logits != NULL, else unused)
 *   idx      [T, k] int32 (device; written when logits != NULL, else read)
 *   x        the [T, row_bytes] rows the later copy reads (device, may be
 *            NULL): prefetched into L2 as a hint when 16-byte aligned
 *   dest     [T, k] int32 (device, written): each pair's rank inside its
 *            block of 64 tokens, -1 for an id outside [0, E)
 *   scratch  ap_dispatch_scratch_bytes(T, k, E) bytes (device, written): the
 *            blocks' expert histograms
 *   counts, live, seg_off  [E] int32 (device, written) or all three NULL:
 *            with them the call also runs the dispatch's expert scan for
 *            capacity and padded (as ap_dispatch_permute), and the scratch
 *            then holds each block's base rank per expert instead of its
 *            histogram; ap_dispatch_stash_ranked(..., scanned = 1) then plans
 *            only the record's pages
 *   d_status device uint32 word (may be NULL): AP_FLAG_BAD_INDEX for an id
 *            outside [0, E)
 * Limits and errors as ap_dispatch_permute (plus AP_EINVAL for k > E with
 * logits, NULL w with logits and T > 0, row_bytes < 0, or only some of
 * counts, live and seg_off). */
ap_status ap_count_rank(const float *logits, float *w, int32_t *idx, int64_t T, int32_t k, int32_t E,
                        const void *x, int64_t row_bytes, int32_t *dest, void *scratch, int64_t scratch_bytes,
                        int32_t capacity, int32_t padded, int32_t *counts, int32_t *live, int32_t *seg_off,
                        uint32_t *d_status, void *stream);

/* ap_dispatch_stash without its count/rank launch (the stash committed by
 * the producer of the rows: torchtitan pull 5541, "AI-Generated Details",
 * first paragraph): dest and scratch must
 * hold the results of ap_count_rank for the same idx, T, k and E, ordered
 * before this call (an event, or the same stream); idx, dest and scratch
 * must not change between the two calls.  scanned = 1: that ap_count_rank
 * call also ran the expert scan into counts, live and seg_off (passed here
 * too, with the same capacity and padded), so the call does not scan again
 * (0 or 1, else AP_EINVAL).  Same arguments, results and errors as
 * ap_dispatch_stash.  Ranks or histograms that do not match idx
 * leave the dispatch rows, the record and the pool's contents unspecified,
 * but no write leaves the dispatch buffer, the pages or the metadata: a
 * pair whose row would fall outside its buffer or page is dropped (dest -1)
 * and AP_FLAG_BAD_COUNT is set. */
ap_status ap_dispatch_stash_ranked(ap_pool *pool, int32_t slot, const void *x, int64_t T, int32_t H,
                                   const int32_t *idx, int32_t k, int32_t E, int32_t capacity, int32_t padded,
                                   int32_t out_dtype, void *xd, float *xd_scale, int64_t xd_rows,
                                   int32_t *counts, int32_t *live, int32_t *seg_off, int32_t *dest,
                                   int32_t *src_tok, void *scratch, int64_t scratch_bytes, uint32_t *d_status,
                                   uint64_t *record_id, int32_t scanned, void *stream);

/* Pop the oldest record of `slot` into dst_planes (host array of nplanes
 * device pointers, each [dst_rows, row_bytes of the push]).  A page whose
 * rows fall outside dst_rows is not copied (AP_FLAG_BAD_COUNT) but still
 * recycled.  record_id (host, may be NULL) receives the popped id.  Returns
 * AP_EEMPTY when the slot has no record. */
ap_status ap_stash_pop(ap_pool *pool, int32_t slot, int32_t nplanes,
                       void *const *dst_planes, int64_t dst_rows,
                       uint64_t *record_id, void *stream);

/* Copy-kernel timing without a profiler.  While set, every push, fused
 * dispatch + push and pop records `before` and `after` (CUDA events, as
 * void *) on the paging stream immediately around its copy kernel, so their
 * elapsed time after the call is that kernel's duration (a push's small
 * plan kernels fall outside; a pop is its copy kernel alone).  Passing NULL,
 * NULL stops it.  The events stay
 * owned by the caller and must outlive the calls that record them. */
ap_status ap_pool_time_copies(ap_pool *pool, void *before, void *after);

/* Records queued in a slot (host-side count, no synchronisation). */
ap_status ap_pool_queue_len(const ap_pool *pool, int32_t slot, int32_t *len);

/* Device address of the sticky flag word (uint32), for device-side consumers
 * such as an optimizer step that skips itself on overflow. */
ap_status ap_pool_flags_device_ptr(const ap_pool *pool, uint32_t **d_flags);

/* ---- read-outs: these synchronise the paging stream ----------------------- */
/* Sticky flags (the only call meant for the training loop).  wait = 1
 * synchronises the paging stream and returns the current flags; wait = 0
 * returns the flags captured by the previous wait = 1 call (or 0). */
ap_status ap_overflow_query(ap_pool *pool, uint32_t *flags, int32_t wait);
/* Whole state block (synchronises). */
ap_status ap_pool_read_state(ap_pool *pool, ap_pool_state *state);
/* Pool occupancy, read outside the CUDA callable like the overflow flags
 * (torchtitan pull 5541, "AI-Generated Details", last paragraph: overflow
 * and pool state are handled later, not inside the copy).
 *   pages_in_use  device pages taken and not yet returned
 *                 (num_pages - free device pages)
 *   high_water    most device pages ever in use since the last reset
 *   spill_in_use  spill pages taken and not yet returned
 * wait = 1 synchronises the paging stream and reads the state block;
 * wait = 0 touches no GPU and returns the figures of the last synchronising
 * read-out (ap_pool_stats with wait = 1, or ap_pool_read_state), zeros
 * before the first.  Any of the three pointers may be NULL. */
ap_status ap_pool_stats(ap_pool *pool, int64_t *pages_in_use,
                        int64_t *high_water, int64_t *spill_in_use,
                        int32_t wait);
/* Free rings: ring [num_pages now] int32 and spill_ring [spill_pages] int32
 * (host, written; spill_ring may be NULL).  Synchronises. */
ap_status ap_pool_read_rings(ap_pool *pool, int32_t *ring,
                             int32_t *spill_ring);
/* Record at queue position qpos (0 = oldest) of a slot: its summary and up
 * to cap page-table entries (device page p -> p, spill page s ->
 * max_num_pages + s, lost -> -1), first rows and row counts (host arrays,
 * each may be NULL).  Synchronises. */
ap_status ap_pool_read_record(ap_pool *pool, int32_t slot, int32_t qpos,
                              ap_record_info *info, int32_t *page_table,
                              int64_t *row0, int32_t *nrows, int64_t cap);

/* ============================================================================
 * Growable device arena: a reserved range of device virtual addresses whose
 * prefix is backed by physical memory on demand (CUDA virtual memory
 * management), so a pool can grow in place without moving the pages it
 * already holds.  The arena is the caller's allocator: the pool calls never
 * create or grow one.  Memory is mapped read-write for the device it was
 * created on, in steps of the allocation granularity.
 * ========================================================================== */
typedef struct ap_arena ap_arena; /* opaque host object */

/* Reserve max_bytes (> 0, rounded up to the granularity) of address range on
 * `device`; nothing is mapped yet.  AP_ENOTSUP when the device or driver
 * lacks virtual memory management. */
ap_status ap_arena_create(ap_arena **out, int64_t max_bytes, int32_t device);
/* Back the first `bytes` of the arena with memory (rounded up to the
 * granularity; never shrinks; AP_EINVAL beyond the reservation).  Mapped
 * bytes keep their contents and address. */
ap_status ap_arena_grow(ap_arena *arena, int64_t bytes);
/* Base address and bytes mapped so far (host, written). */
ap_status ap_arena_info(const ap_arena *arena, void **base, int64_t *mapped_bytes, int64_t *reserved_bytes);
/* Unmap and release everything.  The caller makes sure no queued work still
 * uses the arena (e.g. synchronises the streams that used it). */
ap_status ap_arena_destroy(ap_arena *arena);

/* ============================================================================
 * E4M3 conversion used by the FP8 dispatch, exposed for testing the format:
 * out[i] = e4m3_rn_satfinite(in[i]) (round to nearest even, finite overflow
 * saturates to +-448, NaN -> 0x7F).  in: device float32 [n], out: device
 * uint8 [n].
 * ========================================================================== */
ap_status ap_cast_e4m3(const float *in, uint8_t *out, int64_t n, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* AP_H_ */
