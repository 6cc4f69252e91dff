// Paged activation stash: fixed page pool, free rings, spill, FIFO records.
//
// torchtitan pull 5541, "AI-Generated Details": live counts bound to the
// source that pushes them; one high-priority paging stream serialises every
// free-list change; records stay FIFO per slot; the copy loops run over
// page-aligned multi-token tiles, each tile resolving its page once, and only
// the first tile of a page records it (push) or recycles it (pop); live-prefix
// and page-tail masks keep the payload bytes exact with 64-bit addressing;
// host spill and a sticky overflow flag; a grid bound (default 2048) that
// changes neither the capacity nor the rows copied.  "Verification": wrapped
// allocation and recycling, device counts that change under CUDA-graph replay,
// BF16/FP8 payloads, host spill and overflow.  (Here a pop recycles its pages
// from the record's page table in one CTA instead of each page's first tile;
// see k_pop_copy.)
//
// A fused dispatch + push (k_scan_plan, then k_dispatch_stash_copy or its
// E4M3 form) plans the same way but leaves the page descriptors to the copy
// kernel: the pair that holds row 0 of a page writes its descriptor with its
// page-table entry.  A small record (at most kInlineMaxCounts count/rank
// block counts) skips k_scan_plan: count/rank copies the free-ring counters
// into the record header, every copy block derives the expert scan and the
// page plan it needs from the block counts (inline_plan), and copy block 0
// writes the dispatch outputs, the record and the pool state (inline_commit)
// with exactly the values k_scan_plan would write.
// A push is two launches on the paging stream:
//   k_push_plan (1 CTA): snapshot live/seg_off, page ordinals by a prefix sum of
//     ceil(live/P), one (first row, rows) descriptor per page, and the
//     allocation: pages [0, ndev) come from the device ring at the head
//     snapshot, the next nspill from the spill ring, the rest are lost; head
//     counters advance and sticky flags are set here, once.
//   k_push_copy (grid-stride over tiles): tile -> page ordinal; the page id is
//     read from the ring at head0 + ordinal; tile 0 of the page writes the
//     page-table entry; the tile's rows are copied as one contiguous range per
//     plane.
// A pop is one launch, k_pop_copy: its CTAs copy the pages' live rows back,
// and CTA 0 alone returns the record's pages (its page table, in ordinal
// order) to the rings at their tails and advances the tails: no other CTA
// reads or writes the rings or the counters.
// Nothing here waits on the device: there are no spin loops.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "dispatch_scan.cuh"

namespace ap {
namespace {

struct RecHdr {
    int32_t nseg;
    int32_t pad0;
    int64_t npages, ndev, nspill, nlost;
    uint64_t head0, spill_head0;
    int64_t pad1[9];
};
static_assert(sizeof(RecHdr) == 128, "record header layout");
static_assert(sizeof(ap_pool_state) == 128, "state layout");

struct PageDesc {
    int64_t row0; // first row in the source / destination planes
    int32_t nrows;
    int32_t pad;
};

// Where page ids point.  Device page p (0 <= p < N) lives at pool + p *
// page_bytes; spill page s (0 <= s < SP) has id SB + s and lives at spill +
// s * page_bytes (SB, the most device pages the pool may grow to, keeps spill
// ids fixed while N grows); -1 is a lost page.
struct PageSpace {
    int32_t *ring, *spill_ring;
    uint8_t *pool, *spill;
    int64_t N, SB, SP, page_bytes;
};

__device__ __forceinline__ uint8_t *page_addr(const PageSpace &ps, int64_t id)
{
    return (id < ps.N) ? ps.pool + id * ps.page_bytes : ps.spill + (id - ps.SB) * ps.page_bytes;
}

// Id of page ordinal `ord` of a record being pushed: the device ring entry at
// head0 + ord for the first ndev pages, then the spill ring entry at sh0 +
// (ord - ndev) for the next nspill, else -1 (lost).  A ring entry out of its
// range gives -1 and *corrupt = true.
__device__ __forceinline__ int64_t pushed_page_id(const PageSpace &ps, int64_t ord, int64_t ndev, int64_t nspill,
                                                  uint64_t head0, uint64_t sh0, bool *corrupt)
{
    *corrupt = false;
    if (ord < ndev) {
        const int64_t id = ps.ring[(head0 + (uint64_t)ord) % (uint64_t)ps.N];
        if (id >= 0 && id < ps.N) return id;
        *corrupt = true;
    } else if (ord < ndev + nspill) {
        const int64_t sp = ps.spill_ring[(sh0 + (uint64_t)(ord - ndev)) % (uint64_t)ps.SP];
        if (sp >= 0 && sp < ps.SP) return ps.SB + sp;
        *corrupt = true;
    }
    return -1;
}

struct RecLayout {
    int64_t seg_off, live, pg_base, desc, page_table, stride;
};

__host__ __device__ inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

RecLayout record_layout(const ap_pool_config &c)
{
    RecLayout L;
    int64_t o = sizeof(RecHdr);
    L.seg_off = o;
    o = align_up(o + 4 * (int64_t)c.max_segments, 16);
    L.live = o;
    o = align_up(o + 4 * (int64_t)c.max_segments, 16);
    L.pg_base = o;
    o = align_up(o + 8 * ((int64_t)c.max_segments + 1), 16);
    L.desc = o;
    o = align_up(o + (int64_t)sizeof(PageDesc) * c.max_pages_per_record, 16);
    L.page_table = o;
    o = align_up(o + 4 * c.max_pages_per_record, 256);
    L.stride = o;
    return L;
}

struct MetaLayout {
    int64_t ring, spill_ring, grow_tmp, records, total;
    RecLayout rec;
};

// Most device pages the pool may grow to (spill ids start here).
inline int64_t max_pages_of(const ap_pool_config &c) { return c.max_num_pages > 0 ? c.max_num_pages : c.num_pages; }

MetaLayout meta_layout(const ap_pool_config &c)
{
    MetaLayout M;
    const int64_t nmax = max_pages_of(c);
    M.ring = 256;
    M.spill_ring = align_up(M.ring + 4 * nmax, 256);
    M.grow_tmp = align_up(M.spill_ring + 4 * c.spill_pages, 256); // free-ring copy used by a grow
    M.records = (nmax > c.num_pages) ? align_up(M.grow_tmp + 4 * nmax, 256) : M.grow_tmp;
    M.rec = record_layout(c);
    M.total = M.records + M.rec.stride * (int64_t)c.num_slots * c.max_records_per_slot;
    return M;
}

// Pointers to one record inside the metadata buffer.
struct RecPtr {
    RecHdr *hdr;
    int32_t *seg_off, *live;
    int64_t *pg_base;
    PageDesc *desc;
    int32_t *page_table;
};

RecPtr rec_ptr(uint8_t *meta, const MetaLayout &M, int64_t index)
{
    uint8_t *b = meta + M.records + M.rec.stride * index;
    RecPtr r;
    r.hdr = reinterpret_cast<RecHdr *>(b);
    r.seg_off = reinterpret_cast<int32_t *>(b + M.rec.seg_off);
    r.live = reinterpret_cast<int32_t *>(b + M.rec.live);
    r.pg_base = reinterpret_cast<int64_t *>(b + M.rec.pg_base);
    r.desc = reinterpret_cast<PageDesc *>(b + M.rec.desc);
    r.page_table = reinterpret_cast<int32_t *>(b + M.rec.page_table);
    return r;
}

// ---- kernels -------------------------------------------------------------------
// NMAX: every slot of the device ring is written, also those a grow brings
// into use later (slots at or past N are never read before then).
__global__ void k_reset(ap_pool_state *st, int32_t *ring, int64_t N, int64_t NMAX, int32_t *spill_ring, int64_t SP)
{
    pdl_begin();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < NMAX; i += stride) ring[i] = (int32_t)i;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < SP; i += stride) spill_ring[i] = (int32_t)i;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        st->head = 0;
        st->tail = (uint64_t)N;
        st->spill_head = 0;
        st->spill_tail = (uint64_t)SP;
        st->flags = 0;
        st->copy_done = 0;
        st->high_water = 0;
        st->spill_high_water = 0;
        st->held = 0;
        st->held_high_water = 0;
        st->num_pages = N;
        for (int i = 0; i < 6; ++i) st->pad[i] = 0;
    }
}

// Grow the device pool from N0 to N1 pages (one CTA, on the paging stream):
// the free pages, in the order they would be taken, move to ring positions
// 0 .. free-1 (through tmp, since old and new positions overlap), the new
// pages N0 .. N1-1 follow in id order, and the counters re-base to head = 0.
__global__ void __launch_bounds__(1024) k_grow(ap_pool_state *st, int32_t *ring, int32_t *tmp, int64_t N0, int64_t N1)
{
    pdl_begin();
    const uint64_t head = st->head, tail = st->tail;
    const int64_t avail = (int64_t)(tail - head); // 0 when N0 == 0
    for (int64_t i = threadIdx.x; i < avail; i += blockDim.x) tmp[i] = ring[(head + (uint64_t)i) % (uint64_t)N0];
    __syncthreads();
    for (int64_t i = threadIdx.x; i < avail; i += blockDim.x) ring[i] = tmp[i];
    for (int64_t j = threadIdx.x; j < N1 - N0; j += blockDim.x) ring[avail + j] = (int32_t)(N0 + j);
    __syncthreads();
    if (threadIdx.x == 0) {
        st->head = 0;
        st->tail = (uint64_t)(avail + (N1 - N0));
        st->num_pages = N1;
    }
}

constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemSegs = 2048; // segments whose tables the plan keeps in shared memory

// Descriptor of page ordinal `ord`: its segment is the largest s with
// pg_base[s] <= ord; the page holds rows [pg*P, min(live, (pg+1)*P)) of it.
__device__ __forceinline__ void plan_descriptor(RecPtr rec, const int64_t *pg_base, const int32_t *seg_live,
                                                const int32_t *seg_offs, int nseg, int64_t ord, int P)
{
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pg_base[mid] <= ord) lo = mid;
        else hi = mid - 1;
    }
    const int64_t r0 = (ord - pg_base[lo]) * P;
    int64_t nr = (int64_t)seg_live[lo] - r0;
    if (nr > P) nr = P;
    PageDesc d;
    d.row0 = (int64_t)seg_offs[lo] + r0;
    d.nrows = (int32_t)nr;
    d.pad = 0;
    rec.desc[ord] = d;
}

// Allocation of a record of `total` pages (one thread): the first
// min(total, max_pages) pages come from the device ring at the head snapshot,
// then from the spill ring, the rest are lost; the head counters advance, the
// high-water marks and the sticky flags are updated.
// The state fields a push plan reads, loaded together by the one thread that
// later writes them back (a single round trip instead of one per field; only
// the plan kernel running on the paging stream changes them meanwhile).
struct StateSnap {
    uint64_t head, tail, sh, stl;
    int64_t hw, shw, held, hhw;
    uint32_t flags;
};

__device__ __forceinline__ StateSnap load_state(const ap_pool_state *__restrict__ st)
{
    StateSnap s;
    s.head = st->head;
    s.tail = st->tail;
    s.sh = st->spill_head;
    s.stl = st->spill_tail;
    s.hw = st->high_water;
    s.shw = st->spill_high_water;
    s.held = st->held;
    s.hhw = st->held_high_water;
    s.flags = st->flags;
    return s;
}

__device__ __forceinline__ void plan_allocate(ap_pool_state *__restrict__ st, RecPtr rec, int nseg, int64_t total,
                                              int64_t max_pages, uint32_t f, const StateSnap &snap, int64_t N,
                                              int64_t SP)
{
    const uint64_t head = snap.head, tail = snap.tail, sh = snap.sh, stl = snap.stl;
    const int64_t kept = total < max_pages ? total : max_pages;
    if (total > max_pages) f |= AP_FLAG_RECORD_OVERFLOW;
    const int64_t avail = (int64_t)(tail - head);
    const int64_t savail = (int64_t)(stl - sh);
    const int64_t ndev = kept < avail ? kept : avail;
    int64_t nspill = kept - ndev;
    if (nspill > savail) nspill = savail;
    const int64_t nlost = kept - ndev - nspill;
    if (kept > avail) f |= AP_FLAG_POOL_OVERFLOW;
    if (nlost > 0) f |= AP_FLAG_SPILL_OVERFLOW;
    rec.hdr->nseg = nseg;
    rec.hdr->npages = kept;
    rec.hdr->ndev = ndev;
    rec.hdr->nspill = nspill;
    rec.hdr->nlost = nlost;
    rec.hdr->head0 = head;
    rec.hdr->spill_head0 = sh;
    st->head = head + (uint64_t)ndev;
    st->spill_head = sh + (uint64_t)nspill;
    const int64_t in_use = N - (int64_t)(tail - (head + (uint64_t)ndev));
    if (in_use > snap.hw) st->high_water = in_use;
    const int64_t s_use = SP - (int64_t)(stl - (sh + (uint64_t)nspill));
    if (s_use > snap.shw) st->spill_high_water = s_use;
    const int64_t held = snap.held + kept; // pages of queued records, wherever they went
    st->held = held;
    if (held > snap.hhw) st->held_high_water = held;
    st->flags = snap.flags | f;
}

// have_reg: nseg <= kPlanThreads and thread s already holds segment s's
// offset and live count in reg_off / reg_live (fused scan + plan).
__device__ __forceinline__ void push_plan_body(ap_pool_state *st, RecPtr rec, int nseg,
                                               const int32_t *__restrict__ d_seg_off,
                                               const int32_t *__restrict__ d_live, int64_t src_rows, int P,
                                               int64_t max_pages, int64_t N, int64_t SP, const StateSnap &snap,
                                               bool write_desc, bool have_reg = false, int32_t reg_off = 0,
                                               int32_t reg_live = 0)
{
    __shared__ int64_t s_warp[kPlanThreads / kWarp];
    __shared__ int64_t s_carry;
    __shared__ uint32_t s_flags;
    // segment tables in shared memory when they fit (the descriptor step
    // below searches them once per page)
    __shared__ int64_t s_base[kPlanSmemSegs + 1];
    __shared__ int32_t s_off[kPlanSmemSegs], s_live[kPlanSmemSegs];
    const bool in_smem = nseg <= kPlanSmemSegs;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        s_carry = 0;
        s_flags = 0;
    }
    __syncthreads();
    // 1. snapshot + validation + prefix sum of pages per segment
    for (int base = 0; base < nseg; base += kPlanThreads) {
        const int s = base + tid;
        int64_t n = 0;
        if (s < nseg) {
            const int32_t o = have_reg ? reg_off : d_seg_off[s];
            int32_t l = have_reg ? reg_live : d_live[s];
            if (l < 0 || o < 0 || (int64_t)o + (int64_t)l > src_rows) {
                atomicOr(&s_flags, AP_FLAG_BAD_COUNT);
                l = 0;
            }
            rec.seg_off[s] = o;
            rec.live[s] = l;
            if (in_smem) {
                s_off[s] = o;
                s_live[s] = l;
            }
            n = ((int64_t)l + P - 1) / P;
        }
        int64_t x = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int64_t v = s_warp[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            s_warp[lane] = v;
        }
        __syncthreads();
        const int64_t incl = x + (wid > 0 ? s_warp[wid - 1] : 0);
        if (s < nseg) {
            rec.pg_base[s] = s_carry + incl - n;
            if (in_smem) s_base[s] = s_carry + incl - n;
        }
        __syncthreads();
        if (tid == kPlanThreads - 1) s_carry += incl;
        __syncthreads();
    }
    const int64_t total = s_carry;
    if (tid == 0) rec.pg_base[nseg] = total;
    const int64_t kept = total < max_pages ? total : max_pages;
    __syncthreads();
    // 2. one descriptor per page: segment by binary search over pg_base
    const int64_t *pg_base = in_smem ? s_base : rec.pg_base;
    const int32_t *seg_live = in_smem ? s_live : rec.live;
    const int32_t *seg_offs = in_smem ? s_off : rec.seg_off;
    if (write_desc) // (the fused copy writes them itself, beside the page-table entry)
        for (int64_t ord = tid; ord < kept; ord += kPlanThreads)
            plan_descriptor(rec, pg_base, seg_live, seg_offs, nseg, ord, P);
    // 3. allocation: device pages first, then spill pages, then lost
    if (tid == 0) plan_allocate(st, rec, nseg, total, max_pages, s_flags, snap, N, SP);
}

__global__ void __launch_bounds__(kPlanThreads) k_push_plan(ap_pool_state *st, RecPtr rec, int nseg,
                                                             const int32_t *__restrict__ d_seg_off,
                                                             const int32_t *__restrict__ d_live, int64_t src_rows,
                                                             int P, int64_t max_pages, int64_t N, int64_t SP)
{
    pdl_begin();
    StateSnap snap;
    if (threadIdx.x == 0) snap = load_state(st);
    push_plan_body(st, rec, nseg, d_seg_off, d_live, src_rows, P, max_pages, N, SP, snap, true);
}

// Fused dispatch + stash: the dispatch's expert scan and the record's page
// plan in one CTA (the plan reads the live counts and offsets the scan has
// just written; __syncthreads makes them visible to the whole block).
__global__ void __launch_bounds__(kPlanThreads) k_scan_plan(int32_t *__restrict__ blk, int nblk, int E, int capacity,
                                                             int padded, int32_t *__restrict__ counts,
                                                             int32_t *__restrict__ live,
                                                             int32_t *__restrict__ seg_off, ap_pool_state *st,
                                                             RecPtr rec, int64_t src_rows, int P, int64_t max_pages,
                                                             int64_t N, int64_t SP)
{
    pdl_begin();
    StateSnap snap; // loaded before the scan, so its latency hides under it
    if (threadIdx.x == 0) snap = load_state(st);
    int32_t my_live, my_off;
    scan_body(blk, nblk, E, capacity, padded, counts, live, seg_off, my_live, my_off);
    __syncthreads();
    push_plan_body(st, rec, E, seg_off, live, src_rows, P, max_pages, N, SP, snap, false, E <= kPlanThreads, my_off,
                   my_live);
}

// Fused dispatch + stash whose expert scan already ran (ap_count_rank with the
// scan): the record's page plan alone, from the dispatch's offsets and live
// counts; the copy writes the page descriptors, as after k_scan_plan.
__global__ void __launch_bounds__(kPlanThreads) k_scanned_plan(ap_pool_state *st, RecPtr rec, int nseg,
                                                                const int32_t *__restrict__ seg_off,
                                                                const int32_t *__restrict__ live, int64_t src_rows,
                                                                int P, int64_t max_pages, int64_t N, int64_t SP)
{
    pdl_begin();
    StateSnap snap;
    if (threadIdx.x == 0) snap = load_state(st);
    push_plan_body(st, rec, nseg, seg_off, live, src_rows, P, max_pages, N, SP, snap, false);
}

struct Planes {
    uint8_t *p[2];
    int64_t rb[2];
    int64_t page_off[2];
    int n;
};

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads, 4) k_push_copy(ap_pool_state *st, RecPtr rec, PageSpace ps,
                                                             Planes src, int rows_per_tile, int tiles_per_page)
{
    pdl_begin();
    const int64_t npages = rec.hdr->npages;
    const int64_t ndev = rec.hdr->ndev, nspill = rec.hdr->nspill;
    const uint64_t head0 = rec.hdr->head0, sh0 = rec.hdr->spill_head0;
    const int64_t tiles = npages * tiles_per_page;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t ord = tile / tiles_per_page;
        const int sub = (int)(tile - ord * tiles_per_page);
        const PageDesc d = rec.desc[ord];
        const int64_t r0 = (int64_t)sub * rows_per_tile;
        if (r0 >= d.nrows) continue;
        const int64_t nr = (d.nrows - r0 < rows_per_tile) ? d.nrows - r0 : rows_per_tile;
        // resolve this tile's page once
        bool corrupt;
        const int64_t id = pushed_page_id(ps, ord, ndev, nspill, head0, sh0, &corrupt);
        if (corrupt && threadIdx.x == 0) atomicOr(&st->flags, AP_FLAG_CORRUPT);
        if (sub == 0 && threadIdx.x == 0) rec.page_table[ord] = (int32_t)id; // first tile records the page
        if (id < 0) continue;
        uint8_t *page = page_addr(ps, id);
#pragma unroll
        for (int p = 0; p < 2; ++p)
            if (p < src.n)
                block_copy(page + src.page_off[p] + r0 * src.rb[p], src.p[p] + (d.row0 + r0) * src.rb[p],
                           nr * src.rb[p]);
    }
}

// Pop of the slot's oldest record: its pages' live rows go back to the same
// rows of the destination planes.  CTA 0 also returns the pages to the rings
// they came from, in ordinal order at the tails as this pop found them
// (device pages, then spill pages; a lost or invalid entry returns nothing),
// advances the tails and releases the record's pages.
__global__ void __launch_bounds__(kCopyThreads, 4) k_pop_copy(ap_pool_state *st, RecPtr rec, PageSpace ps,
                                                            Planes dst, int64_t dst_rows, int rows_per_tile,
                                                            int tiles_per_page)
{
    pdl_begin();
    // The first tile's descriptor and page id are loaded together with the
    // record header, before the page count is known: the grid never exceeds
    // the record's page bound times the tiles per page, and that bound is at
    // most the page-table capacity, so the entry exists (it is used only if
    // the tile turns out to be live).
    int64_t tile = blockIdx.x;
    PageDesc d = rec.desc[tile / tiles_per_page];
    int64_t id = rec.page_table[tile / tiles_per_page];
    const int64_t npages = rec.hdr->npages;
    const int64_t ndev = rec.hdr->ndev, nspill = rec.hdr->nspill;
    if (blockIdx.x == 0) {
        const uint64_t tail0 = st->tail, stail0 = st->spill_tail;
        const int64_t held = st->held;
        constexpr int B = 4; // page-table loads in flight per thread
        for (int64_t o0 = threadIdx.x; o0 < npages; o0 += (int64_t)B * blockDim.x) {
            int32_t id[B];
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int64_t ord = o0 + (int64_t)u * blockDim.x;
                id[u] = ord < npages ? rec.page_table[ord] : -1;
            }
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int64_t ord = o0 + (int64_t)u * blockDim.x;
                if (ord >= npages) break;
                if (ord < ndev) {
                    if (id[u] >= 0 && id[u] < ps.N) ps.ring[(tail0 + (uint64_t)ord) % (uint64_t)ps.N] = id[u];
                } else if (ord < ndev + nspill && id[u] >= ps.SB && id[u] < ps.SB + ps.SP) {
                    ps.spill_ring[(stail0 + (uint64_t)(ord - ndev)) % (uint64_t)ps.SP] = (int32_t)(id[u] - ps.SB);
                }
            }
        }
        __syncthreads(); // every thread has read the tails
        if (threadIdx.x == 0) {
            st->tail = tail0 + (uint64_t)ndev;
            st->spill_tail = stail0 + (uint64_t)nspill;
            st->held = held - npages;
        }
    }
    const int64_t tiles = npages * tiles_per_page;
    for (; tile < tiles; tile += gridDim.x) {
        const int64_t ord = tile / tiles_per_page;
        const int sub = (int)(tile - ord * tiles_per_page);
        const PageDesc cur = d;
        const int64_t cur_id = id;
        // the next tile's metadata, in flight while this tile copies
        const int64_t next = tile + gridDim.x;
        if (next < tiles) {
            d = rec.desc[next / tiles_per_page];
            id = rec.page_table[next / tiles_per_page];
        }
        const int64_t r0 = (int64_t)sub * rows_per_tile;
        if (r0 >= cur.nrows) continue;
        const int64_t nr = (cur.nrows - r0 < rows_per_tile) ? cur.nrows - r0 : rows_per_tile;
        const bool ok = (ord < ndev) ? (cur_id >= 0 && cur_id < ps.N)
                                     : (ord < ndev + nspill) ? (cur_id >= ps.SB && cur_id < ps.SB + ps.SP)
                                                             : (cur_id == -1);
        if (!ok) {
            if (threadIdx.x == 0) atomicOr(&st->flags, AP_FLAG_CORRUPT);
            continue;
        }
        if (cur_id < 0) continue;
        if (cur.row0 + cur.nrows > dst_rows) {
            if (threadIdx.x == 0) atomicOr(&st->flags, AP_FLAG_BAD_COUNT);
            continue;
        }
        const uint8_t *page = page_addr(ps, cur_id);
#pragma unroll
        for (int p = 0; p < 2; ++p)
            if (p < dst.n)
                block_copy(dst.p[p] + (cur.row0 + r0) * dst.rb[p], page + dst.page_off[p] + r0 * dst.rb[p],
                           nr * dst.rb[p]);
    }
}

// ---- small records: the expert scan and page plan inside the copy kernel -------
// When the block counts of a record are few (count/rank blocks x experts <=
// kInlineMaxCounts), every copy block derives what the one-CTA scan + plan
// kernel would have written, from the count/rank output, in a prologue: its
// own base rank per expert (the counts of the earlier count/rank blocks), the
// expert totals, live counts, segment offsets, the record's page ordinals
// and the allocation (from the pool's free-ring counters, read after the
// dependency wait).  Block 0 then writes the dispatch outputs and the
// record, and the last block to finish its plan moves the pool state on
// (inline_finish); no other block reads those, and the kernel after this
// one on the paging stream waits for it.  Each block's tokens lie in one
// count/rank block (its first token is a multiple of its token count, which
// divides kTokPerBlk) and the grid covers every token in one pass.
constexpr int kInlineMaxE = 256;
constexpr int kInlineMaxCounts = 16384;

struct InlineArgs {
    int enabled; // 0: a plan kernel ran before the copy; 1: the copy plans the record from the count/rank
                 // block histograms; 2: from the expert scan's block bases, live counts and offsets
    int nblk, padded;
    int32_t *counts, *live; // dispatch outputs (seg_off is the copy kernel's own argument)
    int64_t src_rows;       // rows of the dispatch buffer (both paths: no dispatch row reaches past it)
    int64_t max_pages;
};

struct InlinePlan {
    int32_t base[kInlineMaxE];  // this block's base rank per expert
    int32_t off[kInlineMaxE];   // segment offsets
    int32_t lrec[kInlineMaxE];  // the record's live counts (0 for a segment outside the rows)
    int32_t tot[kInlineMaxE];   // expert totals (counts)
    int32_t ldisp[kInlineMaxE]; // live = min(count, capacity)
    int64_t pg[kInlineMaxE + 1];
    int64_t npages, kept, ndev, nspill;
    uint64_t head0, sh0, tail0, stail0;
    uint32_t bad;
};

// Exclusive scan of v over the threads of a 256-thread block (8 warps);
// returns the thread's exclusive prefix and *total the block's sum.  ws: 8
// shared slots, free again when the call returns.
template <typename V>
__device__ __forceinline__ V block_exclusive_scan256(V v, V *ws, V *total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    V x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[wid] = x;
    __syncthreads();
    V before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const V c = ws[w];
        if (w < wid) before += c;
        all += c;
    }
    __syncthreads();
    *total = all;
    return before + x - v;
}

// The prologue every copy block runs (256 threads).  b: the count/rank block
// of this block's tokens.  Ends with a barrier: pl is complete for the block.
template <bool kVecReads>
__device__ __forceinline__ void inline_plan(InlinePlan &pl, const int32_t *__restrict__ blk, int b, int E,
                                            int capacity, const InlineArgs &ia, const ap_pool_state *st, int P)
{
    constexpr int kPartials = kVecReads ? 1024 : 256;
    __shared__ __align__(16) int32_t s_lt[kPartials], s_all[kPartials]; // partial sums: [row group][expert]
    __shared__ int64_t s_ws[8];
    const int tid = threadIdx.x;
    const int nblk = ia.nblk;
    if (tid == 0) { // the free rings as the previous call left them (the last block commits this call's)
        pl.bad = 0;
        pl.head0 = __ldcg(&st->head);
        pl.sh0 = __ldcg(&st->spill_head);
        pl.tail0 = __ldcg(&st->tail);
        pl.stail0 = __ldcg(&st->spill_tail);
    }
    // each thread sums expert columns over a strided set of rows: the counts
    // of the rows before b (this block's base) and of all rows (totals).  One
    // column per thread takes one round of sixteen loads in flight for up to
    // 16 rows per thread (64 x 64 counts); more rows go four adjacent columns
    // per 16-byte load, in predicated rounds of eight (128 x 128 counts: two),
    // in kernels that can spare the shared memory (kVecReads)
    const int Q1 = blockDim.x / E; // row groups of the one-column reading (>= 1)
    const bool vec =
        kVecReads && nblk > 16 * Q1 && E % 4 == 0 && (reinterpret_cast<uintptr_t>(blk) & 15) == 0;
    const int Q = vec ? blockDim.x / (E / 4) : Q1;
    if (vec && tid / (E / 4) < Q) {
        const int c = tid % (E / 4), q = tid / (E / 4);
        int4 lt = make_int4(0, 0, 0, 0), all = lt;
        for (int r = q; r < nblk; r += 8 * Q) {
            int4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = (r + u * Q < nblk) ? reinterpret_cast<const int4 *>(blk + (int64_t)(r + u * Q) * E)[c]
                                          : make_int4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                all.x += v[u].x, all.y += v[u].y, all.z += v[u].z, all.w += v[u].w;
                if (r + u * Q < b) lt.x += v[u].x, lt.y += v[u].y, lt.z += v[u].z, lt.w += v[u].w;
            }
        }
        reinterpret_cast<int4 *>(s_lt + q * E)[c] = lt;
        reinterpret_cast<int4 *>(s_all + q * E)[c] = all;
    } else if (!vec) {
        const int e = tid % E, q = tid / E;
        int32_t lt = 0, all = 0;
        if (q < Q) {
            int r = q;
            for (; r + 15 * Q < nblk; r += 16 * Q) { // sixteen loads in flight
                int32_t c[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) c[u] = blk[(int64_t)(r + u * Q) * E + e];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    all += c[u];
                    if (r + u * Q < b) lt += c[u];
                }
            }
            for (; r < nblk; r += Q) {
                const int32_t c = blk[(int64_t)r * E + e];
                all += c;
                if (r < b) lt += c;
            }
            s_lt[q * E + e] = lt;
            s_all[q * E + e] = all;
        }
    }
    __syncthreads();
    int32_t total = 0, base = 0;
    if (tid < E) {
        for (int qq = 0; qq < Q; ++qq) {
            base += s_lt[qq * E + tid];
            total += s_all[qq * E + tid];
        }
    }
    const int32_t l = (tid < E) ? ((capacity > 0 && total > capacity) ? capacity : total) : 0;
    // one scan for both prefix sums: live counts in the high half, pages in
    // the low half (page totals stay below 2^31, so nothing carries between)
    const int64_t n0 = (tid < E) ? ((int64_t)l + P - 1) / P : 0;
    int64_t both_sum;
    const int64_t both = block_exclusive_scan256<int64_t>(((int64_t)l << 32) | n0, s_ws, &both_sum);
    const int32_t off = ia.padded ? tid * capacity : (int32_t)(both >> 32);
    // the record's snapshot of the segment: one outside the rows is not copied
    // (the fused call's host checks rule that out; the rescan keeps the rule)
    int32_t lr = l;
    const bool out = tid < E && (l < 0 || off < 0 || (int64_t)off + (int64_t)l > ia.src_rows);
    if (out) {
        atomicOr(&pl.bad, AP_FLAG_BAD_COUNT);
        lr = 0;
    }
    int64_t pg = both & 0xffffffffll, npages = both_sum & 0xffffffffll;
    if (__syncthreads_or(out)) {
        const int64_t n = (tid < E) ? ((int64_t)lr + P - 1) / P : 0;
        pg = block_exclusive_scan256<int64_t>(n, s_ws, &npages);
    }
    if (tid < E) {
        pl.base[tid] = base;
        pl.off[tid] = off;
        pl.lrec[tid] = lr;
        pl.tot[tid] = total;
        pl.ldisp[tid] = l;
        pl.pg[tid] = pg;
    }
    if (tid == 0) {
        // the allocation of k_scan_plan: device pages from the ring, then
        // spill pages, then lost; at most max_pages kept
        pl.pg[E] = npages;
        pl.npages = npages;
        const int64_t kept = npages < ia.max_pages ? npages : ia.max_pages;
        const int64_t avail = (int64_t)(pl.tail0 - pl.head0);
        const int64_t savail = (int64_t)(pl.stail0 - pl.sh0);
        const int64_t ndev = kept < avail ? kept : avail;
        int64_t nspill = kept - ndev;
        if (nspill > savail) nspill = savail;
        pl.kept = kept;
        pl.ndev = ndev;
        pl.nspill = nspill;
    }
    __syncthreads();
}

// The prologue of a copy whose record's expert scan already ran (mode 2: the
// scratch holds each count/rank block's base rank per expert, and seg_off and
// ia.live the dispatch's offsets and live counts): the record's page ordinals
// and the allocation alone.  b: the count/rank block of this block's tokens.
// Ends with a barrier: pl is complete for the block.
__device__ __forceinline__ void inline_plan_scanned(InlinePlan &pl, const int32_t *__restrict__ blk, int b, int E,
                                                    const int32_t *__restrict__ seg_off, const InlineArgs &ia,
                                                    const ap_pool_state *st, int P)
{
    __shared__ int64_t s_ws[8];
    const int tid = threadIdx.x;
    if (tid == 0) { // the free rings as the previous call left them (the last block commits this call's)
        pl.bad = 0;
        pl.head0 = __ldcg(&st->head);
        pl.sh0 = __ldcg(&st->spill_head);
        pl.tail0 = __ldcg(&st->tail);
        pl.stail0 = __ldcg(&st->spill_tail);
    }
    int32_t base = 0, off = 0, l = 0;
    if (tid < E) {
        base = blk[(int64_t)b * E + tid];
        off = seg_off[tid];
        l = ia.live[tid];
    }
    // a segment outside the rows is not copied (as k_scan_plan)
    const bool out = tid < E && (l < 0 || off < 0 || (int64_t)off + (int64_t)l > ia.src_rows);
    const int32_t lr = out ? 0 : l;
    int64_t npages;
    const int64_t pg = block_exclusive_scan256<int64_t>((tid < E) ? ((int64_t)lr + P - 1) / P : 0, s_ws, &npages);
    if (out) atomicOr(&pl.bad, AP_FLAG_BAD_COUNT); // after the scan's barriers: pl.bad is initialised
    if (tid < E) {
        pl.base[tid] = base;
        pl.off[tid] = off;
        pl.lrec[tid] = lr;
        pl.pg[tid] = pg;
    }
    if (tid == 0) {
        pl.pg[E] = npages;
        pl.npages = npages;
        const int64_t kept = npages < ia.max_pages ? npages : ia.max_pages;
        const int64_t avail = (int64_t)(pl.tail0 - pl.head0);
        const int64_t savail = (int64_t)(pl.stail0 - pl.sh0);
        const int64_t ndev = kept < avail ? kept : avail;
        int64_t nspill = kept - ndev;
        if (nspill > savail) nspill = savail;
        pl.kept = kept;
        pl.ndev = ndev;
        pl.nspill = nspill;
    }
    __syncthreads();
}

// Block 0 of an inline-planned copy: the dispatch outputs and the record,
// exactly as k_scan_plan writes them (the pool state is inline_finish's).
__device__ __forceinline__ void inline_commit(const InlinePlan &pl, int E, const InlineArgs &ia,
                                              int32_t *__restrict__ seg_off, const RecPtr &rec)
{
    const int tid = threadIdx.x;
    if (tid < E) {
        if (ia.enabled == 1) { // in mode 2 the expert scan wrote them
            ia.counts[tid] = pl.tot[tid];
            ia.live[tid] = pl.ldisp[tid];
            seg_off[tid] = pl.off[tid];
        }
        rec.seg_off[tid] = pl.off[tid];
        rec.live[tid] = pl.lrec[tid];
        rec.pg_base[tid] = pl.pg[tid];
    }
    if (tid == 0) {
        rec.pg_base[E] = pl.npages;
        rec.hdr->nseg = E;
        rec.hdr->npages = pl.kept;
        rec.hdr->ndev = pl.ndev;
        rec.hdr->nspill = pl.nspill;
        rec.hdr->nlost = pl.kept - pl.ndev - pl.nspill;
        rec.hdr->head0 = pl.head0;
        rec.hdr->spill_head0 = pl.sh0;
    }
}

// Every block of an inline-planned copy, once its plan is complete: counts
// itself in the state's copy_done; the last block to do so (every block has
// read the free rings by then) moves the pool state on, as k_scan_plan does,
// and clears the count for the next call.  The flags are or-ed in, since
// other blocks may still be adding AP_FLAG_CORRUPT.
__device__ __forceinline__ void inline_finish(const InlinePlan &pl, const InlineArgs &ia, ap_pool_state *st,
                                              const PageSpace &ps)
{
    if (threadIdx.x != 0) return;
    if (atomicAdd(&st->copy_done, 1u) + 1u != gridDim.x) return;
    st->copy_done = 0;
    const int64_t kept = pl.kept, ndev = pl.ndev, nspill = pl.nspill;
    uint32_t f = pl.bad;
    if (pl.npages > ia.max_pages) f |= AP_FLAG_RECORD_OVERFLOW;
    if (kept > ndev) f |= AP_FLAG_POOL_OVERFLOW;
    if (kept - ndev - nspill > 0) f |= AP_FLAG_SPILL_OVERFLOW;
    const int64_t hw = __ldcg(&st->high_water), shw = __ldcg(&st->spill_high_water);
    const int64_t held = __ldcg(&st->held) + kept, hhw = __ldcg(&st->held_high_water);
    st->head = pl.head0 + (uint64_t)ndev;
    st->spill_head = pl.sh0 + (uint64_t)nspill;
    const int64_t in_use = ps.N - (int64_t)(pl.tail0 - (pl.head0 + (uint64_t)ndev));
    if (in_use > hw) st->high_water = in_use;
    const int64_t s_use = ps.SP - (int64_t)(pl.stail0 - (pl.sh0 + (uint64_t)nspill));
    if (s_use > shw) st->spill_high_water = s_use;
    st->held = held;
    if (held > hhw) st->held_high_water = held;
    if (f) atomicOr(&st->flags, f);
}

// A pair's dispatch row and, for a kept pair, its place in the record being
// pushed, from the in-block rank k_count_rank left in dest and the block
// bases the scan left in blk (as finalize_dest), in two dependent batches of
// loads: the rank and the expert id, then everything that depends only on
// the expert (block base, segment offset, the record's live count and first
// page ordinal).  The pair's row within its expert segment is its rank.
// Writes the final dest and, for a kept pair, src_tok.
struct PairPlace {
    int32_t d;   // dispatch row, or -1
    int64_t r;   // row within the expert segment (kept pairs)
    int64_t ord; // page ordinal in the record, or -1 (dropped, or past the record's live rows)
    int64_t lv;  // live rows of the expert segment in the record
    bool bad;    // the rank put the row outside the dispatch buffer (dropped; AP_FLAG_BAD_COUNT)
};

__device__ __forceinline__ PairPlace resolve_pair(const int32_t *__restrict__ idx, int32_t *__restrict__ dest,
                                                  int32_t *__restrict__ src_tok, const int32_t *__restrict__ blk,
                                                  const int32_t *__restrict__ seg_off, const RecPtr &rec,
                                                  int64_t t, int j, int k, int E, int capacity, int P, int64_t rows)
{
    PairPlace pp{-1, 0, -1, 0, false};
    const int64_t p = t * k + j;
    const int32_t lr = dest[p];
    const int e = idx[p];
    if (lr < 0 || e < 0 || e >= E) return pp; // an invalid expert id: dest is already -1
    const int32_t base = blk[(t / kTokPerBlk) * E + e];
    const int32_t so = seg_off[e];
    const int64_t lv = rec.live[e], pg0 = rec.pg_base[e];
    const int32_t r = base + lr;
    if ((capacity <= 0 || r < capacity) && (r < 0 || (uint64_t)((int64_t)so + r) >= (uint64_t)rows)) {
        pp.bad = true; // ranks that do not match the counts (ranked input): no row outside xd or a page
    } else if (capacity <= 0 || r < capacity) {
        pp.d = so + r;
        if (src_tok) src_tok[pp.d] = (int32_t)t;
        pp.r = r;
        pp.lv = lv;
        if (r < lv) pp.ord = pg0 + r / P;
    }
    dest[p] = pp.d;
    return pp;
}

// resolve_pair for an inline-planned copy: the block base, segment offset,
// live count and first page ordinal of the pair's expert come from the
// block's plan in shared memory, so only the rank and the expert id are
// loaded.
// lr and e: the pair's in-block rank (dest) and expert id, already loaded.
__device__ __forceinline__ PairPlace resolve_pair_inline(int32_t lr, int e, int32_t *__restrict__ dest,
                                                         int32_t *__restrict__ src_tok, const InlinePlan &pl,
                                                         int64_t t, int j, int k, int E, int capacity, int P,
                                                         int64_t rows)
{
    PairPlace pp{-1, 0, -1, 0, false};
    const int64_t p = t * k + j;
    if (lr < 0 || e < 0 || e >= E) return pp; // an invalid expert id: dest is already -1
    const int32_t r = pl.base[e] + lr;
    if ((capacity <= 0 || r < capacity) && (r < 0 || (uint64_t)((int64_t)pl.off[e] + r) >= (uint64_t)rows)) {
        pp.bad = true; // ranks that do not match the counts (ranked input): no row outside xd or a page
    } else if (capacity <= 0 || r < capacity) {
        pp.d = pl.off[e] + r;
        if (src_tok) src_tok[pp.d] = (int32_t)t;
        pp.r = r;
        pp.lv = pl.lrec[e];
        if (r < pp.lv) pp.ord = pl.pg[e] + r / P;
    }
    dest[p] = pp.d;
    return pp;
}

// Fused dispatch + push: one warp per token reads its BF16 row once and writes
// it both to the dispatch buffer row dest(t, j) and, for a kept pair, to row
// (rank mod P) of page pg_base[e] + rank / P of the record (rank = the pair's
// row within its expert segment).  The pair that holds row 0 of a page records
// the page.  Same bytes, page table and flags as a dispatch followed by a push.
template <typename V>
__global__ void __launch_bounds__(256) k_dispatch_stash_copy(const uint8_t *__restrict__ x, int64_t T, int64_t rb,
                                                             const int32_t *__restrict__ idx,
                                                             int32_t *__restrict__ dest, int k, int E, int capacity,
                                                             const int32_t *__restrict__ blk,
                                                             int32_t *__restrict__ seg_off,
                                                             int32_t *__restrict__ src_tok,
                                                             uint8_t *__restrict__ xd, ap_pool_state *st, RecPtr rec,
                                                             PageSpace ps, int P, InlineArgs ia)
{
    pdl_begin();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    const int64_t nvec = rb / (int64_t)sizeof(V);
    __shared__ InlinePlan pl;
    if (ia.enabled) { // the record is planned here: this block's tokens lie in one count/rank block
        const int b = (int)(((int64_t)blockIdx.x * (blockDim.x / kWarp)) / kTokPerBlk);
        if (ia.enabled == 2) inline_plan_scanned(pl, blk, b, E, seg_off, ia, st, P);
        else inline_plan<true>(pl, blk, b, E, capacity, ia, st, P);
        if (blockIdx.x == 0) inline_commit(pl, E, ia, seg_off, rec);
        inline_finish(pl, ia, st, ps);
    }
    const int64_t npages = ia.enabled ? pl.kept : rec.hdr->npages;
    const int64_t ndev = ia.enabled ? pl.ndev : rec.hdr->ndev, nspill = ia.enabled ? pl.nspill : rec.hdr->nspill;
    const uint64_t head0 = ia.enabled ? pl.head0 : rec.hdr->head0, sh0 = ia.enabled ? pl.sh0 : rec.hdr->spill_head0;
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; t < T; t += warps) {
        int32_t my_d = -1;
        uint8_t *my_page = nullptr; // where this lane's pair lands in the pool (row start), or null
        if (lane < k) {
            const PairPlace pp =
                ia.enabled ? resolve_pair_inline(dest[t * k + lane], idx[t * k + lane], dest, src_tok, pl, t, lane, k,
                                                 E, capacity, P, ia.src_rows)
                           : resolve_pair(idx, dest, src_tok, blk, seg_off, rec, t, lane, k, E, capacity, P,
                                          ia.src_rows);
            if (pp.bad) atomicOr(&st->flags, AP_FLAG_BAD_COUNT);
            my_d = pp.d;
            if (pp.ord >= 0 && pp.ord < npages) {
                bool corrupt;
                const int64_t id = pushed_page_id(ps, pp.ord, ndev, nspill, head0, sh0, &corrupt);
                if (corrupt) atomicOr(&st->flags, AP_FLAG_CORRUPT);
                if (pp.r % P == 0) { // row 0 of the page records it and its descriptor
                    rec.page_table[pp.ord] = (int32_t)id;
                    PageDesc pd;
                    pd.row0 = pp.d;
                    pd.nrows = (int32_t)(pp.lv - pp.r < P ? pp.lv - pp.r : P);
                    pd.pad = 0;
                    rec.desc[pp.ord] = pd;
                }
                if (id >= 0) {
                    uint8_t *page = page_addr(ps, id);
                    my_page = page + (pp.r % P) * rb;
                }
            }
        }
        const V *src = reinterpret_cast<const V *>(x + t * rb);
        constexpr int U = 8; // 8 vectors per lane in flight (a sweep on GB300 favoured 8 over 2 and 4)
        for (int64_t base = 0; base < nvec; base += U * kWarp) { // warp-uniform
            V r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = base + u * kWarp + lane;
                if (v < nvec) r[u] = ld_stream(src + v);
            }
            for (int j = 0; j < k; ++j) {
                const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
                const unsigned long long pg =
                    __shfl_sync(0xffffffffu, (unsigned long long)reinterpret_cast<uintptr_t>(my_page), j);
                if (d < 0) continue;
                V *dst = reinterpret_cast<V *>(xd + (int64_t)d * rb);
                V *pdst = reinterpret_cast<V *>(static_cast<uintptr_t>(pg));
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = base + u * kWarp + lane;
                    if (v < nvec) {
                        st_stream(dst + v, r[u]);
                        if (pdst) st_stream(pdst + v, r[u]);
                    }
                }
            }
        }
    }
}

// Fused dispatch + push for E4M3 payloads, two warps per token: warp h of a
// warp pair holds half h of the row (16-byte vectors [h * half0, ...), at
// most NRH per lane), so twice as many warps share a record's rows.  The two
// warps meet once per token at a named barrier: by then warp 0 has resolved
// the token's pairs (finalize_dest, page ids, page-table entries and
// descriptors of a page's row 0) and both have put their half's amax in
// shared memory (double-buffered by token parity, so a warp that runs ahead
// never overwrites what its partner still reads).  Both then quantise with
// the row's scale (same arithmetic as the E4M3 dispatch) and write their half
// of every kept pair's codes to its dispatch row and page row; warp 0 writes
// the scales (dispatch scale and the page's second plane).
__device__ __forceinline__ void pair_barrier(int id)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(2 * kWarp) : "memory");
}

template <int NRH>
__global__ void __launch_bounds__(256, 4) k_dispatch_stash_e4m3(
    const uint16_t *__restrict__ x, int64_t T, int H, const int32_t *__restrict__ idx, int32_t *__restrict__ dest,
    int k, int E, int capacity, const int32_t *__restrict__ blk, int32_t *__restrict__ seg_off,
    int32_t *__restrict__ src_tok, uint8_t *__restrict__ xd, float *__restrict__ xd_scale, ap_pool_state *st,
    RecPtr rec, PageSpace ps, int P, int64_t plane1_off, InlineArgs ia)
{
    pdl_begin();
    constexpr int kPairs = 256 / (2 * kWarp); // warp pairs per block
    __shared__ uint32_t s_amax[2][kPairs][2];
    __shared__ int32_t s_d[2][kPairs][kWarp];
    __shared__ unsigned long long s_prow[2][kPairs][kWarp];
    __shared__ InlinePlan pl;
    const int lane = (int)lane_id(), wid = threadIdx.x / kWarp;
    const int pr = wid >> 1, h = wid & 1;
    const int nstep = H / 8;
    const int half0 = (nstep + 1) / 2;
    const int s_begin = h ? half0 : 0, s_end = h ? nstep : half0;
    if (ia.enabled) { // the record is planned here: this block's tokens lie in one count/rank block
        const int b = (int)(((int64_t)blockIdx.x * kPairs) / kTokPerBlk);
        if (ia.enabled == 2) inline_plan_scanned(pl, blk, b, E, seg_off, ia, st, P);
        else inline_plan<false>(pl, blk, b, E, capacity, ia, st, P);
        if (blockIdx.x == 0) inline_commit(pl, E, ia, seg_off, rec);
        inline_finish(pl, ia, st, ps);
    }
    const int64_t npages = ia.enabled ? pl.kept : rec.hdr->npages;
    const int64_t ndev = ia.enabled ? pl.ndev : rec.hdr->ndev, nspill = ia.enabled ? pl.nspill : rec.hdr->nspill;
    const uint64_t head0 = ia.enabled ? pl.head0 : rec.hdr->head0, sh0 = ia.enabled ? pl.sh0 : rec.hdr->spill_head0;
    int buf = 0;
    for (int64_t t = (int64_t)blockIdx.x * kPairs + pr; t < T; t += (int64_t)gridDim.x * kPairs, buf ^= 1) {
        // this half's vectors first: their latency overlaps the lookups below
        const int4 *row = reinterpret_cast<const int4 *>(x + t * H);
        int4 v[NRH];
#pragma unroll
        for (int i = 0; i < NRH; ++i) {
            const int s = s_begin + lane + i * kWarp;
            v[i] = (s < s_end) ? ld_stream(row + s) : make_int4(0, 0, 0, 0);
        }
        int32_t my_d = -1;
        float *my_scale = nullptr;
        if (h == 0) {
            uint8_t *my_row = nullptr;
            if (lane < k) {
                const PairPlace pp =
                    ia.enabled ? resolve_pair_inline(dest[t * k + lane], idx[t * k + lane], dest, src_tok, pl, t,
                                                     lane, k, E, capacity, P, ia.src_rows)
                               : resolve_pair(idx, dest, src_tok, blk, seg_off, rec, t, lane, k, E, capacity, P,
                                              ia.src_rows);
                if (pp.bad) atomicOr(&st->flags, AP_FLAG_BAD_COUNT);
                my_d = pp.d;
                if (pp.ord >= 0 && pp.ord < npages) {
                    bool corrupt;
                    const int64_t id = pushed_page_id(ps, pp.ord, ndev, nspill, head0, sh0, &corrupt);
                    if (corrupt) atomicOr(&st->flags, AP_FLAG_CORRUPT);
                    if (pp.r % P == 0) { // row 0 of the page records it and its descriptor
                        rec.page_table[pp.ord] = (int32_t)id;
                        PageDesc pd;
                        pd.row0 = pp.d;
                        pd.nrows = (int32_t)(pp.lv - pp.r < P ? pp.lv - pp.r : P);
                        pd.pad = 0;
                        rec.desc[pp.ord] = pd;
                    }
                    if (id >= 0) {
                        uint8_t *page = page_addr(ps, id);
                        my_row = page + (pp.r % P) * H;
                        my_scale = reinterpret_cast<float *>(page + plane1_off + (pp.r % P) * 4);
                    }
                }
            }
            s_d[buf][pr][lane] = my_d;
            s_prow[buf][pr][lane] = (unsigned long long)reinterpret_cast<uintptr_t>(my_row);
        }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < NRH; ++i) {
            m = absmax_bf16x2(m, (uint32_t)v[i].x);
            m = absmax_bf16x2(m, (uint32_t)v[i].y);
            m = absmax_bf16x2(m, (uint32_t)v[i].z);
            m = absmax_bf16x2(m, (uint32_t)v[i].w);
        }
        const uint32_t half_amax = __reduce_max_sync(0xffffffffu, absmax_bits(m));
        if (lane == 0) s_amax[buf][pr][h] = half_amax;
        pair_barrier(1 + pr);
        const uint32_t a0 = s_amax[buf][pr][0], a1 = s_amax[buf][pr][1];
        float scale, inv;
        e4m3_scales(a0 > a1 ? a0 : a1, scale, inv);
        if (h == 0 && my_d >= 0) {
            xd_scale[my_d] = scale;
            if (my_scale) *my_scale = scale;
        }
#pragma unroll
        for (int i = 0; i < NRH; ++i) { // codes replace the values in place (first 8 bytes)
            const int2 c = quantize8_e4m3(v[i], inv);
            v[i].x = c.x;
            v[i].y = c.y;
        }
        for (int j = 0; j < k; ++j) {
            const int32_t d = s_d[buf][pr][j];
            if (d < 0) continue;
            uint8_t *drow = xd + (int64_t)d * H;
            uint8_t *prow = reinterpret_cast<uint8_t *>(static_cast<uintptr_t>(s_prow[buf][pr][j]));
#pragma unroll
            for (int i = 0; i < NRH; ++i) {
                const int s = s_begin + lane + i * kWarp;
                if (s < s_end) {
                    const int2 c = make_int2(v[i].x, v[i].y);
                    st_stream(reinterpret_cast<int2 *>(drow + (int64_t)s * 8), c);
                    if (prow) st_stream(reinterpret_cast<int2 *>(prow + (int64_t)s * 8), c);
                }
            }
        }
    }
}

// The same for rows that may start 8 bytes off a 16-byte boundary (H not a
// multiple of 16, or a base only 8-byte aligned).  A row of H codes is cut into 16-code units (two 16-byte input vectors each) and, when
// H / 8 is odd, one lone last vector; warp 0 of a warp pair holds the first
// half of the units, warp 1 the rest, one unit per lane per round (at most
// NRU rounds).  Each warp also holds the vector just past its units (its
// lookahead: warp 1's first vector, or the lone last one).  The two warps
// meet once per token at a named barrier: by then warp 0 has resolved the
// token's pairs (finalize_dest, page ids, page-table entries and descriptors
// of a page's row 0) and both have put their half's amax in shared memory
// (double-buffered by token parity, so a warp that runs ahead never
// overwrites what its partner still reads).  Both then quantise with the
// row's scale (same arithmetic as the E4M3 dispatch) and write their units
// of every kept pair's codes to its dispatch row and page row with 16-byte
// stores.  Rows are 8-byte aligned; a destination row 8 bytes off a 16-byte
// boundary gets the aligned 16 bytes that straddle two units (the upper half
// of one unit and the lower half of the next, taken from the next lane or
// the lookahead), plus one 8-byte store at its start.  Warp 1 hands its
// first vector and the lone one to the lookaheads through shared memory at
// the pair barrier.  Warp 0 writes the scales (dispatch scale and the page's
// second plane).
template <int NRU>
__global__ void __launch_bounds__(256, 4) k_dispatch_stash_e4m3_units(
    const uint16_t *__restrict__ x, int64_t T, int H, const int32_t *__restrict__ idx, int32_t *__restrict__ dest,
    int k, int E, int capacity, const int32_t *__restrict__ blk, int32_t *__restrict__ seg_off,
    int32_t *__restrict__ src_tok, uint8_t *__restrict__ xd, float *__restrict__ xd_scale, ap_pool_state *st,
    RecPtr rec, PageSpace ps, int P, int64_t plane1_off, InlineArgs ia)
{
    pdl_begin();
    constexpr int kPairs = 256 / (2 * kWarp); // warp pairs per block
    __shared__ uint32_t s_amax[2][kPairs][2];
    __shared__ int32_t s_d[2][kPairs][kWarp];
    __shared__ unsigned long long s_prow[2][kPairs][kWarp];
    __shared__ int4 s_look[2][kPairs][2]; // raw vectors for the lookaheads: warp 1's first, the lone one
    __shared__ InlinePlan pl;
    const int lane = (int)lane_id(), wid = threadIdx.x / kWarp;
    const int pr = wid >> 1, h = wid & 1;
    const int nstep = H / 8;                           // 16-byte input vectors of a row
    const int nu = nstep >> 1, lone = nstep & 1;       // 16-code units; a lone last vector
    const int u0 = (nu + 1) >> 1;                      // warp 0's units
    const int ub = h ? u0 : 0, un = h ? nu - u0 : u0; // this warp's first unit and unit count
    const int la = h ? (lone ? nstep - 1 : -1) : (2 * u0 < nstep ? 2 * u0 : -1); // lookahead vector
    if (ia.enabled) { // the record is planned here: this block's tokens lie in one count/rank block
        const int b = (int)(((int64_t)blockIdx.x * kPairs) / kTokPerBlk);
        if (ia.enabled == 2) inline_plan_scanned(pl, blk, b, E, seg_off, ia, st, P);
        else inline_plan<false>(pl, blk, b, E, capacity, ia, st, P);
        if (blockIdx.x == 0) inline_commit(pl, E, ia, seg_off, rec);
        inline_finish(pl, ia, st, ps);
    }
    const int64_t npages = ia.enabled ? pl.kept : rec.hdr->npages;
    const int64_t ndev = ia.enabled ? pl.ndev : rec.hdr->ndev, nspill = ia.enabled ? pl.nspill : rec.hdr->nspill;
    const uint64_t head0 = ia.enabled ? pl.head0 : rec.hdr->head0, sh0 = ia.enabled ? pl.sh0 : rec.hdr->spill_head0;
    const int4 zero = make_int4(0, 0, 0, 0);
    int buf = 0;
    for (int64_t t = (int64_t)blockIdx.x * kPairs + pr; t < T; t += (int64_t)gridDim.x * kPairs, buf ^= 1) {
        // this warp's vectors first: their latency overlaps the lookups below
        const int4 *row = reinterpret_cast<const int4 *>(x + t * H);
        int4 v[2 * NRU];
#pragma unroll
        for (int i = 0; i < NRU; ++i) {
            const int w = lane + i * kWarp;
            v[2 * i] = (w < un) ? ld_stream(row + 2 * (ub + w)) : zero;
            v[2 * i + 1] = (w < un) ? ld_stream(row + 2 * (ub + w) + 1) : zero;
        }
        int32_t my_d = -1;
        float *my_scale = nullptr;
        if (h == 0) {
            uint8_t *my_row = nullptr;
            if (lane < k) {
                const PairPlace pp =
                    ia.enabled ? resolve_pair_inline(dest[t * k + lane], idx[t * k + lane], dest, src_tok, pl, t,
                                                     lane, k, E, capacity, P, ia.src_rows)
                               : resolve_pair(idx, dest, src_tok, blk, seg_off, rec, t, lane, k, E, capacity, P,
                                              ia.src_rows);
                if (pp.bad) atomicOr(&st->flags, AP_FLAG_BAD_COUNT);
                my_d = pp.d;
                if (pp.ord >= 0 && pp.ord < npages) {
                    bool corrupt;
                    const int64_t id = pushed_page_id(ps, pp.ord, ndev, nspill, head0, sh0, &corrupt);
                    if (corrupt) atomicOr(&st->flags, AP_FLAG_CORRUPT);
                    if (pp.r % P == 0) { // row 0 of the page records it and its descriptor
                        rec.page_table[pp.ord] = (int32_t)id;
                        PageDesc pd;
                        pd.row0 = pp.d;
                        pd.nrows = (int32_t)(pp.lv - pp.r < P ? pp.lv - pp.r : P);
                        pd.pad = 0;
                        rec.desc[pp.ord] = pd;
                    }
                    if (id >= 0) {
                        uint8_t *page = page_addr(ps, id);
                        my_row = page + (pp.r % P) * H;
                        my_scale = reinterpret_cast<float *>(page + plane1_off + (pp.r % P) * 4);
                    }
                }
            }
            s_d[buf][pr][lane] = my_d;
            s_prow[buf][pr][lane] = (unsigned long long)reinterpret_cast<uintptr_t>(my_row);
        }
        uint32_t m = 0;
        if (h == 1 && lane == 0) { // warp 1 hands its first and lone vectors to the lookaheads
            if (un > 0) s_look[buf][pr][0] = v[0];
            if (lone) {
                const int4 lv = ld_stream(row + nstep - 1);
                s_look[buf][pr][1] = lv;
                m = absmax_bf16x2(m, (uint32_t)lv.x);
                m = absmax_bf16x2(m, (uint32_t)lv.y);
                m = absmax_bf16x2(m, (uint32_t)lv.z);
                m = absmax_bf16x2(m, (uint32_t)lv.w);
            }
        }
#pragma unroll
        for (int i = 0; i < 2 * NRU; ++i) {
            m = absmax_bf16x2(m, (uint32_t)v[i].x);
            m = absmax_bf16x2(m, (uint32_t)v[i].y);
            m = absmax_bf16x2(m, (uint32_t)v[i].z);
            m = absmax_bf16x2(m, (uint32_t)v[i].w);
        }
        const uint32_t half_amax = __reduce_max_sync(0xffffffffu, absmax_bits(m));
        if (lane == 0) s_amax[buf][pr][h] = half_amax;
        pair_barrier(1 + pr);
        const uint32_t a0 = s_amax[buf][pr][0], a1 = s_amax[buf][pr][1];
        float scale, inv;
        e4m3_scales(a0 > a1 ? a0 : a1, scale, inv);
        if (h == 0 && my_d >= 0) {
            xd_scale[my_d] = scale;
            if (my_scale) *my_scale = scale;
        }
#pragma unroll
        for (int i = 0; i < 2 * NRU; ++i) { // codes replace the values in place (first 8 bytes)
            const int2 c = quantize8_e4m3(v[i], inv);
            v[i].x = c.x;
            v[i].y = c.y;
        }
        // warp 0's lookahead is warp 1's first vector, or the lone one when
        // warp 1 has no unit; warp 1's is the lone one
        const int4 lav = (lane == 0 && la >= 0) ? s_look[buf][pr][(h == 1 || 2 * u0 == nstep - 1) ? 1 : 0] : zero;
        const int2 lc = quantize8_e4m3(lav, inv);
        const int la_x = __shfl_sync(0xffffffffu, lc.x, 0), la_y = __shfl_sync(0xffffffffu, lc.y, 0);
        int2 nx[NRU];
        // for a row 8 bytes off: the lower half of the unit after this lane's
        // (next lane, lane 0 of the next round, or the lookahead)
#pragma unroll
        for (int i = 0; i < NRU; ++i) {
            int nxx = __shfl_down_sync(0xffffffffu, v[2 * i].x, 1), nxy = __shfl_down_sync(0xffffffffu, v[2 * i].y, 1);
            if (i + 1 < NRU) {
                const int bx = __shfl_sync(0xffffffffu, v[2 * i + 2].x, 0), by = __shfl_sync(0xffffffffu, v[2 * i + 2].y, 0);
                if (lane == kWarp - 1) {
                    nxx = bx;
                    nxy = by;
                }
            }
            if (lane + i * kWarp + 1 == un) {
                nxx = la_x;
                nxy = la_y;
            }
            nx[i] = make_int2(nxx, nxy);
        }
        for (int j = 0; j < k; ++j) {
            const int32_t d = s_d[buf][pr][j];
            if (d < 0) continue;
            uint8_t *rows2[2] = {xd + (int64_t)d * H,
                                 reinterpret_cast<uint8_t *>(static_cast<uintptr_t>(s_prow[buf][pr][j]))};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint8_t *A = rows2[q];
                if (!A) continue;
                if ((reinterpret_cast<uintptr_t>(A) & 8) == 0) { // 16-byte aligned row
#pragma unroll
                    for (int i = 0; i < NRU; ++i) {
                        const int w = lane + i * kWarp;
                        if (w < un)
                            st_stream(reinterpret_cast<int4 *>(A + 16 * (int64_t)(ub + w)),
                                      make_int4(v[2 * i].x, v[2 * i].y, v[2 * i + 1].x, v[2 * i + 1].y));
                    }
                    if (h == 1 && lane == 0 && lone)
                        st_stream(reinterpret_cast<int2 *>(A + 16 * (int64_t)nu), make_int2(la_x, la_y));
                } else { // 8 bytes off: aligned stores straddle two units
#pragma unroll
                    for (int i = 0; i < NRU; ++i) {
                        const int w = lane + i * kWarp;
                        if (w < un) {
                            uint8_t *c = A + 16 * (int64_t)(ub + w) + 8;
                            if (w + 1 < un || la >= 0)
                                st_stream(reinterpret_cast<int4 *>(c),
                                          make_int4(v[2 * i + 1].x, v[2 * i + 1].y, nx[i].x, nx[i].y));
                            else
                                st_stream(reinterpret_cast<int2 *>(c), make_int2(v[2 * i + 1].x, v[2 * i + 1].y));
                        }
                    }
                    if (lane == 0) { // the row's first 8 bytes
                        if (h == 0 && un > 0) st_stream(reinterpret_cast<int2 *>(A), make_int2(v[0].x, v[0].y));
                        if (h == 1 && lone && nu == 0) st_stream(reinterpret_cast<int2 *>(A), make_int2(la_x, la_y));
                    }
                }
            }
        }
    }
}

} // namespace
} // namespace ap

// ---- host runtime ------------------------------------------------------------------
namespace {

struct HostRec {
    uint64_t id;
    int64_t index; // record index in the metadata buffer
    int32_t nplanes;
    int64_t rb[2];
    int32_t rows_per_tile, tiles_per_page;
    int64_t bound_pages; // upper bound of the record's pages (grid sizing)
};

} // namespace

struct ap_pool {
    ap_pool_config cfg;
    uint8_t *dev_pool = nullptr;
    uint8_t *dev_meta = nullptr;
    uint8_t *host_spill = nullptr;
    uint8_t *spill_dev = nullptr;
    cudaStream_t stream = nullptr;
    ap::MetaLayout M;
    int32_t max_ctas = 2048;
    HostRec *q = nullptr; // [S][R]
    int32_t *q_head = nullptr, *q_count = nullptr;
    uint64_t next_id = 1;
    void *pinned = nullptr; // small pinned host buffer for read-outs
    uint32_t last_flags = 0;
    ap_pool_state last_state{}; // the last synchronising read-out of the state block (ap_pool_stats)
    bool have_state = false;
    cudaEvent_t copy_before = nullptr, copy_after = nullptr; // ap_pool_time_copies
};

namespace {

using ap::fail;

ap_status check_config(const ap_pool_config *c)
{
    if (!c) return fail(AP_EINVAL, "pool config is NULL");
    if (c->page_tokens < 1) return fail(AP_EINVAL, "page_tokens must be >= 1");
    if (c->page_bytes < 16 || c->page_bytes % 16) return fail(AP_EINVAL, "page_bytes must be a positive multiple of 16");
    const int64_t nmax = ap::max_pages_of(*c);
    if (c->num_pages < 0 || c->max_num_pages < 0 || nmax < 1 || c->num_pages > nmax || c->spill_pages < 0 ||
        nmax + c->spill_pages >= (int64_t(1) << 31))
        return fail(AP_EINVAL, "need 0 <= num_pages <= max_num_pages (>= 1) and max_num_pages + spill_pages < 2^31");
    if (c->num_slots < 1 || c->max_records_per_slot < 1) return fail(AP_EINVAL, "num_slots and max_records_per_slot must be >= 1");
    if (c->max_segments < 1 || c->max_segments > (1 << 20)) return fail(AP_EINVAL, "max_segments must lie in [1, 2^20]");
    if (c->max_pages_per_record < 1 || c->max_pages_per_record >= (int64_t(1) << 31))
        return fail(AP_EINVAL, "max_pages_per_record must lie in [1, 2^31)");
    if (c->max_ctas < 0) return fail(AP_EINVAL, "max_ctas must be >= 0");
    if (c->reserved != 0) return fail(AP_EINVAL, "reserved must be 0");
    return AP_OK;
}

int resolve_max_ctas(int32_t cfg_value)
{
    if (cfg_value > 0) return cfg_value;
    const char *env = getenv("AP_STASH_MAX_CTAS");
    if (env && *env) {
        char *end = nullptr;
        const long v = strtol(env, &end, 10);
        if (end && *end == '\0' && v >= 1 && v <= (1L << 30)) return (int)v;
    }
    return 2048;
}

bool plane_fit(const ap_pool *p, int32_t nplanes, const int64_t *rb, int64_t *page_off)
{
    if (nplanes < 1 || nplanes > 2) return false;
    const int64_t P = p->cfg.page_tokens;
    if (rb[0] < 1 || (nplanes == 2 && rb[1] < 1)) return false;
    page_off[0] = 0;
    int64_t need = P * rb[0];
    page_off[1] = 0;
    if (nplanes == 2) {
        page_off[1] = ap::align_up(P * rb[0], 16);
        need = page_off[1] + P * rb[1];
    }
    return need <= p->cfg.page_bytes;
}

// Records the caller's timing event (if set) on the paging stream.
void mark(const ap_pool *p, cudaEvent_t ev)
{
    if (ev) (void)cudaEventRecord(ev, p->stream);
}

// Rows per copy tile: about 32 KB of plane 0, rounded to the nearest whole
// row (so that rows just over a divisor of 32 KB, such as 2056-byte E4M3
// rows, fill the copy's full eight-vector passes rather than leaving most of
// a pass to its tail), at least one row and at most a page.
int64_t tile_rows(int64_t rb0, int64_t P)
{
    int64_t rpt = (32768 + rb0 / 2) / rb0;
    if (rpt < 1) rpt = 1;
    if (rpt > P) rpt = P;
    return rpt;
}

ap::PageSpace page_space(const ap_pool *p)
{
    ap::PageSpace ps;
    ps.ring = reinterpret_cast<int32_t *>(p->dev_meta + p->M.ring);
    ps.spill_ring = reinterpret_cast<int32_t *>(p->dev_meta + p->M.spill_ring);
    ps.pool = p->dev_pool;
    ps.spill = p->spill_dev;
    ps.N = p->cfg.num_pages;
    ps.SB = ap::max_pages_of(p->cfg);
    ps.SP = p->cfg.spill_pages;
    ps.page_bytes = p->cfg.page_bytes;
    return ps;
}

ap_status sync_read(ap_pool *p, void *host, const void *dev, size_t bytes)
{
    cudaError_t e = cudaMemcpyAsync(host, dev, bytes, cudaMemcpyDeviceToHost, p->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
    if (e != cudaSuccess) return ap::cuda_fail(e, "pool read-out");
    return AP_OK;
}

} // namespace

extern "C" ap_status ap_pool_required_bytes(const ap_pool_config *cfg, int64_t *dev_pool_bytes,
                                            int64_t *dev_meta_bytes, int64_t *host_spill_bytes)
{
    ap_status s = check_config(cfg);
    if (s != AP_OK) return s;
    const ap::MetaLayout M = ap::meta_layout(*cfg);
    if (dev_pool_bytes) *dev_pool_bytes = cfg->num_pages * cfg->page_bytes;
    if (dev_meta_bytes) *dev_meta_bytes = M.total;
    if (host_spill_bytes) *host_spill_bytes = cfg->spill_pages * cfg->page_bytes;
    return AP_OK;
}

extern "C" ap_status ap_pool_init(ap_pool **out, const ap_pool_config *cfg, void *dev_pool, void *dev_meta,
                                  void *host_spill, void *paging_stream)
{
    AP_NVTX_RANGE("ap_pool_init");
    if (!out) return fail(AP_EINVAL, "pool_init: out is NULL");
    *out = nullptr;
    ap_status s = check_config(cfg);
    if (s != AP_OK) return s;
    if (!dev_meta || (!dev_pool && cfg->num_pages > 0))
        return fail(AP_EINVAL, "pool_init: NULL pool or metadata buffer");
    if ((reinterpret_cast<uintptr_t>(dev_pool) | reinterpret_cast<uintptr_t>(dev_meta)) & 255)
        return fail(AP_EINVAL, "pool_init: pool and metadata buffers must be 256-byte aligned");
    if ((cfg->spill_pages > 0) != (host_spill != nullptr))
        return fail(AP_EINVAL, "pool_init: host_spill must be given iff spill_pages > 0");
    uint8_t *spill_dev = nullptr;
    if (host_spill) {
        // pinned host memory is mapped into the device address space; its
        // attributes give the device-side address (also for interior pointers)
        cudaPointerAttributes attr;
        cudaError_t e = cudaPointerGetAttributes(&attr, host_spill);
        if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) {
            (void)cudaGetLastError();
            return fail(AP_EINVAL, "pool_init: host_spill is not mapped pinned host memory (%s)",
                        e != cudaSuccess ? cudaGetErrorString(e) : "not page-locked");
        }
        spill_dev = static_cast<uint8_t *>(attr.devicePointer);
    }
    ap_pool *p = new (std::nothrow) ap_pool();
    if (!p) return fail(AP_EINVAL, "pool_init: out of host memory");
    p->cfg = *cfg;
    p->dev_pool = static_cast<uint8_t *>(dev_pool);
    p->dev_meta = static_cast<uint8_t *>(dev_meta);
    p->host_spill = static_cast<uint8_t *>(host_spill);
    p->spill_dev = spill_dev;
    p->stream = static_cast<cudaStream_t>(paging_stream);
    p->M = ap::meta_layout(*cfg);
    p->max_ctas = resolve_max_ctas(cfg->max_ctas);
    const int64_t nrec = (int64_t)cfg->num_slots * cfg->max_records_per_slot;
    p->q = new (std::nothrow) HostRec[nrec];
    p->q_head = new (std::nothrow) int32_t[cfg->num_slots]();
    p->q_count = new (std::nothrow) int32_t[cfg->num_slots]();
    if (!p->q || !p->q_head || !p->q_count) {
        ap_pool_destroy(p);
        return fail(AP_EINVAL, "pool_init: out of host memory");
    }
    cudaError_t e = cudaMallocHost(&p->pinned, 256);
    if (e != cudaSuccess) {
        p->pinned = nullptr;
        ap_pool_destroy(p);
        return ap::cuda_fail(e, "pool_init: pinned read-out buffer");
    }
    s = ap_pool_reset(p, paging_stream);
    if (s != AP_OK) {
        ap_pool_destroy(p);
        return s;
    }
    *out = p;
    return AP_OK;
}

extern "C" ap_status ap_pool_reset(ap_pool *p, void *stream)
{
    AP_NVTX_RANGE("ap_pool_reset");
    if (!p) return fail(AP_EINVAL, "pool_reset: NULL pool");
    if (static_cast<cudaStream_t>(stream) != p->stream) return fail(AP_ESTREAM, "pool_reset: not the paging stream");
    for (int32_t s = 0; s < p->cfg.num_slots; ++s) {
        p->q_head[s] = 0;
        p->q_count[s] = 0;
    }
    p->last_flags = 0;
    const int64_t nmax = ap::max_pages_of(p->cfg);
    const int64_t n = nmax > p->cfg.spill_pages ? nmax : p->cfg.spill_pages;
    int64_t grid = (n + 255) / 256;
    if (grid > 1024) grid = 1024;
    if (grid < 1) grid = 1;
    ap::launch(ap::k_reset, (unsigned)grid, 256, 0, p->stream, reinterpret_cast<ap_pool_state *>(p->dev_meta),
                                                      reinterpret_cast<int32_t *>(p->dev_meta + p->M.ring),
                                                      p->cfg.num_pages, nmax,
                                                      reinterpret_cast<int32_t *>(p->dev_meta + p->M.spill_ring),
                                                      p->cfg.spill_pages);
    AP_CHECK_LAUNCH("pool reset launch");
    return AP_OK;
}

extern "C" ap_status ap_pool_grow(ap_pool *p, int64_t num_pages, void *dev_pool, void *stream)
{
    AP_NVTX_RANGE("ap_pool_grow");
    if (!p) return fail(AP_EINVAL, "pool_grow: NULL pool");
    if (static_cast<cudaStream_t>(stream) != p->stream) return fail(AP_ESTREAM, "pool_grow: not the paging stream");
    const int64_t n0 = p->cfg.num_pages, nmax = ap::max_pages_of(p->cfg);
    if (num_pages < n0 || num_pages > nmax)
        return fail(AP_EINVAL, "pool_grow: %lld pages outside [%lld, %lld]", (long long)num_pages, (long long)n0,
                    (long long)nmax);
    uint8_t *pool = static_cast<uint8_t *>(dev_pool);
    if (num_pages > 0 && !pool) return fail(AP_EINVAL, "pool_grow: NULL pool memory");
    if (reinterpret_cast<uintptr_t>(pool) & 255) return fail(AP_EINVAL, "pool_grow: pool memory not 256-byte aligned");
    if (n0 > 0 && pool != p->dev_pool)
        return fail(AP_EINVAL, "pool_grow: the pool memory must keep its address once it holds pages");
    if (num_pages == n0) return AP_OK;
    ap::launch(ap::k_grow, 1, 1024, 0, p->stream, reinterpret_cast<ap_pool_state *>(p->dev_meta),
                                          reinterpret_cast<int32_t *>(p->dev_meta + p->M.ring),
                                          reinterpret_cast<int32_t *>(p->dev_meta + p->M.grow_tmp), n0, num_pages);
    AP_CHECK_LAUNCH("pool grow launch");
    p->cfg.num_pages = num_pages;
    p->dev_pool = pool;
    return AP_OK;
}

extern "C" ap_status ap_pool_time_copies(ap_pool *p, void *before, void *after)
{
    if (!p) return fail(AP_EINVAL, "pool_time_copies: NULL pool");
    if ((before == nullptr) != (after == nullptr)) return fail(AP_EINVAL, "pool_time_copies: give both events or neither");
    p->copy_before = static_cast<cudaEvent_t>(before);
    p->copy_after = static_cast<cudaEvent_t>(after);
    return AP_OK;
}

extern "C" ap_status ap_pool_destroy(ap_pool *p)
{
    if (!p) return AP_OK;
    if (p->pinned) cudaFreeHost(p->pinned);
    delete[] p->q;
    delete[] p->q_head;
    delete[] p->q_count;
    delete p;
    return AP_OK;
}

extern "C" ap_status ap_pool_max_ctas(const ap_pool *p, int32_t *max_ctas)
{
    if (!p || !max_ctas) return fail(AP_EINVAL, "pool_max_ctas: NULL argument");
    *max_ctas = p->max_ctas;
    return AP_OK;
}

extern "C" ap_status ap_pool_set_max_ctas(ap_pool *p, int32_t max_ctas)
{
    if (!p || max_ctas < 0) return fail(AP_EINVAL, "pool_set_max_ctas: bad argument");
    p->max_ctas = resolve_max_ctas(max_ctas);
    return AP_OK;
}

extern "C" ap_status ap_stash_push(ap_pool *p, int32_t slot, int32_t nplanes, const void *const *src_planes,
                                   const int64_t *row_bytes, int64_t src_rows, int32_t nseg,
                                   const int32_t *d_seg_off, const int32_t *d_live, uint64_t *record_id,
                                   void *stream)
{
    AP_NVTX_RANGE("ap_stash_push");
    if (!p) return fail(AP_EINVAL, "stash_push: NULL pool");
    if (static_cast<cudaStream_t>(stream) != p->stream) return fail(AP_ESTREAM, "stash_push: not the paging stream");
    if (slot < 0 || slot >= p->cfg.num_slots) return fail(AP_EINVAL, "stash_push: slot %d out of range", slot);
    if (!src_planes || !row_bytes) return fail(AP_EINVAL, "stash_push: NULL plane arrays");
    if (nseg < 0 || nseg > p->cfg.max_segments)
        return fail(AP_EINVAL, "stash_push: nseg %d outside [0, %d]", nseg, p->cfg.max_segments);
    if (src_rows < 0) return fail(AP_EINVAL, "stash_push: src_rows < 0");
    int64_t rb[2] = {row_bytes[0], nplanes == 2 ? row_bytes[1] : 0};
    int64_t page_off[2] = {0, 0};
    if (!plane_fit(p, nplanes, rb, page_off))
        return fail(AP_EINVAL, "stash_push: %d plane(s) of the given row bytes do not fit a page", nplanes);
    for (int i = 0; i < nplanes; ++i)
        if (!src_planes[i] && src_rows > 0) return fail(AP_EINVAL, "stash_push: NULL source plane");
    if (nseg > 0 && (!d_seg_off || !d_live)) return fail(AP_EINVAL, "stash_push: NULL seg_off/live");
    if (p->q_count[slot] >= p->cfg.max_records_per_slot) return fail(AP_EQFULL, "stash_push: slot %d queue full", slot);

    const int32_t pos = (p->q_head[slot] + p->q_count[slot]) % p->cfg.max_records_per_slot;
    const int64_t index = (int64_t)slot * p->cfg.max_records_per_slot + pos;
    HostRec &h = p->q[index];
    h.id = p->next_id;
    h.index = index;
    h.nplanes = nplanes;
    h.rb[0] = rb[0];
    h.rb[1] = rb[1];
    const int64_t P = p->cfg.page_tokens;
    const int64_t rpt = tile_rows(rb[0], P);
    h.rows_per_tile = (int32_t)rpt;
    h.tiles_per_page = (int32_t)((P + rpt - 1) / rpt);
    int64_t bound = nseg + (src_rows + P - 1) / P;
    if (bound > p->cfg.max_pages_per_record) bound = p->cfg.max_pages_per_record;
    h.bound_pages = bound;

    ap::RecPtr rec = ap::rec_ptr(p->dev_meta, p->M, index);
    ap_pool_state *st = reinterpret_cast<ap_pool_state *>(p->dev_meta);
    ap::launch(ap::k_push_plan, 1, ap::kPlanThreads, 0, p->stream, st, rec, nseg, d_seg_off, d_live, src_rows,
                                                           p->cfg.page_tokens, p->cfg.max_pages_per_record,
                                                           p->cfg.num_pages, p->cfg.spill_pages);
    AP_CHECK_LAUNCH("stash push plan launch");
    ap::Planes pl;
    for (int i = 0; i < 2; ++i) {
        pl.p[i] = (i < nplanes) ? const_cast<uint8_t *>(static_cast<const uint8_t *>(src_planes[i])) : nullptr;
        pl.rb[i] = rb[i];
        pl.page_off[i] = page_off[i];
    }
    pl.n = nplanes;
    int64_t grid = bound * h.tiles_per_page;
    if (grid > p->max_ctas) grid = p->max_ctas;
    if (grid < 1) grid = 1;
    mark(p, p->copy_before);
    ap::launch(ap::k_push_copy, (unsigned)grid, ap::kCopyThreads, 0, p->stream, st, rec, page_space(p), pl, h.rows_per_tile,
                                                                        h.tiles_per_page);
    AP_CHECK_LAUNCH("stash push copy launch");
    mark(p, p->copy_after);
    p->next_id += 1;
    p->q_count[slot] += 1;
    if (record_id) *record_id = h.id;
    return AP_OK;
}

namespace {

// Fused dispatch + push; with logits != NULL the routing (into idx and w) is
// done by the count/rank launch itself.
ap_status dispatch_stash_impl(ap_pool *p, int32_t slot, const float *logits, float *w, const void *x, int64_t T,
                              int32_t H, int32_t *idx, int32_t k, int32_t E, int32_t capacity, int32_t padded,
                              int32_t out_dtype, void *xd, float *xd_scale, int64_t xd_rows, int32_t *counts,
                              int32_t *live, int32_t *seg_off, int32_t *dest, int32_t *src_tok, void *scratch,
                              int64_t scratch_bytes, uint32_t *d_status, uint64_t *record_id, void *stream,
                              bool ranked = false, bool scanned = false)
{
    using namespace ap;
    if (!p) return fail(AP_EINVAL, "dispatch_stash: NULL pool");
    if (static_cast<cudaStream_t>(stream) != p->stream) return fail(AP_ESTREAM, "dispatch_stash: not the paging stream");
    if (slot < 0 || slot >= p->cfg.num_slots) return fail(AP_EINVAL, "dispatch_stash: slot %d out of range", slot);
    ap_status s = dispatch_check("dispatch_stash", x, T, H, idx, k, E, capacity, padded, xd, xd_rows, counts, live,
                                 seg_off, dest, scratch, scratch_bytes);
    if (s != AP_OK) return s;
    if (E > p->cfg.max_segments)
        return fail(AP_EINVAL, "dispatch_stash: E=%d segments > max_segments %d", E, p->cfg.max_segments);
    if (out_dtype != AP_DTYPE_BF16 && out_dtype != AP_DTYPE_E4M3)
        return fail(AP_EINVAL, "dispatch_stash: unknown out_dtype %d", out_dtype);
    const bool fp8 = out_dtype == AP_DTYPE_E4M3;
    const int nplanes = fp8 ? 2 : 1;
    int64_t rb[2] = {fp8 ? (int64_t)H : (int64_t)H * 2, fp8 ? 4 : 0};
    int64_t page_off[2] = {0, 0};
    if (!plane_fit(p, nplanes, rb, page_off))
        return fail(AP_EINVAL, "dispatch_stash: the rows of H=%d do not fit a page", H);
    if (fp8 && T > 0 && !xd_scale) return fail(AP_EINVAL, "dispatch_stash: E4M3 needs xd_scale");
    if (p->q_count[slot] >= p->cfg.max_records_per_slot)
        return fail(AP_EQFULL, "dispatch_stash: slot %d queue full", slot);
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xd) |
                         reinterpret_cast<uintptr_t>(p->dev_pool) | reinterpret_cast<uintptr_t>(p->spill_dev) |
                         (uintptr_t)rb[0] | (uintptr_t)p->cfg.page_bytes;
    if (!fp8 && T > 0 && (al & 15) != 0 && (al & 7) != 0)
        return fail(AP_ENOTSUP, "dispatch_stash: rows must be 8-byte aligned (H %% 4 == 0)");
    if (fp8 && T > 0 && (H % 8 != 0 || H > 256 * 16 || (reinterpret_cast<uintptr_t>(x) & 15) != 0 || (al & 7) != 0))
        return fail(AP_ENOTSUP, "dispatch_stash: E4M3 needs H %% 8 == 0, H <= 4096 and aligned buffers");
    if (logits && k > E) return fail(AP_EINVAL, "route_dispatch_stash: k=%d > E=%d", k, E);
    if (logits && T > 0 && !w) return fail(AP_EINVAL, "route_dispatch_stash: NULL weights");
    cudaStream_t st = p->stream;
    const int32_t pos = (p->q_head[slot] + p->q_count[slot]) % p->cfg.max_records_per_slot;
    const int64_t index = (int64_t)slot * p->cfg.max_records_per_slot + pos;
    ap::RecPtr rec = ap::rec_ptr(p->dev_meta, p->M, index);
    ap_pool_state *stt = reinterpret_cast<ap_pool_state *>(p->dev_meta);
    // few block counts: the copy kernel plans the record itself (no scan + plan launch)
    const bool inl = T > 0 && (int64_t)dispatch_blocks(T) * E <= ap::kInlineMaxCounts && E <= ap::kInlineMaxE;
    if (!ranked) { // else dest and scratch hold ap_count_rank's results for idx
        s = logits ? dispatch_route_count_rank(logits, T, E, k, idx, w, scratch, dest, st, x, (int64_t)H * 2)
                   : dispatch_count_rank(T, idx, k, E, scratch, dest, d_status, st, x, (int64_t)H * 2);
        if (s != AP_OK) return s;
    }

    HostRec &h = p->q[index];
    h.id = p->next_id;
    h.index = index;
    h.nplanes = nplanes;
    h.rb[0] = rb[0];
    h.rb[1] = rb[1];
    const int64_t P = p->cfg.page_tokens;
    const int64_t rpt = tile_rows(rb[0], P);
    h.rows_per_tile = (int32_t)rpt;
    h.tiles_per_page = (int32_t)((P + rpt - 1) / rpt);
    int64_t bound = E + (xd_rows + P - 1) / P;
    if (bound > p->cfg.max_pages_per_record) bound = p->cfg.max_pages_per_record;
    h.bound_pages = bound;
    ap::InlineArgs ia{};
    ia.src_rows = xd_rows; // the copy kernels' bound on a dispatch row
    if (inl) {
        ia.enabled = scanned ? 2 : 1;
        ia.nblk = dispatch_blocks(T);
        ia.padded = padded;
        ia.counts = counts;
        ia.live = live;
        ia.max_pages = p->cfg.max_pages_per_record;
    } else if (scanned) { // the expert scan ran with the count/rank: the page plan alone
        ap::launch(ap::k_scanned_plan, 1, ap::kPlanThreads, 0, st, stt, rec, E, static_cast<const int32_t *>(seg_off),
                   static_cast<const int32_t *>(live), xd_rows, p->cfg.page_tokens, p->cfg.max_pages_per_record,
                   p->cfg.num_pages, p->cfg.spill_pages);
        AP_CHECK_LAUNCH("dispatch_stash plan launch");
    } else {
        ap::launch(ap::k_scan_plan, 1, ap::kPlanThreads, 0, st, static_cast<int32_t *>(scratch), dispatch_blocks(T),
                   E, capacity, padded, counts, live, seg_off, stt, rec, xd_rows, p->cfg.page_tokens,
                   p->cfg.max_pages_per_record, p->cfg.num_pages, p->cfg.spill_pages);
        AP_CHECK_LAUNCH("dispatch_stash scan + plan launch");
    }
    if (T > 0) {
        // an inline-planned copy covers every token in one pass (each block's
        // tokens in one count/rank block); otherwise the grid is capped and
        // blocks stride over the tokens
        const int64_t want = (T + 7) / 8;
        const int64_t cap = inl ? want : (int64_t)sm_count() * 16;
        const int grid = (int)(want < cap ? want : cap);
        const ap::PageSpace ps = page_space(p);
        const uint8_t *xs = static_cast<const uint8_t *>(x);
        mark(p, p->copy_before);
        uint8_t *xo = static_cast<uint8_t *>(xd);
        const int32_t *blk = static_cast<const int32_t *>(scratch);
        if (fp8) {
            const uint16_t *xs16 = static_cast<const uint16_t *>(x);
            const int64_t want2 = (T + 3) / 4; // four tokens (warp pairs) per block
            const int64_t cap2 = inl ? want2 : (int64_t)sm_count() * 16;
            const int grid2 = (int)(want2 < cap2 ? want2 : cap2);
            // every row 16-byte aligned (H and every base are): one vector per
            // lane and round, 8-byte code stores; otherwise 16-code units and
            // aligned 16-byte stores (a warp holds at most 32 * NRU units, so
            // H / 8 <= 128 * NRU + 1 vectors)
            const bool aligned16 = H % 16 == 0 && (al & 15) == 0;
            const int nvec = H / 8;
#define AP_LAUNCH_E4M3(KERNEL)                                                                                    \
    ap::launch(KERNEL, grid2, 256, 0, st, xs16, T, H, idx, dest, k, E, capacity, blk, seg_off, src_tok, xo,       \
               xd_scale, stt, rec, ps, p->cfg.page_tokens, page_off[1], ia)
            if (aligned16) {
                if (H <= 512) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3<1>);
                else if (H <= 1024) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3<2>);
                else if (H <= 2048) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3<4>);
                else if (H <= 2304) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3<5>);
                else AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3<8>);
            } else if (nvec <= 129) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3_units<1>);
            else if (nvec <= 257) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3_units<2>);
            else if (nvec <= 385) AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3_units<3>);
            else AP_LAUNCH_E4M3(ap::k_dispatch_stash_e4m3_units<4>);
#undef AP_LAUNCH_E4M3
        } else if ((al & 15) == 0)
            ap::launch(ap::k_dispatch_stash_copy<int4>, grid, 256, 0, st, xs, T, rb[0], idx, dest, k, E, capacity, blk,
                       seg_off, src_tok, xo, stt, rec, ps, p->cfg.page_tokens, ia);
        else
            ap::launch(ap::k_dispatch_stash_copy<int2>, grid, 256, 0, st, xs, T, rb[0], idx, dest, k, E, capacity, blk,
                       seg_off, src_tok, xo, stt, rec, ps, p->cfg.page_tokens, ia);
        AP_CHECK_LAUNCH("dispatch_stash copy launch");
        mark(p, p->copy_after);
    }
    p->next_id += 1;
    p->q_count[slot] += 1;
    if (record_id) *record_id = h.id;
    return AP_OK;
}

} // namespace

extern "C" ap_status ap_dispatch_stash(ap_pool *p, int32_t slot, const void *x, int64_t T, int32_t H,
                                       const int32_t *idx, int32_t k, int32_t E, int32_t capacity, int32_t padded,
                                       int32_t out_dtype, void *xd, float *xd_scale, int64_t xd_rows,
                                       int32_t *counts, int32_t *live, int32_t *seg_off, int32_t *dest,
                                       int32_t *src_tok, void *scratch, int64_t scratch_bytes, uint32_t *d_status,
                                       uint64_t *record_id, void *stream)
{
    AP_NVTX_RANGE("ap_dispatch_stash");
    return dispatch_stash_impl(p, slot, nullptr, nullptr, x, T, H, const_cast<int32_t *>(idx), k, E, capacity,
                               padded, out_dtype, xd, xd_scale, xd_rows, counts, live, seg_off, dest, src_tok,
                               scratch, scratch_bytes, d_status, record_id, stream);
}

extern "C" ap_status ap_route_dispatch_stash(ap_pool *p, int32_t slot, const float *logits, float *w, const void *x,
                                             int64_t T, int32_t H, int32_t *idx, int32_t k, int32_t E,
                                             int32_t capacity, int32_t padded, int32_t out_dtype, void *xd,
                                             float *xd_scale, int64_t xd_rows, int32_t *counts, int32_t *live,
                                             int32_t *seg_off, int32_t *dest, int32_t *src_tok, void *scratch,
                                             int64_t scratch_bytes, uint32_t *d_status, uint64_t *record_id,
                                             void *stream)
{
    AP_NVTX_RANGE("ap_route_dispatch_stash");
    if (T > 0 && !logits) return ap::fail(AP_EINVAL, "route_dispatch_stash: NULL logits");
    static const float kNoLogits = 0.f; // T == 0: nothing to route, still the routing variant
    return dispatch_stash_impl(p, slot, logits ? logits : &kNoLogits, w, x, T, H, idx, k, E, capacity, padded,
                               out_dtype, xd, xd_scale, xd_rows, counts, live, seg_off, dest, src_tok, scratch,
                               scratch_bytes, d_status, record_id, stream);
}

extern "C" ap_status ap_dispatch_stash_ranked(ap_pool *p, int32_t slot, const void *x, int64_t T, int32_t H,
                                              const int32_t *idx, int32_t k, int32_t E, int32_t capacity,
                                              int32_t padded, int32_t out_dtype, void *xd, float *xd_scale,
                                              int64_t xd_rows, int32_t *counts, int32_t *live, int32_t *seg_off,
                                              int32_t *dest, int32_t *src_tok, void *scratch, int64_t scratch_bytes,
                                              uint32_t *d_status, uint64_t *record_id, int32_t scanned,
                                              void *stream)
{
    AP_NVTX_RANGE("ap_dispatch_stash_ranked");
    if (scanned != 0 && scanned != 1) return ap::fail(AP_EINVAL, "dispatch_stash_ranked: scanned must be 0 or 1");
    return dispatch_stash_impl(p, slot, nullptr, nullptr, x, T, H, const_cast<int32_t *>(idx), k, E, capacity,
                               padded, out_dtype, xd, xd_scale, xd_rows, counts, live, seg_off, dest, src_tok,
                               scratch, scratch_bytes, d_status, record_id, stream, true, scanned != 0);
}

extern "C" ap_status ap_stash_pop(ap_pool *p, int32_t slot, int32_t nplanes, void *const *dst_planes,
                                  int64_t dst_rows, uint64_t *record_id, void *stream)
{
    AP_NVTX_RANGE("ap_stash_pop");
    if (!p) return fail(AP_EINVAL, "stash_pop: NULL pool");
    if (static_cast<cudaStream_t>(stream) != p->stream) return fail(AP_ESTREAM, "stash_pop: not the paging stream");
    if (slot < 0 || slot >= p->cfg.num_slots) return fail(AP_EINVAL, "stash_pop: slot %d out of range", slot);
    if (p->q_count[slot] == 0) return fail(AP_EEMPTY, "stash_pop: slot %d is empty", slot);
    const int64_t index = (int64_t)slot * p->cfg.max_records_per_slot + p->q_head[slot];
    const HostRec &h = p->q[index];
    if (nplanes != h.nplanes) return fail(AP_EINVAL, "stash_pop: record has %d plane(s), got %d", h.nplanes, nplanes);
    if (!dst_planes || dst_rows < 0) return fail(AP_EINVAL, "stash_pop: bad destination");
    for (int i = 0; i < nplanes; ++i)
        if (!dst_planes[i]) return fail(AP_EINVAL, "stash_pop: NULL destination plane");
    int64_t page_off[2] = {0, 0};
    plane_fit(p, h.nplanes, h.rb, page_off);
    ap::RecPtr rec = ap::rec_ptr(p->dev_meta, p->M, index);
    ap_pool_state *st = reinterpret_cast<ap_pool_state *>(p->dev_meta);
    ap::Planes pl;
    for (int i = 0; i < 2; ++i) {
        pl.p[i] = (i < nplanes) ? static_cast<uint8_t *>(dst_planes[i]) : nullptr;
        pl.rb[i] = h.rb[i];
        pl.page_off[i] = page_off[i];
    }
    pl.n = nplanes;
    int64_t grid = h.bound_pages * h.tiles_per_page;
    if (grid > p->max_ctas) grid = p->max_ctas;
    if (grid < 1) grid = 1;
    mark(p, p->copy_before);
    ap::launch(ap::k_pop_copy, (unsigned)grid, ap::kCopyThreads, 0, p->stream, st, rec, page_space(p), pl, dst_rows,
                                                                       h.rows_per_tile, h.tiles_per_page);
    AP_CHECK_LAUNCH("stash pop copy launch");
    mark(p, p->copy_after);
    if (record_id) *record_id = h.id;
    p->q_head[slot] = (p->q_head[slot] + 1) % p->cfg.max_records_per_slot;
    p->q_count[slot] -= 1;
    return AP_OK;
}

extern "C" ap_status ap_pool_queue_len(const ap_pool *p, int32_t slot, int32_t *len)
{
    if (!p || !len) return fail(AP_EINVAL, "pool_queue_len: NULL argument");
    if (slot < 0 || slot >= p->cfg.num_slots) return fail(AP_EINVAL, "pool_queue_len: slot out of range");
    *len = p->q_count[slot];
    return AP_OK;
}

extern "C" ap_status ap_pool_flags_device_ptr(const ap_pool *p, uint32_t **d_flags)
{
    if (!p || !d_flags) return fail(AP_EINVAL, "pool_flags_device_ptr: NULL argument");
    *d_flags = &reinterpret_cast<ap_pool_state *>(p->dev_meta)->flags;
    return AP_OK;
}

extern "C" ap_status ap_overflow_query(ap_pool *p, uint32_t *flags, int32_t wait)
{
    AP_NVTX_RANGE("ap_overflow_query");
    if (!p || !flags) return fail(AP_EINVAL, "overflow_query: NULL argument");
    if (wait) {
        ap_status s = sync_read(p, p->pinned, &reinterpret_cast<ap_pool_state *>(p->dev_meta)->flags, 4);
        if (s != AP_OK) return s;
        memcpy(&p->last_flags, p->pinned, 4);
    }
    *flags = p->last_flags;
    return AP_OK;
}

extern "C" ap_status ap_pool_read_state(ap_pool *p, ap_pool_state *state)
{
    AP_NVTX_RANGE("ap_pool_read_state");
    if (!p || !state) return fail(AP_EINVAL, "pool_read_state: NULL argument");
    ap_status s = sync_read(p, p->pinned, p->dev_meta, sizeof(ap_pool_state));
    if (s != AP_OK) return s;
    memcpy(state, p->pinned, sizeof(ap_pool_state));
    p->last_flags = state->flags;
    p->last_state = *state;
    p->have_state = true;
    return AP_OK;
}

extern "C" ap_status ap_pool_stats(ap_pool *p, int64_t *pages_in_use, int64_t *high_water, int64_t *spill_in_use,
                                   int32_t wait)
{
    AP_NVTX_RANGE("ap_pool_stats");
    if (!p) return fail(AP_EINVAL, "pool_stats: NULL pool");
    if (wait) {
        ap_pool_state st;
        ap_status s = ap_pool_read_state(p, &st);
        if (s != AP_OK) return s;
    }
    const ap_pool_state &st = p->last_state;
    const bool h = p->have_state; // zeros before the first read-out
    if (pages_in_use) *pages_in_use = h ? st.num_pages - (int64_t)(st.tail - st.head) : 0;
    if (high_water) *high_water = h ? st.high_water : 0;
    if (spill_in_use) *spill_in_use = h ? p->cfg.spill_pages - (int64_t)(st.spill_tail - st.spill_head) : 0;
    return AP_OK;
}

extern "C" ap_status ap_pool_read_rings(ap_pool *p, int32_t *ring, int32_t *spill_ring)
{
    AP_NVTX_RANGE("ap_pool_read_rings");
    if (!p || !ring) return fail(AP_EINVAL, "pool_read_rings: NULL argument");
    ap_status s = sync_read(p, ring, p->dev_meta + p->M.ring, 4 * (size_t)p->cfg.num_pages);
    if (s == AP_OK && spill_ring && p->cfg.spill_pages > 0)
        s = sync_read(p, spill_ring, p->dev_meta + p->M.spill_ring, 4 * (size_t)p->cfg.spill_pages);
    return s;
}

extern "C" ap_status ap_pool_read_record(ap_pool *p, int32_t slot, int32_t qpos, ap_record_info *info,
                                         int32_t *page_table, int64_t *row0, int32_t *nrows, int64_t cap)
{
    AP_NVTX_RANGE("ap_pool_read_record");
    if (!p) return fail(AP_EINVAL, "pool_read_record: NULL pool");
    if (slot < 0 || slot >= p->cfg.num_slots || qpos < 0 || qpos >= p->q_count[slot])
        return fail(AP_EINVAL, "pool_read_record: no record at slot %d position %d", slot, qpos);
    const int64_t index =
        (int64_t)slot * p->cfg.max_records_per_slot + (p->q_head[slot] + qpos) % p->cfg.max_records_per_slot;
    ap::RecPtr rec = ap::rec_ptr(p->dev_meta, p->M, index);
    ap::RecHdr hdr;
    ap_status s = sync_read(p, &hdr, rec.hdr, sizeof(hdr));
    if (s != AP_OK) return s;
    if (info) {
        info->record_id = p->q[index].id;
        info->slot = slot;
        info->nseg = hdr.nseg;
        info->npages = hdr.npages;
        info->ndev = hdr.ndev;
        info->nspill = hdr.nspill;
        info->nlost = hdr.nlost;
    }
    int64_t n = hdr.npages < cap ? hdr.npages : cap;
    if (n <= 0) return AP_OK;
    if (page_table) {
        s = sync_read(p, page_table, rec.page_table, 4 * (size_t)n);
        if (s != AP_OK) return s;
    }
    if (row0 || nrows) {
        ap::PageDesc *tmp = static_cast<ap::PageDesc *>(malloc(sizeof(ap::PageDesc) * (size_t)n));
        if (!tmp) return fail(AP_EINVAL, "pool_read_record: out of host memory");
        s = sync_read(p, tmp, rec.desc, sizeof(ap::PageDesc) * (size_t)n);
        if (s == AP_OK)
            for (int64_t i = 0; i < n; ++i) {
                if (row0) row0[i] = tmp[i].row0;
                if (nrows) nrows[i] = tmp[i].nrows;
            }
        free(tmp);
    }
    return s;
}
