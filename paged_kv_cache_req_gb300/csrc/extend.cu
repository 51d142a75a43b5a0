// pkv_extend: attention of many query tokens per request through the page table
// (extend / chunked prefill, speculative target-verify, and the mixed
// causal/full segments of a diffusion row), on the 5th-generation tensor cores.
//
// Query row j of request b sees the keys [0, kv_end[j]) of that request (by
// default the causal bound of the request's last positions).  A work item is
// (request, kv head, block of 128 query rows, chunk of keys): the rows are the
// (token, query head) pairs of 128 / g consecutive tokens times the g query
// heads sharing the kv head, so every K/V tile serves the whole block.  The
// two halves of each 128-key tile go to two softmax groups, each with its own
// online-softmax state and accumulator: one Q K^T of N = 128 serves both, and
// the tensor cores run the next tile's Q K^T and the groups' P V while the
// groups compute their exponentials.  Per CTA:
//   warps 8, 15  producers of K and of V tiles, each through a ring of its own
//              (2 and 3 stages, 4 each at head_dim 64), so K runs ahead as soon as a Q K^T
//              has run while V waits for P V: one TMA box per page per slab, one
//              copy per lane, pool rows looked up 32 boxes at a time; pages under
//              8 keys are gathered row by row with cp.async instead.  Warp 8 also
//              claims the CTA's items and publishes them to every warp;
//   warp 9     loads the q blocks (one 3-D box per 64-dim slab, rows
//              token-major; at head_dim 64 into two buffers, the next item's
//              while this one runs), and issues S = Q K^T (M = 128, N = 128) for tile n into
//              one of two 128-column score buffers in TMEM;
//   warp 10    O_g += P_g V_g (K = 64 keys, N = head_dim) for each group g:
//              its half of the tile's keys into its own accumulator, P read
//              from the group's half of the score buffer;
//   warps 0-7  two groups of four warps, one query row per thread: group g
//              takes keys 64 g ... 64 g + 63 of every tile: mask keys at or
//              past the row's bound, online softmax (base 2, running max
//              raised only past 2^8), P written over those scores;
//   warps 11-14 epilogue: combine the two groups' (m, l, O) by log-sum-exp,
//              normalise and write the item while the groups run the next.
// Per-request values sit in shared memory (when they fit), so moving from one
// item to the next costs no global loads.  Items whose block is cut into
// several key chunks write fp32 (o, lse) partials that ext_merge_kernel
// combines.  Every wait is bounded (~2 s).
#include <algorithm>

#include "pkv_internal.cuh"
#include "tc05.cuh"

namespace pkv {
namespace ext {

constexpr int kRows = 128, kTile = 128;   // query rows per block, keys per tile
constexpr int kChunkUnit = 64;             // a caller's kv_chunk is a multiple of this
constexpr int kThreads = 512;              // warps 0-7 softmax (two groups), 8 K producer, 9 q.k, 10 P.V,
                                           // 11-14 epilogue, 15 V producer
constexpr int kProducerWarp = 8, kQkWarp = 9, kPvWarp = 10, kEpiWarp0 = 11, kVProducerWarp = 15;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kLazy = 8.f;
constexpr int kRing = 8;                   // slots of the item queue
constexpr int kItemReaders = 16;           // warps that read every queued item

template <int D>
struct Cfg {
    // Shared memory at head_dim 128 (192 KB of 227): one q block (the next item's
    // is requested when this one's last Q K^T has completed), a 2-stage K ring and
    // a 3-stage V ring.  V is consumed a softmax later than K, so its deeper ring
    // lets its copies run further ahead; this split timed 1-3 % faster than two q
    // blocks with two stages each.
    static constexpr int kQBufs = D == 128 ? 1 : 2;            // q blocks: this item's (and the next)
    static constexpr int kKStages = D == 128 ? 2 : 4;          // depth of the K ring
    static constexpr int kVStages = D == 128 ? 3 : 4;          // depth of the V ring
    static constexpr int kSl = D / 64;                         // 64-dim slabs
    static constexpr int kQBytes = kSl * kRows * 128;          // one q block, SW128 K-major
    static constexpr int kKBytes = kSl * kTile * 128;          // one K (or V) tile
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQBufs * kQBytes;    // K ring, then V ring
    static constexpr int kOffBar = kOffKV + (kKStages + kVStages) * kKBytes;
    static constexpr int kNumBars = 56;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;    // tmem slot, abort flag, scan scratch
    static constexpr int kOffStats = kOffMisc + 128;           // [2 items][2 groups][128 rows] of (m, l) for the epilogue
    static constexpr int kOffRing = kOffStats + 4 * kRows * 8; // the CTA's next items, as the producer claims them
    static constexpr int kOffTable = kOffRing + kRing * 64;
    static constexpr int kFixedSmem = kOffTable + 1024;        // + request tables + alignment slack
    static constexpr uint32_t kColS = 0;                       // two 128-column score buffers (a 64-column half per group), P over S
    static constexpr uint32_t kColO = 2 * kTile;               // the two groups' D-column accumulators
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kColO + 2 * D <= kTmemCols, "tensor memory");
};

struct Params {
    int32_t layout, batch, hq, hkv, g, g_shift, T;
    int32_t ps_shift, ps_mask, box_rows, bt_width, chunk, max_len;
    float scale_log2;
    int64_t num_pages, kv_indices_len, total_q;
    const int32_t *qo_indptr, *kv_end, *kv_indptr, *kv_indices, *kv_last, *block_table, *seq_lens;
    uint16_t *out;
    float *lse, *part_o, *part_lse;
    int32_t *err;
    uint64_t wait_ns;          // bound of every mbarrier wait (pkv_set_wait_limit)
    int32_t cache_requests;   // per-request values kept in shared memory (they fit)
    int32_t *counter;         // items handed out past the first wave (zeroed before the launch)
    int32_t *goff, *ioff;     // [B + 1] first (kv head, query block) group / first item of each request,
                              // written by CTA 0 for the merge kernel
    const uint16_t *k_pool, *v_pool;   // pages under 8 keys: rows gathered with cp.async
    int64_t k_stride, v_stride;        // elements between pool rows
    // PKV_LAYOUT_REQ_TO_TOKEN: the token table itself
    const int32_t *r2t, *req_pool_idx, *kv_start;
    int64_t r2t_rows, r2t_stride, r2t_width;
};

// Keys of request b (0 and a flag for malformed inputs).
__device__ __forceinline__ int key_count(const Params &p, int b, int64_t &base, bool report) {
    int64_t L, cap;
    if (p.layout == PKV_LAYOUT_CSR) {
        const int64_t lo = p.kv_indptr[b], hi = p.kv_indptr[b + 1], n = hi - lo;
        const int last = n > 0 ? p.kv_last[b] : 0;
        base = lo;
        if (lo < 0 || n < 0 || hi > p.kv_indices_len || (n > 0 && (last < 1 || last > (1 << p.ps_shift)))) {
            if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
            base = 0;
            return 0;
        }
        L = n > 0 ? ((n - 1) << p.ps_shift) + last : 0;
        cap = L;
    } else if (p.layout == PKV_LAYOUT_REQ_TO_TOKEN) {
        // the request's keys are columns s .. s + L - 1 of its row ("From slots to a page table")
        const int64_t row = p.req_pool_idx[b], st = p.kv_start ? p.kv_start[b] : 0;
        L = p.seq_lens[b];
        if (row < 0 || row >= p.r2t_rows || st < 0 || (st & p.ps_mask) || L < 0 || st + L > p.r2t_width) {
            if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
            base = 0;
            return 0;
        }
        base = row * p.r2t_stride + st;
        cap = L;
    } else {
        base = static_cast<int64_t>(b) * p.bt_width;
        L = p.seq_lens[b];
        cap = static_cast<int64_t>(p.bt_width) << p.ps_shift;
    }
    const int64_t limit = min(cap, static_cast<int64_t>(p.max_len));
    if (L < 0 || L > limit) {
        if (report) raise_flag(p.err, L < 0 ? PKV_DEVERR_RANGE : PKV_DEVERR_CAPACITY);
        L = L < 0 ? 0 : limit;
    }
    return static_cast<int>(L);
}

// Query rows of request b (0 for a malformed qo_indptr).
__device__ __forceinline__ int q_count(const Params &p, int b, bool report) {
    const int64_t lo = p.qo_indptr[b], hi = p.qo_indptr[b + 1];
    if (lo < 0 || hi < lo || hi > p.total_q) {
        if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
        return 0;
    }
    return static_cast<int>(hi - lo);
}

// Key bound of query block qblk: the causal bound of its last token, or all keys
// when the caller gives its own bounds (the rows then mask the rest).
__device__ __forceinline__ int block_keys(const Params &p, int L, int n, int qblk) {
    if (p.kv_end) return L;
    const int last = min(n, (qblk + 1) * p.T);
    return max(0, L - n + last);
}

__device__ __forceinline__ int chunks_of(const Params &p, int kmax) { return max(1, (kmax + p.chunk - 1) / p.chunk); }

// Items of request b: hkv x sum over its query blocks of their key chunks.
__device__ __forceinline__ int per_head_items(const Params &p, int L, int n) {
    const int nq = (n + p.T - 1) / p.T;
    int s = 0;
    for (int q = 0; q < nq; ++q) s += chunks_of(p, block_keys(p, L, n, q));
    return s;
}

// Shared-memory tables of one launch: off[b] = first item of request b (B + 1
// entries) and, when they fit, each request's key count, query rows, first
// query row and page-list base, so that finding an item costs no global loads.
struct Tables {
    int *off, *keys, *nq, *qo0, *base;   // keys..base null when not cached
};

struct Req {
    int L, n, qo0;
    int64_t base;
};

// Request b from the inputs (flags raised only with `report`); causal rows need their keys.
__device__ __forceinline__ Req load_req(const Params &p, int b, bool report) {
    Req r;
    r.L = key_count(p, b, r.base, report);
    r.n = q_count(p, b, report);
    if (!p.kv_end && r.n > r.L) {
        if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
        r.n = 0;
    }
    r.qo0 = r.n > 0 ? p.qo_indptr[b] : 0;
    return r;
}

__device__ __forceinline__ Req get_req(const Params &p, const Tables &t, int b) {
    if (!t.keys) return load_req(p, b, false);
    Req r;
    r.L = t.keys[b];
    r.n = t.nq[b];
    r.qo0 = t.qo0[b];
    // cached for the CSR and token-table layouts (the host caches only when it fits an int)
    r.base = p.layout == PKV_LAYOUT_BLOCK_TABLE ? static_cast<int64_t>(b) * p.bt_width : static_cast<int64_t>(t.base[b]);
    return r;
}

struct Item {
    int64_t base, w;
    int b, kh, qblk, c, L, n, qo0, nch, k0, k1, n_tiles;
};

__device__ __forceinline__ Item locate(const Params &p, const Tables &t, int64_t w) {
    Item it;
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (t.off[mid] <= w) lo = mid; else hi = mid;
    }
    it.b = lo;
    it.w = w;
    const Req r = get_req(p, t, lo);
    it.L = r.L;
    it.n = r.n;
    it.qo0 = r.qo0;
    it.base = r.base;
    const int nq = (it.n + p.T - 1) / p.T;
    const bool one = p.chunk >= it.L;   // every query block is a single chunk
    const int per = one ? nq : per_head_items(p, it.L, it.n);
    int rem = static_cast<int>(w - t.off[it.b]);
    it.kh = rem / per;
    rem -= it.kh * per;
    // a request's query blocks in decreasing order (causal blocks shrink towards the first
    // token), so the items handed out last are the smallest and the CTAs finish together
    int q = 0;   // place of the block in that order
    if (one) {
        q = rem;
        rem = 0;
    } else {
        for (;; ++q) {
            const int c = chunks_of(p, block_keys(p, it.L, it.n, nq - 1 - q));
            if (rem < c) break;
            rem -= c;
        }
    }
    it.qblk = nq - 1 - q;
    it.c = rem;
    const int kmax = block_keys(p, it.L, it.n, it.qblk);
    it.nch = chunks_of(p, kmax);
    // the block's nch pieces are made equal (a multiple of 64 keys, at most p.chunk)
    const int span = ((kmax + it.nch - 1) / it.nch + kTile - 1) / kTile * kTile;
    it.k0 = it.c * span;
    it.k1 = min(kmax, it.k0 + span);
    it.n_tiles = it.k1 > it.k0 ? (it.k1 - it.k0 + kTile - 1) / kTile : 0;
    return it;
}

// Every CTA builds the same tables (CTA 0 reports malformed inputs).
__device__ __forceinline__ void build_tables(const Params &p, const Tables &t, int *scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.batch;
    const int seg = (B + kThreads - 1) / kThreads;
    const int lo = min(B, tid * seg), hi = min(B, lo + seg);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
        const Req r = load_req(p, b, blockIdx.x == 0);
        local += p.hkv * per_head_items(p, r.L, r.n);
        if (t.keys) {
            t.keys[b] = r.L;
            t.nq[b] = r.n;
            t.qo0[b] = r.qo0;
            t.base[b] = static_cast<int>(r.base);
        }
    }
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += scratch[w];
    int run = wbase + incl - local;
    for (int b = lo; b < hi; ++b) {
        t.off[b] = run;
        const Req r = t.keys ? get_req(p, t, b) : load_req(p, b, false);
        run += p.hkv * per_head_items(p, r.L, r.n);
    }
    if (tid == kThreads - 1) t.off[B] = wbase + incl;
    __syncthreads();
    if (blockIdx.x == 0) {   // the merge kernel's tables: items and groups per request, as prefixes
        int gl = 0;
        for (int b = lo; b < hi; ++b) {
            const Req r = t.keys ? get_req(p, t, b) : load_req(p, b, false);
            gl += p.hkv * ((r.n + p.T - 1) / p.T);
        }
        int gi = gl;
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, gi, o);
            if (lane >= o) gi += x;
        }
        if (lane == 31) scratch[warp] = gi;
        __syncthreads();
        int gbase = 0;
        for (int w = 0; w < warp; ++w) gbase += scratch[w];
        int grun = gbase + gi - gl;
        for (int b = lo; b < hi; ++b) {
            p.goff[b] = grun;
            p.ioff[b] = t.off[b];
            const Req r = t.keys ? get_req(p, t, b) : load_req(p, b, false);
            grun += p.hkv * ((r.n + p.T - 1) / p.T);
        }
        if (tid == kThreads - 1) {
            p.goff[B] = gbase + gi;
            p.ioff[B] = t.off[B];
        }
        __syncthreads();
    }
}

// Bounded wait with the CTA-wide abort flag: gives up once another warp gave up or
// `limit_ns` have passed (checked after the second poll and every 64 polls).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *err,
                                         uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 1) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                raise_flag(err, PKV_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool warp_wait(bool ok, uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err, uint64_t limit_ns) {
    return __all_sync(0xffffffffu, ok && wait_bar(bar, parity, abort_flag, err, limit_ns));
}
// Bounded wait that ignores the abort flag: drains work this CTA started.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return;
        if ((i & 63) == 63 && global_ns() - t0 > 2000000000ull) return;
    }
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes in one 64-bit register, and the paired FMA / add on them (one
// instruction for two values on this architecture).
__device__ __forceinline__ uint64_t pair(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float2 unpair(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Three-input maximum (one instruction on this architecture).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

enum Bar {
    kQFull0 = 0, kQEmpty0 = 2, kKFull0 = 4, kKEmpty0 = kKFull0 + 4, kVFull0 = kKEmpty0 + 4, kVEmpty0 = kVFull0 + 4,
    kSFull0 = kVEmpty0 + 4, kSFree0 = kSFull0 + 2, kPFull0 = kSFree0 + 2, kODone0 = kPFull0 + 4, kOFree0 = kODone0 + 2,
    kStatFull0 = kOFree0 + 2, kItemFull0 = kStatFull0 + 2, kItemEmpty0 = kItemFull0 + kRing,
    kFinalQk = kItemEmpty0 + kRing, kFinalPv, kBarCount
};

// Keys 64 g ... 64 g + 63 of every 128-key tile go to softmax group g, by their place
// in the item, so an item's result does not depend on which CTA runs it.  Tile n of
// the CTA's sequence uses score buffer n mod 2 (its use n / 2), and group g hands
// its P over to P V through barrier kPFull0 + 2 g + n mod 2: a group runs at most
// two tiles ahead of P V (it needs the score buffer), so a barrier never completes
// a second phase before its waiter has seen the first.

// Item k of this CTA's sequence from the queue (w < 0: no more items, or an
// abort).  Every reader warp takes every item once, in order, and frees its slot.
__device__ __forceinline__ Item ring_read(const Item *ring, uint64_t *bars, uint32_t k, bool &ok,
                                          volatile int *abort_flag, int32_t *err, uint64_t limit_ns) {
    ok = warp_wait(ok, &bars[kItemFull0 + k % kRing], (k / kRing) & 1, abort_flag, err, limit_ns);
    Item it;
    if (ok) {
        it = ring[k % kRing];
    } else {
        it.w = -1;
        it.n_tiles = 0;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bars[kItemEmpty0 + k % kRing]);
    return it;
}

// Sixteen warps: four of them on one SM sub-partition share its 16K registers, so
// at most 128 registers a thread.
template <int D>
__global__ void __maxnreg__(128)
ext_kernel(const Params p, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
           const __grid_constant__ CUtensorMap tmv) {
    using C = Cfg<D>;
    constexpr int kKStages = C::kKStages, kVStages = C::kVStages, kQBufs = C::kQBufs;
    static_assert(kBarCount <= C::kNumBars && kKStages <= 4 && kVStages <= 4 && kQBufs <= 2, "barrier slots");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem + C::kOffQ;
    unsigned char *sKV = smem + C::kOffKV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    int *scan = reinterpret_cast<int *>(smem + C::kOffMisc + 16);
    float2 *stats = reinterpret_cast<float2 *>(smem + C::kOffStats);
    Tables tb;
    tb.off = reinterpret_cast<int *>(smem + C::kOffTable);
    if (p.cache_requests) {
        tb.keys = tb.off + p.batch + 1;
        tb.nq = tb.keys + p.batch;
        tb.qo0 = tb.nq + p.batch;
        tb.base = tb.qo0 + p.batch;
    } else {
        tb.keys = tb.nq = tb.qo0 = tb.base = nullptr;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kQFull0 + i], 1);
            mbar_init(&bars[kQEmpty0 + i], 1);
            mbar_init(&bars[kODone0 + i], 1);
            mbar_init(&bars[kOFree0 + i], 4);
            mbar_init(&bars[kStatFull0 + i], 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kSFull0 + i], 1);   // score buffer i: q.k done
            mbar_init(&bars[kSFree0 + i], 1);   // score buffer i: both groups' P V that read P over it done
        }
        for (int i = 0; i < 4; ++i) mbar_init(&bars[kPFull0 + i], 4);   // group i / 2's four warps stored P in buffer i % 2
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars[kKFull0 + s], 1);
            mbar_init(&bars[kKEmpty0 + s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars[kVFull0 + s], 1);
            mbar_init(&bars[kVEmpty0 + s], 1);
        }
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&bars[kItemFull0 + s], 1);
            mbar_init(&bars[kItemEmpty0 + s], kItemReaders);
        }
        mbar_init(&bars[kFinalQk], 1);
        mbar_init(&bars[kFinalPv], 1);
        mbar_init_fence();
    }
    if (warp == kQkWarp) {
        tc05::tmem_alloc(tslot, C::kTmemCols);
        tc05::tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    pdl_wait();          // lengths, bounds, q and the pools may come from the previous kernel
    pdl_launch_next();
    build_tables(p, tb, scan);
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tbase = *tslot;
    const int64_t total = tb.off[p.batch];
    Item *ring = reinterpret_cast<Item *>(smem + C::kOffRing);

    if (warp == kProducerWarp || warp == kVProducerWarp) {
        // ------------------------------------------------------------ producers: K (warp 8), V (warp 15)
        // A box is `box` keys of one page; a tile is `nbox` boxes.  Each warp fills
        // its own ring, in tile order: K runs ahead as soon as a Q K^T has freed a
        // stage, while V waits for P V.  The pool rows of an item's boxes are looked
        // up 32 at a time, one window ahead (lane j holds box 32 win + j), so no
        // page-table load sits between two tile issues.  The TMA unit's time per box
        // bounds this loop, so nothing is prefetched into L2.
        const bool is_v = warp == kVProducerWarp;
        const int box = p.box_rows;
        const int nbox = kTile / box;
        const int32_t *tab = p.layout == PKV_LAYOUT_CSR ? p.kv_indices : p.block_table;
        // one copy per lane: lane = (box j, slab), at most 32 per tile
        const int nops = nbox * C::kSl;
        const int j_box = (lane / C::kSl) & (nbox - 1), sl_op = lane % C::kSl;
        uint64_t *fulls = &bars[is_v ? kVFull0 : kKFull0], *empties = &bars[is_v ? kVEmpty0 : kKEmpty0];
        unsigned char *ring_base = sKV + (is_v ? kKStages * C::kKBytes : 0);
        const uint32_t stages = is_v ? kVStages : kKStages;   // depth of this warp's ring
        const uint16_t *pool = is_v ? p.v_pool : p.k_pool;
        const int64_t pool_stride = is_v ? p.v_stride : p.k_stride;
        uint32_t n = 0, kpub = 0, issued = 0;   // tiles; tiles whose copies were issued
        bool ok = true;
        // Pages under 8 keys: the warp gathers a tile's rows itself with 16-byte
        // cp.async copies (one commit group per tile), written in the same swizzled
        // layout the TMA boxes produce.  A tile's full barrier is arrived once its
        // group has completed and the warp has fenced its writes for the tensor
        // cores' async proxy; up to two tiles stay in flight (`pend`).
        const bool gather = box < 8;
        uint32_t pend = 0, n_arr = 0;   // tiles in flight; the oldest of them
        auto settle_one = [&]() {
            if (pend >= 3) cp_async_wait<2>();
            else if (pend == 2) cp_async_wait<1>();
            else cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&fulls[n_arr % stages]);
            ++n_arr;
            --pend;
        };
        auto settle_all = [&]() { while (pend > 0) settle_one(); };
        // The queue (warp 8): the CTA's first item is blockIdx.x; later ones are
        // claimed from a global counter (dynamic balance), two items ahead of the one
        // being issued, decoded here and published to every reader warp.  A negative
        // w ends it.
        auto publish = [&](int64_t w) {
            settle_all();   // the readers of the queue may be waiting for these tiles
            const uint32_t slot = kpub % kRing;
            ok = warp_wait(ok, &bars[kItemEmpty0 + slot], ((kpub / kRing) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
            Item qi;
            if (w >= 0 && w < total) {
                qi = locate(p, tb, w);
            } else {
                qi.w = -1;
                qi.n_tiles = 0;
            }
            if (lane == 0 && ok) {
                ring[slot] = qi;
                mbar_arrive(&bars[kItemFull0 + slot]);
            }
            __syncwarp();
            ++kpub;
        };
        bool more = false;
        if (!is_v) {
            more = blockIdx.x < total;
            publish(more ? static_cast<int64_t>(blockIdx.x) : -1);
            if (more) {
                int got = 0;
                if (lane == 0) got = atomicAdd(p.counter, 1);
                const int64_t w1 = static_cast<int64_t>(gridDim.x) + __shfl_sync(0xffffffffu, got, 0);
                more = w1 < total;
                publish(more ? w1 : -1);
            }
        }
        for (uint32_t k = 0; ok; ++k) {
            if (is_v) settle_all();   // this warp may wait below for an item not yet published
            const Item it = ring_read(ring, bars, k, ok, abort_flag, p.err, p.wait_ns);
            if (it.w < 0) break;
            int got = 0;   // the claim's latency hides behind this item's tiles
            if (more && lane == 0) got = atomicAdd(p.counter, 1);
            if (it.n_tiles > 0) {
                // pool row of box bx: -1 past the item's keys, -2 for a page outside the pool
                // pool row of key k of the item: -2 for a page outside the pool, -3 for a
                // token-table page start that is not a multiple of the page size
                auto pool_row = [&](int k) -> int {
                    if (p.layout == PKV_LAYOUT_REQ_TO_TOKEN) {   // the slot of the page's first key, + the offset
                        const int first = __ldg(p.r2t + it.base + (k & ~p.ps_mask));
                        if (first < 0 || first >= (p.num_pages << p.ps_shift)) return -2;
                        if (first & p.ps_mask) return -3;
                        return first + (k & p.ps_mask);
                    }
                    const int page = __ldg(tab + it.base + (k >> p.ps_shift));
                    if (page < 0 || page >= p.num_pages) return -2;
                    return static_cast<int>((static_cast<int64_t>(page) << p.ps_shift) + (k & p.ps_mask));
                };
                // pool row of box bx: -1 past the item's keys
                auto box_row = [&](int bx) -> int {
                    const int kb = it.k0 + bx * box;
                    return kb >= it.k1 ? -1 : pool_row(kb);
                };
                if (gather) {
                    constexpr int kRowsPerLane = kTile / 32;
                    for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                        const int kt0 = it.k0 + ti * kTile;
                        // pool row of key j of the tile: -1 past the item's keys
                        auto key_row = [&](int j) -> int {
                            const int kk = kt0 + j;
                            return kk >= it.k1 ? -1 : pool_row(kk);
                        };
                        int rr[kRowsPerLane];
                        bool bad_range = false, bad_start = false;
#pragma unroll
                        for (int q = 0; q < kRowsPerLane; ++q) {
                            rr[q] = key_row(lane + 32 * q);
                            bad_range |= rr[q] == -2;
                            bad_start |= rr[q] == -3;
                        }
                        if (bad_range && !is_v) raise_flag(p.err, PKV_DEVERR_RANGE);
                        if (bad_start && !is_v) raise_flag(p.err, PKV_DEVERR_CONTIG);
                        const int s = static_cast<int>(n % stages);
                        // the stage frees once the Q K^T / P V of tile n - stages ran, which
                        // waits for that tile's full barrier: settle it first
                        while (pend > stages - 1) settle_one();
                        if (lane == 0) ok = wait_bar(&empties[s], ((n / stages) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                        if (!ok) break;
                        constexpr int CPR = D / 8;       // 16-byte chunks per row
                        constexpr int KPI = 32 / CPR;    // rows per warp instruction
                        const int c = lane % CPR, sl = c >> 3, cc = c & 7;
                        unsigned char *st = ring_base + s * C::kKBytes;
#pragma unroll 4
                        for (int j0 = 0; j0 < kTile; j0 += KPI) {
                            const int j = j0 + lane / CPR;
                            int row = -1;
#pragma unroll
                            for (int q = 0; q < kRowsPerLane; ++q) {
                                const int a = __shfl_sync(0xffffffffu, rr[q], j & 31);
                                if ((j >> 5) == q) row = a;
                            }
                            const bool live = row >= 0;
                            const int off = sl * kTile * 128 + j * 128 + ((cc ^ (j & 7)) << 4);
                            const int64_t col = static_cast<int64_t>(it.kh) * D + c * 8;
                            cp_async_16(st + off, live ? pool + row * pool_stride + col : pool, live ? 16 : 0);
                        }
                        cp_async_commit();
                        ++issued;
                        ++pend;
                        if (pend > 2) settle_one();
                    }
                } else {
                    int win = 0;
                    int cur = box_row(lane), nxt = box_row(32 + lane);
                    for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                        if (((ti * nbox) >> 5) != win) {
                            ++win;
                            cur = nxt;
                            nxt = box_row(32 * (win + 1) + lane);
                        }
                        // pool row of this lane's box (a tile's boxes share one window: win or win + 1)
                        const int bx0 = ti * nbox;
                        int row = __shfl_sync(0xffffffffu, (bx0 >> 5) == win ? cur : nxt, (bx0 & 31) + j_box);
                        if (lane >= nops) row = -1;
                        if (row <= -2 && sl_op == 0 && !is_v) raise_flag(p.err, row == -2 ? PKV_DEVERR_RANGE : PKV_DEVERR_CONTIG);
                        const int s = static_cast<int>(n % stages);
                        const uint32_t valid = __ballot_sync(0xffffffffu, row >= 0);
                        unsigned char *dst = ring_base + s * C::kKBytes + sl_op * kTile * 128 + j_box * box * 128;
                        if (lane == 0) ok = wait_bar(&empties[s], ((n / stages) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                        if (!ok) break;
                        if (row <= -2) {   // a bad page reads as zeros
                            for (int o = 0; o < box * 128; o += 16) *reinterpret_cast<uint4 *>(dst + o) = make_uint4(0, 0, 0, 0);
                            fence_proxy_async_smem();   // for the tensor cores and later TMA writes
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive_expect_tx(&fulls[s], __popc(valid) * static_cast<uint32_t>(box) * 128u);
                        __syncwarp();
                        if (row >= 0) tma_load_2d(dst, is_v ? &tmv : &tmk, it.kh * D + sl_op * 64, row, &fulls[s]);
                        ++issued;
                    }
                }
            }
            if (more) {
                const int64_t w2 = static_cast<int64_t>(gridDim.x) + __shfl_sync(0xffffffffu, got, 0);
                more = w2 < total;
                publish(more ? w2 : -1);
            }
        }
        settle_all();
        if (lane == 0)   // drain: the copies this warp issued have landed
            for (uint32_t k = issued > stages ? issued - stages : 0; k < issued; ++k)
                drain_wait(&fulls[k % stages], (k / stages) & 1);
        __syncwarp();
    } else if (warp == kQkWarp) {
        // ------------------------------------------------------------ S = Q K^T
        // This warp also loads the q blocks.  With two buffers, item i + 1's block is
        // requested once item i's first tile is issued (its buffer was freed by the
        // completion of item i - 1's last q.k), so q never waits at an item boundary;
        // with one, it is requested once item i's last q.k has completed.
        const uint32_t idesc = tc05::idesc_bf16_f32(kRows, kTile, false, false);
        uint32_t n = 0, iq = 0, q_issued = 0;
        bool ok = true;
        auto load_q = [&](const Item &qi, uint32_t slot_use) {   // slot_use: how many q loads came before
            const int sl = slot_use % kQBufs;
            ok = warp_wait(ok, &bars[kQEmpty0 + sl], ((slot_use / kQBufs) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
            if (ok && lane == 0) {
                mbar_arrive_expect_tx(&bars[kQFull0 + sl], C::kQBytes);
                const int tok = qi.qo0 + qi.qblk * p.T;
                for (int k = 0; k < C::kSl; ++k)
                    tma_load_3d(sQ + sl * C::kQBytes + k * kRows * 128, &tmq, k * 64, qi.kh * p.g, tok,
                                &bars[kQFull0 + sl]);
            }
            __syncwarp();
            if (ok) ++q_issued;
        };
        uint32_t kr = 0;
        Item it = ring_read(ring, bars, kr++, ok, abort_flag, p.err, p.wait_ns);
        bool q_req = false;   // it's q block already requested
        while (it.w >= 0 && ok) {
            const Item nx = ring_read(ring, bars, kr++, ok, abort_flag, p.err, p.wait_ns);   // may be the end
            bool nx_req = false;
            if (it.n_tiles > 0) {
                if (!q_req) load_q(it, iq);
                const int sl = iq % kQBufs;
                ok = warp_wait(ok, &bars[kQFull0 + sl], (iq / kQBufs) & 1, abort_flag, p.err, p.wait_ns);
                for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                    // score buffer n mod 2 is free once both groups' P V of tile n - 2 are done
                    const int s = n % kKStages, b = n & 1;
                    ok = warp_wait(ok, &bars[kKFull0 + s], (n / kKStages) & 1, abort_flag, p.err, p.wait_ns);
                    ok = warp_wait(ok, &bars[kSFree0 + b], ((n >> 1) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                    if (!ok) break;
                    tc05::fence_after_sync();
                    if (lane == 0) {
                        const uint64_t kd = tc05::smem_desc(sKV + s * C::kKBytes, 16, 1024);
                        const uint64_t qd = tc05::smem_desc(sQ + sl * C::kQBytes, 16, 1024);
    #pragma unroll
                        for (int k2 = 0; k2 < C::kSl; ++k2)
    #pragma unroll
                            for (int k = 0; k < 4; ++k)   // slab: q +16 KB, K +16 KB; k-step +32 bytes
                                tc05::mma_ss(tbase + C::kColS + b * kTile,
                                             qd + static_cast<uint64_t>((k2 * kRows * 128 + k * 32) >> 4),
                                             kd + static_cast<uint64_t>((k2 * kTile * 128 + k * 32) >> 4), idesc,
                                             (k2 | k) ? 1u : 0u);
                        tc05::commit(&bars[kSFull0 + b]);
                        tc05::commit(&bars[kKEmpty0 + s]);
                        if (ti == it.n_tiles - 1) tc05::commit(&bars[kQEmpty0 + sl]);
                    }
                    __syncwarp();
                    if (ti == (kQBufs == 2 ? 0 : it.n_tiles - 1) && nx.w >= 0 && nx.n_tiles > 0) {
                        load_q(nx, iq + 1);
                        nx_req = true;
                    }
                }
                ++iq;
            }
            it = nx;
            q_req = nx_req;
        }
        if (lane == 0) {
            // q loads issued but not waited for have landed before shared memory is released
            for (uint32_t k = iq; k < q_issued; ++k) drain_wait(&bars[kQFull0 + k % kQBufs], (k / kQBufs) & 1);
            tc05::commit(&bars[kFinalQk]);
            drain_wait(&bars[kFinalQk], 0);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ O_g += P_g V_g
        // Group g's half of tile n (keys 64 g ... 64 g + 63) into its accumulator.  An
        // item's first tile starts both accumulators afresh, once the epilogue has read
        // the previous item's.
        const uint32_t idesc = tc05::idesc_bf16_f32(kRows, D, false, true);
        uint32_t n = 0, io = 0;
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            const Item it = ring_read(ring, bars, k, ok, abort_flag, p.err, p.wait_ns);
            if (it.w < 0) break;
            if (it.n_tiles == 0) continue;
            for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                const int s = n % kVStages, b = n & 1;
                ok = warp_wait(ok, &bars[kVFull0 + s], (n / kVStages) & 1, abort_flag, p.err, p.wait_ns);
                if (!ok) break;
                unsigned char *v = sKV + (kKStages + s) * C::kKBytes;
                const int n_valid = it.k1 - (it.k0 + ti * kTile);
                if (n_valid < kTile) {   // key rows past the chunk hold stale data: zero them
                    for (int i = lane; i < (kTile - n_valid) * C::kSl * 8; i += 32) {
                        const int key = n_valid + i / (C::kSl * 8);
                        const int sl = (i / 8) % C::kSl, c = i % 8;
                        *reinterpret_cast<uint4 *>(v + sl * kTile * 128 + key * 128 + (c << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (ti == 0 && io > 0)
                    ok = warp_wait(ok, &bars[kOFree0 + ((io - 1) & 1)], ((io - 1) >> 1) & 1, abort_flag, p.err, p.wait_ns);
                for (int g = 0; g < 2 && ok; ++g) {
                    ok = warp_wait(ok, &bars[kPFull0 + 2 * g + b], (n >> 1) & 1, abort_flag, p.err, p.wait_ns);
                    if (!ok) break;
                    tc05::fence_after_sync();
                    if (lane == 0) {
                        const uint64_t vd = tc05::smem_desc(v + g * 64 * 128, kTile * 128, 1024);
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // 16 keys: +2048 bytes of V, +8 columns of P
                            tc05::mma_ts(tbase + C::kColO + g * D, tbase + C::kColS + b * kTile + g * 64 + k * 8,
                                         vd + static_cast<uint64_t>((k * 2048) >> 4), idesc,
                                         (ti == 0 && k == 0) ? 0u : 1u);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) {
                    tc05::commit(&bars[kSFree0 + b]);
                    tc05::commit(&bars[kVEmpty0 + s]);
                    if (ti == it.n_tiles - 1) tc05::commit(&bars[kODone0 + (io & 1)]);
                }
                __syncwarp();
            }
            ++io;
        }
        if (lane == 0) {
            tc05::commit(&bars[kFinalPv]);
            drain_wait(&bars[kFinalPv], 0);
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------------ epilogue (one row per thread)
        // Once an item's last P V is done and both groups have left the row's (m, l),
        // combines the groups: o = (2^(mA - M) OA + 2^(mB - M) OB) / (2^(mA - M) lA +
        // 2^(mB - M) lB) with M = max(mA, mB), writes the bf16 row (or the fp32 split
        // partial) and frees the accumulators, while the groups already run the next
        // item.  A group without keys in the item (l = 0) is left out: its
        // accumulator was not written for this item.
        const int quarter = warp & 3;                 // TMEM lanes this warp may read
        const int r = quarter * 32 + lane;
        const uint32_t trow = tc05::taddr(tbase, quarter * 32, 0);
        const int tok = r >> p.g_shift, hh = r & (p.g - 1);
        uint32_t io = 0;
        bool ok = true;
        for (uint32_t k = 0;; ++k) {
            const Item it = ring_read(ring, bars, k, ok, abort_flag, p.err, p.wait_ns);
            if (it.w < 0) break;
            if (it.n_tiles == 0) continue;
            const int ko = io & 1;
            ok = warp_wait(ok, &bars[kStatFull0 + ko], (io >> 1) & 1, abort_flag, p.err, p.wait_ns);
            const float2 sa = stats[(ko * 2) * kRows + r], sb2 = stats[(ko * 2 + 1) * kRows + r];
            ok = warp_wait(ok, &bars[kODone0 + ko], (io >> 1) & 1, abort_flag, p.err, p.wait_ns);
            tc05::fence_after_sync();
            const float M = fmaxf(sa.x, sb2.x);
            const float wa = sa.y > 0.f ? ex2(sa.x - M) : 0.f, wb = sb2.y > 0.f ? ex2(sb2.x - M) : 0.f;
            const float den = sa.y * wa + sb2.y * wb;
            const float inv = den > 0.f ? 1.f / den : 0.f;
            const float ca = wa * inv, cb2 = wb * inv;
            const int tq = it.qblk * p.T + tok;
            const bool valid = tq < it.n;
            const int64_t qrow = static_cast<int64_t>(it.qo0) + tq;
            const int head = it.kh * p.g + hh;
            const bool single = it.nch == 1;
            const int64_t prow = it.w * kRows + r;
#pragma unroll 1
            for (int cb = 0; cb < D / 16; cb += 2) {
                float oa[2][16], ob[2][16];
                if (ok) {
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        tc05::ld_x16(trow + C::kColO + (cb + q2) * 16, oa[q2]);
                        tc05::ld_x16(trow + C::kColO + D + (cb + q2) * 16, ob[q2]);
                    }
                    tc05::wait_ld();
                }
                if (valid) {
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        float ov[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            // selects, not products: an accumulator left out may hold anything
                            const float xa = ok && wa != 0.f ? oa[q2][e] * ca : 0.f;
                            const float xb = ok && wb != 0.f ? ob[q2][e] * cb2 : 0.f;
                            ov[e] = xa + xb;
                        }
                        const int col = (cb + q2) * 16;
                        if (single) {
                            uint32_t h2[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) h2[e] = pack_bf16x2(ov[2 * e], ov[2 * e + 1]);
                            uint4 *o = reinterpret_cast<uint4 *>(p.out + (qrow * p.hq + head) * D + col);
                            o[0] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
                            o[1] = make_uint4(h2[4], h2[5], h2[6], h2[7]);
                        } else {
                            float4 *o = reinterpret_cast<float4 *>(p.part_o + prow * D + col);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[e] = make_float4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
                        }
                    }
                }
            }
            if (valid) {
                const float lse2 = den > 0.f ? M + log2f(den) : -INFINITY;
                if (single) {
                    if (p.lse) p.lse[qrow * p.hq + head] = lse2 * kLn2;
                } else {
                    p.part_lse[prow] = lse2;
                }
            }
            tc05::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kOFree0 + ko]);
            ++io;
        }
    } else {
        // ------------------------------------------------------------ softmax (one row per thread)
        // Group grp = warp / 4 takes keys 64 grp ... 64 grp + 63 of every tile, keeping
        // its own (m, l) and accumulator; warp w reads TMEM lanes 32 (w mod 4) ...
        const int grp = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tc05::taddr(tbase, quarter * 32, 0);
        const int tok = r >> p.g_shift, hh = r & (p.g - 1);
        uint32_t io = 0, n = 0;   // items and tiles so far
        bool ok = true;
        // the row's key bound; its load for the next item is issued an item early
        auto row_bound = [&](const Item &qi) -> int {
            const int tq = qi.qblk * p.T + tok;
            if (tq >= qi.n) return 0;
            int kend = p.kv_end ? __ldg(p.kv_end + static_cast<int64_t>(qi.qo0) + tq) : qi.L - qi.n + tq + 1;
            if (kend < 0 || kend > qi.L) {
                if (qi.c == 0 && qi.kh == 0) raise_flag(p.err, PKV_DEVERR_RANGE);
                kend = 0;
            }
            return kend;
        };
        uint32_t kr = 0;
        Item it = ring_read(ring, bars, kr++, ok, abort_flag, p.err, p.wait_ns);
        int kend = it.w >= 0 ? row_bound(it) : 0;
        while (it.w >= 0) {
            const Item nx = ring_read(ring, bars, kr++, ok, abort_flag, p.err, p.wait_ns);   // may be the end
            const int kend_nx = nx.w >= 0 ? row_bound(nx) : 0;
            const int tq = it.qblk * p.T + tok;                  // token within the request
            const bool valid = tq < it.n;
            const int64_t qrow = static_cast<int64_t>(it.qo0) + tq;
            const int head = it.kh * p.g + hh;
            float m = -INFINITY, l = 0.f;
            if (it.n_tiles == 0) {   // no keys: out = 0, lse = -inf
                if (grp == 0 && valid && it.nch == 1) {
                    uint4 *o = reinterpret_cast<uint4 *>(p.out + (qrow * p.hq + head) * D);
                    for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
                    if (p.lse) p.lse[qrow * p.hq + head] = -INFINITY;
                }
                it = nx;
                kend = kend_nx;
                continue;
            }
            const int ko = io & 1;
            for (int ti = 0; ti < it.n_tiles; ++ti, ++n) {
                const int b = n & 1;
                const int key0 = it.k0 + ti * kTile + grp * 64;   // this group's half of the tile
                // rows past the block's tokens are never written: they only mask the
                // keys past the chunk (stale data), which keeps full halves select-free
                const int vis = max(0, min(min(valid ? kend : it.k1, it.k1) - key0, 64));
                const uint32_t sc = trow + C::kColS + b * kTile + grp * 64;
                ok = warp_wait(ok, &bars[kSFull0 + b], (n >> 1) & 1, abort_flag, p.err, p.wait_ns);
                float x[64];
                if (ok) {
                    tc05::fence_after_sync();
                    tc05::ld_x64(sc, x);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) x[j] = 0.f;
                }
                // keys at or past the row's bound read as -inf (no selects when the
                // whole half is inside every row's bound); max over a tree
                if (!__all_sync(0xffffffffu, vis == 64)) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) x[j] = j < vis ? x[j] : -INFINITY;
                }
                float mx;
                {   // a tree of three-input maxima: 64 -> 22 -> 8 -> 3 -> 1
                    float t[22];
#pragma unroll
                    for (int j = 0; j < 21; ++j) t[j] = fmax3(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
                    t[21] = x[63];
                    float u[8];
#pragma unroll
                    for (int j = 0; j < 7; ++j) u[j] = fmax3(t[3 * j], t[3 * j + 1], t[3 * j + 2]);
                    u[7] = t[21];
                    mx = fmax3(fmax3(u[0], u[1], u[2]), fmax3(u[3], u[4], u[5]), fmaxf(u[6], u[7])) *
                         p.scale_log2;   // scores are unscaled up to here (the scale is positive)
                }
                const bool raise = mx > m + kLazy || (m == -INFINITY && mx != -INFINITY);
                const float corr = raise ? ex2(m - mx) : 1.f;
                if (__any_sync(0xffffffffu, raise && m != -INFINITY) && ok) {
                    // the group's accumulator is final for tile n - 1 (of this item: m is
                    // finite) once that tile's P V completed; rescale the row
                    const uint32_t np = n - 1;
                    ok = warp_wait(ok, &bars[kSFree0 + (np & 1)], (np >> 1) & 1, abort_flag, p.err, p.wait_ns);
                    tc05::fence_after_sync();
#pragma unroll 1
                    for (int cc = 0; cc < D / 16 && ok; ++cc) {
                        float ov[16];
                        tc05::ld_x16(trow + C::kColO + grp * D + cc * 16, ov);
                        tc05::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) ov[e] *= corr;
                        tc05::st_x16(trow + C::kColO + grp * D + cc * 16, ov);
                    }
                    tc05::wait_st();
                }
                if (raise) {
                    l *= corr;
                    m = mx;
                }
                uint32_t h0[16], h1[16];
                // a row with no keys yet (m = -inf) has only -inf scores: offset 0 gives p = 0
                const float nm = m == -INFINITY ? 0.f : -m;
                // scaling and the row sum two keys per instruction (the softmax groups
                // are bound by instruction issue)
                const uint64_t sc2 = pair(p.scale_log2, p.scale_log2), nm2 = pair(nm, nm);
                uint64_t acc = pair(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 16; ++j) {   // p = 2^(scale log2(e) s - m)
                    const float2 ya = unpair(fma2(pair(x[2 * j], x[2 * j + 1]), sc2, nm2));
                    const float2 yb = unpair(fma2(pair(x[32 + 2 * j], x[32 + 2 * j + 1]), sc2, nm2));
                    const float a0 = ex2(ya.x), a1 = ex2(ya.y), b0 = ex2(yb.x), b1 = ex2(yb.y);
                    acc = add2(acc, pair(a0, a1));
                    acc = add2(acc, pair(b0, b1));
                    h0[j] = pack_bf16x2(a0, a1);
                    h1[j] = pack_bf16x2(b0, b1);
                }
                const float2 ls = unpair(acc);
                l += ls.x + ls.y;
                if (ok) {   // P (bf16 pairs) over the first 32 columns of the scores just read
                    tc05::st_x16_u32(sc, h0);
                    tc05::st_x16_u32(sc + 16, h1);
                    tc05::wait_st();
                }
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kPFull0 + 2 * grp + b]);
            }
            // hand (m, l) to the epilogue warps; the buffer is free once they are done
            // with the item two back
            ok = warp_wait(ok, &bars[kOFree0 + ko], ((io >> 1) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
            stats[(ko * 2 + grp) * kRows + r] = make_float2(m, l);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kStatFull0 + ko]);
            ++io;
            it = nx;
            kend = kend_nx;
        }
    }

    tc05::fence_before_sync();
    __syncthreads();
    if (warp == kQkWarp) {
        tc05::fence_after_sync();
        tc05::tmem_dealloc(tbase, C::kTmemCols);
    }
}

// Log-sum-exp merge of the key chunks of one (request, kv head, query block):
// one CTA per such group (found in the prefix tables the attention kernel left),
// rows x head_dim.
template <int D>
__global__ void __launch_bounds__(256) ext_merge_kernel(const Params p, int64_t groups) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    const int64_t gi = blockIdx.x;
    if (gi >= groups) return;
    // the group's request by binary search over the prefix tables, then its first item
    if (gi >= p.goff[p.batch]) return;
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.goff[mid] <= gi) lo = mid; else hi = mid;
    }
    const int b = lo;
    const Req rq = load_req(p, b, false);
    const int L = rq.L, n = rq.n;
    const int nq = (n + p.T - 1) / p.T;
    const int rem = static_cast<int>(gi - p.goff[b]);
    const int kh = rem / nq, qblk = rem % nq;
    const int nch = chunks_of(p, block_keys(p, L, n, qblk));
    if (nch <= 1) return;
    int64_t w0 = p.ioff[b] + static_cast<int64_t>(kh) * per_head_items(p, L, n);
    for (int q = qblk + 1; q < nq; ++q) w0 += chunks_of(p, block_keys(p, L, n, q));   // blocks before it in item order
    for (int i = threadIdx.x; i < kRows * (D / 4); i += blockDim.x) {
        const int r = i / (D / 4), d4 = i % (D / 4);
        const int tok = r >> p.g_shift, hh = r & (p.g - 1);
        const int tb = qblk * p.T + tok;
        if (tb >= n) continue;
        float M = -INFINITY;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, p.part_lse[(w0 + c) * kRows + r]);
        float den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int c = 0; c < nch; ++c) {
                const float lc = p.part_lse[(w0 + c) * kRows + r];
                if (lc == -INFINITY) continue;
                const float wgt = ex2(lc - M);
                const float4 x = reinterpret_cast<const float4 *>(p.part_o + ((w0 + c) * kRows + r) * D)[d4];
                acc.x = fmaf(wgt, x.x, acc.x);
                acc.y = fmaf(wgt, x.y, acc.y);
                acc.z = fmaf(wgt, x.z, acc.z);
                acc.w = fmaf(wgt, x.w, acc.w);
                den += wgt;
            }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const int64_t qrow = static_cast<int64_t>(rq.qo0) + tb;
        const int head = kh * p.g + hh;
        uint2 o;
        o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        reinterpret_cast<uint2 *>(p.out + (qrow * p.hq + head) * D)[d4] = o;
        if (d4 == 0 && p.lse) p.lse[qrow * p.hq + head] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
}

// ------------------------------------------------------------------ span planner
// One CTA per request: its segments' positions and key bounds, rows counted from
// the sum of the segment lengths of the requests before it.
__global__ void __launch_bounds__(256)
span_plan_kernel(int32_t batch, const int32_t *__restrict__ seg_indptr, const int32_t *__restrict__ seg_kind,
                 const int32_t *__restrict__ seg_start, const int32_t *__restrict__ seg_end, int32_t *__restrict__ qo,
                 int32_t *__restrict__ q_pos, int32_t *__restrict__ kv_end, int64_t cap, int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    __shared__ long long scratch[32];
    const int b = blockIdx.x;
    auto seg_len = [&](int s) -> long long {
        const int64_t a = seg_start[s], e = seg_end[s];
        return (a < 0 || e < a || (seg_kind[s] != 0 && seg_kind[s] != 1)) ? 0 : e - a;
    };
    long long before = 0;
    for (int s = threadIdx.x; s < seg_indptr[b]; s += blockDim.x) before += seg_len(s);
    before = block_sum(before, scratch);
    long long mine = 0;
    for (int s = seg_indptr[b] + threadIdx.x; s < seg_indptr[b + 1]; s += blockDim.x) mine += seg_len(s);
    mine = block_sum(mine, scratch);
    if (threadIdx.x == 0) {
        if (b == 0) qo[0] = 0;
        qo[b + 1] = static_cast<int32_t>(before + mine);
        if (before + mine > cap) raise_flag(err, PKV_DEVERR_CAPACITY);
    }
    long long j = before;
    for (int s = seg_indptr[b]; s < seg_indptr[b + 1]; ++s) {   // segments in order, positions in parallel
        const int64_t a = seg_start[s], e = seg_end[s];
        if (a < 0 || e < a || (seg_kind[s] != 0 && seg_kind[s] != 1)) {
            if (threadIdx.x == 0) raise_flag(err, PKV_DEVERR_RANGE);
            continue;
        }
        for (int64_t t = threadIdx.x; t < e - a; t += blockDim.x) {
            if (j + t >= cap) break;
            q_pos[j + t] = static_cast<int32_t>(a + t);
            kv_end[j + t] = static_cast<int32_t>(seg_kind[s] == 0 ? a + t + 1 : e);
        }
        j += e - a;
    }
}

// ------------------------------------------------------------------ host side
struct Plan {
    int g, T, chunk, nch_max;
    int64_t items_max, groups_max;
    size_t part_o_bytes, part_lse_bytes;
    static constexpr size_t kCounterBytes = 256;   // the item counter, after the partials
    size_t table_bytes;                            // then the merge kernel's two prefix tables
};

static bool make_plan(const pkv_extend_args *a, Plan &pl) {
    pl.g = a->num_q_heads / a->num_kv_heads;
    pl.T = kRows / pl.g;
    const int64_t blocks_max = a->total_q / pl.T + a->batch;      // query blocks, upper bound
    pl.groups_max = static_cast<int64_t>(a->num_kv_heads) * blocks_max;
    const int64_t L = std::max(1, a->max_seq_len);
    if (a->kv_chunk > 0) {
        // whole tiles: a block's pieces are then never empty ((pieces - 1) x piece < keys)
        pl.chunk = (a->kv_chunk + kTile - 1) / kTile * kTile;
    } else {   // split the keys only when the query blocks alone leave SMs idle
        // (an SM count of 0, when no device answers, plans as for one SM)
        const int64_t target = 2 * std::max<int64_t>(1, sm_count());
        const int64_t groups = std::max<int64_t>(1, static_cast<int64_t>(a->num_kv_heads) *
                                                        std::max<int64_t>(a->batch, a->total_q / pl.T));
        const int64_t want = std::max<int64_t>(1, (target + groups - 1) / groups);
        int64_t c = (L + want - 1) / want;
        c = std::max<int64_t>(512, (c + kTile - 1) / kTile * kTile);
        // long rows of uneven length: cap an item at 4096 keys so no single item
        // outlasts the others' share
        if (L > 8192) c = std::min<int64_t>(c, 4096);
        pl.chunk = static_cast<int>(std::min<int64_t>(c, (L + kTile - 1) / kTile * kTile));
    }
    pl.nch_max = static_cast<int>((L + pl.chunk - 1) / pl.chunk);
    pl.items_max = pl.groups_max * pl.nch_max;
    if (pl.items_max > INT32_MAX / kRows) return false;
    if (pl.nch_max <= 1) {
        pl.part_o_bytes = pl.part_lse_bytes = 0;
    } else {
        const int64_t rows = pl.items_max * kRows;
        pl.part_o_bytes = (static_cast<size_t>(rows) * a->head_dim * 4 + 255) / 256 * 256;
        pl.part_lse_bytes = (static_cast<size_t>(rows) * 4 + 255) / 256 * 256;
    }
    pl.table_bytes = (2 * (static_cast<size_t>(a->batch) + 1) * 4 + 255) / 256 * 256;
    return true;
}

static pkv_status validate(const pkv_extend_args *a, bool check_ptrs) {
    if (a->batch < 0 || a->num_q_heads < 1 || a->num_kv_heads < 1 || a->total_q < 0 || a->max_seq_len < 0 ||
        a->num_slots < 0)
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: negative or zero size");
    if (a->num_q_heads % a->num_kv_heads) return fail(PKV_ERR_INVALID_ARG, "pkv_extend: Hq not a multiple of Hkv");
    const int g = a->num_q_heads / a->num_kv_heads;
    if (!is_pow2(g) || g > 16) return fail(PKV_ERR_UNSUPPORTED, "pkv_extend: Hq/Hkv must be 1, 2, 4, 8 or 16");
    if (a->head_dim != 64 && a->head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "pkv_extend: head_dim 64 or 128");
    if (!is_pow2(a->page_size) || a->page_size > 1024)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_extend: page_size must be a power of two in [1, 1024]");
    if (a->layout != PKV_LAYOUT_CSR && a->layout != PKV_LAYOUT_BLOCK_TABLE && a->layout != PKV_LAYOUT_REQ_TO_TOKEN)
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: layout must be CSR, BLOCK_TABLE or REQ_TO_TOKEN");
    if (a->layout == PKV_LAYOUT_REQ_TO_TOKEN &&
        (a->r2t_rows < 0 || a->r2t_width < 0 || a->r2t_row_stride < a->r2t_width || a->r2t_width > INT32_MAX))
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: bad req_to_token shape");
    if (a->kv_chunk < 0 || a->kv_chunk % kChunkUnit) return fail(PKV_ERR_INVALID_ARG, "pkv_extend: kv_chunk multiple of 64");
    const int64_t rowq = static_cast<int64_t>(a->num_kv_heads) * a->head_dim;
    if (a->k_row_stride < rowq || a->v_row_stride < rowq || a->k_row_stride % 8 || a->v_row_stride % 8)
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: pool row strides must hold Hkv x head_dim and be 16-byte aligned");
    if (a->num_slots > INT32_MAX || a->total_q > INT32_MAX)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_extend: more than 2^31 pool rows or query rows");
    if (a->batch == 0 || !check_ptrs) return PKV_OK;
    if (!a->q || !a->k_pool || !a->v_pool || !a->out || !a->qo_indptr)
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: null q/k_pool/v_pool/out/qo_indptr");
    if (!aligned(a->q, 16) || !aligned(a->k_pool, 16) || !aligned(a->v_pool, 16) || !aligned(a->out, 16))
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: q, pools and out must be 16-byte aligned");
    if (a->layout == PKV_LAYOUT_CSR && (!a->kv_indptr || !a->kv_indices || !a->kv_last_page_len))
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: CSR layout needs kv_indptr/kv_indices/kv_last_page_len");
    if (a->layout == PKV_LAYOUT_BLOCK_TABLE && (!a->block_table || !a->seq_lens || a->block_table_width < 0))
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: block-table layout needs block_table and seq_lens");
    if (a->layout == PKV_LAYOUT_REQ_TO_TOKEN && (!a->req_to_token || !a->req_pool_idx || !a->seq_lens))
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: token-table layout needs req_to_token, req_pool_idx, seq_lens");
    return PKV_OK;
}

template <int D>
static pkv_status launch_t(const pkv_extend_args *a, const Plan &pl, void *ws, int32_t *err, cudaStream_t s) {
    using C = Cfg<D>;
    Params p{};
    p.layout = a->layout;
    p.batch = a->batch;
    p.hq = a->num_q_heads;
    p.hkv = a->num_kv_heads;
    p.g = pl.g;
    p.g_shift = ilog2(pl.g);
    p.T = pl.T;
    p.ps_shift = ilog2(a->page_size);
    p.ps_mask = a->page_size - 1;
    p.box_rows = std::min(a->page_size, kTile);
    p.bt_width = a->block_table_width;
    p.chunk = pl.chunk;
    p.max_len = a->max_seq_len;
    p.scale_log2 = a->sm_scale * kLog2e;
    p.num_pages = a->num_slots >> p.ps_shift;
    p.kv_indices_len = a->kv_indices_len;
    p.total_q = a->total_q;
    p.qo_indptr = a->qo_indptr;
    p.kv_end = a->kv_end;
    p.kv_indptr = a->kv_indptr;
    p.kv_indices = a->kv_indices;
    p.kv_last = a->kv_last_page_len;
    p.block_table = a->block_table;
    p.seq_lens = a->seq_lens;
    p.out = static_cast<uint16_t *>(a->out);
    p.lse = a->lse;
    p.part_o = static_cast<float *>(ws);
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(ws) + pl.part_o_bytes);
    p.counter = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + pl.part_o_bytes + pl.part_lse_bytes);
    p.goff = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + pl.part_o_bytes + pl.part_lse_bytes +
                                         Plan::kCounterBytes);
    p.ioff = p.goff + a->batch + 1;
    p.err = err;
    p.wait_ns = wait_limit_ns();
    p.k_pool = static_cast<const uint16_t *>(a->k_pool);
    p.v_pool = static_cast<const uint16_t *>(a->v_pool);
    p.k_stride = a->k_row_stride;
    p.v_stride = a->v_row_stride;
    p.r2t = a->req_to_token;
    p.req_pool_idx = a->req_pool_idx;
    p.kv_start = a->kv_start;
    p.r2t_rows = a->r2t_rows;
    p.r2t_stride = a->r2t_row_stride;
    p.r2t_width = a->r2t_width;

    CUtensorMap tmq, tmk, tmv;
    {   // q [total_q, Hq, D]: boxes of 64 dims x g heads x T tokens = 128 rows of 128 bytes
        const uint64_t dq[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a->num_q_heads),
                                static_cast<uint64_t>(std::max<int64_t>(a->total_q, 1))};
        const uint64_t sq[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a->num_q_heads) * D * 2};
        const uint32_t bq[3] = {64, static_cast<uint32_t>(pl.g), static_cast<uint32_t>(pl.T)};
        if (!encode_tmap_bf16(&tmq, a->q, 3, dq, sq, bq))
            return fail(PKV_ERR_CUDA, "pkv_extend: cuTensorMapEncodeTiled rejected q");
        // pool rows as a 2-D tensor (kv heads x head_dim wide): a box is 64 dims of one
        // kv head over a page's rows
        const uint64_t dk[2] = {static_cast<uint64_t>(a->num_kv_heads) * D, static_cast<uint64_t>(a->num_slots)};
        const uint64_t sk[1] = {static_cast<uint64_t>(a->k_row_stride) * 2};
        const uint64_t sv[1] = {static_cast<uint64_t>(a->v_row_stride) * 2};
        const uint32_t bk[2] = {64, static_cast<uint32_t>(p.box_rows)};
        if (!encode_tmap_bf16(&tmk, a->k_pool, 2, dk, sk, bk) || !encode_tmap_bf16(&tmv, a->v_pool, 2, dk, sv, bk))
            return fail(PKV_ERR_CUDA, "pkv_extend: cuTensorMapEncodeTiled rejected the pools");
    }
    std::atomic<int64_t> *m_lim = device_memo(reinterpret_cast<const void *>(ext_kernel<D>));
    if (!m_lim) return fail(PKV_ERR_CUDA, "pkv_extend: cannot query the current device");
    if (m_lim->load() == 0) {   // kernel attributes are per device
        int optin = 0, dev = 0;
        cudaFuncAttributes fa{};
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, ext_kernel<D>) != cudaSuccess)
            return fail(PKV_ERR_CUDA, "pkv_extend: cannot query shared-memory limits");
        const size_t l = static_cast<size_t>(optin) - fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(ext_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(l)) !=
            cudaSuccess)
            return fail(PKV_ERR_CUDA, "pkv_extend: cannot raise the shared-memory limit");
        m_lim->store(static_cast<int64_t>(l));
    }
    const size_t lim = static_cast<size_t>(m_lim->load());
    // item table (B + 1 ints), plus four ints per request when they fit as well
    size_t smem = C::kFixedSmem + (static_cast<size_t>(a->batch) + 1) * 4;
    if (smem > lim) return fail(PKV_ERR_UNSUPPORTED, "pkv_extend: batch too large for the on-chip item table");
    const size_t cached = smem + static_cast<size_t>(a->batch) * 16;
    // a token-table base (row x stride + start) is cached as an int only when every one fits
    const bool bases_fit = a->layout != PKV_LAYOUT_REQ_TO_TOKEN || a->r2t_rows * a->r2t_row_stride <= INT32_MAX;
    p.cache_requests = cached <= lim && bases_fit ? 1 : 0;
    if (p.cache_requests) smem = cached;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(pl.items_max, sm_count()));
    if (cudaMemsetAsync(p.counter, 0, sizeof(int32_t), s) != cudaSuccess)
        return fail(PKV_ERR_CUDA, "pkv_extend: cannot reset the item counter");
    ext_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p, tmq, tmk, tmv);
    pkv_status st = check_launch("pkv_extend (attention kernel)");
    if (st != PKV_OK || pl.nch_max <= 1) return st;
    return launch_status(launch_chained(ext_merge_kernel<D>, dim3(static_cast<unsigned>(pl.groups_max)), dim3(256), 0, s,
                                        p, pl.groups_max),
                         "pkv_extend (merge kernel)");
}

}  // namespace ext
}  // namespace pkv

extern "C" size_t pkv_extend_workspace_size(const pkv_extend_args *args) {
    using namespace pkv::ext;
    if (!args || validate(args, false) != PKV_OK) return 0;
    Plan pl;
    if (!make_plan(args, pl)) return 0;
    return pl.part_o_bytes + pl.part_lse_bytes + Plan::kCounterBytes + pl.table_bytes;
}

extern "C" pkv_status pkv_extend(const pkv_extend_args *args, void *workspace, size_t workspace_bytes,
                                 int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    using namespace pkv::ext;
    if (!args) return fail(PKV_ERR_INVALID_ARG, "pkv_extend: null args");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_extend: err_flags is required");
    pkv_status st = validate(args, true);
    if (st != PKV_OK) return st;
    if (args->batch == 0 || args->total_q == 0) return ok();
    Plan pl;
    if (!make_plan(args, pl)) return fail(PKV_ERR_UNSUPPORTED, "pkv_extend: too many work items");
    const size_t need = pl.part_o_bytes + pl.part_lse_bytes + Plan::kCounterBytes + pl.table_bytes;
    if (workspace_bytes < need)
        return fail(PKV_ERR_CAPACITY, "pkv_extend: workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (!workspace || !aligned(workspace, 256))
        return fail(PKV_ERR_INVALID_ARG, "pkv_extend: workspace must be non-null and 256-byte aligned");
    auto s = reinterpret_cast<cudaStream_t>(stream);
    return args->head_dim == 128 ? launch_t<128>(args, pl, workspace, err_flags, s)
                                 : launch_t<64>(args, pl, workspace, err_flags, s);
}

extern "C" pkv_status pkv_span_plan(int32_t batch, const int32_t *seg_indptr, const int32_t *seg_kind,
                                    const int32_t *seg_start, const int32_t *seg_end, int32_t *qo_indptr,
                                    int32_t *q_pos, int32_t *kv_end, int64_t cap, int32_t *err_flags,
                                    pkv_stream_t stream) {
    using namespace pkv;
    if (batch < 0 || cap < 0) return fail(PKV_ERR_INVALID_ARG, "pkv_span_plan: negative size");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_span_plan: err_flags is required");
    if (batch == 0) return ok();
    if (!seg_indptr || !seg_kind || !seg_start || !seg_end || !qo_indptr || (cap > 0 && (!q_pos || !kv_end)))
        return fail(PKV_ERR_INVALID_ARG, "pkv_span_plan: null input");
    return launch_status(launch_chained(ext::span_plan_kernel, dim3(batch), dim3(256), 0,
                                        reinterpret_cast<cudaStream_t>(stream), batch, seg_indptr, seg_kind, seg_start,
                                        seg_end, qo_indptr, q_pos, kv_end, cap, err_flags),
                         "pkv_span_plan");
}
