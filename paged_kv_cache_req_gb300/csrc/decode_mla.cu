// pkv_decode for MLA: 128 query heads per item attending over one latent KV
// head through a page table, on the 5th-generation tensor cores.
//
// Each latent row holds kv_lora_rank + rope dims (512 + 64); keys are the whole
// row, values its first 512 entries (AttentionBackend notes: FlashMLA metadata
// with num_kv_heads 1, kv_lora_rank and qk_rope_head_dim; block table padded
// with -1, page_size 64).  For a decode token the work per key is
// 128 x (576 + 512) x 2 flops on 1152 bytes, close to the HBM/tensor ridge.
//
// Work is spread as equal spans of the concatenated key-tile sequence, one
// span per CTA pair (see next_seg); a request cut by a span boundary is merged
// from its split partials by a second kernel.
//
// The fp32 output accumulator of 128 heads x 512 dims fills all of an SM's
// tensor memory, so a 2-CTA cluster shares each segment (request, 128-head
// group, run of 64-key tiles): CTA r owns value dims [256 r, 256 r + 256) and
// rope dims [512 + 32 r, 512 + 32 r + 32).  It computes the partial scores over
// those 288 dims and accumulates its 256 output dims.  The two partial score
// tiles (128 heads x 64 keys) are swapped as fp16 through distributed shared
// memory one tile ahead, so both CTAs hold bitwise-identical full scores and run
// the same softmax; nothing is loaded or multiplied twice.
//
// Per CTA: warps 0-15 softmax (four threads per head row, 16 keys each), warp 16
// producer (TMA boxes per page and 64-dim slab into 4 stages of 36 KB, with tiles
// three ahead prefetched into L2; for pages under 8 keys a second instance of the
// kernel gathers rows with cp.async), warp 17 issues S = Q K^T, warp 18 O += P V.
// Tensor memory holds two 64-column score buffers, O (256 columns), q over the
// CTA's first 128 dims (64 columns, the A operand of eight of the 18 q.k MMAs)
// and two 32-column P buffers (the A operand of P V); q over the other 160 dims
// comes from shared memory.  The online softmax works in base 2 with the running
// max raised only past 2^8 headroom, so O rescales in TMEM are rare; the softmax
// warps also normalise O and write the output or the split partials.
// Every wait is bounded (~2 s) and an abort flag lets the CTA drain instead of
// hanging.
#include <algorithm>
#include <cmath>
#include <mutex>

#include <cuda_fp16.h>

#include "pkv_internal.cuh"
#include "tc05.cuh"

namespace pkv {
namespace mla {

constexpr int kDqk = 576, kDv = 512, kHeads = 128, kTile = 64;
constexpr int kVSlabs = 4;                 // 256 value dims per CTA: four 64-dim slabs
constexpr int kStages = 4;
constexpr int kSoftmaxWarps = 16;          // four threads per head row: keys 16 qt .. 16 qt + 15 in warps 4 qt .. 4 qt + 3
constexpr int kThreads = 608;              // warps 0-15 softmax, 16 producer, 17 q.k MMAs, 18 P.V MMAs
constexpr int kProducerWarp = 16, kMmaWarp = 17, kPvWarp = 18;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;              // two 64-column score tiles
constexpr uint32_t kColO = 128;            // 256-column output accumulator
constexpr uint32_t kColQ = 384;            // q over this CTA's first 128 dims, the MMA A operand (64 columns)
constexpr uint32_t kColP = 448;            // P (bf16 probabilities), A operand of P V: two buffers of 32 columns
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kLazy = 8.f;

// shared-memory carve-up (bytes from a 1024-aligned base)
constexpr int kSlabBytes = kTile * 128;                     // 8 KB: 64 keys x 64 dims, 128-byte swizzle
constexpr int kRopeBytes = kTile * 64;                      // 4 KB: 64 keys x 32 rope dims, 64-byte swizzle
constexpr int kStageBytes = kVSlabs * kSlabBytes + kRopeBytes;   // 36 KB
constexpr int kOffKV = 0;
constexpr int kXBytes = kHeads * kTile * 2;                // one tile of peer partial scores, fp16
constexpr int kXSlots = 2;
constexpr int kOffX = kOffKV + kStages * kStageBytes;       // kXSlots slots, each [8 chunks][128 heads] x 16 B
constexpr int kOffQ = kOffX + kXSlots * kXBytes;            // q over the CTA's dims 128-255: two SW128 slabs
constexpr int kOffQr = kOffQ + 2 * kHeads * 128;            // q over the CTA's 32 rope dims, 64-byte swizzle
constexpr int kOffBar = kOffQr + kHeads * 64;
constexpr int kNumBars = 24;
constexpr int kOffMisc = kOffBar + kNumBars * 8;            // tmem slot, abort flag, scan scratch (one int per warp)
constexpr int kOffRed = kOffMisc + 128;                     // row-max / row-sum exchange of a row's four threads
constexpr int kOffTable = kOffRed + 2 * 4 * kHeads * 4;
constexpr int kFixedSmem = kOffTable + 1024;                // + item table + alignment slack

struct Params {
    int32_t layout;
    int32_t batch, hq, hgroups;
    int32_t ps_shift, ps_mask;
    float scale_log2;
    int32_t span_tiles;    // tiles per span of the concatenated tile sequence; 0: total / pairs, rounded up
    int32_t max_len;       // keys a request may have (the caller's max_seq_len)
    int32_t bt_width;
    int32_t box_rows;
    int64_t num_slots, num_pages, kv_indices_len;
    const int32_t *kv_indptr, *kv_indices, *kv_last, *block_table, *seq_lens, *cu_seqlens;
    const uint16_t *q;
    uint16_t *out;
    float *lse;
    float *part_o, *part_lse;  // [span][2 slots][128 heads] x (512 | 1), base-2 lse
    int32_t *meta;             // [0]: tiles per span, [1 + v]: first tile of row v (rows + 1 entries)
    int32_t *err;
    uint64_t wait_ns;          // bound of every mbarrier wait (pkv_set_wait_limit)
    const uint16_t *pool;      // latent rows (read directly when pages are under 8 keys)
    int64_t pool_stride;       // elements between latent rows
};

// Marks the 16 floats as written here, so that no use of registers an asynchronous
// TMEM load fills is scheduled before the wait that follows that load.
__device__ __forceinline__ void reg_fence16(float (&v)[16]) {
    asm volatile(""
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                   "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]),
                   "+f"(v[15]));
}

// bit casts between a 32-bit word and a pair of fp16 values (by value, so arrays stay in registers)
__device__ __forceinline__ __half2 u2h2(uint32_t u) {
    __half2_raw r;
    r.x = static_cast<unsigned short>(u & 0xffffu);
    r.y = static_cast<unsigned short>(u >> 16);
    return __half2(r);
}
__device__ __forceinline__ uint32_t h22u(__half2 h) {
    const __half2_raw r = static_cast<__half2_raw>(h);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int key_count(const Params &p, int b, int64_t &base, bool report) {
    int64_t L, cap;
    if (p.layout == PKV_LAYOUT_CSR) {
        const int64_t lo = p.kv_indptr[b], hi = p.kv_indptr[b + 1];
        const int64_t n = hi - lo;
        const int last = n > 0 ? p.kv_last[b] : 0;
        base = lo;
        if (lo < 0 || n < 0 || hi > p.kv_indices_len || (n > 0 && (last < 1 || last > (1 << p.ps_shift)))) {
            if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
            base = 0;
            return 0;
        }
        L = n > 0 ? ((n - 1) << p.ps_shift) + last : 0;
        cap = L;
    } else if (p.layout == PKV_LAYOUT_BLOCK_TABLE) {
        base = static_cast<int64_t>(b) * p.bt_width;
        L = p.seq_lens[b];
        cap = static_cast<int64_t>(p.bt_width) << p.ps_shift;
    } else {
        base = p.cu_seqlens[b];
        L = static_cast<int64_t>(p.cu_seqlens[b + 1]) - base;
        cap = L;
    }
    const int64_t limit = min(cap, static_cast<int64_t>(p.max_len));
    if (L < 0 || L > limit) {
        if (report) raise_flag(p.err, L < 0 ? PKV_DEVERR_RANGE : PKV_DEVERR_CAPACITY);
        L = L < 0 ? 0 : limit;
    }
    return static_cast<int>(L);
}

// ---- work distribution ----
// A row is one (request, 128-head group): v = b * hgroups + hg, with
// ceil(L_b / 64) key tiles.  The rows' tiles, concatenated in row order, are cut
// into spans of equal length (the last may be shorter); CTA pair `pair` takes
// spans pair, pair + npairs, ...  So every pair gets the same number of tiles
// whatever the length mix, and crosses few row boundaries.  The piece of a row
// inside one span is a segment.  A segment holding its whole row writes the
// final output; otherwise it is a split whose (o, lse) partial goes to slot 0
// of its span (the segment opens the span) or slot 1 (it closes the span), and
// the merge kernel combines a row's splits.
struct Seg {
    int b, hg, L, key_begin, key_end, n_tiles;
    int part;  // -1: the whole row; else the partial's index, span * 2 + slot
    int64_t base;
};

struct Cursor {
    int s, t;  // current span, next tile (index into the concatenated sequence)
};

// A row with keys enters the concatenated sequence as kSegCost stand-in tiles (the
// cost of starting a segment: loading its q, the pipeline's refill, the epilogue)
// followed by its real tiles, so that spans of equal length also even out the
// segment starts a pair makes.  Stand-in tiles produce no work.
constexpr int kSegCost = 4;

__device__ __forceinline__ int row_tiles(const Params &p, int v, bool report) {
    int64_t base;
    const int L = key_count(p, v / p.hgroups, base, report);
    return L > 0 ? (L + kTile - 1) / kTile + kSegCost : 0;
}

// R[v] = first tile (stand-ins included) of row v, R[V] = total; every CTA builds
// the same table.
__device__ __forceinline__ void build_row_table(const Params &p, int V, int *R, int *scratch, bool report) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = (V + kThreads - 1) / kThreads;
    const int lo = min(V, tid * seg), hi = min(V, lo + seg);
    int local = 0;
    for (int v = lo; v < hi; ++v) local += row_tiles(p, v, report && v % p.hgroups == 0);
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
    for (int v = lo; v < hi; ++v) {
        R[v] = run;
        run += row_tiles(p, v, false);
    }
    if (tid == kThreads - 1) R[V] = wbase + incl;
    __syncthreads();
}

// The next segment of this pair's spans (false when there is none left).  A
// segment is the real tiles of one row inside one span; a span that holds only
// stand-in tiles of a row holds no segment of it.  A split segment's partial goes to
// slot 0 of its span when it is the span's first segment (its row began at or
// before the span's first tile), else to slot 1.
__device__ __forceinline__ bool next_seg(const Params &p, const int *R, int V, int per, int S, int npairs, Cursor &c,
                                         Seg &g) {
    const int T = R[V];
    while (c.s < S) {
        const int s_begin = c.s * per;
        const int s_end = min(T, s_begin + per);
        while (c.t < s_end) {
            int lo = 0, hi = V;  // R[lo] <= t < R[hi]: row lo holds tile t
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (R[mid] <= c.t) lo = mid; else hi = mid;
            }
            const int v = lo;
            const int real0 = R[v] + kSegCost;       // the row's first real tile
            const int t0 = max(c.t, real0);
            const int t1 = min(s_end, R[v + 1]);
            c.t = t1;
            if (t0 >= t1) continue;                  // only stand-in tiles of row v in this span
            g.b = v / p.hgroups;
            g.hg = v % p.hgroups;
            g.L = key_count(p, g.b, g.base, false);
            g.key_begin = (t0 - real0) * kTile;
            g.key_end = min(g.L, (t1 - real0) * kTile);
            g.n_tiles = t1 - t0;
            g.part = (t0 == real0 && t1 == R[v + 1]) ? -1 : c.s * 2 + (R[v] <= s_begin ? 0 : 1);
            return true;
        }
        c.s += npairs;
        c.t = c.s * per;
    }
    return false;
}

// Bounded wait (local or cluster-scope acquire) with the CTA-wide abort flag: gives
// up once another warp gave up or `limit_ns` have passed (checked after the second
// poll and every 64 polls).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *err,
                                         uint64_t limit_ns, bool cluster_scope = false) {
    auto poll = [&]() { return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll()) return true;
    if (*abort_flag) return false;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (poll()) return true;
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

// Warp-wide bounded wait (every lane polls; measured faster than one polling lane
// with the others parked).  `ok` is warp-uniform; so is the result.
__device__ __forceinline__ bool warp_wait(bool ok, uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err, uint64_t limit_ns, bool cluster_scope = false) {
    return __all_sync(0xffffffffu, ok && wait_bar(bar, parity, abort_flag, err, limit_ns, cluster_scope));
}

// Bounded wait that ignores the abort flag: used only to drain work this CTA
// itself started (MMAs, TMA copies) before its TMEM and shared memory go away.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return;
        if ((i & 63) == 63 && global_ns() - t0 > 2000000000ull) return;
    }
}

enum Bar {
    kQFull = 0, kQEmpty, kKvFull0, kKvEmpty0 = kKvFull0 + kStages, kSFull0 = kKvEmpty0 + kStages, kSFree0 = kSFull0 + 2,
    kPFull0 = kSFree0 + 2, kPFree0 = kPFull0 + 2, kXFull0 = kPFree0 + 2, kODone = kXFull0 + kXSlots, kOFree,
    kFinal, kFinalPv, kBarCount
};
static_assert(kBarCount <= kNumBars, "barrier slots");
static_assert(16 + 4 * (kThreads / 32) <= kOffRed - kOffMisc, "scan scratch");

template <bool kGather>   // pages under 8 keys: rows gathered with cp.async instead of TMA boxes
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_kernel(const Params p, const __grid_constant__ CUtensorMap tmkv, const __grid_constant__ CUtensorMap tmrope) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sKV = smem + kOffKV;
    float *sX = reinterpret_cast<float *>(smem + kOffX);
    unsigned char *sQ = smem + kOffQ;
    unsigned char *sQr = smem + kOffQr;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    int *scan = reinterpret_cast<int *>(smem + kOffMisc + 16);
    int *R = reinterpret_cast<int *>(smem + kOffTable);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int slab0 = 4 * static_cast<int>(rank);   // first 64-dim slab of the latent row owned by this CTA
    const int rope0 = 512 + 32 * static_cast<int>(rank);   // first of the CTA's 32 rope dims

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(&bars[kQFull], kSoftmaxWarps); // the softmax warps after writing q into TMEM
        mbar_init(&bars[kQEmpty], 1);            // MMA commit after an item's last q.k
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[kKvFull0 + s], 1);
            mbar_init(&bars[kKvEmpty0 + s], 1);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(&bars[kSFull0 + b2], 1);
            mbar_init(&bars[kSFree0 + b2], kSoftmaxWarps);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(&bars[kPFull0 + b2], kSoftmaxWarps);
            mbar_init(&bars[kPFree0 + b2], 1);
        }
        for (int x = 0; x < kXSlots; ++x) mbar_init(&bars[kXFull0 + x], 1);  // own expect_tx arrive + peer bytes
        mbar_init(&bars[kODone], 1);
        mbar_init(&bars[kOFree], kSoftmaxWarps);
        mbar_init(&bars[kFinal], 1);
        mbar_init(&bars[kFinalPv], 1);
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tc05::tmem_alloc(tslot, kTmemCols);
        tc05::tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tmkv);
        prefetch_tmap(&tmrope);
    }
    pdl_wait();          // lengths, tables, q and the pool may come from the previous kernel
    pdl_launch_next();
    const int V = p.batch * p.hgroups;
    build_row_table(p, V, R, scan, blockIdx.x == 0);   // contains __syncthreads
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    cluster_sync_all();                // the peer's barriers exist before any remote arrive
    const uint32_t tbase = *tslot;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int T = R[V];
    const int per = p.span_tiles > 0 ? p.span_tiles : max(1, (T + npairs - 1) / npairs);
    const int S = (T + per - 1) / per;
    if (blockIdx.x == 0) {             // the merge kernel reads the plan back
        for (int v = tid; v <= V; v += kThreads) p.meta[1 + v] = R[v];
        if (tid == 0) p.meta[0] = per;
    }

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer: K/V tiles
        // Lane j < 64 / box handles box j of a tile: one page lookup, then the CTA's
        // four 64-dim slabs and its 32 rope dims of those rows.  Tiles kPrefetch
        // ahead of the one being loaded are first pulled into L2, so a stage's own
        // loads (issued once the stage is free) wait on L2 rather than on HBM.
        const int box = p.box_rows;
        const int nbox = kTile / box;
        const uint32_t box_bytes = static_cast<uint32_t>(box) * 128u;
        constexpr int kPrefetch = 3;
        uint32_t n = 0;
        bool ok = true;
        Cursor cur{pair, pair * per};
        Seg it{};
        // pool row of this lane's box of tile ti (-1: past the end, -2: bad page id)
        auto box_row = [&](int ti, bool report) -> int {
            if (lane >= nbox) return -1;
            const int tb = it.key_begin + ti * kTile + lane * box;
            if (tb >= it.key_end) return -1;
            if (p.layout == PKV_LAYOUT_VARLEN) return static_cast<int>(it.base + tb);
            const int32_t *tab = p.layout == PKV_LAYOUT_CSR ? p.kv_indices : p.block_table;
            const int page = __ldg(tab + it.base + (tb >> p.ps_shift));
            if (page < 0 || page >= p.num_pages) {
                if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
                return -2;
            }
            return static_cast<int>((static_cast<int64_t>(page) << p.ps_shift) + (tb & p.ps_mask));
        };
        auto prefetch = [&](int ti) {
            const int r = box_row(ti, false);
            if (r >= 0) {
                tma_prefetch_2d(&tmrope, rope0, r);
                for (int sl = 0; sl < kVSlabs; ++sl) tma_prefetch_2d(&tmkv, (slab0 + sl) * 64, r);
            }
        };
        // Pages under 8 keys: the warp gathers each tile's rows with 16-byte cp.async
        // copies into the layout the TMA boxes would produce (128-byte swizzle for the
        // value slabs, 64-byte for the rope rows), one commit group per tile; a
        // tile's full barrier is arrived once its group completed and the writes are
        // fenced for the tensor cores' async proxy.  Up to two tiles stay in flight.
        // The next segment's q (this CTA's 288 dims of 128 heads: four 128-byte lines
        // and one rope line per head) into L2 while this segment's last tile loads, a
        // few tiles before the softmax warps read it.  (Earlier, the streaming K/V
        // would evict it again.)
        auto prefetch_next_q = [&]() {
            Cursor c2 = cur;
            Seg nx;
            if (!next_seg(p, R, V, per, S, npairs, c2, nx)) return;
            const char *qb = reinterpret_cast<const char *>(p.q + (static_cast<int64_t>(nx.b) * p.hq + nx.hg * kHeads) * kDqk);
            for (int i = lane; i < kHeads * 5; i += 32) {
                const int h = i / 5, k = i % 5;
                prefetch_l2(qb + h * (kDqk * 2) + (k < 4 ? slab0 * 128 + k * 128 : rope0 * 2));
            }
        };
        constexpr bool gather = kGather;
        uint32_t pend = 0, n_arr = 0;
        auto settle_one = [&]() {
            if (pend >= 3) cp_async_wait<2>();
            else if (pend == 2) cp_async_wait<1>();
            else cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kKvFull0 + n_arr % kStages]);
            ++n_arr;
            --pend;
        };
        while (ok && next_seg(p, R, V, per, S, npairs, cur, it)) {
            if constexpr (gather) {
                for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                    const int kt0 = it.key_begin + ti * kTile;
                    auto key_row = [&](int j) -> int {   // -1 past the segment, -2 outside the pool
                        const int kk = kt0 + j;
                        if (kk >= it.key_end) return -1;
                        if (p.layout == PKV_LAYOUT_VARLEN) return static_cast<int>(it.base + kk);
                        const int32_t *tab = p.layout == PKV_LAYOUT_CSR ? p.kv_indices : p.block_table;
                        const int page = __ldg(tab + it.base + (kk >> p.ps_shift));
                        if (page < 0 || page >= p.num_pages) return -2;
                        return static_cast<int>((static_cast<int64_t>(page) << p.ps_shift) + (kk & p.ps_mask));
                    };
                    const int r0 = key_row(lane), r1 = key_row(lane + 32);
                    if (r0 == -2 || r1 == -2) raise_flag(p.err, PKV_DEVERR_RANGE);
                    const int s = n % kStages;
                    if (lane == 0) ok = wait_bar(&bars[kKvEmpty0 + s], ((n / kStages) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    unsigned char *st = sKV + s * kStageBytes;
                    // value slabs: lane = 16-byte chunk (slab lane / 8, chunk lane % 8) of one key row
                    const int sl = lane >> 3, cc = lane & 7;
#pragma unroll 4
                    for (int j = 0; j < kTile; ++j) {
                        const int a0 = __shfl_sync(0xffffffffu, r0, j & 31), a1 = __shfl_sync(0xffffffffu, r1, j & 31);
                        const int row = j < 32 ? a0 : a1;
                        const bool live = row >= 0;
                        cp_async_16(st + sl * kSlabBytes + j * 128 + ((cc ^ (j & 7)) << 4),
                                    live ? p.pool + row * p.pool_stride + (slab0 + sl) * 64 + cc * 8 : p.pool,
                                    live ? 16 : 0);
                    }
                    // rope rows: 4 chunks of 64 bytes per key, 8 keys per instruction
#pragma unroll
                    for (int j0 = 0; j0 < kTile; j0 += 8) {
                        const int j = j0 + (lane >> 2), c = lane & 3;
                        const int a0 = __shfl_sync(0xffffffffu, r0, j & 31), a1 = __shfl_sync(0xffffffffu, r1, j & 31);
                        const int row = j < 32 ? a0 : a1;
                        const bool live = row >= 0;
                        cp_async_16(st + kVSlabs * kSlabBytes + j * 64 + ((c ^ ((j >> 1) & 3)) << 4),
                                    live ? p.pool + row * p.pool_stride + rope0 + c * 8 : p.pool, live ? 16 : 0);
                    }
                    cp_async_commit();
                    ++pend;
                    if (pend > 2) settle_one();
                    if (ti == it.n_tiles - 1) prefetch_next_q();
                }
                continue;
            }
            for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                // a segment's first tile is loaded before anything is prefetched (its
                // page lookups are the only loads ahead of it); later tiles prefetch the
                // tile kPrefetch ahead while they wait for a free stage
                if (ti > 0 && ti + kPrefetch < it.n_tiles) prefetch(ti + kPrefetch);
                const int row = box_row(ti, true);
                const int s = n % kStages;
                if (lane == 0) ok = wait_bar(&bars[kKvEmpty0 + s], ((n / kStages) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (row == -2) {   // a page outside the pool reads as zeros (the flag is raised by box_row)
                    unsigned char *st = sKV + s * kStageBytes;
                    for (int sl = 0; sl < kVSlabs; ++sl)
                        for (uint32_t o = 0; o < box_bytes; o += 16)
                            *reinterpret_cast<uint4 *>(st + sl * kSlabBytes + lane * box_bytes + o) = make_uint4(0, 0, 0, 0);
                    for (int o = 0; o < box * 64; o += 16)
                        *reinterpret_cast<uint4 *>(st + kVSlabs * kSlabBytes + lane * box * 64 + o) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_smem();   // for the tensor cores and later TMA writes
                }
                const uint32_t valid = __ballot_sync(0xffffffffu, row >= 0);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars[kKvFull0 + s], __popc(valid) * static_cast<uint32_t>(box) *
                                                                   static_cast<uint32_t>(kVSlabs * 128 + 64));
                __syncwarp();
                if (row >= 0) {
                    unsigned char *st = sKV + s * kStageBytes;
                    tma_load_2d(st + kVSlabs * kSlabBytes + lane * box * 64, &tmrope, rope0, row, &bars[kKvFull0 + s]);
                    for (int sl = 0; sl < kVSlabs; ++sl)
                        tma_load_2d(st + sl * kSlabBytes + lane * box_bytes, &tmkv, (slab0 + sl) * 64, row,
                                    &bars[kKvFull0 + s]);
                }
                if (ti == 0)
                    for (int k = 1; k <= kPrefetch && k < it.n_tiles; ++k) prefetch(k);
                if (ti == it.n_tiles - 1) prefetch_next_q();
            }
        }
        while (pend > 0) settle_one();
        // drain: the copies this warp issued have landed before shared memory is released
        if (lane == 0)
            for (uint32_t k = n > kStages ? n - kStages : 0; k < n; ++k)
                drain_wait(&bars[kKvFull0 + k % kStages], (k / kStages) & 1);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ q.k MMAs (one thread)
        // S(n) = Q K(n)^T into score buffer n % 2 as soon as it is free (the softmax
        // warps have read S(n - 2)) and K/V tile n has landed; never waits for P V.
        // q over the CTA's dims 0-127 comes from TMEM, dims 128-255 and the 32 rope
        // dims from shared memory.
        const uint32_t id_qk = tc05::idesc_bf16_f32(kHeads, kTile, false, false);
        uint32_t n = 0, ic = 0;
        bool ok = true;
        Cursor cur{pair, pair * per};
        Seg it{};
        while (ok && next_seg(p, R, V, per, S, npairs, cur, it)) {
            ok = warp_wait(ok, &bars[kQFull], ic & 1, abort_flag, p.err, p.wait_ns);
            for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                const int s = n % kStages;
                ok = warp_wait(ok, &bars[kKvFull0 + s], (n / kStages) & 1, abort_flag, p.err, p.wait_ns);
                ok = warp_wait(ok, &bars[kSFree0 + (n & 1)], ((n >> 1) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                if (!ok) break;
                tc05::fence_after_sync();
                if (lane == 0) {
                    const uint32_t d = tbase + kColS + (n & 1) * kTile;
                    const uint64_t kdesc = tc05::smem_desc(sKV + s * kStageBytes, 16, 1024);
                    const uint64_t qdesc = tc05::smem_desc(sQ, 16, 1024);
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // slab: +8 KB, k-step: +32 bytes (16 dims) / +8 TMEM columns
                            tc05::mma_ts(d, tbase + kColQ + sl * 32 + k * 8,
                                         kdesc + static_cast<uint64_t>((sl * kSlabBytes + k * 32) >> 4), id_qk,
                                         (sl | k) ? 1u : 0u);
#pragma unroll
                    for (int sl = 2; sl < 4; ++sl)
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // q slab: +16 KB (128 rows)
                            tc05::mma_ss(d, qdesc + static_cast<uint64_t>(((sl - 2) * kHeads * 128 + k * 32) >> 4),
                                         kdesc + static_cast<uint64_t>((sl * kSlabBytes + k * 32) >> 4), id_qk, 1u);
                    // the rope dims: 64-byte rows, 64-byte swizzle (layout type 4), 8-row groups 512 bytes apart
                    const uint64_t rq = tc05::smem_desc(sQr, 16, 512, 4);
                    const uint64_t rk = tc05::smem_desc(sKV + s * kStageBytes + kVSlabs * kSlabBytes, 16, 512, 4);
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        tc05::mma_ss(d, rq + static_cast<uint64_t>((k * 32) >> 4), rk + static_cast<uint64_t>((k * 32) >> 4),
                                     id_qk, 1u);
                    tc05::commit(&bars[kSFull0 + (n & 1)]);
                    if (ti == it.n_tiles - 1) tc05::commit(&bars[kQEmpty]);
                }
                __syncwarp();
            }
            ++ic;
        }
        // drain: every MMA this warp issued has completed before TMEM is freed
        if (lane == 0) {
            tc05::commit(&bars[kFinal]);
            drain_wait(&bars[kFinal], 0);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ P V MMAs (one thread)
        const uint32_t id_pv = tc05::idesc_bf16_f32(kHeads, 256, false, true);
        uint32_t n = 0, ic = 0;
        bool ok = true;
        Cursor cur{pair, pair * per};
        Seg it{};
        while (ok && next_seg(p, R, V, per, S, npairs, cur, it)) {
            for (int ti = 0; ti < it.n_tiles && ok; ++ti, ++n) {
                ok = warp_wait(ok, &bars[kPFull0 + (n & 1)], (n >> 1) & 1, abort_flag, p.err, p.wait_ns);
                if (!ok) break;
                unsigned char *st = sKV + (n % kStages) * kStageBytes;
                const int n_valid = it.key_end - (it.key_begin + ti * kTile);
                if (n_valid < kTile) {
                    // key rows past the end hold stale data: zero their value dims
                    for (int i = lane; i < (kTile - n_valid) * kVSlabs * 8; i += 32) {
                        const int key = n_valid + i / (kVSlabs * 8);
                        const int sl = (i / 8) % kVSlabs, c = i % 8;
                        *reinterpret_cast<uint4 *>(st + sl * kSlabBytes + key * 128 + (c << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (ti == 0) ok = warp_wait(ok, &bars[kOFree], (ic & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                if (!ok) break;
                tc05::fence_after_sync();
                if (lane == 0) {
                    const uint64_t vdesc = tc05::smem_desc(st, kSlabBytes, 1024);
#pragma unroll
                    for (int k = 0; k < kTile / 16; ++k)   // 16 keys per MMA: +2048 bytes of V rows, +8 columns of P
                        tc05::mma_ts(tbase + kColO, tbase + kColP + (n & 1) * 32 + k * 8,
                                     vdesc + static_cast<uint64_t>(k * 2048 >> 4),
                                     id_pv, (ti == 0 && k == 0) ? 0u : 1u);
                    tc05::commit(&bars[kPFree0 + (n & 1)]);
                    tc05::commit(&bars[kKvEmpty0 + n % kStages]);
                    if (ti == it.n_tiles - 1) tc05::commit(&bars[kODone]);
                }
                __syncwarp();
            }
            ++ic;
        }
        if (lane == 0) {
            tc05::commit(&bars[kFinalPv]);
            drain_wait(&bars[kFinalPv], 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        // Thread (row, qt) owns head `row` (TMEM lane) and, of every tile, keys
        // [16 qt, 16 qt + 16); of O the value columns [64 qt, +64); of q a quarter of
        // each of its three parts.  The four threads of a row sit in warps
        // (row / 32) + 4 qt and combine their row maxima and sums through shared
        // memory and a 128-thread named barrier.
        const int row = (warp & 3) * 32 + lane;
        const int qt = warp >> 2;
        // The softmax warps run one tile ahead: in the iteration of tile n they load
        // S(n + 1), wait for and read the peer's partial of tile n, send their own
        // partial of tile n + 1, then do tile n's softmax, so the exchange of n + 1
        // overlaps the math of n on both CTAs.  Tile t travels in slot t % 2 of the
        // receiver's buffer.  The peer writes tile t only after it has received our
        // tile t - 1, which we send only after reading tile t - 2 out of the same
        // slot (program order; the complete_tx of st.async has release semantics at
        // cluster scope, the peer's wait on it acquire), so no release message is
        // needed.
        const uint32_t x_peer = mapa(smem_u32(sX), peer);
        const uint32_t xf_peer0 = mapa(smem_u32(&bars[kXFull0]), peer);
        float *red = reinterpret_cast<float *>(smem + kOffRed);   // [2 buffers][4 quarters][128 rows]
        const uint32_t trow = tc05::taddr(tbase, (warp & 3) * 32, 0);
        const int row_bar = 2 + (warp & 3);                       // named barrier of the row's four warps
        uint32_t n = 0, ic = 0;
        bool ok = true;
        // q of segment `jt` -> TMEM (the CTA's dims 0-127: 32 per thread), the two
        // SW128 slabs (dims 128-255: 32 per thread) and the SW64 rope rows (8 per
        // thread), once the previous segment's q.k MMAs are done with them.
        auto load_q = [&](const Seg &jt, uint32_t jc) {
            const int64_t qrow = static_cast<int64_t>(jt.b) * p.hq + jt.hg * kHeads + row;
            const uint16_t *qb = p.q + qrow * kDqk;
            const uint4 *qt4 = reinterpret_cast<const uint4 *>(qb + slab0 * 64 + qt * 32);
            const uint4 *qs4 = reinterpret_cast<const uint4 *>(qb + slab0 * 64 + 128 + qt * 32);
            const uint4 *qr4 = reinterpret_cast<const uint4 *>(qb + rope0 + qt * 8);
            ok = warp_wait(ok, &bars[kQEmpty], (jc & 1) ^ 1, abort_flag, p.err, p.wait_ns);
            tc05::fence_after_sync();
            uint4 qv[9];
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[i] = __ldg(qt4 + i);
#pragma unroll
            for (int i = 0; i < 4; ++i) qv[4 + i] = __ldg(qs4 + i);
            qv[8] = __ldg(qr4);
            if (ok) {
                const uint32_t w[16] = {qv[0].x, qv[0].y, qv[0].z, qv[0].w, qv[1].x, qv[1].y, qv[1].z, qv[1].w,
                                        qv[2].x, qv[2].y, qv[2].z, qv[2].w, qv[3].x, qv[3].y, qv[3].z, qv[3].w};
                tc05::st_x16_u32(trow + kColQ + qt * 16, w);
            }
            // slab qt / 2, 16-byte chunks 4 (qt % 2) + i of the row at chunk ^ (row & 7)
            unsigned char *slab = sQ + (qt >> 1) * kHeads * 128 + row * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4 *>(slab + ((((qt & 1) * 4 + i) ^ (row & 7)) << 4)) = qv[4 + i];
            // rope chunk qt of the 64-byte row at chunk ^ ((row >> 1) & 3)
            *reinterpret_cast<uint4 *>(sQr + row * 64 + ((qt ^ ((row >> 1) & 3)) << 4)) = qv[8];
            fence_proxy_async_smem();     // the MMAs read these through the async proxy
            tc05::wait_st();
            tc05::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kQFull]);
        };
        // rows without keys: out = 0, lse = -inf
        for (int v = pair; v < V; v += npairs) {
            if (R[v] != R[v + 1]) continue;
            const int64_t orow = static_cast<int64_t>(v / p.hgroups) * p.hq + (v % p.hgroups) * kHeads + row;
            uint4 *o = reinterpret_cast<uint4 *>(p.out + orow * kDv + rank * 256 + qt * 64);
            for (int i = 0; i < 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
            if (rank == 0 && qt == 0 && p.lse) p.lse[orow] = -INFINITY;
        }
        bool q_loaded = false;
        Cursor cs{pair, pair * per};
        Seg it{};
        while (next_seg(p, R, V, per, S, npairs, cs, it)) {
            const int head = it.hg * kHeads + row;
            const int64_t orow = static_cast<int64_t>(it.b) * p.hq + head;
            if (!q_loaded) load_q(it, ic);
            q_loaded = false;
            float m = -INFINITY, l = 0.f;   // running max (log2 units, scaled) and this thread's part of the sum
            // Partial scores of tile t over this CTA's dims for this thread's 16 keys,
            // rounded to fp16 (unscaled: the scale is applied in the exponent), as 8
            // half2 in nxt[].  Both CTAs round their own partial the same way, so own
            // + peer is bitwise identical in the two CTAs.  (Macros rather than
            // lambdas keep the arrays in registers.)  The exchange barrier of tile t
            // is armed only while the warp is live: once the CTA gave up, the tiles it
            // skips must not arrive again on a phase still waiting for bytes that
            // will never come.
#define PKV_MLA_FETCH_ISSUE(t)                                                                                   \
    do {                                                                                                       \
        if (tid == 0 && ok) mbar_arrive_expect_tx(&bars[kXFull0 + (t) % kXSlots], kXBytes);                    \
        ok = warp_wait(ok, &bars[kSFull0 + ((t) & 1)], ((t) >> 1) & 1, abort_flag, p.err, p.wait_ns);                     \
        if (ok) {                                                                                              \
            tc05::fence_after_sync();                                                                          \
            tc05::ld_x16(trow + kColS + ((t) & 1) * kTile + qt * 16, a_);                                      \
        } else {                                                                                               \
            _Pragma("unroll") for (int j = 0; j < 16; ++j) a_[j] = 0.f;                                        \
        }                                                                                                      \
    } while (0)
            // the load lands: free the score buffer, round to fp16 into nxt[]
#define PKV_MLA_FETCH_DONE(t)                                                                                    \
    do {                                                                                                       \
        tc05::wait_ld();                                                                                       \
        reg_fence16(a_);                                                                                       \
        tc05::fence_before_sync();                                                                             \
        __syncwarp();                                                                                          \
        if (lane == 0) mbar_arrive(&bars[kSFree0 + ((t) & 1)]);                                               \
        _Pragma("unroll") for (int j = 0; j < 8; ++j) nxt[j] = h22u(__floats2half2_rn(a_[2 * j], a_[2 * j + 1])); \
    } while (0)
            // this thread's 16 keys of tile t (2 x 16 B) -> slot t % kXSlots of the peer
#define PKV_MLA_SEND(t)                                                                                          \
    do {                                                                                                       \
        if (ok) {                                                                                              \
            const uint32_t dst_ = x_peer + ((t) % kXSlots) * kXBytes;                                          \
            const uint32_t bar_ = xf_peer0 + ((t) % kXSlots) * 8;                                              \
            _Pragma("unroll") for (int c = 0; c < 2; ++c)                                                      \
                st_async_v4(dst_ + ((qt * 2 + c) * kHeads + row) * 16, __uint_as_float(nxt[4 * c]),            \
                            __uint_as_float(nxt[4 * c + 1]), __uint_as_float(nxt[4 * c + 2]),                  \
                            __uint_as_float(nxt[4 * c + 3]), bar_);                                            \
        }                                                                                                      \
    } while (0)
            uint32_t cur[8], nxt[8];
            float a_[16];
            PKV_MLA_FETCH_ISSUE(n);
            PKV_MLA_FETCH_DONE(n);
            PKV_MLA_SEND(n);
#pragma unroll
            for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
            for (int ti = 0; ti < it.n_tiles; ++ti, ++n) {
                const bool ahead = ti + 1 < it.n_tiles;
                // the scores of tile n + 1 load while the peer's partial of tile n is read
                if (ahead) PKV_MLA_FETCH_ISSUE(n + 1);
                // ---- the peer's partial of tile n (this thread's 16 keys) ----
                const int xs = n % kXSlots;
                ok = warp_wait(ok, &bars[kXFull0 + xs], (n / kXSlots) & 1, abort_flag, p.err, p.wait_ns);
                const int n_valid = it.key_end - (it.key_begin + ti * kTile);
                // own + peer partial in half2 (the same bits in both CTAs)
                __half2 x2[8];
                {
                    const uint4 *xr = reinterpret_cast<const uint4 *>(reinterpret_cast<unsigned char *>(sX) + xs * kXBytes);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint4 w4 = make_uint4(0, 0, 0, 0);
                        if (ok) w4 = xr[(qt * 2 + c) * kHeads + row];
                        x2[4 * c] = __hadd2(u2h2(cur[4 * c]), u2h2(w4.x));
                        x2[4 * c + 1] = __hadd2(u2h2(cur[4 * c + 1]), u2h2(w4.y));
                        x2[4 * c + 2] = __hadd2(u2h2(cur[4 * c + 2]), u2h2(w4.z));
                        x2[4 * c + 3] = __hadd2(u2h2(cur[4 * c + 3]), u2h2(w4.w));
                    }
                }
                // slot n % 2 is read: tile n + 1 may go out (the peer answers it with
                // tile n + 2 into this slot)
                if (ahead) {
                    PKV_MLA_FETCH_DONE(n + 1);
                    PKV_MLA_SEND(n + 1);
                }
                if (n_valid < kTile) {   // keys past the end: -inf
                    const __half2 ninf = __halves2half2(__ushort_as_half(0xfc00), __ushort_as_half(0xfc00));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int key = qt * 16 + 2 * j;
                        if (key >= n_valid) x2[j] = ninf;
                        else if (key + 1 >= n_valid) x2[j] = __halves2half2(__low2half(x2[j]), __ushort_as_half(0xfc00));
                    }
                }
                // row max of the tile: this thread's 16 keys, then the row's other three
                // threads' through shared memory
                float mx;
                {
                    __half2 m2 = x2[0];
#pragma unroll
                    for (int j = 1; j < 8; ++j) m2 = __hmax2(m2, x2[j]);
                    const float2 mf = __half22float2(m2);
                    float *mb = red + (n & 1) * 4 * kHeads;
                    mb[qt * kHeads + row] = fmaxf(mf.x, mf.y);
                    named_bar_sync(row_bar, 128);
                    mx = fmaxf(fmaxf(mb[row], mb[kHeads + row]), fmaxf(mb[2 * kHeads + row], mb[3 * kHeads + row])) *
                         p.scale_log2;
                }
                // ---- online softmax over this tile's keys (log2 units) ----
                const bool raise = mx > m + kLazy || (m == -INFINITY && mx != -INFINITY);
                const float corr = raise ? ex2(m - mx) : 1.f;
                if (__any_sync(0xffffffffu, raise && m != -INFINITY) && ok) {
                    // O is final for tile n - 1 (m finite: it belongs to this segment)
                    // once its P V completed; then rescale this thread's 64 value columns
                    ok = warp_wait(ok, &bars[kPFree0 + ((n - 1) & 1)], ((n - 1) >> 1) & 1, abort_flag, p.err, p.wait_ns);
                    tc05::fence_after_sync();
#pragma unroll 1
                    for (int cc = 0; cc < 4 && ok; ++cc) {
                        float ov[16];
                        tc05::ld_x16(trow + kColO + qt * 64 + cc * 16, ov);
                        tc05::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) ov[e] *= corr;
                        tc05::st_x16(trow + kColO + qt * 64 + cc * 16, ov);
                    }
                    tc05::wait_st();
                }
                if (raise) {
                    l *= corr;
                    m = mx;
                }
                uint32_t h[8];
                float lsum = 0.f;
                const float nm = -m;
#pragma unroll
                for (int j = 0; j < 8; ++j) {   // p = 2^(scale log2(e) x - m)
                    const float2 xf = __half22float2(x2[j]);
                    const float p0 = m == -INFINITY ? 0.f : ex2(fmaf(xf.x, p.scale_log2, nm));
                    const float p1 = m == -INFINITY ? 0.f : ex2(fmaf(xf.y, p.scale_log2, nm));
                    lsum += p0 + p1;
                    h[j] = pack_bf16x2(p0, p1);
                }
                l += lsum;
                // this thread's 16 keys of P (8 bf16 pairs) into buffer n & 1, free once
                // the P V of tile n - 2 completed
                ok = warp_wait(ok, &bars[kPFree0 + (n & 1)], ((n >> 1) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
                if (ok) {
                    tc05::fence_after_sync();
                    tc05::st_x8_u32(trow + kColP + (n & 1) * 32 + qt * 8, h);
                    tc05::wait_st();
                }
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kPFull0 + (n & 1)]);
#pragma unroll
                for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
            }
#undef PKV_MLA_FETCH_ISSUE
#undef PKV_MLA_FETCH_DONE
#undef PKV_MLA_SEND
            // ---- the next segment's q goes in now, so its q.k overlaps this epilogue ----
            {
                Cursor c2 = cs;
                Seg nt;
                if (next_seg(p, R, V, per, S, npairs, c2, nt)) {
                    load_q(nt, ic + 1);
                    q_loaded = true;
                }
            }
            // ---- epilogue: normalise O and write the output (or the split partial) ----
            // l of the whole row = the four threads' partial sums (m is the same in all).
            // Buffer n & 1: not the last tile's max buffer, and free since that tile's barrier.
            float *lb = red + (n & 1) * 4 * kHeads;
            lb[qt * kHeads + row] = l;
            named_bar_sync(row_bar, 128);
            l = (lb[row] + lb[kHeads + row]) + (lb[2 * kHeads + row] + lb[3 * kHeads + row]);
            named_bar_sync(row_bar, 128);
            ok = warp_wait(ok, &bars[kODone], ic & 1, abort_flag, p.err, p.wait_ns);
            tc05::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool single = it.part < 0;
            const int64_t prow = static_cast<int64_t>(it.part) * kHeads + row;
#pragma unroll 1
            for (int cb = 0; cb < 4; cb += 2) {
                float ov[2][16];
                if (ok) {
                    tc05::ld_x16(trow + kColO + qt * 64 + cb * 16, ov[0]);
                    tc05::ld_x16(trow + kColO + qt * 64 + (cb + 1) * 16, ov[1]);
                    tc05::wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) ov[0][e] = ov[1][e] = 0.f;
                }
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    const int col = rank * 256 + qt * 64 + (cb + q2) * 16;
                    if (single) {
                        uint32_t hh[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) hh[e] = pack_bf16x2(ov[q2][2 * e] * inv, ov[q2][2 * e + 1] * inv);
                        uint4 *o = reinterpret_cast<uint4 *>(p.out + orow * kDv + col);
                        o[0] = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        o[1] = make_uint4(hh[4], hh[5], hh[6], hh[7]);
                    } else {
                        // partial layout [part][128 chunks of 4 dims][128 heads] x 16 B: a warp's
                        // store covers 32 consecutive heads of one chunk, 512 contiguous bytes
                        float4 *o = reinterpret_cast<float4 *>(p.part_o) +
                                    (static_cast<int64_t>(it.part) * (kDv / 4) + col / 4) * kHeads + row;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e * kHeads] = make_float4(ov[q2][4 * e] * inv, ov[q2][4 * e + 1] * inv,
                                                        ov[q2][4 * e + 2] * inv, ov[q2][4 * e + 3] * inv);
                    }
                }
            }
            if (rank == 0 && qt == 0) {
                const float lse2 = m + log2f(l);
                if (single) {
                    if (p.lse) p.lse[orow] = lse2 * kLn2;
                } else {
                    p.part_lse[prow] = lse2;
                }
            }
            tc05::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kOFree]);
            ++ic;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc05::fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // both CTAs have issued everything they will issue
    // In a launch that gave up (either CTA), a partial score the peer sent with st.async
    // before it stopped may not have been waited for: give such stores time to land
    // before either CTA releases its shared memory.  (Every send is waited for
    // otherwise.)
    if (*abort_flag || ld_cluster_s32(mapa(smem_u32(const_cast<int *>(abort_flag)), peer)) != 0) {
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 20000ull) {
        }
    }
    cluster_sync_all();   // the peer no longer touches this CTA's shared memory
    if (warp == kMmaWarp) {
        tc05::fence_after_sync();
        tc05::tmem_dealloc(tbase, kTmemCols);
    }
}

// Log-sum-exp merge of the splits of MLA rows: one CTA per (row, 16 heads);
// base-2 lse in the workspace.  The decode kernel left the span length and the
// row table in meta, from which the CTA finds the spans its row crosses.
__global__ void __launch_bounds__(256) mla_merge_kernel(const Params p, int max_splits) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    extern __shared__ float wsm[];  // [16][max_splits]
    __shared__ float den_s[16], mx_s[16];
    const int v = blockIdx.x, h0 = blockIdx.y * 16;
    const int per = p.meta[0];
    const int r0 = p.meta[1 + v], r1 = p.meta[2 + v];   // the row's tiles, stand-ins first
    if (r1 <= r0 + kSegCost || per < 1) return;
    const int s_first = (r0 + kSegCost) / per, s_last = (r1 - 1) / per;
    const int n = s_last - s_first + 1;
    if (n <= 1) return;  // the row sat inside one span: the decode kernel wrote it
    if (n > max_splits) {
        if (threadIdx.x == 0 && blockIdx.y == 0) raise_flag(p.err, PKV_DEVERR_CAPACITY);
        return;
    }
    // split i of the row is slot 1 of its span when another row's segment opens the
    // span (only the first split can be: its row began after the span's first tile)
    auto part = [&](int i) -> int64_t {
        const int s = s_first + i;
        return static_cast<int64_t>(s) * 2 + ((i == 0 && r0 > s * per) ? 1 : 0);
    };
    for (int i = threadIdx.x; i < 16 * n; i += blockDim.x) {
        const int h = i / n, c = i % n;
        wsm[h * max_splits + c] = p.part_lse[part(c) * kHeads + h0 + h];
    }
    __syncthreads();
    if (threadIdx.x < 16) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int c = 0; c < n; ++c) M = fmaxf(M, wsm[h * max_splits + c]);
        float den = 0.f;
        for (int c = 0; c < n; ++c) {
            const float wgt = ex2(wsm[h * max_splits + c] - M);
            wsm[h * max_splits + c] = wgt;
            den += wgt;
        }
        den_s[h] = den;
        mx_s[h] = M;
    }
    __syncthreads();
    const int64_t orow0 = static_cast<int64_t>(v / p.hgroups) * p.hq + (v % p.hgroups) * kHeads + h0;
    // partials are [part][chunk of 4 dims][head]: consecutive threads take consecutive heads
    for (int i = threadIdx.x; i < 16 * (kDv / 4); i += blockDim.x) {
        const int h = i % 16, d4 = i / 16;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < n; ++c) {
            const float wgt = wsm[h * max_splits + c];
            const float4 x = reinterpret_cast<const float4 *>(p.part_o)[(part(c) * (kDv / 4) + d4) * kHeads + h0 + h];
            acc.x = fmaf(wgt, x.x, acc.x);
            acc.y = fmaf(wgt, x.y, acc.y);
            acc.z = fmaf(wgt, x.z, acc.z);
            acc.w = fmaf(wgt, x.w, acc.w);
        }
        const float inv = 1.f / den_s[h];
        uint2 o;
        o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        reinterpret_cast<uint2 *>(p.out + (orow0 + h) * kDv)[d4] = o;
        if (d4 == 0 && p.lse) p.lse[orow0 + h] = (mx_s[h] + log2f(den_s[h])) * kLn2;
    }
}

// ------------------------------------------------------------------ host side
struct Plan {
    int hgroups, span_tiles, max_spans, max_splits;
    size_t part_o_bytes, part_lse_bytes, meta_bytes;
};

// Spans: kv_chunk / 64 tiles each when the caller fixes kv_chunk, else one span
// per CTA pair (at most one pair per two SMs).  Each span holds at most two
// partials.
static bool make_plan(const pkv_decode_args *a, Plan &pl) {
    pl.hgroups = a->num_q_heads / kHeads;
    const int64_t rows = static_cast<int64_t>(a->batch) * pl.hgroups;
    // tiles a row can take in the concatenated sequence, its stand-ins included
    const int64_t tiles_max = (static_cast<int64_t>(std::max(0, a->max_seq_len)) + kTile - 1) / kTile + kSegCost;
    if (rows * tiles_max > INT32_MAX / 4) return false;
    int64_t spans;
    if (a->kv_chunk > 0) {
        pl.span_tiles = a->kv_chunk / kTile;
        spans = std::max<int64_t>(1, (rows * tiles_max + pl.span_tiles - 1) / pl.span_tiles);
    } else {
        pl.span_tiles = 0;
        spans = std::max(1, sm_count() / 2);
    }
    if (spans > INT32_MAX / 4) return false;
    pl.max_spans = static_cast<int>(spans);
    const int64_t per_min = std::max(1, pl.span_tiles);
    pl.max_splits = static_cast<int>(std::min<int64_t>(spans, (tiles_max + per_min - 1) / per_min + 1));
    pl.part_o_bytes = (static_cast<size_t>(spans) * 2 * kHeads * kDv * 4 + 255) / 256 * 256;
    pl.part_lse_bytes = (static_cast<size_t>(spans) * 2 * kHeads * 4 + 255) / 256 * 256;
    pl.meta_bytes = (static_cast<size_t>(rows + 2) * 4 + 255) / 256 * 256;
    return true;
}

pkv_status validate(const pkv_decode_args *a, bool check_ptrs) {
    if (a->batch < 0 || a->num_q_heads < 1 || a->max_seq_len < 0 || a->num_slots < 0)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): negative or zero size");
    if (a->num_kv_heads != 1) return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): num_kv_heads must be 1");
    if (a->head_dim_qk != kDqk || a->head_dim_v != kDv)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): head_dim_qk 576 and head_dim_v 512 are supported");
    if (a->num_q_heads % kHeads)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): num_q_heads must be a multiple of 128");
    if (a->layout != PKV_LAYOUT_VARLEN && (!is_pow2(a->page_size) || a->page_size > 1024))
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): page_size must be a power of two in [1, 1024]");
    if (a->kv_chunk < 0 || a->kv_chunk % kTile)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): kv_chunk must be a multiple of 64");
    if (a->layout == PKV_LAYOUT_REQ_TO_TOKEN || a->k_new || a->v_new)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): the token-table layout and the fused store are GQA only");
    if (a->layout != PKV_LAYOUT_CSR && a->layout != PKV_LAYOUT_BLOCK_TABLE && a->layout != PKV_LAYOUT_VARLEN)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): unknown layout");
    if (a->k_row_stride < kDqk || a->k_row_stride % 8)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): latent row stride must be >= 576 and 16-byte aligned");
    if (a->num_slots > INT32_MAX) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): pool larger than 2^31 rows");
    if (a->batch == 0 || !check_ptrs) return PKV_OK;
    if (!a->q || !a->k_pool || !a->out) return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): null q/k_pool/out");
    if (a->v_pool && a->v_pool != a->k_pool)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): values come from the latent pool; pass v_pool = NULL");
    if (!aligned(a->q, 16) || !aligned(a->k_pool, 16) || !aligned(a->out, 16))
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): q, latent pool and out must be 16-byte aligned");
    switch (a->layout) {
        case PKV_LAYOUT_CSR:
            if (!a->kv_indptr || !a->kv_indices || !a->kv_last_page_len)
                return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): CSR layout needs kv_indptr/kv_indices/kv_last_page_len");
            break;
        case PKV_LAYOUT_BLOCK_TABLE:
            if (!a->block_table || !a->seq_lens || a->block_table_width < 0)
                return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): block-table layout needs block_table and seq_lens");
            break;
        default:
            if (!a->cu_seqlens) return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): varlen layout needs cu_seqlens");
    }
    return PKV_OK;
}

size_t workspace_size(const pkv_decode_args *a) {
    Plan pl;
    if (a->batch == 0 || !make_plan(a, pl)) return 0;
    return pl.part_o_bytes + pl.part_lse_bytes + pl.meta_bytes;
}

// Opt-in shared memory (raised once) and the most co-resident CTA pairs of one
// instantiation of the decode kernel.
template <bool G>
static pkv_status kernel_limits(size_t &lim_out, int &pairs_out) {
    std::atomic<int64_t> *m_lim = device_memo(reinterpret_cast<const void *>(mla_decode_kernel<G>), 0);
    std::atomic<int64_t> *m_pairs = device_memo(reinterpret_cast<const void *>(mla_decode_kernel<G>), 1);
    if (!m_lim || !m_pairs) return fail(PKV_ERR_CUDA, "pkv_decode(MLA): cannot query the current device");
    if (m_lim->load() == 0 || m_pairs->load() == 0) {
        int optin = 0, dev = 0;
        cudaFuncAttributes fa{};
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, mla_decode_kernel<G>) != cudaSuccess)
            return fail(PKV_ERR_CUDA, "pkv_decode(MLA): cannot query shared-memory limits");
        const size_t l = static_cast<size_t>(optin) - fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(mla_decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(l)) != cudaSuccess)
            return fail(PKV_ERR_CUDA, "pkv_decode(MLA): cannot raise the shared-memory limit");
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2 * std::max(1, sm_count() / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = l;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<G>, &cfg) != cudaSuccess || n < 1)
            n = std::max(1, sm_count() / 2);
        m_pairs->store(n);
        m_lim->store(static_cast<int64_t>(l));
    }
    lim_out = static_cast<size_t>(m_lim->load());
    pairs_out = static_cast<int>(m_pairs->load());
    return PKV_OK;
}

pkv_status launch(const pkv_decode_args *a, void *ws, size_t ws_bytes, int32_t *err, cudaStream_t s) {
    Plan pl;
    if (!make_plan(a, pl)) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): batch x max_seq_len too large");
    const size_t need = pl.part_o_bytes + pl.part_lse_bytes + pl.meta_bytes;
    if (ws_bytes < need) return fail(PKV_ERR_CAPACITY, "pkv_decode(MLA): workspace of %zu bytes, %zu needed", ws_bytes, need);
    if (!ws || !aligned(ws, 256))
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode(MLA): workspace must be non-null and 256-byte aligned");
    const size_t msmem = static_cast<size_t>(16) * pl.max_splits * 4;
    if (msmem > 200 * 1024) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): too many splits for the merge");
    Params p{};
    p.layout = a->layout;
    p.batch = a->batch;
    p.hq = a->num_q_heads;
    p.hgroups = pl.hgroups;
    const int ps = a->layout == PKV_LAYOUT_VARLEN ? kTile : a->page_size;
    p.ps_shift = ilog2(ps);
    p.ps_mask = ps - 1;
    p.scale_log2 = a->sm_scale * kLog2e;
    p.span_tiles = pl.span_tiles;
    p.max_len = a->max_seq_len;
    p.bt_width = a->block_table_width;
    p.box_rows = std::min(ps, kTile);
    p.num_slots = a->num_slots;
    p.num_pages = a->num_slots >> p.ps_shift;
    p.kv_indices_len = a->kv_indices_len;
    p.kv_indptr = a->kv_indptr;
    p.kv_indices = a->kv_indices;
    p.kv_last = a->kv_last_page_len;
    p.block_table = a->block_table;
    p.seq_lens = a->seq_lens;
    p.cu_seqlens = a->cu_seqlens;
    p.q = static_cast<const uint16_t *>(a->q);
    p.out = static_cast<uint16_t *>(a->out);
    p.lse = a->lse;
    p.part_o = static_cast<float *>(ws);
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(ws) + pl.part_o_bytes);
    p.meta = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + pl.part_o_bytes + pl.part_lse_bytes);
    p.err = err;
    p.wait_ns = wait_limit_ns();
    p.pool = static_cast<const uint16_t *>(a->k_pool);
    p.pool_stride = a->k_row_stride;
    if (a->layout == PKV_LAYOUT_VARLEN) p.ps_shift = 0, p.ps_mask = 0;

    // TMA map of the latent pool as [num_slots rows, 576] (box box_rows x 64 dims, 128-byte swizzle).
    CUtensorMap tmkv;
    const uint64_t dk[2] = {static_cast<uint64_t>(kDqk), static_cast<uint64_t>(a->num_slots)};
    const uint64_t sk[1] = {static_cast<uint64_t>(a->k_row_stride) * 2};
    const uint32_t bk[2] = {64, static_cast<uint32_t>(p.box_rows)};
    if (!encode_tmap_bf16(&tmkv, a->k_pool, 2, dk, sk, bk))
        return fail(PKV_ERR_CUDA, "pkv_decode(MLA): cuTensorMapEncodeTiled rejected the latent pool");
    // the same pool as 32-dim boxes with 64-byte swizzle: each CTA's half of the rope dims
    CUtensorMap tmrope;
    const uint32_t br[2] = {32, static_cast<uint32_t>(p.box_rows)};
    if (!encode_tmap_bf16(&tmrope, a->k_pool, 2, dk, sk, br, 64))
        return fail(PKV_ERR_CUDA, "pkv_decode(MLA): cuTensorMapEncodeTiled rejected the latent pool (rope view)");

    const bool gather = p.box_rows < 8;
    size_t lim = 0;
    int max_pairs = 0;
    pkv_status st = gather ? kernel_limits<true>(lim, max_pairs) : kernel_limits<false>(lim, max_pairs);
    if (st != PKV_OK) return st;
    const size_t smem = kFixedSmem + (static_cast<size_t>(a->batch) * pl.hgroups + 1) * 4;
    if (smem > lim) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(MLA): batch too large for the on-chip item table");
    const int pairs = std::max(1, std::min(max_pairs, pl.max_spans));
    st = launch_status(gather ? launch_chained(mla_decode_kernel<true>, dim3(2 * pairs), dim3(kThreads), smem, s, p,
                                               tmkv, tmrope)
                              : launch_chained(mla_decode_kernel<false>, dim3(2 * pairs), dim3(kThreads), smem, s, p,
                                               tmkv, tmrope),
                       "pkv_decode(MLA split kernel)");
    if (st != PKV_OK) return st;
    if (msmem > 48 * 1024 &&
        cudaFuncSetAttribute(mla_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(msmem)) !=
            cudaSuccess)
        return fail(PKV_ERR_CUDA, "pkv_decode(MLA): cannot raise the merge shared-memory limit");
    return launch_status(launch_chained(mla_merge_kernel, dim3(a->batch * pl.hgroups, kHeads / 16), dim3(256), msmem, s, p,
                                        pl.max_splits),
                         "pkv_decode(MLA merge kernel)");
}

}  // namespace mla
}  // namespace pkv
