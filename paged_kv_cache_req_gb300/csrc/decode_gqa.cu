// pkv_decode for GQA / MHA: one query token per request attending through a page table.
//
// Work decomposition (split-KV): a work item is (request b, key piece c, kv head
// kh, head slice hs).  A request of L keys is cut into n = ceil(L / chunk) equal
// pieces (multiples of 64 keys); the item covers piece c of kv head kh for the
// query heads of the slice that share kh (up to 16: the whole GQA group), so every
// K/V tile is read from HBM once per group.  Items are ordered request-major with
// the kv heads of one piece adjacent (they read the same pool pages) and are
// handed out round-robin to a persistent grid of SM-count x occupancy CTAs; each
// CTA derives the item list from the device-side lengths in its prologue, so no
// host synchronisation is needed.  Small batches (a few items per CTA) are cut
// instead into equal spans of 64-key tiles (see "work items" below), with the
// rows that a span boundary cuts combined by merge_spans_kernel.  The slot of key
// t is page_table[b][t / ps] * ps + t % ps ("From slots to a page table").
//
// decode_tma_kernel (pages of >= 8 keys, and contiguous varlen rows): one producer
// warp issues a TMA box per page and 64-dim slab (128-byte swizzle) into a ring of
// 64-key stages (3 at head_dim 128, 4 at 64), completion counted in bytes on the
// stage's mbarrier, running ahead across items.  decode_cp_async_kernel (pages of
// 1-4 keys): every thread gathers 16-byte row chunks with cp.async into the same
// layout.  Math (four warps, 16 keys of each tile per warp, each with its own
// online softmax in base 2 whose running max is raised only past 2^8): for GQA
// groups, S = q K^T and O += P V are m16n8k16 bf16 MMAs with the group's heads as
// the MMA rows (K via ldmatrix, V via ldmatrix.trans); for one head per kv head,
// CUDA cores with 8 lanes per key and xor-shuffle reductions.  The warps' states
// are combined at the end of the item.  A request with one piece writes bf16
// output directly; longer ones write fp32 partials and their log-sum-exp,
// combined by merge_kernel.  Every wait is bounded (~2 s).
#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "pkv_internal.cuh"

namespace pkv {
namespace gqa {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 64;   // keys per pipeline stage
constexpr int kStages = 3;
constexpr int kMaxRows = 16; // query heads per CTA (tensor-core path); the CUDA-core path takes <= 4
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;

struct Params {
    int32_t layout;
    int32_t batch, hq, hkv, g, gc, hsplit;
    int32_t ps_shift, ps_mask;
    float scale_log2;
    int32_t chunk, n_chunks_max;
    int32_t spans;      // 0: pieces of `chunk` keys dealt round-robin; else the number of equal spans
    int32_t bt_width;
    int64_t num_slots, num_pages, k_stride, v_stride, kv_indices_len;
    int32_t box_rows;   // TMA box height (keys per box)
    const uint16_t *q, *k_pool, *v_pool;
    const int32_t *kv_indptr, *kv_indices, *kv_last, *block_table, *seq_lens, *cu_seqlens;
    uint16_t *out;
    float *lse;
    float *part_o, *part_lse;
    int32_t *err;
    uint64_t wait_ns;   // bound of every mbarrier wait (pkv_set_wait_limit)
    // PKV_LAYOUT_REQ_TO_TOKEN: the token table itself
    const int32_t *r2t, *req_pool_idx, *kv_start;
    int64_t r2t_rows, r2t_stride, r2t_width;
    // fused store: the new token's rows (nullptr: none), written into the pools
    const uint16_t *k_new, *v_new;
    uint16_t *k_pool_w, *v_pool_w;
    // span mode: [0] tiles per span, then one int4 per span (see SpanCut)
    int32_t *meta;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Key count of request b (clamped to what its page table can address) and the
// base offset of its page list.
__device__ __forceinline__ int key_count(const Params &p, int b, int64_t &base, bool report, bool *clamped = nullptr) {
    int64_t L, cap;
    if (clamped) *clamped = false;
    if (p.layout == PKV_LAYOUT_REQ_TO_TOKEN) {
        // keys at columns s .. s + L - 1 of the request's row; base = offset of column s
        const int64_t row = p.req_pool_idx[b];
        const int64_t s = p.kv_start ? p.kv_start[b] : 0;
        L = p.seq_lens[b];
        if (row < 0 || row >= p.r2t_rows || s < 0 || L < 0 || s + L > p.r2t_width || (s & p.ps_mask)) {
            if (report) raise_flag(p.err, PKV_DEVERR_RANGE);
            base = 0;
            return 0;
        }
        base = row * p.r2t_stride + s;
        cap = L;
    } else if (p.layout == PKV_LAYOUT_CSR) {
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
    const int64_t limit = min(cap, static_cast<int64_t>(p.chunk) * p.n_chunks_max);
    if (L < 0 || L > limit) {
        if (report) raise_flag(p.err, L < 0 ? PKV_DEVERR_RANGE : PKV_DEVERR_CAPACITY);
        if (clamped) *clamped = true;
        L = L < 0 ? 0 : limit;
    }
    return static_cast<int>(L);
}

// Pool slot of key t (base from key_count): -1 when its page lies outside the pool,
// -2 when the token table gives a page start that is not a multiple of the page size.
__device__ __forceinline__ int64_t slot_of(const Params &p, int64_t base, int t) {
    if (p.layout == PKV_LAYOUT_VARLEN) {
        const int64_t s = base + t;
        return (s >= 0 && s < p.num_slots) ? s : -1;
    }
    if (p.layout == PKV_LAYOUT_REQ_TO_TOKEN) {
        // the slot of the page's first position, then the offset inside the page
        const int64_t first = __ldg(p.r2t + base + (t & ~p.ps_mask));
        if (first < 0 || first >= (p.num_pages << p.ps_shift)) return -1;
        if (first & p.ps_mask) return -2;
        return first + (t & p.ps_mask);
    }
    const int32_t *tab = p.layout == PKV_LAYOUT_CSR ? p.kv_indices : p.block_table;
    const int page = __ldg(tab + base + (t >> p.ps_shift));
    if (page < 0 || page >= p.num_pages) return -1;
    return (static_cast<int64_t>(page) << p.ps_shift) + (t & p.ps_mask);
}

// Tile layout in shared memory: a 64-key tile of one kv head is D/64 slabs of
// [64 keys x 128 B]; 16-byte chunk c of key row r sits at chunk (c ^ (r & 7))
// of its 128-byte row (the TMA 128-byte swizzle).  The eight rows an ldmatrix
// reads, or the eight lanes of a SIMT read, land in eight bank groups.
template <int D>
__device__ __forceinline__ int toff(int key, int c) {
    return (c >> 3) * (kTile * 64) + key * 64 + (((c & 7) ^ (key & 7)) << 3);
}

template <int D>
struct Tile {
    static constexpr int kElems = kTile * D;          // one K (or V) tile
    static constexpr int kBytes = kElems * 2;
    static constexpr int kSlabs = D / 64;
    static constexpr int kStageBytes = 2 * kBytes;    // K + V
};

// ---------------------------------------------------------------- work items
// Two ways to cut the work into items, both derived by every CTA from the
// device-side lengths (no host synchronisation):
//
// Pieces (p.spans == 0): request b's keys are cut into n = ceil(L / chunk) equal
// pieces and item (b, c, kh, hs) is piece c of kv head kh for head slice hs.  Items
// are numbered request-major (pieces, then kv heads, then slices) and dealt
// round-robin to the CTAs, so the items of one request run at about the same time
// and pages that several requests share (a common prefix) are read while they are
// still in L2.  This is the choice for large batches, where every CTA gets many
// items and round-robin evens them out.
//
// Spans (p.spans = S > 0; small batches): for each unit u = (kv head kh, head
// slice hs) the requests' rows form one sequence of 64-key tiles, each row entering
// as kSegCost stand-in tiles (the cost of starting an item: its q, the epilogue)
// followed by its real tiles.  Each unit's sequence is cut into S / U equal spans
// (U units), span s = j * U + u, and CTA c takes spans c, c + grid, ...; an item
// is the real tiles of one row inside one span.  With two or three items per
// CTA, dealing whole pieces leaves some CTAs with half again the average work;
// equal spans leave them within a few tiles of each other.  (Three stand-in tiles:
// a traced item start and finish cost about what 2-3 tiles take.)  Cutting every
// unit's sequence at the same places keeps U neighbouring CTAs on the same keys of
// different kv heads at the same time, so the DRAM rows of a key (all kv heads side
// by side) are read together, as in the piece order.  A row that a span
// boundary cuts writes one fp32 partial per span: to slot 0 of its span when it is
// the span's first item (its row began at or before the span's first tile), else
// to slot 1 (only the span's last item can be cut there); merge_spans_kernel
// combines them.
constexpr int kSegCost = 3;

// Work units of request b with L keys: items (pieces, all units) or tiles of one
// unit's row (spans).
__device__ __forceinline__ int request_units(const Params &p, int L) {
    if (p.spans) return L > 0 ? (L + kTile - 1) / kTile + kSegCost : 0;
    return max(1, (L + p.chunk - 1) / p.chunk) * p.hkv * p.hsplit;
}

// off[b] = first unit of request b (exclusive scan of its units), off[B] = total.
// Every CTA builds the same table from the lengths, with `nthreads` threads (a
// multiple of 32) and one barrier id; `report` raises the requests' range and
// capacity flags (spans: CTA 0; pieces report as they are located).
__device__ __forceinline__ void build_item_table(const Params &p, int *off, int *scratch, int nthreads, bool report) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.batch;
    const int seg = (B + nthreads - 1) / nthreads;
    const int lo = min(B, tid * seg), hi = min(B, lo + seg);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
        int64_t base;
        local += request_units(p, key_count(p, b, base, report));
    }
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += scratch[w];
    int run = wbase + incl - local;
    for (int b = lo; b < hi; ++b) {
        off[b] = run;
        int64_t base;
        run += request_units(p, key_count(p, b, base, false));
    }
    if (tid == nthreads - 1) off[B] = wbase + incl;
    __syncthreads();
}

struct Item {
    int b, kh, hs, L, head0, t_begin, t_end;
    int part;     // -1: the item is its row's only one and writes bf16 output; else its fp32 partial
    int64_t base;
    bool store;   // fused store: this item's keys end with the request's new token
};

// Request holding unit w: the last b with off[b] <= w (empty requests are skipped).
__device__ __forceinline__ int request_of(const int *off, int batch, int w) {
    int lo = 0, hi = batch;  // off[lo] <= w < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= w) lo = mid; else hi = mid;
    }
    return lo;
}

// Spans of one unit's sequence, and the tiles of each.
__device__ __forceinline__ int unit_spans(const Params &p) { return p.spans / (p.hkv * p.hsplit); }
__device__ __forceinline__ int span_tiles(const Params &p, const int *off) {
    const int sk = unit_spans(p);
    return max(1, (off[p.batch] + sk - 1) / sk);
}

// Pieces: item w.
template <int GC>
__device__ __forceinline__ Item locate(const Params &p, const int *off, int w, bool report) {
    Item it;
    it.b = request_of(off, p.batch, w);
    int rem = w - off[it.b];
    it.hs = rem % p.hsplit;
    rem /= p.hsplit;
    it.kh = rem % p.hkv;
    const int c = rem / p.hkv;
    bool clamped = false;
    it.L = key_count(p, it.b, it.base, report && c == 0 && it.kh == 0 && it.hs == 0, &clamped);
    const int n_chunks = max(1, (it.L + p.chunk - 1) / p.chunk);
    it.head0 = it.kh * p.g + it.hs * GC;
    // the request's n_chunks pieces are made equal (a multiple of 64 keys, at most
    // p.chunk), so its last piece is not a stub that leaves the others waiting
    const int piece = ((it.L + n_chunks - 1) / n_chunks + kTile - 1) / kTile * kTile;
    it.t_begin = c * piece;
    it.t_end = min(it.L, it.t_begin + piece);
    it.part = n_chunks == 1 ? -1
                            : static_cast<int>(((static_cast<int64_t>(it.b) * p.hkv + it.kh) * p.hsplit + it.hs) *
                                                   p.n_chunks_max + c);
    it.store = p.k_new != nullptr && !clamped && it.L > 0 && it.t_end == it.L;
    return it;
}

// A CTA's walk over its items: pieces w = blockIdx.x, + gridDim.x, ...; spans
// s = blockIdx.x, + gridDim.x, ..., each from its first tile (w = next tile of
// the span's unit sequence).
struct Cursor {
    int w, s;
};

__device__ __forceinline__ Cursor first_cursor(const Params &p, const int *off) {
    const int c = static_cast<int>(blockIdx.x);
    return p.spans ? Cursor{(c / (p.hkv * p.hsplit)) * span_tiles(p, off), c} : Cursor{c, 0};
}

// The CTA's next item (false when there is none left).  Pieces may be empty
// (t_end <= t_begin: a request without keys); span items never are.
template <int GC>
__device__ __forceinline__ bool next_item(const Params &p, const int *off, Cursor &c, Item &it, bool report) {
    const int total = off[p.batch];
    if (!p.spans) {
        if (c.w >= total) return false;
        it = locate<GC>(p, off, c.w, report);
        c.w += gridDim.x;
        return true;
    }
    const int per = span_tiles(p, off), U = p.hkv * p.hsplit;
    while (c.s < p.spans) {
        const int u = c.s % U;
        const int s_begin = (c.s / U) * per;
        const int s_end = min(total, s_begin + per);
        while (c.w < s_end) {
            const int b = request_of(off, p.batch, c.w);
            bool clamped = false;
            int64_t base;
            const int L = key_count(p, b, base, false, &clamped);
            const int r0 = off[b], r1 = off[b + 1];     // the row's tiles, stand-ins first
            const int real0 = r0 + kSegCost;
            const int t0 = max(c.w, real0), t1 = min(s_end, r1);
            c.w = t1;
            if (t0 >= t1) continue;   // only stand-in tiles of this row in this span
            it.b = b;
            it.hs = u % p.hsplit;
            it.kh = u / p.hsplit;
            it.L = L;
            it.base = base;
            it.head0 = it.kh * p.g + it.hs * GC;
            it.t_begin = (t0 - real0) * kTile;
            it.t_end = min(L, (t1 - real0) * kTile);
            it.part = (t0 == real0 && t1 == r1) ? -1 : c.s * 2 + (r0 <= s_begin ? 0 : 1);
            it.store = p.k_new != nullptr && !clamped && it.t_end == L;
            return true;
        }
        c.s += gridDim.x;
        c.w = (c.s / U) * per;
    }
    return false;
}

// Span mode: what merge_spans_kernel needs about the row that the first tile of
// span s cuts, {request, unit, first tile of the row, tiles of the row} (tiles
// within the unit's sequence), or b = -1 when that tile cuts no row or the row was
// already cut by an earlier span boundary (each cut row is merged once, for its
// first cut).
struct SpanCut {
    int b, u, r0, rs;
};

__device__ __forceinline__ SpanCut span_cut(const Params &p, const int *off, int s) {
    const int per = span_tiles(p, off), U = p.hkv * p.hsplit;
    const int u = s % U, j = s / U;
    const int x = j * per;
    SpanCut cut{-1, 0, 0, 0};
    if (j < 1 || x >= off[p.batch]) return cut;
    const int b = request_of(off, p.batch, x);
    const int r0 = off[b];
    const int real0 = r0 + kSegCost;
    // cut: real tiles on both sides of x; first cut: the row's first real tile lies in span j - 1
    if (real0 < x && real0 / per == j - 1) cut = SpanCut{b, u, r0, off[b + 1] - r0};
    return cut;
}

// Fused store of the new token (key L - 1 of the request, kv head kh): the pool rows
// are written here, with plain stores (run by one warp of the item).  The key itself
// is masked out of its tile (whatever the tile load read from its stale slot is
// ignored) and added to the warp's softmax state afterwards from k_new / v_new
// (Math::add_key), so the tile loop is the same code with or without the store.
template <int D>
__device__ __forceinline__ void store_new_rows(const Params &p, const Item &it) {
    const int lane = threadIdx.x & 31;
    const int64_t slot = slot_of(p, it.base, it.L - 1);
    if (slot < 0) return;   // the loads of that page raised the flag
    const int64_t row = (static_cast<int64_t>(it.b) * p.hkv + it.kh) * D;
    for (int i = lane; i < 2 * (D / 8); i += 32) {
        const bool is_v = i >= D / 8;
        const int c = is_v ? i - D / 8 : i;
        const uint4 val = __ldg(reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) + row + c * 8));
        uint16_t *dst = is_v ? p.v_pool_w + slot * p.v_stride : p.k_pool_w + slot * p.k_stride;
        *reinterpret_cast<uint4 *>(dst + it.kh * D + c * 8) = val;
    }
}

// Valid keys of the tile starting at t0 for the math: with the fused store the new
// token (the item's last key) is left out of its tile.
__device__ __forceinline__ int tile_keys(const Item &it, int t0) {
    const int n = it.t_end - t0;
    return (it.store && n <= kTile) ? n - 1 : n;
}

template <int D, int GC>
__device__ __forceinline__ void write_empty(const Params &p, const Item &it) {
    for (int i = threadIdx.x; i < GC * D; i += kThreads) {
        const int h = i / D, d = i % D;
        p.out[(static_cast<int64_t>(it.b) * p.hq + it.head0 + h) * D + d] = 0;
        if (d == 0 && p.lse) p.lse[static_cast<int64_t>(it.b) * p.hq + it.head0 + h] = -INFINITY;
    }
}

// Combines the per-warp states left in red_* (base-2 running max m, sum l,
// unnormalised o; rows GC apart per warp) and writes the item's output or
// split partial.  Run by the kThreads math threads.
template <int D, int GC>
__device__ __forceinline__ void finish_item(const Params &p, const Item &it, const float *red_o, const float *red_m,
                                            const float *red_l) {
    const int64_t pidx = it.part;
    for (int i = threadIdx.x; i < GC * D; i += kThreads) {
        const int h = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, red_m[ww * GC + h]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
            const float mw = red_m[ww * GC + h];
            const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
            num = fmaf(red_o[(ww * GC + h) * D + d], sc, num);
            den = fmaf(red_l[ww * GC + h], sc, den);
        }
        const float val = num / den;
        if (it.part < 0) {
            p.out[(static_cast<int64_t>(it.b) * p.hq + it.head0 + h) * D + d] =
                __bfloat16_as_ushort(__float2bfloat16_rn(val));
            if (d == 0 && p.lse) p.lse[static_cast<int64_t>(it.b) * p.hq + it.head0 + h] = (M + log2f(den)) * kLn2;
        } else {
            p.part_o[(pidx * GC + h) * D + d] = val;
            if (d == 0) p.part_lse[pidx * GC + h] = M + log2f(den);
        }
    }
}

template <int D, int GC>
struct RedLayout {
    static constexpr int kBytes = kWarps * GC * D * 4 + 2 * kWarps * GC * 4;
};

// ---------------------------------------------------------------- tensor-core math (GQA groups)
// Per 64-key tile each warp owns 16 keys.  S = Q K^T is an m16n8k16 bf16 MMA
// with the group's query heads as the 16 rows (rows past the group are zero),
// the warp's keys as columns (two n8 tiles) and head_dim as the reduction;
// K comes from the swizzled tile with ldmatrix.  The fp32 scores go through a
// per-warp online softmax (base 2; the running max is raised only when a row
// grows by more than 2^8, so rescales are rare and p <= 256), are rounded to
// bf16 in registers and reused directly as the A operand of O += P V (V read
// with ldmatrix.trans).
template <int D, int GC>
struct MmaState {
    static constexpr int KS = D / 16;
    static constexpr int NT = D / 8;
    static constexpr bool kRows8 = GC > 8;
    uint32_t qa[KS][4];
    float o[NT][4];
    float m0, m1, l0, l1;
};

template <int D, int GC>
__device__ __forceinline__ void mma_begin(MmaState<D, GC> &st, const Params &p, const Item &it) {
    const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const uint32_t *q0 =
        reinterpret_cast<const uint32_t *>(p.q + (static_cast<int64_t>(it.b) * p.hq + it.head0 + g) * D);
    const uint32_t *q8 =
        reinterpret_cast<const uint32_t *>(p.q + (static_cast<int64_t>(it.b) * p.hq + it.head0 + g + 8) * D);
#pragma unroll
    for (int ks = 0; ks < MmaState<D, GC>::KS; ++ks) {
        st.qa[ks][0] = g < GC ? __ldg(q0 + ks * 8 + tig) : 0u;
        st.qa[ks][2] = g < GC ? __ldg(q0 + ks * 8 + 4 + tig) : 0u;
        st.qa[ks][1] = (MmaState<D, GC>::kRows8 && g + 8 < GC) ? __ldg(q8 + ks * 8 + tig) : 0u;
        st.qa[ks][3] = (MmaState<D, GC>::kRows8 && g + 8 < GC) ? __ldg(q8 + ks * 8 + 4 + tig) : 0u;
    }
#pragma unroll
    for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt) st.o[nt][0] = st.o[nt][1] = st.o[nt][2] = st.o[nt][3] = 0.f;
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
}

template <int D, int GC>
__device__ __forceinline__ void mma_tile(MmaState<D, GC> &st, const uint16_t *kt, const uint16_t *vt, int n_valid,
                                         float scale_log2) {
    constexpr bool kRows8 = MmaState<D, GC>::kRows8;
    constexpr float kLazy = 8.f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3;
    const int key0 = warp * 16;
    float sc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        const int key = key0 + j * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, kt + toff<D>(key, kk * 4 + (lane >> 3)));
            mma_bf16_16816(sc[j], st.qa[2 * kk], b0, b1);
            mma_bf16_16816(sc[j], st.qa[2 * kk + 1], b2, b3);
        }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = key0 + j * 8 + tig * 2 + (e & 1);
            sc[j][e] = key < n_valid ? sc[j][e] * scale_log2 : -INFINITY;
        }
    float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    if (mx0 > st.m0 + kLazy || (st.m0 == -INFINITY && mx0 != -INFINITY)) {
        const float corr = ex2(st.m0 - mx0);
        st.l0 *= corr;
#pragma unroll
        for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt) { st.o[nt][0] *= corr; st.o[nt][1] *= corr; }
        st.m0 = mx0;
    }
    if (kRows8) {
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        if (mx1 > st.m1 + kLazy || (st.m1 == -INFINITY && mx1 != -INFINITY)) {
            const float corr = ex2(st.m1 - mx1);
            st.l1 *= corr;
#pragma unroll
            for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt) { st.o[nt][2] *= corr; st.o[nt][3] *= corr; }
            st.m1 = mx1;
        }
    }
    uint32_t pa[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float p0 = st.m0 == -INFINITY ? 0.f : ex2(sc[j][0] - st.m0);
        const float p1 = st.m0 == -INFINITY ? 0.f : ex2(sc[j][1] - st.m0);
        const float p2 = (!kRows8 || st.m1 == -INFINITY) ? 0.f : ex2(sc[j][2] - st.m1);
        const float p3 = (!kRows8 || st.m1 == -INFINITY) ? 0.f : ex2(sc[j][3] - st.m1);
        st.l0 += p0 + p1;
        st.l1 += p2 + p3;
        pa[2 * j] = pack_bf16x2(p0, p1);
        pa[2 * j + 1] = pack_bf16x2(p2, p3);
    }
#pragma unroll
    for (int nn = 0; nn < D / 16; ++nn) {
        const int mi = lane >> 3;
        const int key = key0 + (mi & 1) * 8 + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(b0, b1, b2, b3, vt + toff<D>(key, nn * 2 + (mi >> 1)));
        mma_bf16_16816(st.o[2 * nn], pa, b0, b1);
        mma_bf16_16816(st.o[2 * nn + 1], pa, b2, b3);
    }
}

template <int D, int GC>
__device__ __forceinline__ void mma_store(MmaState<D, GC> &st, float *red_o, float *red_m, float *red_l) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 1);
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 2);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 1);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 2);
    if (g < GC) {
#pragma unroll
        for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt)
            *reinterpret_cast<float2 *>(&red_o[(warp * GC + g) * D + nt * 8 + tig * 2]) =
                make_float2(st.o[nt][0], st.o[nt][1]);
        if (tig == 0) {
            red_m[warp * GC + g] = st.m0;
            red_l[warp * GC + g] = st.l0;
        }
    }
    if (MmaState<D, GC>::kRows8 && g + 8 < GC) {
#pragma unroll
        for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt)
            *reinterpret_cast<float2 *>(&red_o[(warp * GC + g + 8) * D + nt * 8 + tig * 2]) =
                make_float2(st.o[nt][2], st.o[nt][3]);
        if (tig == 0) {
            red_m[warp * GC + g + 8] = st.m1;
            red_l[warp * GC + g + 8] = st.l1;
        }
    }
}

// One more key, given as bf16 rows kn / vn in global memory, added to this warp's
// state (the fused store's new token).  The thread holds q of rows g and g + 8 in
// the A-fragment layout: dims 16 ks + 2 tig + {0, 1} and + 8; the four threads of a
// row reduce their partial dot products with xor-shuffles.  P stays in fp32; l is
// counted once per row (by tig 0), as the row sum is reduced over tig at the end.
template <int D, int GC>
__device__ __forceinline__ void mma_add_key(MmaState<D, GC> &st, const uint16_t *kn, const uint16_t *vn,
                                            float scale_log2) {
    constexpr bool kRows8 = MmaState<D, GC>::kRows8;
    constexpr float kLazy = 8.f;
    const int lane = threadIdx.x & 31, tig = lane & 3;
    const uint32_t *k32 = reinterpret_cast<const uint32_t *>(kn);
    float d0 = 0.f, d1 = 0.f;
#pragma unroll
    for (int ks = 0; ks < MmaState<D, GC>::KS; ++ks) {
        const uint32_t klo = __ldg(k32 + ks * 8 + tig), khi = __ldg(k32 + ks * 8 + 4 + tig);
        d0 = fmaf(bf16_lo(st.qa[ks][0]), bf16_lo(klo), d0);
        d0 = fmaf(bf16_hi(st.qa[ks][0]), bf16_hi(klo), d0);
        d0 = fmaf(bf16_lo(st.qa[ks][2]), bf16_lo(khi), d0);
        d0 = fmaf(bf16_hi(st.qa[ks][2]), bf16_hi(khi), d0);
        d1 = fmaf(bf16_lo(st.qa[ks][1]), bf16_lo(klo), d1);
        d1 = fmaf(bf16_hi(st.qa[ks][1]), bf16_hi(klo), d1);
        d1 = fmaf(bf16_lo(st.qa[ks][3]), bf16_lo(khi), d1);
        d1 = fmaf(bf16_hi(st.qa[ks][3]), bf16_hi(khi), d1);
    }
    d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
    d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
    d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
    d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
    const float s0 = d0 * scale_log2, s1 = d1 * scale_log2;
    if (s0 > st.m0 + kLazy || st.m0 == -INFINITY) {
        const float corr = ex2(st.m0 - s0);
        st.l0 *= corr;
#pragma unroll
        for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt) { st.o[nt][0] *= corr; st.o[nt][1] *= corr; }
        st.m0 = s0;
    }
    if (kRows8 && (s1 > st.m1 + kLazy || st.m1 == -INFINITY)) {
        const float corr = ex2(st.m1 - s1);
        st.l1 *= corr;
#pragma unroll
        for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt) { st.o[nt][2] *= corr; st.o[nt][3] *= corr; }
        st.m1 = s1;
    }
    const float p0 = ex2(s0 - st.m0);
    const float p1 = kRows8 ? ex2(s1 - st.m1) : 0.f;
    if (tig == 0) {
        st.l0 += p0;
        st.l1 += p1;
    }
    const uint32_t *v32 = reinterpret_cast<const uint32_t *>(vn);
#pragma unroll
    for (int nt = 0; nt < MmaState<D, GC>::NT; ++nt) {
        const uint32_t vv = __ldg(v32 + nt * 4 + tig);   // dims 8 nt + 2 tig, + 1
        st.o[nt][0] = fmaf(p0, bf16_lo(vv), st.o[nt][0]);
        st.o[nt][1] = fmaf(p0, bf16_hi(vv), st.o[nt][1]);
        st.o[nt][2] = fmaf(p1, bf16_lo(vv), st.o[nt][2]);
        st.o[nt][3] = fmaf(p1, bf16_hi(vv), st.o[nt][3]);
    }
}

// ---------------------------------------------------------------- CUDA-core math (one head per kv head)
// Each warp takes 16 keys of a tile; 8 lanes share a key (each lane owns D/8
// dims), reduce q.k with three xor-shuffles, and keep their own online-softmax
// state (base 2, scale * log2 e folded into q).
template <int D, int GC>
struct SimtState {
    static constexpr int NC = D / 64;
    float q[GC][NC][8];
    float o[GC][NC][8];
    float m[GC], l[GC];
};

template <int D, int GC>
__device__ __forceinline__ void simt_begin(SimtState<D, GC> &st, const Params &p, const Item &it) {
    const int part = threadIdx.x & 7;
#pragma unroll
    for (int h = 0; h < GC; ++h)
#pragma unroll
        for (int ci = 0; ci < SimtState<D, GC>::NC; ++ci) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                p.q + (static_cast<int64_t>(it.b) * p.hq + it.head0 + h) * D + (part + 8 * ci) * 8));
            widen8(raw, st.q[h][ci]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                st.q[h][ci][e] *= p.scale_log2;
                st.o[h][ci][e] = 0.f;
            }
        }
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        st.m[h] = -INFINITY;
        st.l[h] = 0.f;
    }
}

template <int D, int GC>
__device__ __forceinline__ void simt_tile(SimtState<D, GC> &st, const uint16_t *kt, const uint16_t *vt, int n_valid) {
    constexpr int NC = SimtState<D, GC>::NC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, grp = lane >> 3, part = lane & 7;
    float s[4][GC];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int key = warp * 16 + j * 4 + grp;
#pragma unroll
        for (int h = 0; h < GC; ++h) s[j][h] = 0.f;
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(kt + toff<D>(key, part + 8 * ci));
            float kf[8];
            widen8(raw, kf);
#pragma unroll
            for (int h = 0; h < GC; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) s[j][h] = fmaf(st.q[h][ci][e], kf[e], s[j][h]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            float v = s[j][h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            s[j][h] = (warp * 16 + j * 4 + grp < n_valid) ? v : -INFINITY;
        }
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        const float mt = fmaxf(fmaxf(s[0][h], s[1][h]), fmaxf(s[2][h], s[3][h]));
        if (mt > st.m[h]) {
            const float corr = ex2(st.m[h] - mt);  // m = -inf gives 0
            st.l[h] *= corr;
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                for (int e = 0; e < 8; ++e) st.o[h][ci][e] *= corr;
            st.m[h] = mt;
        }
        const bool live = st.m[h] != -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s[j][h] = live ? ex2(s[j][h] - st.m[h]) : 0.f;
            st.l[h] += s[j][h];
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int key = warp * 16 + j * 4 + grp;
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(vt + toff<D>(key, part + 8 * ci));
            float vf[8];
            widen8(raw, vf);
#pragma unroll
            for (int h = 0; h < GC; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) st.o[h][ci][e] = fmaf(s[j][h], vf[e], st.o[h][ci][e]);
        }
    }
}

template <int D, int GC>
__device__ __forceinline__ void simt_store(SimtState<D, GC> &st, float *red_o, float *red_m, float *red_l) {
    constexpr int NC = SimtState<D, GC>::NC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, grp = lane >> 3, part = lane & 7;
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        float mw = fmaxf(st.m[h], __shfl_xor_sync(0xffffffffu, st.m[h], 8));
        mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
        const float corr = (st.m[h] == -INFINITY) ? 0.f : ex2(st.m[h] - mw);
        float lw = st.l[h] * corr;
        lw += __shfl_xor_sync(0xffffffffu, lw, 8);
        lw += __shfl_xor_sync(0xffffffffu, lw, 16);
#pragma unroll
        for (int ci = 0; ci < NC; ++ci)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float v = st.o[h][ci][e] * corr;
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                st.o[h][ci][e] = v;
            }
        st.m[h] = mw;
        st.l[h] = lw;
    }
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < GC; ++h) {
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                for (int e = 0; e < 8; ++e) red_o[(warp * GC + h) * D + (part + 8 * ci) * 8 + e] = st.o[h][ci][e];
            if (part == 0) {
                red_m[warp * GC + h] = st.m[h];
                red_l[warp * GC + h] = st.l[h];
            }
        }
    }
}

// One more key (the fused store's new token) added to the state of lane group 0
// (lanes 0-7: each owns D / 8 dims; q is already scaled by scale * log2 e).  The
// groups' states are combined in simt_store, so one group taking the key counts it
// once.
template <int D, int GC>
__device__ __forceinline__ void simt_add_key(SimtState<D, GC> &st, const uint16_t *kn, const uint16_t *vn) {
    constexpr int NC = SimtState<D, GC>::NC;
    const int lane = threadIdx.x & 31, grp = lane >> 3, part = lane & 7;
    float s[GC];
#pragma unroll
    for (int h = 0; h < GC; ++h) s[h] = 0.f;
#pragma unroll
    for (int ci = 0; ci < NC; ++ci) {
        float kf[8];
        widen8(__ldg(reinterpret_cast<const uint4 *>(kn + (part + 8 * ci) * 8)), kf);
#pragma unroll
        for (int h = 0; h < GC; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[h] = fmaf(st.q[h][ci][e], kf[e], s[h]);
    }
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 2);
        s[h] += __shfl_xor_sync(0xffffffffu, s[h], 4);
    }
    if (grp != 0) return;
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        if (s[h] > st.m[h]) {
            const float corr = ex2(st.m[h] - s[h]);   // m = -inf gives 0
            st.l[h] *= corr;
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                for (int e = 0; e < 8; ++e) st.o[h][ci][e] *= corr;
            st.m[h] = s[h];
        }
        s[h] = ex2(s[h] - st.m[h]);
        st.l[h] += s[h];
    }
#pragma unroll
    for (int ci = 0; ci < NC; ++ci) {
        float vf[8];
        widen8(__ldg(reinterpret_cast<const uint4 *>(vn + (part + 8 * ci) * 8)), vf);
#pragma unroll
        for (int h = 0; h < GC; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) st.o[h][ci][e] = fmaf(s[h], vf[e], st.o[h][ci][e]);
    }
}

template <int D, int GC, bool MMA>
struct Math;
template <int D, int GC>
struct Math<D, GC, true> {
    using State = MmaState<D, GC>;
    static __device__ __forceinline__ void begin(State &s, const Params &p, const Item &it) { mma_begin<D, GC>(s, p, it); }
    static __device__ __forceinline__ void tile(State &s, const uint16_t *k, const uint16_t *v, int n, float sc) {
        mma_tile<D, GC>(s, k, v, n, sc);
    }
    static __device__ __forceinline__ void store(State &s, float *o, float *m, float *l) { mma_store<D, GC>(s, o, m, l); }
    static __device__ __forceinline__ void add_key(State &s, const uint16_t *kn, const uint16_t *vn, float sc) {
        mma_add_key<D, GC>(s, kn, vn, sc);
    }
};
template <int D, int GC>
struct Math<D, GC, false> {
    using State = SimtState<D, GC>;
    static __device__ __forceinline__ void begin(State &s, const Params &p, const Item &it) { simt_begin<D, GC>(s, p, it); }
    static __device__ __forceinline__ void tile(State &s, const uint16_t *k, const uint16_t *v, int n, float) {
        simt_tile<D, GC>(s, k, v, n);
    }
    static __device__ __forceinline__ void store(State &s, float *o, float *m, float *l) { simt_store<D, GC>(s, o, m, l); }
    static __device__ __forceinline__ void add_key(State &s, const uint16_t *kn, const uint16_t *vn, float) {
        simt_add_key<D, GC>(s, kn, vn);
    }
};

// The fused store's new token: math warp 0 adds it to its state (it was left out of
// the item's last tile) and writes its rows into the pools.
template <int D, int GC, bool MMA>
__device__ __forceinline__ void add_new_key(typename Math<D, GC, MMA>::State &st, const Params &p, const Item &it) {
    if (!it.store || (threadIdx.x >> 5) != 0) return;
    const int64_t row = (static_cast<int64_t>(it.b) * p.hkv + it.kh) * D;
    Math<D, GC, MMA>::add_key(st, p.k_new + row, p.v_new + row, p.scale_log2);
    store_new_rows<D>(p, it);
}

// ---------------------------------------------------------------- cp.async kernel (page_size < 8)
// Issue the cp.async copies of one 64-key tile (K and V) of kv head kh; keys
// past t1, and keys whose page is outside the pool, are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile_cp_async(const Params &p, uint16_t *ks, uint16_t *vs, int64_t base, int t0,
                                                   int t1, int kh) {
    constexpr int CPR = D / 8;              // 16-byte chunks per row
    constexpr int RPP = kThreads / CPR;     // rows per pass
    const int chunk = threadIdx.x % CPR;
    const int row0 = threadIdx.x / CPR;
#pragma unroll
    for (int i = 0; i < kTile / RPP; ++i) {
        const int key = row0 + i * RPP;
        const int t = t0 + key;
        int64_t slot = -1;
        if (t < t1) {
            slot = slot_of(p, base, t);
            if (slot < 0 && chunk == 0) raise_flag(p.err, slot == -2 ? PKV_DEVERR_CONTIG : PKV_DEVERR_RANGE);
        }
        const bool ok = slot >= 0;
        const uint16_t *ksrc = ok ? p.k_pool + slot * p.k_stride + kh * D + chunk * 8 : p.k_pool;
        const uint16_t *vsrc = ok ? p.v_pool + slot * p.v_stride + kh * D + chunk * 8 : p.v_pool;
        const int dst = toff<D>(key, chunk);
        cp_async_16(ks + dst, ksrc, ok ? 16 : 0);
        cp_async_16(vs + dst, vsrc, ok ? 16 : 0);
    }
}

template <int D, int GC, bool MMA>
__global__ void __launch_bounds__(kThreads, 2) decode_cp_async_kernel(const Params p) {
    using T = Tile<D>;
    using M = Math<D, GC, MMA>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint16_t *tiles = reinterpret_cast<uint16_t *>(smem);
    float *red_o = reinterpret_cast<float *>(smem + kStages * T::kStageBytes);
    float *red_m = red_o + kWarps * GC * D;
    float *red_l = red_m + kWarps * GC;
    int *off = reinterpret_cast<int *>(smem + kStages * T::kStageBytes + RedLayout<D, GC>::kBytes);
    __shared__ int scan_scratch[kWarps];

    pdl_wait();          // lengths, tables and pool rows may come from the previous kernel
    pdl_launch_next();
    build_item_table(p, off, scan_scratch, kThreads, false);   // pieces only (p.spans == 0)

    Cursor cur = first_cursor(p, off);
    Item it;
    while (next_item<GC>(p, off, cur, it, threadIdx.x == 0)) {
        if (it.t_end <= it.t_begin) {
            write_empty<D, GC>(p, it);
            continue;
        }
        typename M::State st;
        M::begin(st, p, it);
        const int n_tiles = (it.t_end - it.t_begin + kTile - 1) / kTile;
#pragma unroll
        for (int s = 0; s < kStages - 1; ++s) {
            if (s < n_tiles) {
                uint16_t *kst = tiles + s * 2 * T::kElems;
                load_tile_cp_async<D>(p, kst, kst + T::kElems, it.base, it.t_begin + s * kTile, it.t_end, it.kh);
            }
            cp_async_commit();
        }
        for (int ti = 0; ti < n_tiles; ++ti) {
            cp_async_wait<kStages - 2>();
            __syncthreads();
            {
                const int nt_ = ti + kStages - 1;
                if (nt_ < n_tiles) {
                    uint16_t *kst = tiles + (nt_ % kStages) * 2 * T::kElems;
                    load_tile_cp_async<D>(p, kst, kst + T::kElems, it.base, it.t_begin + nt_ * kTile, it.t_end,
                                          it.kh);
                }
                cp_async_commit();
            }
            const uint16_t *kt = tiles + (ti % kStages) * 2 * T::kElems;
            M::tile(st, kt, kt + T::kElems, tile_keys(it, it.t_begin + ti * kTile), p.scale_log2);
        }
        cp_async_wait<0>();
        add_new_key<D, GC, MMA>(st, p, it);
        M::store(st, red_o, red_m, red_l);
        __syncthreads();
        finish_item<D, GC>(p, it, red_o, red_m, red_l);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- TMA kernel (page_size >= 8, varlen)
// Warp-specialised: warps 0-3 do the math, warp 4 (one lane) is the producer.
// The producer walks the same item sequence as the math warps and, for every
// 64-key tile, issues one TMA box per page (box = min(ps, 64) keys x 64 dims,
// 128-byte swizzle; D = 128 takes two boxes per page) into a free stage, with
// completion counted in bytes on that stage's full barrier.  It runs up to
// kTmaStages tiles ahead, across item boundaries, so the next item's K/V is in
// flight while the math warps reduce and write the current one.  Math warps
// release a stage through its empty barrier.  Key rows past the item's end
// (and rows of pages that do not exist) may hold stale data: K is masked by
// the scores' select, V rows are zeroed by the warp that reads them.
// Bounded mbarrier wait shared by the producer and the math warps: gives up
// when another warp already gave up (abort flag) or once `limit_ns` have passed
// (checked after the second poll and every 64 polls), raising
// PKV_DEVERR_TIMEOUT; afterwards no warp of the CTA waits again.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int32_t *err,
                                              uint64_t limit_ns) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
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

// Bounded wait that ignores the abort flag: lets the TMA copies a warp issued land
// before its CTA exits (~2 s at most, whatever the wait limit).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return;
        if ((i & 63) == 63 && global_ns() - t0 > 2000000000ull) return;
    }
}

// Stages of the TMA kernel: two CTAs per SM at head_dim 128; three at 64, whose
// 16 KB stages leave room for a third CTA with four stages each (more tiles in
// flight per SM than two CTAs of five: 7-8 % faster on the Whisper-shaped step).
template <int D>
struct TmaCfg {
    static constexpr int kStagesN = D == 128 ? 3 : 4;
    static constexpr int kCtasPerSm = D == 128 ? 2 : 3;
};

// Two CTAs per SM (the shared memory of D = 128 with up to 8 heads per group allows
// it) put three of the pair's ten warps on one SM sub-partition, whose share of the
// register file is 16K: hence at most 168 registers a thread there.
template <int D, int GC, bool MMA>
__global__ void __launch_bounds__(kThreads + 32, 1) __maxnreg__((D == 128 && GC < 16) ? 168 : 255)
decode_tma_kernel(const Params p, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using T = Tile<D>;
    using M = Math<D, GC, MMA>;
    constexpr int S = TmaCfg<D>::kStagesN;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint16_t *tiles = reinterpret_cast<uint16_t *>(smem);
    float *red_o = reinterpret_cast<float *>(smem + S * T::kStageBytes);
    float *red_m = red_o + kWarps * GC * D;
    float *red_l = red_m + kWarps * GC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * T::kStageBytes + RedLayout<D, GC>::kBytes);
    uint64_t *empty = full + S;
    int *scan = reinterpret_cast<int *>(empty + S);
    volatile int *abort_flag = scan + 7;
    int *off = scan + 8;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init_fence();
    }
    if (warp == kWarps && lane == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    pdl_wait();          // lengths, tables and pool rows may come from the previous kernel
    pdl_launch_next();
    build_item_table(p, off, scan, kThreads + 32, p.spans != 0 && blockIdx.x == 0);

    if (warp == kWarps) {
        // ---------------- producer ----------------
        // Lane j owns box j of every tile (kTile / box <= 8 boxes).  The page ids
        // of tile n+1 are loaded before tile n is issued, so the table lookups
        // overlap the wait for a free stage.
        const int box = p.box_rows;
        const int nbox = kTile / box;
        const uint32_t box_bytes = static_cast<uint32_t>(box) * 128u;
        const bool own = lane < nbox;
        // cursor over (item, tile), skipping empty items
        Cursor cur = first_cursor(p, off);
        int ti = 0;
        Item it{};
        bool have = false;
        // With the token table every page start sits in its own part of the request's
        // row, so the lookups miss L2 far more often than in a packed page list: when
        // the cursor reaches an item, the page starts of this CTA's following item are
        // pulled into L2 (one 128-byte line holds 32 positions).
        auto prefetch_pages = [&]() {
            if (p.layout != PKV_LAYOUT_REQ_TO_TOKEN) return;
            Cursor c2 = cur;
            Item nx;
            if (!next_item<GC>(p, off, c2, nx, false) || nx.t_end <= nx.t_begin) return;
            const int step = max(1, 32 >> p.ps_shift);   // pages per line
            const int last = (nx.t_end - 1) >> p.ps_shift;
            for (int pg = (nx.t_begin >> p.ps_shift) + lane * step; pg <= last; pg += 32 * step)
                prefetch_l2(p.r2t + nx.base + (static_cast<int64_t>(pg) << p.ps_shift));
        };
        // Token table: the warp holds the slots of a window of 32 * kBatch page starts
        // (lane j: pages pg0 + j, pg0 + j + 32, ...), loaded at once when the cursor
        // enters an item and again when a tile passes the window, so a tile's lookup
        // is a register shuffle instead of a load that would wait on L2 one tile ahead.
        constexpr int kBatch = 4;
        int firsts[kBatch];
        int pg0 = 0;
        const bool batched = p.layout == PKV_LAYOUT_REQ_TO_TOKEN;
        auto load_firsts = [&](int t) {   // window from the page of key t
            pg0 = t >> p.ps_shift;
            const int npg = ((it.t_end - 1) >> p.ps_shift) - pg0 + 1;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int pg = lane + 32 * k;
                firsts[k] = pg < npg ? __ldg(p.r2t + it.base + (static_cast<int64_t>(pg0 + pg) << p.ps_shift)) : -1;
            }
        };
        auto next_nonempty = [&]() {
            Item nx;
            while (next_item<GC>(p, off, cur, nx, false)) {
                if (nx.t_end > nx.t_begin) {
                    it = nx;
                    // the item's q rows into L2 a few tiles before the math warps load them,
                    // and with the fused store the new token's K and V rows, which warp 0
                    // adds to its softmax state after the tile loop
                    constexpr int kQLines = (GC * D * 2 + 127) / 128;
                    if (lane < kQLines)
                        prefetch_l2(reinterpret_cast<const char *>(p.q + (static_cast<int64_t>(it.b) * p.hq + it.head0) * D) +
                                    lane * 128);
                    if (it.store && lane < 2 * (D / 64)) {
                        const uint16_t *nrow = (lane < D / 64 ? p.k_new : p.v_new) + (static_cast<int64_t>(it.b) * p.hkv + it.kh) * D;
                        prefetch_l2(reinterpret_cast<const char *>(nrow) + (lane % (D / 64)) * 128);
                    }
                    prefetch_pages();
                    if (batched) load_firsts(it.t_begin);
                    return true;
                }
            }
            return false;
        };
        have = next_nonempty();
        // row of this lane's box for the cursor's tile (-1: no box, -2: page outside the
        // pool, -3: a token-table page start that is not page-aligned)
        auto lookup = [&]() -> int {
            if (have && batched) {   // warp-uniform: every lane takes part in the shuffles
                const int tb = it.t_begin + ti * kTile + lane * box;
                const int pi = own && tb < it.t_end ? (tb >> p.ps_shift) - pg0 : 0;
                int first = -1;
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int v = __shfl_sync(0xffffffffu, firsts[k], pi & 31);
                    if ((pi >> 5) == k) first = v;
                }
                if (!own || tb >= it.t_end) return -1;
                if (first < 0 || first >= (p.num_pages << p.ps_shift)) return -2;
                if (first & p.ps_mask) return -3;
                return first + (tb & p.ps_mask);
            }
            if (!have || !own) return -1;
            const int tb = it.t_begin + ti * kTile + lane * box;
            if (tb >= it.t_end) return -1;
            if (p.layout == PKV_LAYOUT_VARLEN) return static_cast<int>(it.base + tb);
            const int32_t *tab = p.layout == PKV_LAYOUT_CSR ? p.kv_indices : p.block_table;
            const int page = __ldg(tab + it.base + (tb >> p.ps_shift));
            if (page < 0 || page >= p.num_pages) return -2;
            return static_cast<int>((static_cast<int64_t>(page) << p.ps_shift) + (tb & p.ps_mask));
        };
        int row = lookup();
        uint32_t n = 0;
        for (; have; ++n) {
            const int kh = it.kh;
            // advance the cursor and start the next tile's lookups
            const int n_tiles = (it.t_end - it.t_begin + kTile - 1) / kTile;
            if (++ti >= n_tiles) {
                ti = 0;
                have = next_nonempty();
            } else if (batched && ((it.t_begin + ti * kTile + kTile - 1) >> p.ps_shift) - pg0 >= 32 * kBatch) {
                load_firsts(it.t_begin + ti * kTile);
            }
            const int next_row = lookup();
            const int s = n % S;
            bool ok = true;
            if (lane == 0) ok = wait_or_abort(&empty[s], ((n / S) & 1) ^ 1, abort_flag, p.err, p.wait_ns);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            if (row <= -2) {   // a bad page reads as zeros (and raises the flag)
                raise_flag(p.err, row == -2 ? PKV_DEVERR_RANGE : PKV_DEVERR_CONTIG);
                unsigned char *kst = smem + s * T::kStageBytes;
                for (int h = 0; h < T::kSlabs; ++h)
                    for (uint32_t o = 0; o < box_bytes; o += 16) {
                        *reinterpret_cast<uint4 *>(kst + h * (kTile * 128) + lane * box_bytes + o) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(kst + T::kBytes + h * (kTile * 128) + lane * box_bytes + o) =
                            make_uint4(0, 0, 0, 0);
                    }
                fence_proxy_async_smem();   // before later TMA writes into this stage
            }
            const uint32_t valid = __ballot_sync(0xffffffffu, row >= 0);
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], __popc(valid) * box_bytes * T::kSlabs * 2u);
            __syncwarp();
            if (row >= 0) {
                unsigned char *kst = smem + s * T::kStageBytes;
                unsigned char *vst = kst + T::kBytes;
#pragma unroll
                for (int h = 0; h < T::kSlabs; ++h) {
                    tma_load_3d(kst + h * (kTile * 128) + lane * box_bytes, &tmk, h * 64, kh, row, &full[s]);
                    tma_load_3d(vst + h * (kTile * 128) + lane * box_bytes, &tmv, h * 64, kh, row, &full[s]);
                }
            }
            row = next_row;
        }
        // drain: the copies of the last (at most S) tiles issued land before the CTA
        // may exit; consumers that gave up no longer wait for them
        if (lane == 0)
            for (uint32_t k = n > static_cast<uint32_t>(S) ? n - S : 0; k < n; ++k) drain_wait(&full[k % S], (k / S) & 1);
        __syncwarp();
        return;
    }

    // ---------------- math warps ----------------
    if (p.spans) {
        // rows without keys take no tiles: their outputs are written here, and the
        // merge's view of the spans (tiles per span, the row each boundary cuts)
        for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
            if (off[b + 1] != off[b]) continue;
            Item e{};
            e.b = b;
            for (int u = 0; u < p.hkv * p.hsplit; ++u) {
                e.head0 = (u / p.hsplit) * p.g + (u % p.hsplit) * GC;
                write_empty<D, GC>(p, e);
            }
        }
        if (tid == 0 && blockIdx.x == 0) p.meta[0] = span_tiles(p, off);
        for (int s = blockIdx.x + tid * gridDim.x; s < p.spans; s += gridDim.x * kThreads) {
            const SpanCut c = span_cut(p, off, s);
            reinterpret_cast<int4 *>(p.meta + 4)[s] = make_int4(c.b, c.u, c.r0, c.rs);
        }
    }
    uint32_t n = 0;
    Cursor cur = first_cursor(p, off);
    Item it;
    while (next_item<GC>(p, off, cur, it, tid == 0)) {
        if (it.t_end <= it.t_begin) {
            write_empty<D, GC>(p, it);
            continue;
        }
        typename M::State st;
        M::begin(st, p, it);
        const int n_tiles = (it.t_end - it.t_begin + kTile - 1) / kTile;
        for (int ti = 0; ti < n_tiles; ++ti, ++n) {
            const int s = n % S;
            if (!wait_or_abort(&full[s], (n / S) & 1, abort_flag, p.err, p.wait_ns)) {
                // abandoned launch: keep releasing stages and reaching barriers, compute nothing
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                continue;
            }
            uint16_t *kt = tiles + s * 2 * T::kElems;
            uint16_t *vt = kt + T::kElems;
            const int n_valid = tile_keys(it, it.t_begin + ti * kTile);
            if (n_valid < kTile) {
                // zero the V rows of this warp's keys past the end (stale or never loaded)
                for (int i = lane; i < 16 * (D / 8); i += 32) {
                    const int key = warp * 16 + i / (D / 8);
                    if (key >= n_valid)
                        *reinterpret_cast<uint4 *>(vt + toff<D>(key, i % (D / 8))) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            M::tile(st, kt, vt, n_valid, p.scale_log2);
            if (n_valid < kTile) fence_proxy_async_smem();  // generic writes before the next TMA into this stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        add_new_key<D, GC, MMA>(st, p, it);
        M::store(st, red_o, red_m, red_l);
        named_bar_sync(1, kThreads);
        finish_item<D, GC>(p, it, red_o, red_m, red_l);
        named_bar_sync(1, kThreads);
    }
}

// ---------------------------------------------------------------- merge
// Log-sum-exp merge of a request's chunk partials (base-2 lse inside the workspace).
template <int D, int GC>
__global__ void __launch_bounds__(kThreads) merge_kernel(const Params p) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    extern __shared__ float wsm[];  // [GC][n_chunks_max] weights
    const int idx = blockIdx.x;
    const int hs = idx % p.hsplit;
    const int kh = (idx / p.hsplit) % p.hkv;
    const int b = idx / (p.hsplit * p.hkv);
    int64_t base;
    const int L = key_count(p, b, base, false);
    const int n = (L + p.chunk - 1) / p.chunk;
    if (n <= 1) return;
    const int64_t pbase = ((static_cast<int64_t>(b) * p.hkv + kh) * p.hsplit + hs) * p.n_chunks_max;
    __shared__ float den_s[kMaxRows], mx_s[kMaxRows];
    for (int i = threadIdx.x; i < GC * n; i += kThreads) {
        const int h = i / n, c = i % n;
        wsm[h * p.n_chunks_max + c] = p.part_lse[(pbase + c) * GC + h];
    }
    __syncthreads();
    if (threadIdx.x < GC) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int c = 0; c < n; ++c) M = fmaxf(M, wsm[h * p.n_chunks_max + c]);
        float den = 0.f;
        for (int c = 0; c < n; ++c) {
            const float wgt = ex2(wsm[h * p.n_chunks_max + c] - M);
            wsm[h * p.n_chunks_max + c] = wgt;
            den += wgt;
        }
        den_s[h] = den;
        mx_s[h] = M;
    }
    __syncthreads();
    const int head0 = kh * p.g + hs * GC;
    for (int i = threadIdx.x; i < GC * D; i += kThreads) {
        const int h = i / D, d = i % D;
        float acc = 0.f;
        for (int c = 0; c < n; ++c)
            acc = fmaf(wsm[h * p.n_chunks_max + c], p.part_o[((pbase + c) * GC + h) * D + d], acc);
        acc /= den_s[h];
        p.out[(static_cast<int64_t>(b) * p.hq + head0 + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        if (d == 0 && p.lse) p.lse[static_cast<int64_t>(b) * p.hq + head0 + h] = (mx_s[h] + log2f(den_s[h])) * kLn2;
    }
}

// Span mode: log-sum-exp merge of the rows cut by span boundaries, one CTA per
// span s (the row whose first cut is the span's first tile; see span_cut).  The
// row's real tiles lie in spans s - 1 .. of its unit; its item in span s - 1 wrote
// slot 1 of that span when another row opened the span, every later one slot 0.
template <int D, int GC>
__global__ void __launch_bounds__(kThreads) merge_spans_kernel(const Params p) {
    pdl_wait();          // the split kernel's partials and span records
    pdl_launch_next();
    extern __shared__ float wsm[];  // [GC][spans] weights
    __shared__ float den_s[kMaxRows], mx_s[kMaxRows];
    const int s = blockIdx.x;
    const int4 cut = reinterpret_cast<const int4 *>(p.meta + 4)[s];
    if (cut.x < 0) return;
    const int b = cut.x, u = cut.y, r0 = cut.z, rs = cut.w;
    const int per = p.meta[0];
    const int U = p.hkv * p.hsplit;
    const int j_first = s / U - 1, j_last = (r0 + rs - 1) / per;   // spans of the row within its unit
    const int n = j_last - j_first + 1;
    auto part = [&](int i) -> int64_t {
        return static_cast<int64_t>((j_first + i) * U + u) * 2 + ((i == 0 && r0 > j_first * per) ? 1 : 0);
    };
    for (int i = threadIdx.x; i < GC * n; i += kThreads) {
        const int h = i / n, c = i % n;
        wsm[h * p.spans + c] = p.part_lse[part(c) * GC + h];
    }
    __syncthreads();
    if (threadIdx.x < GC) {
        const int h = threadIdx.x;
        float M = -INFINITY;
        for (int c = 0; c < n; ++c) M = fmaxf(M, wsm[h * p.spans + c]);
        float den = 0.f;
        for (int c = 0; c < n; ++c) {
            const float wgt = ex2(wsm[h * p.spans + c] - M);
            wsm[h * p.spans + c] = wgt;
            den += wgt;
        }
        den_s[h] = den;
        mx_s[h] = M;
    }
    __syncthreads();
    const int head0 = (u / p.hsplit) * p.g + (u % p.hsplit) * GC;
    for (int i = threadIdx.x; i < GC * D; i += kThreads) {
        const int h = i / D, d = i % D;
        float acc = 0.f;
        for (int c = 0; c < n; ++c) acc = fmaf(wsm[h * p.spans + c], p.part_o[(part(c) * GC + h) * D + d], acc);
        acc /= den_s[h];
        p.out[(static_cast<int64_t>(b) * p.hq + head0 + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        if (d == 0 && p.lse) p.lse[static_cast<int64_t>(b) * p.hq + head0 + h] = (mx_s[h] + log2f(den_s[h])) * kLn2;
    }
}

// ------------------------------------------------------------------ host side
struct Plan {
    bool mma, tma;
    int gc, hsplit, chunk, n_chunks_max;
    int spans;   // 0: pieces
    size_t part_o_bytes, part_lse_bytes, meta_bytes;
    size_t bytes() const { return part_o_bytes + part_lse_bytes + meta_bytes; }
};

// Equal spans replace round-robin pieces when even the longest possible requests
// would give each span at most this many tiles (a few items per CTA).
constexpr int64_t kSpanTilesMax = 128;

static int choose_chunk(const pkv_decode_args *a, int units) {
    // Fewest equal chunks of the longest request (each a multiple of 64 keys, at most
    // 1024) that still give about two waves of work items when the requests average
    // half of max_seq_len.  Equal chunks keep the items of one request alike, and a
    // request short enough for one chunk needs no merge at all.
    const int64_t target = 2ll * std::max(1, sm_count()) * 2;
    const int64_t L = std::max<int64_t>(1, a->max_seq_len);
    const int64_t half = std::max<int64_t>(1, L / 2);
    for (int64_t n = std::max<int64_t>(1, (L + 1023) / 1024); n <= L; ++n) {
        const int64_t c = ((L + n - 1) / n + kTile - 1) / kTile * kTile;
        if (c > 1024) continue;
        if (c <= kTile) break;
        const int64_t items = static_cast<int64_t>(a->batch) * units * ((half + c - 1) / c);
        if (items >= target) return static_cast<int>(c);
    }
    return kTile;
}

static pkv_status make_plan(const pkv_decode_args *a, Plan &pl) {
    const int g = a->num_q_heads / a->num_kv_heads;
    // GQA groups go to the tensor-core kernel (up to 16 heads as MMA rows);
    // a single head per kv head (MHA) stays on CUDA cores.
    pl.mma = g >= 2;
    pl.gc = pl.mma ? std::min(g, kMaxRows) : 1;
    pl.hsplit = g / pl.gc;
    pl.chunk = a->kv_chunk > 0 ? a->kv_chunk : choose_chunk(a, a->num_kv_heads * pl.hsplit);
    pl.n_chunks_max = std::max(1, (a->max_seq_len + pl.chunk - 1) / pl.chunk);
    // Whole pages of >= 8 keys (or contiguous rows) stream in as TMA boxes; smaller
    // pages are gathered row by row with cp.async.
    pl.tma = (a->layout == PKV_LAYOUT_VARLEN || a->page_size >= 8) && a->num_slots <= INT32_MAX;
    // Spans (TMA kernel, library-chosen split): one per CTA the SMs hold (two per SM,
    // three at head_dim 64), the same number for every unit (kv head, head slice).
    const int64_t units = static_cast<int64_t>(a->num_kv_heads) * pl.hsplit;
    const int64_t per_sm = a->head_dim_qk == 64 ? TmaCfg<64>::kCtasPerSm : TmaCfg<128>::kCtasPerSm;
    const int64_t spans = units * (per_sm * std::max(1, sm_count()) / units);
    const int64_t tiles_ub = static_cast<int64_t>(a->batch) * units * ((a->max_seq_len + kTile - 1) / kTile + kSegCost);
    pl.spans = (pl.tma && a->kv_chunk == 0 && a->batch > 0 && spans > 0 && tiles_ub <= kSpanTilesMax * spans)
                   ? static_cast<int>(spans) : 0;
    pl.meta_bytes = 0;
    if (pl.spans) {
        const int64_t parts = 2 * spans * pl.gc;   // two slots per span
        pl.part_o_bytes = (static_cast<size_t>(parts) * a->head_dim_v * 4 + 255) / 256 * 256;
        pl.part_lse_bytes = (static_cast<size_t>(parts) * 4 + 255) / 256 * 256;
        pl.meta_bytes = (static_cast<size_t>(spans + 1) * 16 + 255) / 256 * 256;
    } else if (pl.n_chunks_max == 1) {
        pl.part_o_bytes = pl.part_lse_bytes = 0;
    } else {
        const int64_t parts = static_cast<int64_t>(a->batch) * a->num_kv_heads * pl.hsplit * pl.n_chunks_max * pl.gc;
        pl.part_o_bytes = (static_cast<size_t>(parts) * a->head_dim_v * 4 + 255) / 256 * 256;
        pl.part_lse_bytes = (static_cast<size_t>(parts) * 4 + 255) / 256 * 256;
    }
    return PKV_OK;
}

pkv_status validate(const pkv_decode_args *a, bool check_ptrs) {
    if (a->batch < 0 || a->num_q_heads < 1 || a->num_kv_heads < 1 || a->max_seq_len < 0 || a->num_slots < 0)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: negative or zero size");
    if (a->num_q_heads % a->num_kv_heads)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: num_q_heads must be a multiple of num_kv_heads");
    const int g = a->num_q_heads / a->num_kv_heads;
    if (a->head_dim_qk != a->head_dim_v || (a->head_dim_qk != 64 && a->head_dim_qk != 128))
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(GQA): head_dim must be 64 or 128 for both q/k and v");
    if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode(GQA): Hq/Hkv must be 1, 2, 4, 8 or 16");
    if (a->layout != PKV_LAYOUT_VARLEN && (!is_pow2(a->page_size) || a->page_size > 1024))
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: page_size must be a power of two <= 1024");
    if (a->kv_chunk < 0 || a->kv_chunk % kTile)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: kv_chunk must be a multiple of 64");
    if (a->batch == 0 || !check_ptrs) return PKV_OK;
    if (!a->q || !a->k_pool || !a->v_pool || !a->out)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: null q/k_pool/v_pool/out");
    switch (a->layout) {
        case PKV_LAYOUT_CSR:
            if (!a->kv_indptr || !a->kv_indices || !a->kv_last_page_len)
                return fail(PKV_ERR_INVALID_ARG, "pkv_decode: CSR layout needs kv_indptr/kv_indices/kv_last_page_len");
            break;
        case PKV_LAYOUT_BLOCK_TABLE:
            if (!a->block_table || !a->seq_lens || a->block_table_width < 0)
                return fail(PKV_ERR_INVALID_ARG, "pkv_decode: block-table layout needs block_table and seq_lens");
            break;
        case PKV_LAYOUT_VARLEN:
            if (!a->cu_seqlens) return fail(PKV_ERR_INVALID_ARG, "pkv_decode: varlen layout needs cu_seqlens");
            break;
        case PKV_LAYOUT_REQ_TO_TOKEN:
            if (!a->req_to_token || !a->req_pool_idx || !a->seq_lens)
                return fail(PKV_ERR_INVALID_ARG, "pkv_decode: token-table layout needs req_to_token, req_pool_idx, seq_lens");
            if (a->r2t_rows < 0 || a->r2t_width < 0 || a->r2t_row_stride < a->r2t_width || a->r2t_width > INT32_MAX)
                return fail(PKV_ERR_INVALID_ARG, "pkv_decode: bad req_to_token shape");
            break;
        default:
            return fail(PKV_ERR_INVALID_ARG, "pkv_decode: unknown layout");
    }
    if ((a->k_new == nullptr) != (a->v_new == nullptr))
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: k_new and v_new go together");
    if (a->k_new && a->layout == PKV_LAYOUT_VARLEN)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: the fused store needs a pool layout (not VARLEN)");
    if (a->k_new && (!aligned(a->k_new, 16) || !aligned(a->v_new, 16)))
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: k_new and v_new must be 16-byte aligned");
    const int64_t row = static_cast<int64_t>(a->num_kv_heads) * a->head_dim_qk;
    if (a->k_row_stride < row || a->v_row_stride < row)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: pool row stride smaller than a row");
    if (!aligned(a->q, 16) || !aligned(a->k_pool, 16) || !aligned(a->v_pool, 16) || a->k_row_stride % 8 ||
        a->v_row_stride % 8)
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: q, pools and row strides must be 16-byte aligned");
    return PKV_OK;
}

size_t workspace_size(const pkv_decode_args *a) {
    Plan pl;
    make_plan(a, pl);
    return pl.bytes();
}

// Opt-in dynamic shared memory of a kernel (device limit minus its static part), set once.
template <typename K>
static pkv_status smem_limit(K kernel, size_t &lim) {
    int optin = 0, dev = 0;
    cudaFuncAttributes fa{};
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
        return fail(PKV_ERR_CUDA, "pkv_decode: cannot query shared-memory limits");
    lim = static_cast<size_t>(optin) - fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(lim)) != cudaSuccess)
        return fail(PKV_ERR_CUDA, "pkv_decode: cannot raise the shared-memory limit to %zu bytes", lim);
    return PKV_OK;
}

// smem_limit once per device (kernel attributes are per device); the limit is cached.
template <typename K>
static pkv_status device_smem_limit(K kernel, size_t &lim) {
    std::atomic<int64_t> *m = device_memo(reinterpret_cast<const void *>(kernel));
    if (!m) return fail(PKV_ERR_CUDA, "pkv_decode: cannot query the current device");
    if (m->load() == 0) {
        pkv_status st = smem_limit(kernel, lim);
        if (st != PKV_OK) return st;
        m->store(static_cast<int64_t>(lim));
    }
    lim = static_cast<size_t>(m->load());
    return PKV_OK;
}

template <typename K>
static int persistent_grid(K kernel, int threads, size_t smem, const Params &p) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess || occ < 1) occ = 1;
    const int64_t upper = p.spans ? p.spans : static_cast<int64_t>(p.batch) * p.hkv * p.hsplit * p.n_chunks_max;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(upper, static_cast<int64_t>(sm_count()) * occ)));
}

template <int D, int GC>
static pkv_status launch_merge(const Params &p, cudaStream_t s) {
    if (p.spans) {
        const size_t msmem = static_cast<size_t>(GC) * p.spans * 4;   // at most 16 x 3 x SMs weights
        return launch_status(launch_chained(merge_spans_kernel<D, GC>, dim3(p.spans), dim3(kThreads), msmem, s, p),
                             "pkv_decode(GQA span merge kernel)");
    }
    if (p.n_chunks_max == 1) return PKV_OK;
    const size_t msmem = static_cast<size_t>(GC) * p.n_chunks_max * 4;
    if (msmem > 200 * 1024) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: too many splits for the merge");
    if (msmem > 48 * 1024) {
        // the raised limit is per device: remember the largest one set on this device
        std::atomic<int64_t> *m = device_memo(reinterpret_cast<const void *>(merge_kernel<D, GC>));
        if (!m) return fail(PKV_ERR_CUDA, "pkv_decode: cannot query the current device");
        if (m->load() < static_cast<int64_t>(msmem)) {
            if (cudaFuncSetAttribute(merge_kernel<D, GC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(msmem)) != cudaSuccess)
                return fail(PKV_ERR_CUDA, "pkv_decode: cannot raise the merge shared-memory limit");
            int64_t cur = m->load();
            while (cur < static_cast<int64_t>(msmem) && !m->compare_exchange_weak(cur, static_cast<int64_t>(msmem))) {
            }
        }
    }
    return launch_status(launch_chained(merge_kernel<D, GC>, dim3(p.batch * p.hkv * p.hsplit), dim3(kThreads), msmem, s, p),
                         "pkv_decode(GQA merge kernel)");
}

template <int D, int GC, bool MMA>
static pkv_status launch_t(const Params &p, const pkv_decode_args *a, bool tma, cudaStream_t s) {
    using T = Tile<D>;
    pkv_status st;
    if (tma) {
        const auto kernel = decode_tma_kernel<D, GC, MMA>;
        size_t lim = 0;
        if ((st = device_smem_limit(kernel, lim)) != PKV_OK) return st;
        const size_t smem = 1024 + TmaCfg<D>::kStagesN * T::kStageBytes + RedLayout<D, GC>::kBytes +
                            2 * TmaCfg<D>::kStagesN * 8 + 32 + (static_cast<size_t>(p.batch) + 1) * 4;
        if (smem > lim) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: batch too large for the on-chip item table");
        CUtensorMap tmk, tmv;
        const uint64_t rows = static_cast<uint64_t>(a->num_slots);
        const uint64_t dk[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(p.hkv), rows};
        const uint64_t sk[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(p.k_stride) * 2};
        const uint64_t sv[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(p.v_stride) * 2};
        const uint32_t box[3] = {64, 1, static_cast<uint32_t>(p.box_rows)};
        if (!encode_tmap_bf16(&tmk, a->k_pool, 3, dk, sk, box) || !encode_tmap_bf16(&tmv, a->v_pool, 3, dk, sv, box))
            return fail(PKV_ERR_CUDA, "pkv_decode: cuTensorMapEncodeTiled rejected the pool layout");
        const int grid = persistent_grid(kernel, kThreads + 32, smem, p);
        st = launch_status(launch_chained(kernel, dim3(grid), dim3(kThreads + 32), smem, s, p, tmk, tmv),
                           "pkv_decode(GQA split kernel)");
    } else {
        const auto kernel = decode_cp_async_kernel<D, GC, MMA>;
        size_t lim = 0;
        if ((st = device_smem_limit(kernel, lim)) != PKV_OK) return st;
        const size_t smem = kStages * T::kStageBytes + RedLayout<D, GC>::kBytes + (static_cast<size_t>(p.batch) + 1) * 4;
        if (smem > lim) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: batch too large for the on-chip item table");
        const int grid = persistent_grid(kernel, kThreads, smem, p);
        st = launch_status(launch_chained(kernel, dim3(grid), dim3(kThreads), smem, s, p), "pkv_decode(GQA split kernel)");
    }
    if (st != PKV_OK) return st;
    return launch_merge<D, GC>(p, s);
}

template <int D>
static pkv_status launch_d(const Plan &pl, const Params &p, const pkv_decode_args *a, bool tma, cudaStream_t s) {
    if (!pl.mma) return launch_t<D, 1, false>(p, a, tma, s);
    switch (pl.gc) {
        case 2: return launch_t<D, 2, true>(p, a, tma, s);
        case 4: return launch_t<D, 4, true>(p, a, tma, s);
        case 8: return launch_t<D, 8, true>(p, a, tma, s);
        default: return launch_t<D, 16, true>(p, a, tma, s);
    }
}

pkv_status launch(const pkv_decode_args *a, void *ws, size_t ws_bytes, int32_t *err, cudaStream_t s) {
    Plan pl;
    make_plan(a, pl);
    if (ws_bytes < pl.bytes())
        return fail(PKV_ERR_CAPACITY, "pkv_decode: workspace of %zu bytes, %zu needed", ws_bytes, pl.bytes());
    if (pl.bytes() && (!ws || !aligned(ws, 256)))
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: workspace must be non-null and 256-byte aligned");
    if (static_cast<int64_t>(pl.chunk) * pl.n_chunks_max > INT32_MAX / 2 ||
        static_cast<int64_t>(a->batch) * a->num_kv_heads * pl.hsplit * pl.n_chunks_max > INT32_MAX)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: max_seq_len too large");
    Params p{};
    p.layout = a->layout;
    p.batch = a->batch;
    p.hq = a->num_q_heads;
    p.hkv = a->num_kv_heads;
    p.g = a->num_q_heads / a->num_kv_heads;
    p.gc = pl.gc;
    p.hsplit = pl.hsplit;
    const int ps = a->layout == PKV_LAYOUT_VARLEN ? 1 : a->page_size;
    p.ps_shift = ilog2(ps);
    p.ps_mask = ps - 1;
    p.scale_log2 = a->sm_scale * kLog2e;
    p.chunk = pl.chunk;
    p.n_chunks_max = pl.n_chunks_max;
    p.bt_width = a->block_table_width;
    p.num_slots = a->num_slots;
    p.num_pages = a->num_slots >> p.ps_shift;
    p.k_stride = a->k_row_stride;
    p.v_stride = a->v_row_stride;
    p.kv_indices_len = a->kv_indices_len;
    p.q = static_cast<const uint16_t *>(a->q);
    p.k_pool = static_cast<const uint16_t *>(a->k_pool);
    p.v_pool = static_cast<const uint16_t *>(a->v_pool);
    p.kv_indptr = a->kv_indptr;
    p.kv_indices = a->kv_indices;
    p.kv_last = a->kv_last_page_len;
    p.block_table = a->block_table;
    p.seq_lens = a->seq_lens;
    p.cu_seqlens = a->cu_seqlens;
    p.out = static_cast<uint16_t *>(a->out);
    p.lse = a->lse;
    p.part_o = static_cast<float *>(ws);
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(ws) + pl.part_o_bytes);
    p.spans = pl.spans;
    p.meta = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + pl.part_o_bytes + pl.part_lse_bytes);
    p.err = err;
    p.wait_ns = wait_limit_ns();
    p.r2t = a->req_to_token;
    p.req_pool_idx = a->req_pool_idx;
    p.kv_start = a->kv_start;
    p.r2t_rows = a->r2t_rows;
    p.r2t_stride = a->r2t_row_stride;
    p.r2t_width = a->r2t_width;
    p.k_new = static_cast<const uint16_t *>(a->k_new);
    p.v_new = static_cast<const uint16_t *>(a->v_new);
    // the fused store writes into the caller's pools (documented: writable when k_new is set)
    p.k_pool_w = const_cast<uint16_t *>(p.k_pool);
    p.v_pool_w = const_cast<uint16_t *>(p.v_pool);
    const bool tma = pl.tma;
    p.box_rows = a->layout == PKV_LAYOUT_VARLEN ? kTile : std::min(a->page_size, kTile);
    return a->head_dim_qk == 128 ? launch_d<128>(pl, p, a, tma, s) : launch_d<64>(pl, p, a, tma, s);
}

}  // namespace gqa

// MLA entry points live in decode_mla.cu.
namespace mla {
pkv_status validate(const pkv_decode_args *a, bool check_ptrs);
size_t workspace_size(const pkv_decode_args *a);
pkv_status launch(const pkv_decode_args *a, void *ws, size_t ws_bytes, int32_t *err, cudaStream_t s);
}  // namespace mla

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_size(const pkv_decode_args *args) {
    using namespace pkv;
    if (!args) return 0;
    if (args->kind == PKV_KIND_MLA) return mla::validate(args, false) == PKV_OK ? mla::workspace_size(args) : 0;
    if (args->kind != PKV_KIND_GQA || gqa::validate(args, false) != PKV_OK) return 0;
    return gqa::workspace_size(args);
}

extern "C" pkv_status pkv_decode(const pkv_decode_args *args, void *workspace, size_t workspace_bytes,
                                 int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (!args) return fail(PKV_ERR_INVALID_ARG, "pkv_decode: null args");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_decode: err_flags is required");
    auto s = reinterpret_cast<cudaStream_t>(stream);
    pkv_status st;
    if (args->kind == PKV_KIND_MLA) {
        st = mla::validate(args, true);
        if (st != PKV_OK) return st;
        if (args->batch == 0) return ok();
        return mla::launch(args, workspace, workspace_bytes, err_flags, s);
    }
    if (args->kind != PKV_KIND_GQA) return fail(PKV_ERR_INVALID_ARG, "pkv_decode: unknown kind");
    st = gqa::validate(args, true);
    if (st != PKV_OK) return st;
    if (args->batch == 0) return ok();
    return gqa::launch(args, workspace, workspace_bytes, err_flags, s);
}

// ---------------------------------------------------------------------------
// pkv_decode_no_alloc: GQA/MHA decode whose split-KV scratch is a fixed
// device array inside this library instead of a caller-provided workspace.
//
// Some callers cannot call cudaMalloc at all: code loaded into a host
// process whose device memory is entirely owned by another allocator (for
// example a serving engine that reserved the rest of HBM for its KV pool at
// start-up), or a latency-critical loop where a first-touch allocation could
// block.  For them the partial outputs and log-sum-exp values of the split
// plan live in g_no_alloc_scratch below.  Every GPU that loads this library
// holds the array until the process exits.
namespace pkv {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
__device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

// Device address of the array, resolved once per device.  In host code the
// symbol is only a host-side stand-in, so the kernel must receive this address.
pkv_status no_alloc_scratch_address(void **out) {
    static std::mutex mu;
    static std::vector<void *> by_device;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "pkv_decode_no_alloc: cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(by_device.size())) by_device.resize(dev + 1, nullptr);
    if (!by_device[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(PKV_ERR_CUDA, "pkv_decode_no_alloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        by_device[dev] = p;
    }
    *out = by_device[dev];
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_decode_no_alloc(const pkv_decode_args *args, int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (!args) return fail(PKV_ERR_INVALID_ARG, "pkv_decode_no_alloc: null args");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_decode_no_alloc: err_flags is required");
    if (args->kind != PKV_KIND_GQA)
        return fail(PKV_ERR_UNSUPPORTED, "pkv_decode_no_alloc: only GQA/MHA decode has a built-in scratch");
    pkv_status st = gqa::validate(args, true);
    if (st != PKV_OK) return st;
    if (args->batch == 0) return ok();
    const size_t need = gqa::workspace_size(args);
    if (need > kNoAllocScratchBytes)
        return fail(PKV_ERR_CAPACITY,
                    "pkv_decode_no_alloc: split plan needs %zu bytes of scratch, the built-in array holds %zu "
                    "(use pkv_decode with a caller workspace, or a larger kv_chunk / smaller batch)",
                    need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    st = no_alloc_scratch_address(&scratch);
    if (st != PKV_OK) return st;
    return gqa::launch(args, scratch, kNoAllocScratchBytes, err_flags, reinterpret_cast<cudaStream_t>(stream));
}
