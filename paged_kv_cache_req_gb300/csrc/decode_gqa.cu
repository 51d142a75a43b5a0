// pkv_decode for GQA / MHA: one query token per request attending through a page table.
//
// Work decomposition (split-KV): a work item is (request b, key chunk c, kv head
// kh, head slice hs).  It covers keys [c*chunk, min(L, (c+1)*chunk)) of kv head kh
// for up to 4 of the query heads that share kh, so every K/V tile is read from
// HBM once for the whole GQA group.  Items are ordered request-major with the
// kv heads of one chunk adjacent (they read the same pool pages) and are
// handed out round-robin to a persistent grid of SM-count x occupancy CTAs;
// each CTA derives the item list from the lengths in its prologue, so no host
// synchronisation is needed.
//
// Inside an item, 64-key tiles of K and V stream through a 3-stage cp.async
// pipeline (16-byte chunks; 16 lanes cover one 256-byte row, so a warp copies
// two rows per instruction).  The slot of key t is
// page_table[b][t / ps] * ps + t % ps ("From slots to a page table").  Each
// warp takes 16 keys of a tile; 8 lanes share a key (each lane owns 16 of the
// 128 dims), reduce q.k with three xor-shuffles, and keep their own online-
// softmax state (base-2, scale * log2 e folded into q).  States are combined
// across lane groups and warps at the end of the item.  A request with one
// chunk writes bf16 output directly; longer ones write fp32 partials and their
// log-sum-exp, combined by merge_kernel.
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
constexpr int kMaxGc = 4;   // query heads per CTA
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;

struct Params {
    int32_t layout;
    int32_t batch, hq, hkv, g, gc, hsplit;
    int32_t ps_shift, ps_mask;
    float scale_log2;
    int32_t chunk, n_chunks_max;
    int32_t bt_width;
    int64_t num_slots, num_pages, k_stride, v_stride, kv_indices_len;
    const uint16_t *q, *k_pool, *v_pool;
    const int32_t *kv_indptr, *kv_indices, *kv_last, *block_table, *seq_lens, *cu_seqlens;
    uint16_t *out;
    float *lse;
    float *part_o, *part_lse;
    int32_t *err;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Key count of request b (clamped to what its page table can address) and the
// base offset of its page list.
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
    const int64_t limit = min(cap, static_cast<int64_t>(p.chunk) * p.n_chunks_max);
    if (L < 0 || L > limit) {
        if (report) raise_flag(p.err, L < 0 ? PKV_DEVERR_RANGE : PKV_DEVERR_CAPACITY);
        L = L < 0 ? 0 : limit;
    }
    return static_cast<int>(L);
}

__device__ __forceinline__ int64_t slot_of(const Params &p, int64_t base, int t) {
    if (p.layout == PKV_LAYOUT_VARLEN) {
        const int64_t s = base + t;
        return (s >= 0 && s < p.num_slots) ? s : -1;
    }
    const int32_t *tab = p.layout == PKV_LAYOUT_CSR ? p.kv_indices : p.block_table;
    const int page = __ldg(tab + base + (t >> p.ps_shift));
    if (page < 0 || page >= p.num_pages) return -1;
    return (static_cast<int64_t>(page) << p.ps_shift) + (t & p.ps_mask);
}

template <int D>
struct Smem {
    static constexpr int kRowElems = D;                         // one kv head of one key
    static constexpr int kTileElems = kTile * D;
    static constexpr int kStageBytes = 2 * kTileElems * 2;       // K + V
    static constexpr int kRedOBytes = kWarps * kMaxGc * D * 4;
    static constexpr int kFixedBytes = kStages * kStageBytes + kRedOBytes + 2 * kWarps * kMaxGc * 4;
};

// Issue the cp.async copies of one 64-key tile (K and V) of kv head kh.
template <int D>
__device__ __forceinline__ void load_tile(const Params &p, uint16_t *ks, uint16_t *vs, int64_t base, int t0, int t1,
                                          int kh) {
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
            if (slot < 0 && chunk == 0) raise_flag(p.err, PKV_DEVERR_RANGE);
        }
        const bool ok = slot >= 0;
        const uint16_t *ksrc = ok ? p.k_pool + slot * p.k_stride + kh * D + chunk * 8 : p.k_pool;
        const uint16_t *vsrc = ok ? p.v_pool + slot * p.v_stride + kh * D + chunk * 8 : p.v_pool;
        cp_async_16(ks + key * D + chunk * 8, ksrc, ok ? 16 : 0);
        cp_async_16(vs + key * D + chunk * 8, vsrc, ok ? 16 : 0);
    }
}

template <int D, int GC>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const Params p) {
    constexpr int NC = D / 64;  // 16-byte chunks per lane: chunk index part + 8*ci
    using S = Smem<D>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint16_t *tiles = reinterpret_cast<uint16_t *>(smem);
    float *red_o = reinterpret_cast<float *>(smem + kStages * S::kStageBytes);
    float *red_m = red_o + kWarps * kMaxGc * D;
    float *red_l = red_m + kWarps * kMaxGc;
    int *off = reinterpret_cast<int *>(red_l + kWarps * kMaxGc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 3, part = lane & 7;
    const int per_chunk = p.hkv * p.hsplit;

    // ---- prologue: item offsets off[b] = sum_{j<b} items(j) (exclusive scan) ----
    {
        const int B = p.batch;
        const int seg = (B + kThreads - 1) / kThreads;
        const int lo = min(B, tid * seg), hi = min(B, lo + seg);
        int local = 0;
        for (int b = lo; b < hi; ++b) {
            int64_t base;
            const int L = key_count(p, b, base, false);
            local += max(1, (L + p.chunk - 1) / p.chunk) * per_chunk;
        }
        int incl = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) red_m[warp] = __int_as_float(incl);
        __syncthreads();
        int wbase = 0;
        for (int w = 0; w < warp; ++w) wbase += __float_as_int(red_m[w]);
        int run = wbase + incl - local;
        for (int b = lo; b < hi; ++b) {
            off[b] = run;
            int64_t base;
            const int L = key_count(p, b, base, false);
            run += max(1, (L + p.chunk - 1) / p.chunk) * per_chunk;
        }
        if (tid == kThreads - 1) off[B] = wbase + incl;
        __syncthreads();
    }
    const int total = off[p.batch];

    for (int w = blockIdx.x; w < total; w += gridDim.x) {
        // ---- locate the item ----
        int lo = 0, hi = p.batch;  // find b with off[b] <= w < off[b+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (off[mid] <= w) lo = mid; else hi = mid;
        }
        const int b = lo;
        int rem = w - off[b];
        const int hs = rem % p.hsplit;
        rem /= p.hsplit;
        const int kh = rem % p.hkv;
        const int c = rem / p.hkv;
        int64_t base;
        const int L = key_count(p, b, base, tid == 0 && c == 0 && kh == 0 && hs == 0);
        const int n_chunks = max(1, (L + p.chunk - 1) / p.chunk);
        const int head0 = kh * p.g + hs * GC;
        const int t_begin = c * p.chunk;
        const int t_end = min(L, t_begin + p.chunk);

        if (t_end <= t_begin) {  // empty request: zero output, lse = -inf
            for (int i = tid; i < GC * D; i += kThreads) {
                const int h = i / D, d = i % D;
                p.out[(static_cast<int64_t>(b) * p.hq + head0 + h) * D + d] = 0;
                if (d == 0 && p.lse) p.lse[static_cast<int64_t>(b) * p.hq + head0 + h] = -INFINITY;
            }
            continue;
        }

        // ---- q slice in registers, pre-scaled into the base-2 domain ----
        float qr[GC][NC][8];
#pragma unroll
        for (int h = 0; h < GC; ++h)
#pragma unroll
            for (int ci = 0; ci < NC; ++ci) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
                    p.q + (static_cast<int64_t>(b) * p.hq + head0 + h) * D + (part + 8 * ci) * 8));
                widen8(raw, qr[h][ci]);
#pragma unroll
                for (int e = 0; e < 8; ++e) qr[h][ci][e] *= p.scale_log2;
            }
        float o[GC][NC][8];
        float m[GC], l[GC];
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][ci][e] = 0.f;
        }

        // ---- pipelined tile loop ----
        const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;
#pragma unroll
        for (int s = 0; s < kStages - 1; ++s) {
            if (s < n_tiles) {
                uint16_t *ks = tiles + s * 2 * S::kTileElems;
                load_tile<D>(p, ks, ks + S::kTileElems, base, t_begin + s * kTile, t_end, kh);
            }
            cp_async_commit();
        }
        for (int it = 0; it < n_tiles; ++it) {
            cp_async_wait<kStages - 2>();
            __syncthreads();
            {
                const int nt = it + kStages - 1;
                if (nt < n_tiles) {
                    uint16_t *ks = tiles + (nt % kStages) * 2 * S::kTileElems;
                    load_tile<D>(p, ks, ks + S::kTileElems, base, t_begin + nt * kTile, t_end, kh);
                }
                cp_async_commit();
            }
            const uint16_t *ks = tiles + (it % kStages) * 2 * S::kTileElems;
            const uint16_t *vs = ks + S::kTileElems;
            const int n_valid = t_end - (t_begin + it * kTile);

            float s[4][GC];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = warp * 16 + j * 4 + grp;
#pragma unroll
                for (int h = 0; h < GC; ++h) s[j][h] = 0.f;
#pragma unroll
                for (int ci = 0; ci < NC; ++ci) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(ks + key * D + (part + 8 * ci) * 8);
                    float kf[8];
                    widen8(raw, kf);
#pragma unroll
                    for (int h = 0; h < GC; ++h)
#pragma unroll
                        for (int e = 0; e < 8; ++e) s[j][h] = fmaf(qr[h][ci][e], kf[e], s[j][h]);
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
                if (mt > m[h]) {
                    const float corr = ex2(m[h] - mt);  // m = -inf gives 0
                    l[h] *= corr;
#pragma unroll
                    for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[h][ci][e] *= corr;
                    m[h] = mt;
                }
                const bool live = m[h] != -INFINITY;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[j][h] = live ? ex2(s[j][h] - m[h]) : 0.f;
                    l[h] += s[j][h];
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = warp * 16 + j * 4 + grp;
#pragma unroll
                for (int ci = 0; ci < NC; ++ci) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(vs + key * D + (part + 8 * ci) * 8);
                    float vf[8];
                    widen8(raw, vf);
#pragma unroll
                    for (int h = 0; h < GC; ++h)
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[h][ci][e] = fmaf(s[j][h], vf[e], o[h][ci][e]);
                }
            }
        }
        cp_async_wait<0>();

        // ---- combine the four lane groups of each warp ----
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            float mw = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], 8));
            mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
            const float corr = (m[h] == -INFINITY) ? 0.f : ex2(m[h] - mw);
            float lw = l[h] * corr;
            lw += __shfl_xor_sync(0xffffffffu, lw, 8);
            lw += __shfl_xor_sync(0xffffffffu, lw, 16);
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float v = o[h][ci][e] * corr;
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    o[h][ci][e] = v;
                }
            m[h] = mw;
            l[h] = lw;
        }
        if (grp == 0) {
#pragma unroll
            for (int h = 0; h < GC; ++h) {
#pragma unroll
                for (int ci = 0; ci < NC; ++ci)
#pragma unroll
                    for (int e = 0; e < 8; ++e) red_o[(warp * kMaxGc + h) * D + (part + 8 * ci) * 8 + e] = o[h][ci][e];
                if (part == 0) {
                    red_m[warp * kMaxGc + h] = m[h];
                    red_l[warp * kMaxGc + h] = l[h];
                }
            }
        }
        __syncthreads();

        // ---- combine warps and write ----
        const int64_t pidx = ((static_cast<int64_t>(b) * p.hkv + kh) * p.hsplit + hs) * p.n_chunks_max + c;
        for (int i = tid; i < GC * D; i += kThreads) {
            const int h = i / D, d = i % D;
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, red_m[ww * kMaxGc + h]);
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
                const float mw = red_m[ww * kMaxGc + h];
                const float sc = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                num = fmaf(red_o[(ww * kMaxGc + h) * D + d], sc, num);
                den = fmaf(red_l[ww * kMaxGc + h], sc, den);
            }
            const float val = num / den;
            if (n_chunks == 1) {
                p.out[(static_cast<int64_t>(b) * p.hq + head0 + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
                if (d == 0 && p.lse) p.lse[static_cast<int64_t>(b) * p.hq + head0 + h] = (M + log2f(den)) * kLn2;
            } else {
                p.part_o[(pidx * GC + h) * D + d] = val;
                if (d == 0) p.part_lse[pidx * GC + h] = M + log2f(den);
            }
        }
        __syncthreads();
    }
}

// Log-sum-exp merge of a request's chunk partials (base-2 lse inside the workspace).
template <int D, int GC>
__global__ void __launch_bounds__(kThreads) merge_kernel(const Params p) {
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
    __shared__ float den_s[kMaxGc], mx_s[kMaxGc];
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
        for (int c = 0; c < n; ++c) acc = fmaf(wsm[h * p.n_chunks_max + c], p.part_o[((pbase + c) * GC + h) * D + d], acc);
        acc /= den_s[h];
        p.out[(static_cast<int64_t>(b) * p.hq + head0 + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        if (d == 0 && p.lse) p.lse[static_cast<int64_t>(b) * p.hq + head0 + h] = (mx_s[h] + log2f(den_s[h])) * kLn2;
    }
}

// ------------------------------------------------------------------ host side
struct Plan {
    int gc, hsplit, chunk, n_chunks_max;
    size_t part_o_bytes, part_lse_bytes;
};

static int choose_chunk(const pkv_decode_args *a, int units) {
    // Largest chunk (<= 1024 keys) that still gives ~4 waves of work when the
    // requests average half of max_seq_len.
    const int64_t target = 4ll * std::max(1, sm_count()) * 2;
    const int64_t L = std::max<int64_t>(1, a->max_seq_len);
    for (int c = 1024; c > kTile; c >>= 1) {
        const int64_t items = static_cast<int64_t>(a->batch) * units * ((L + c - 1) / c);
        if (items / 2 >= target) return c;
    }
    return kTile;
}

static pkv_status make_plan(const pkv_decode_args *a, Plan &pl) {
    const int g = a->num_q_heads / a->num_kv_heads;
    pl.gc = std::min(g, kMaxGc);
    pl.hsplit = g / pl.gc;
    pl.chunk = a->kv_chunk > 0 ? a->kv_chunk : choose_chunk(a, a->num_kv_heads * pl.hsplit);
    pl.n_chunks_max = std::max(1, (a->max_seq_len + pl.chunk - 1) / pl.chunk);
    if (pl.n_chunks_max == 1) {
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
        default:
            return fail(PKV_ERR_INVALID_ARG, "pkv_decode: unknown layout");
    }
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
    return pl.part_o_bytes + pl.part_lse_bytes;
}

template <int D, int GC>
static pkv_status launch_t(const Params &p, cudaStream_t s) {
    using S = Smem<D>;
    const size_t smem = S::kFixedBytes + (static_cast<size_t>(p.batch) + 1) * 4;
    static int configured_smem = 0;
    if (configured_smem < 227 * 1024) {
        if (cudaFuncSetAttribute(decode_kernel<D, GC>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
            cudaSuccess)
            return fail(PKV_ERR_CUDA, "pkv_decode: cannot raise the shared-memory limit");
        configured_smem = 227 * 1024;
    }
    if (smem > 227 * 1024) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: batch too large for the on-chip item table");
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel<D, GC>, kThreads, smem) != cudaSuccess ||
        occ < 1)
        occ = 1;
    const int64_t upper = static_cast<int64_t>(p.batch) * p.hkv * p.hsplit * p.n_chunks_max;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(upper, static_cast<int64_t>(sm_count()) * occ)));
    decode_kernel<D, GC><<<grid, kThreads, smem, s>>>(p);
    pkv_status st = check_launch("pkv_decode(GQA split kernel)");
    if (st != PKV_OK || p.n_chunks_max == 1) return st;
    const size_t msmem = static_cast<size_t>(GC) * p.n_chunks_max * 4;
    if (msmem > 200 * 1024) return fail(PKV_ERR_UNSUPPORTED, "pkv_decode: too many splits for the merge");
    if (msmem > 48 * 1024) {
        if (cudaFuncSetAttribute(merge_kernel<D, GC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(std::min<size_t>(msmem, 227 * 1024))) != cudaSuccess)
            return fail(PKV_ERR_CUDA, "pkv_decode: cannot raise the merge shared-memory limit");
    }
    merge_kernel<D, GC><<<p.batch * p.hkv * p.hsplit, kThreads, msmem, s>>>(p);
    return check_launch("pkv_decode(GQA merge kernel)");
}

pkv_status launch(const pkv_decode_args *a, void *ws, size_t ws_bytes, int32_t *err, cudaStream_t s) {
    Plan pl;
    make_plan(a, pl);
    if (ws_bytes < pl.part_o_bytes + pl.part_lse_bytes)
        return fail(PKV_ERR_CAPACITY, "pkv_decode: workspace of %zu bytes, %zu needed", ws_bytes,
                    pl.part_o_bytes + pl.part_lse_bytes);
    if (pl.part_o_bytes && (!ws || !aligned(ws, 256)))
        return fail(PKV_ERR_INVALID_ARG, "pkv_decode: workspace must be non-null and 256-byte aligned");
    if (static_cast<int64_t>(pl.chunk) * pl.n_chunks_max > INT32_MAX / 2)
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
    p.err = err;
    const int D = a->head_dim_qk;
    if (D == 128) {
        if (pl.gc == 1) return launch_t<128, 1>(p, s);
        if (pl.gc == 2) return launch_t<128, 2>(p, s);
        return launch_t<128, 4>(p, s);
    }
    if (pl.gc == 1) return launch_t<64, 1>(p, s);
    if (pl.gc == 2) return launch_t<64, 2>(p, s);
    return launch_t<64, 4>(p, s);
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
