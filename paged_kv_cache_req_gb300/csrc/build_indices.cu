// pkv_build_indices: per-request page lists from the token-granular req_to_token table.
//
// Work items are (request, span): a span is about 2048 positions of one request,
// a whole number of pages, so a long row is read by many CTAs at once rather than
// walked by one.  The grid is persistent (a few CTAs per SM) and every CTA takes
// items w = blockIdx.x, blockIdx.x + gridDim.x, ... in request order.  The
// kv_indptr offset of a request is the sum of the page counts before it: each CTA
// streams the page counts of all requests once, 2048 at a time (eight independent
// loads per thread, then a block-wide scan), carrying the running total, and
// takes its items of those requests with their offsets from shared memory.  The
// whole grid thus reads O(batch x CTAs) counts, linear in the batch, where
// re-summing per item would be quadratic.  Inside a span each thread reads eight
// positions with independent loads; position t compares its slot with the slot of
// its page's first position, which checks page alignment and contiguity ("From
// slots to a page table": the stride-and-divide derivation relies on tokens being
// contiguous inside a page), and the thread owning a page's first position writes
// the page id.
#include <algorithm>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
constexpr int kSpanTarget = kThreads * kUnroll;
constexpr int kChunk = kThreads * kUnroll;     // requests per step of the offset scan

// Positions per CTA: a whole number of pages, close to kSpanTarget.
int64_t span_for(int32_t ps) { return ps >= kSpanTarget ? ps : static_cast<int64_t>(ps) * (kSpanTarget / ps); }

// Exclusive block-wide prefix of one value per thread; *total gets the sum.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long *warp_sums, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const long long x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    long long before = 0, all = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        const long long x = warp_sums[w];
        if (w < warp) before += x;
        all += x;
    }
    *total = all;
    __syncthreads();   // warp_sums may be reused
    return before + incl - v;
}

__global__ void __launch_bounds__(kThreads)
build_indices_kernel(const int32_t *__restrict__ r2t, int64_t r2t_rows, int64_t row_stride, int64_t width,
                     const int32_t *__restrict__ req_pool_idx, const int32_t *__restrict__ seq_lens,
                     const int32_t *__restrict__ kv_start, int32_t batch, int32_t ps, int64_t num_pool_pages,
                     int64_t span, int64_t spans, int32_t *__restrict__ kv_indptr, int32_t *__restrict__ kv_indices,
                     int64_t cap, int32_t *__restrict__ last_page_len, int32_t *__restrict__ block_table,
                     int32_t bt_width, int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    __shared__ long long warp_sums[kThreads / 32];
    __shared__ long long off_s[kChunk];   // kv_indptr offset of each request of the chunk
    if (blockIdx.x == 0 && threadIdx.x == 0 && kv_indptr) kv_indptr[0] = 0;
    if (batch <= 0) return;

    // Page count of request j, or -1 when its row/region lies outside the table
    // (such a request contributes no pages).
    auto pages_of = [&](int j) -> long long {
        const int64_t row = req_pool_idx[j];
        const int64_t s = kv_start ? kv_start[j] : 0;
        const int64_t L = seq_lens[j];
        const bool ok = row >= 0 && row < r2t_rows && s >= 0 && L >= 0 && s + L <= width;
        return ok ? (L + ps - 1) / ps : -1;
    };
    const int64_t items = static_cast<int64_t>(batch) * spans;
    const int64_t pool_slots = num_pool_pages * ps;
    const bool pow2 = (ps & (ps - 1)) == 0;
    const int shift = __ffs(ps) - 1;
    int64_t w = blockIdx.x;
    long long carry = 0;   // pages of the requests before the chunk
    for (int c0 = 0; c0 < batch && w < items; c0 += kChunk) {
        // ---- offsets of requests c0 .. c0 + kChunk - 1: thread i sums requests c0 + 8i .. 8i + 7
        if (kv_indptr) {
            long long n8[kUnroll];
            long long mine = 0;
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int j = c0 + threadIdx.x * kUnroll + k;
                n8[k] = j < batch ? max(pages_of(j), 0LL) : 0;
                mine += n8[k];
            }
            long long total = 0;
            long long run = carry + block_exclusive_scan(mine, warp_sums, &total);
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                off_s[threadIdx.x * kUnroll + k] = run;
                run += n8[k];
            }
            carry += total;
            __syncthreads();
        }
        // ---- this CTA's items of those requests
        for (; w < items && w / spans < c0 + kChunk; w += gridDim.x) {
            const int b = static_cast<int>(w / spans);
            const int64_t c = w % spans;
            const long long n_or_bad = pages_of(b);
            const bool valid = n_or_bad >= 0;
            const long long n = valid ? n_or_bad : 0;
            const int64_t L = valid ? seq_lens[b] : 0;
            const int64_t t_begin = c * span;
            const int64_t t_end = min(L, t_begin + span);
            const int64_t p_begin = t_begin / ps, p_end = (t_begin + span) / ps;
            const long long before = kv_indptr ? off_s[b - c0] : 0;

            if (block_table) {
                const int64_t pad_end = min(static_cast<int64_t>(bt_width), p_end);
                for (int64_t p = max(static_cast<int64_t>(n), p_begin) + threadIdx.x; p < pad_end; p += kThreads)
                    block_table[static_cast<int64_t>(b) * bt_width + p] = -1;
            }
            if (c == 0 && threadIdx.x == 0) {
                if (!valid) raise_flag(err, PKV_DEVERR_RANGE);
                if (kv_indptr) kv_indptr[b + 1] = static_cast<int32_t>(before + n);
                if (last_page_len) last_page_len[b] = L > 0 ? static_cast<int32_t>(L - (n - 1) * ps) : 0;
                if (kv_indices && before + n > cap) raise_flag(err, PKV_DEVERR_CAPACITY);
                if (block_table && n > bt_width) raise_flag(err, PKV_DEVERR_CAPACITY);
            }
            if (t_begin >= t_end) continue;   // nothing of this request in this span

            const int32_t *row = r2t + req_pool_idx[b] * row_stride + (kv_start ? kv_start[b] : 0);
            const int te = static_cast<int>(t_end);  // width <= INT32_MAX (checked on the host)
            int bad = 0;
            for (int base = static_cast<int>(t_begin) + threadIdx.x; base < te; base += kThreads * kUnroll) {
                int32_t slot[kUnroll] = {}, head[kUnroll] = {};
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int t = base + k * kThreads;
                    if (t < te) {
                        const int off = pow2 ? (t & (ps - 1)) : (t % ps);
                        slot[k] = __ldg(row + t);
                        head[k] = __ldg(row + (t - off));  // slot of this page's first position
                    }
                }
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int t = base + k * kThreads;
                    if (t >= te) continue;
                    const int off = pow2 ? (t & (ps - 1)) : (t % ps);
                    const int64_t h = head[k];
                    if (off == 0) {
                        if (h < 0 || h >= pool_slots) {
                            bad |= PKV_DEVERR_RANGE;
                            continue;
                        }
                        if ((pow2 ? (h & (ps - 1)) : (h % ps)) != 0) bad |= PKV_DEVERR_CONTIG;
                        const int pg = pow2 ? (t >> shift) : (t / ps);
                        const int32_t page = static_cast<int32_t>(pow2 ? (h >> shift) : (h / ps));
                        if (kv_indices && before + pg < cap) kv_indices[before + pg] = page;
                        if (block_table && pg < bt_width) block_table[static_cast<int64_t>(b) * bt_width + pg] = page;
                    } else if (slot[k] != h + off) {
                        bad |= PKV_DEVERR_CONTIG;
                    }
                }
            }
            if (bad) raise_flag(err, bad);
        }
        __syncthreads();   // off_s is rewritten by the next chunk
    }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_build_indices(const int32_t *req_to_token, int64_t r2t_rows, int64_t r2t_row_stride,
                                        int64_t r2t_width, const int32_t *req_pool_idx, const int32_t *seq_lens,
                                        const int32_t *kv_start, int32_t batch, int32_t page_size,
                                        int64_t num_pool_pages, int32_t *kv_indptr, int32_t *kv_indices,
                                        int64_t kv_indices_cap, int32_t *kv_last_page_len, int32_t *block_table,
                                        int32_t block_table_width, int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (batch < 0 || page_size < 1 || r2t_rows < 0 || r2t_width < 0 || r2t_row_stride < r2t_width ||
        num_pool_pages < 0 || kv_indices_cap < 0 || block_table_width < 0)
        return fail(PKV_ERR_INVALID_ARG, "pkv_build_indices: negative or inconsistent size");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_build_indices: err_flags is required");
    const bool csr = kv_indptr || kv_indices || kv_last_page_len;
    if (csr && !(kv_indptr && kv_indices && kv_last_page_len))
        return fail(PKV_ERR_INVALID_ARG, "pkv_build_indices: kv_indptr, kv_indices, kv_last_page_len go together");
    if (!csr && !block_table) return fail(PKV_ERR_INVALID_ARG, "pkv_build_indices: no output requested");
    if (batch > 0 && (!req_to_token || !req_pool_idx || !seq_lens))
        return fail(PKV_ERR_INVALID_ARG, "pkv_build_indices: null input table");
    if (num_pool_pages > INT32_MAX) return fail(PKV_ERR_UNSUPPORTED, "pkv_build_indices: more than 2^31 pages");
    if (r2t_width > INT32_MAX) return fail(PKV_ERR_UNSUPPORTED, "pkv_build_indices: rows wider than 2^31 columns");
    // Spans cover every position a row can hold and every block-table column.
    const int64_t span = span_for(page_size);
    const int64_t covered = std::max<int64_t>(r2t_width, static_cast<int64_t>(block_table_width) * page_size);
    const int64_t spans = std::max<int64_t>(1, (covered + span - 1) / span);
    // Persistent grid: at most 8 CTAs per SM, each streaming the batch's page counts once.
    const int64_t items = static_cast<int64_t>(std::max(batch, 1)) * spans;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(items, 8ll * std::max(1, sm_count())));
    return launch_status(launch_chained(build_indices_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0,
                                        reinterpret_cast<cudaStream_t>(stream), req_to_token, r2t_rows, r2t_row_stride,
                                        r2t_width, req_pool_idx, seq_lens, kv_start, batch, page_size, num_pool_pages,
                                        span, spans, kv_indptr, kv_indices, kv_indices_cap, kv_last_page_len,
                                        block_table, block_table_width, err_flags),
                         "pkv_build_indices");
}
