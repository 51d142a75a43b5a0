// Slot bookkeeping on the device: pkv_alloc_extend (the paged allocator's
// alloc_extend / alloc_decode growth path) and pkv_write_req_to_token (the row
// writer, write_cache_indices / write_req_to_token_pool), so a step needs no
// host round trip between scheduling and attention.
//
// Allocation runs in one CTA: every request's page and token counts are
// validated and prefix-summed in shared memory, the whole step is refused
// before anything is written when it does not fit (the allocator's None), and
// then every new position finds its request by binary search and computes its
// slot: the slots after last_loc while the partly used last page lasts, then
// page free_pages[head + P_b + k] for the k-th new page of request b, P_b being
// the new pages of the requests before it.
#include <algorithm>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kAllocThreads = 1024;
constexpr int kWriteThreads = 256;
constexpr int kWriteSpan = 4096;       // row columns per CTA of the row writer

// Bitwise OR of v over the block; every thread gets the result.
__device__ __forceinline__ int block_or(int v, int *scratch32) {
    v = __reduce_or_sync(0xffffffffu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch32[warp] = v;
    __syncthreads();
    int r = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) r |= scratch32[i];
    return r;
}

// Exclusive prefix sums of a[0 .. n) into out[0 .. n], out[n] = total; one block,
// each thread owning a contiguous run of entries.
__device__ void block_scan(const int32_t *a, int32_t *out, int n, int *warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    const int seg = (n + nt - 1) / nt;
    const int lo = min(n, tid * seg), hi = min(n, lo + seg);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += a[i];
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int i = lo; i < hi; ++i) {
        out[i] = run;
        run += a[i];
    }
    if (tid == nt - 1) out[n] = base + incl;
    __syncthreads();
}

__global__ void __launch_bounds__(kAllocThreads)
alloc_extend_kernel(const int32_t *__restrict__ prefix_lens, const int32_t *__restrict__ seq_lens,
                    const int32_t *__restrict__ last_loc, int32_t batch, int32_t ps, int64_t num_pool_pages,
                    const int32_t *__restrict__ free_pages, int64_t free_pages_len, int32_t *__restrict__ free_state,
                    int32_t *__restrict__ out, int64_t out_cap, int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    extern __shared__ int32_t sh[];
    int32_t *pages = sh;                       // [batch] new pages of each request
    int32_t *toks = sh + (batch + 1);          // [batch] new positions of each request
    int32_t *P = toks + (batch + 1);           // exclusive prefix sums of pages, P[batch] = total
    int32_t *E = P + (batch + 1);              // exclusive prefix sums of toks
    __shared__ int ored[32];
    __shared__ int warp_tot[32];
    __shared__ long long red[32];
    const int tid = threadIdx.x;
    int bad = 0;
    long long my_pages = 0, my_toks = 0;
    for (int b = tid; b < batch; b += kAllocThreads) {
        const int64_t p = prefix_lens[b], s = seq_lens[b];
        int np = 0, nt = 0;
        if (p < 0 || s < p || s > INT32_MAX / 2) {
            bad |= PKV_DEVERR_RANGE;
        } else {
            if (p % ps != 0) {   // the partly used page must hold position p - 1 at its offset
                const int64_t ll = last_loc[b];
                if (ll < 0 || ll >= num_pool_pages * ps) bad |= PKV_DEVERR_RANGE;
                else if (ll % ps != (p - 1) % ps) bad |= PKV_DEVERR_CONTIG;
            }
            np = static_cast<int>((s + ps - 1) / ps - (p + ps - 1) / ps);
            nt = static_cast<int>(s - p);
        }
        pages[b] = np;
        toks[b] = nt;
        my_pages += np;
        my_toks += nt;
    }
    bad = block_or(bad, ored);
    const long long total_pages = block_sum(my_pages, red);
    const long long total_toks = block_sum(my_toks, red);
    if (!bad && total_toks > INT32_MAX) bad = PKV_DEVERR_RANGE;
    const int64_t head = free_state[0], count = free_state[1];
    bool fits = total_toks <= out_cap && total_pages <= count && head >= 0 && head + total_pages <= free_pages_len;
    if (!bad && fits) {
        int range = 0;
        for (int64_t k = tid; k < total_pages; k += kAllocThreads) {
            const int32_t pg = free_pages[head + k];
            if (pg < 0 || pg >= num_pool_pages) range = PKV_DEVERR_RANGE;
        }
        bad = block_or(range, ored);
    }
    if (bad || !fits) {   // malformed or does not fit: write nothing, change nothing (uniform branch)
        if (tid == 0) raise_flag(err, bad ? bad : PKV_DEVERR_CAPACITY);
        return;
    }
    block_scan(pages, P, batch, warp_tot);
    block_scan(toks, E, batch, warp_tot);
    for (int64_t o = tid; o < total_toks; o += kAllocThreads) {
        int lo = 0, hi = batch;   // E[lo] <= o < E[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (E[mid] <= o) lo = mid; else hi = mid;
        }
        const int b = lo;
        const int64_t p = prefix_lens[b];
        const int64_t t = p + (o - E[b]);
        const int64_t aligned_p = (p + ps - 1) / ps * ps;
        int64_t slot;
        if (t < aligned_p) slot = static_cast<int64_t>(last_loc[b]) + (t - p + 1);
        else slot = static_cast<int64_t>(free_pages[head + P[b] + (t - aligned_p) / ps]) * ps + t % ps;
        out[o] = static_cast<int32_t>(slot);
    }
    if (tid == 0) {
        free_state[0] = static_cast<int32_t>(head + total_pages);
        free_state[1] = static_cast<int32_t>(count - total_pages);
    }
}

// Grid (request, span of kWriteSpan columns).  CTA (b, c) finds its offset into
// out_cache_loc by summing the extend lengths of the requests before it, then
// writes the columns of its span: prefix slots below prefix_len, new slots above.
__global__ void __launch_bounds__(kWriteThreads)
write_req_to_token_kernel(int32_t *__restrict__ r2t, int64_t r2t_rows, int64_t row_stride, int64_t width,
                          const int32_t *__restrict__ req_pool_idx, const int32_t *__restrict__ kv_start,
                          const int32_t *__restrict__ prefix_lens, const int32_t *__restrict__ seq_lens,
                          const int32_t *const *__restrict__ prefix_slots, const int32_t *__restrict__ out_cache_loc,
                          int32_t batch, int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    __shared__ long long scratch[32];
    const int b = blockIdx.x;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kWriteSpan;
    const int64_t p = prefix_lens[b], s = seq_lens[b];
    const int64_t row = req_pool_idx[b], st = kv_start ? kv_start[b] : 0;
    if (row < 0 || row >= r2t_rows || st < 0 || p < 0 || s < p || st + s > width) {
        if (threadIdx.x == 0 && blockIdx.y == 0) raise_flag(err, PKV_DEVERR_RANGE);
        return;
    }
    if (c0 >= s) return;   // uniform over the CTA
    long long before = 0;
    for (int j = threadIdx.x; j < b; j += kWriteThreads) {
        const int64_t pj = prefix_lens[j], sj = seq_lens[j];
        before += sj > pj ? sj - pj : 0;
    }
    before = block_sum(before, scratch);
    int32_t *dst = r2t + row * row_stride + st;
    const int32_t *pre = prefix_slots ? prefix_slots[b] : nullptr;
    const int64_t c1 = min(s, c0 + kWriteSpan);
    for (int64_t t = c0 + threadIdx.x; t < c1; t += kWriteThreads) {
        if (t < p) {
            if (pre) dst[t] = pre[t];
        } else {
            dst[t] = out_cache_loc[before + (t - p)];
        }
    }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_alloc_extend(const int32_t *prefix_lens, const int32_t *seq_lens, const int32_t *last_loc,
                                       int32_t batch, int32_t page_size, int64_t num_pool_pages,
                                       const int32_t *free_pages, int64_t free_pages_len, int32_t *free_state,
                                       int32_t *out_cache_loc, int64_t out_cap, int32_t *err_flags,
                                       pkv_stream_t stream) {
    using namespace pkv;
    if (batch < 0 || page_size < 1 || num_pool_pages < 0 || free_pages_len < 0 || out_cap < 0)
        return fail(PKV_ERR_INVALID_ARG, "pkv_alloc_extend: negative size");
    if (!err_flags || !free_state) return fail(PKV_ERR_INVALID_ARG, "pkv_alloc_extend: null err_flags or free_state");
    if (batch > 0 && (!prefix_lens || !seq_lens || !last_loc || !out_cache_loc || (free_pages_len > 0 && !free_pages)))
        return fail(PKV_ERR_INVALID_ARG, "pkv_alloc_extend: null input");
    if (batch > 8192) return fail(PKV_ERR_UNSUPPORTED, "pkv_alloc_extend: more than 8192 requests in one step");
    if (num_pool_pages > INT32_MAX / page_size) return fail(PKV_ERR_UNSUPPORTED, "pkv_alloc_extend: pool above 2^31 slots");
    if (batch == 0) return ok();
    const size_t smem = static_cast<size_t>(batch + 1) * 4 * sizeof(int32_t);
    if (smem > 48 * 1024 && cudaFuncSetAttribute(alloc_extend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem)) != cudaSuccess)
        return fail(PKV_ERR_CUDA, "pkv_alloc_extend: cannot raise the shared-memory limit");
    return launch_status(
        launch_chained(alloc_extend_kernel, dim3(1), dim3(kAllocThreads), smem, reinterpret_cast<cudaStream_t>(stream),
                       prefix_lens, seq_lens, last_loc, batch, page_size, num_pool_pages, free_pages, free_pages_len,
                       free_state, out_cache_loc, out_cap, err_flags),
        "pkv_alloc_extend");
}

extern "C" pkv_status pkv_write_req_to_token(int32_t *req_to_token, int64_t r2t_rows, int64_t r2t_row_stride,
                                             int64_t r2t_width, const int32_t *req_pool_idx, const int32_t *kv_start,
                                             const int32_t *prefix_lens, const int32_t *seq_lens,
                                             const int32_t *const *prefix_slots, const int32_t *out_cache_loc,
                                             int32_t batch, int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (batch < 0 || r2t_rows < 0 || r2t_width < 0 || r2t_row_stride < r2t_width)
        return fail(PKV_ERR_INVALID_ARG, "pkv_write_req_to_token: negative or inconsistent size");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_write_req_to_token: err_flags is required");
    if (batch > 0 && (!req_to_token || !req_pool_idx || !prefix_lens || !seq_lens || !out_cache_loc))
        return fail(PKV_ERR_INVALID_ARG, "pkv_write_req_to_token: null input");
    if (batch == 0) return ok();
    const int64_t spans = std::max<int64_t>(1, (r2t_width + kWriteSpan - 1) / kWriteSpan);
    if (spans > 65535) return fail(PKV_ERR_UNSUPPORTED, "pkv_write_req_to_token: rows too wide");
    return launch_status(launch_chained(write_req_to_token_kernel, dim3(batch, static_cast<unsigned>(spans)),
                                        dim3(kWriteThreads), 0, reinterpret_cast<cudaStream_t>(stream), req_to_token,
                                        r2t_rows, r2t_row_stride, r2t_width, req_pool_idx, kv_start, prefix_lens,
                                        seq_lens, prefix_slots, out_cache_loc, batch, err_flags),
                         "pkv_write_req_to_token");
}
