// Row movement: pkv_store (scatter new K/V rows into pool slots),
// pkv_ragged_gather (pack token-granular K/V rows into contiguous varlen buffers)
// and pkv_encoder_merge (gather encoder-cache blocks into positioned hidden rows).
//
// All three are pure indexed copies of whole rows.  One warp moves one row with
// 16-byte vector accesses (the mini-sglang store kernel's "one warp per token,
// 16 bytes per move"); every row start is checked to be 16-byte aligned on the
// host, otherwise a 2-byte element path is used.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kStoreThreads = 256;
constexpr int kGatherThreads = 256;

// Copies `elems` bf16 elements from src to dst with one warp.
template <bool kVec>
__device__ __forceinline__ void warp_copy_row(uint16_t *__restrict__ dst, const uint16_t *__restrict__ src,
                                              int64_t elems, int lane) {
    if (kVec) {
        const int64_t n16 = elems / 8;
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (int64_t i = lane; i < n16; i += 32) st_stream_16(d + i, ld_stream_16(s + i));
    } else {
        for (int64_t i = lane; i < elems; i += 32) dst[i] = src[i];
    }
}

template <bool kVec>
__global__ void __launch_bounds__(kStoreThreads)
store_kernel(uint16_t *__restrict__ k_pool, uint16_t *__restrict__ v_pool, int64_t num_slots, int64_t k_stride,
             int64_t v_stride, int64_t k_elems, int64_t v_elems, const uint16_t *__restrict__ k_new,
             const uint16_t *__restrict__ v_new, const int32_t *__restrict__ slot_mapping, int32_t n,
             int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    const int warp = (blockIdx.x * kStoreThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int rows_per_token = v_pool ? 2 : 1;
    if (warp >= n * rows_per_token) return;
    const int i = warp / rows_per_token;
    const bool is_v = (warp % rows_per_token) == 1;
    const int64_t slot = slot_mapping[i];
    if (slot < 0) return;  // padded token
    if (slot >= num_slots) {
        if (lane == 0 && !is_v) raise_flag(err, PKV_DEVERR_RANGE);
        return;
    }
    if (is_v)
        warp_copy_row<kVec>(v_pool + slot * v_stride, v_new + i * v_elems, v_elems, lane);
    else
        warp_copy_row<kVec>(k_pool + slot * k_stride, k_new + i * k_elems, k_elems, lane);
}

// Zeroes `elems` bf16 elements at dst with one warp.
template <bool kVec>
__device__ __forceinline__ void warp_zero_row(uint16_t *__restrict__ dst, int64_t elems, int lane) {
    if (kVec) {
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (int64_t i = lane; i < elems / 8; i += 32) st_stream_16(d + i, make_uint4(0, 0, 0, 0));
    } else {
        for (int64_t i = lane; i < elems; i += 32) dst[i] = 0;
    }
}

constexpr int kGatherChunk = kGatherThreads * 8;   // requests per step of the offset scan

// Exclusive block-wide prefix of one value per thread; *total gets the sum.
__device__ __forceinline__ long long gather_block_scan(long long v, long long *warp_sums, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
    for (int o = 1; o < 32; o <<= 1) {
        const long long x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    long long before = 0, all = 0;
    for (int w = 0; w < kGatherThreads / 32; ++w) {
        const long long x = warp_sums[w];
        if (w < warp) before += x;
        all += x;
    }
    *total = all;
    __syncthreads();
    return before + incl - v;
}

// Work items are (request b, split y); the grid is persistent and every CTA takes
// items blockIdx.x, blockIdx.x + gridDim.x, ... in request order.  cu_seqlens[b] is
// the sum of the lengths before b: each CTA streams all lengths once, 2048 at a
// time, carrying the running total (linear in the batch over the whole grid).  The
// warps of item (b, y) copy rows t = y*W + w, y*W + w + splits*W, ... of request b.
// A request whose row or region lies outside the table, and a slot outside the
// pool, raise PKV_DEVERR_RANGE and leave zeros in the rows reserved for them, as a
// bad key reads as zeros in pkv_decode.
template <bool kVec>
__global__ void __launch_bounds__(kGatherThreads)
ragged_gather_kernel(const uint16_t *__restrict__ k_pool, const uint16_t *__restrict__ v_pool, int64_t num_slots,
                     int64_t pool_stride, int64_t row_elems, const int32_t *__restrict__ r2t, int64_t r2t_rows,
                     int64_t row_stride, int64_t width, const int32_t *__restrict__ req_pool_idx,
                     const int32_t *__restrict__ kv_start, const int32_t *__restrict__ seq_lens, int32_t batch,
                     int64_t splits, uint16_t *__restrict__ k_out, uint16_t *__restrict__ v_out, int64_t cap,
                     int32_t *__restrict__ cu_seqlens, int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    __shared__ long long warp_sums[kGatherThreads / 32];
    __shared__ long long off_s[kGatherChunk];
    if (blockIdx.x == 0 && threadIdx.x == 0) cu_seqlens[0] = 0;
    if (batch <= 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int W = kGatherThreads / 32;
    const int64_t items = static_cast<int64_t>(batch) * splits;
    int64_t w = blockIdx.x;
    long long carry = 0;
    for (int c0 = 0; c0 < batch && w < items; c0 += kGatherChunk) {
        long long n8[8];
        long long mine = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int j = c0 + threadIdx.x * 8 + k;
            n8[k] = j < batch ? max(seq_lens[j], 0) : 0;
            mine += n8[k];
        }
        long long total = 0;
        long long run = carry + gather_block_scan(mine, warp_sums, &total);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            off_s[threadIdx.x * 8 + k] = run;
            run += n8[k];
        }
        carry += total;
        __syncthreads();
        for (; w < items && w / splits < c0 + kGatherChunk; w += gridDim.x) {
            const int b = static_cast<int>(w / splits);
            const int64_t y = w % splits;
            const long long before = off_s[b - c0];
            const int64_t row = req_pool_idx[b];
            const int64_t s = kv_start ? kv_start[b] : 0;
            int64_t L = max(seq_lens[b], 0);
            const bool valid = row >= 0 && row < r2t_rows && s >= 0 && s + L <= width && seq_lens[b] >= 0;
            if (y == 0 && threadIdx.x == 0) {
                cu_seqlens[b + 1] = static_cast<int32_t>(before + L);
                if (before + L > cap) raise_flag(err, PKV_DEVERR_CAPACITY);
                if (!valid) raise_flag(err, PKV_DEVERR_RANGE);
            }
            if (before + L > cap) L = cap > before ? cap - before : 0;
            const int32_t *rrow = valid ? r2t + row * row_stride + s : nullptr;
            for (int64_t t = y * W + warp; t < L; t += splits * W) {
                const int64_t o = before + t;
                const int64_t slot = valid ? __ldg(rrow + t) : -1;
                if (slot < 0 || slot >= num_slots) {
                    if (valid && lane == 0) raise_flag(err, PKV_DEVERR_RANGE);
                    warp_zero_row<kVec>(k_out + o * row_elems, row_elems, lane);
                    if (v_pool) warp_zero_row<kVec>(v_out + o * row_elems, row_elems, lane);
                    continue;
                }
                warp_copy_row<kVec>(k_out + o * row_elems, k_pool + slot * pool_stride, row_elems, lane);
                if (v_pool) warp_copy_row<kVec>(v_out + o * row_elems, v_pool + slot * pool_stride, row_elems, lane);
            }
        }
        __syncthreads();   // off_s is rewritten by the next chunk
    }
}

constexpr int kMergeThreads = 256;

// One warp per (block slot i, token j) of the position map: position
// positions[i][j] in [0, num_tokens) receives row j of block block_ids[i];
// sentinel positions (>= num_tokens) write nothing.  Rows move as 16-byte
// streaming vectors, four per lane in flight (or bytes when unaligned).
template <bool kVec>
__global__ void __launch_bounds__(kMergeThreads, 4)
encoder_merge_kernel(const uint8_t *__restrict__ buffer, int64_t num_blocks, int64_t block_size, int64_t row_bytes,
                     const int32_t *__restrict__ block_ids, const int64_t *__restrict__ positions, int64_t entries,
                     uint8_t *__restrict__ hidden, int64_t num_tokens, int64_t hidden_stride,
                     unsigned long long *__restrict__ filled, int32_t *__restrict__ err) {
    pdl_wait();          // inputs may come from the previous kernel of the stream
    pdl_launch_next();
    __shared__ int cnt;
    if (threadIdx.x == 0) cnt = 0;
    __syncthreads();
    const int64_t e = static_cast<int64_t>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (e < entries) {
        const int64_t pos = positions[e];
        if (pos < num_tokens) {
            const int64_t i = e / block_size, j = e % block_size;
            const int64_t blk = block_ids[i];
            if (pos < 0 || blk < 0 || blk >= num_blocks) {
                if (lane == 0) raise_flag(err, PKV_DEVERR_RANGE);
            } else {
                const uint8_t *src = buffer + (blk * block_size + j) * row_bytes;
                uint8_t *dst = hidden + pos * hidden_stride;
                if (kVec) {
                    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
                    const int64_t n16 = row_bytes >> 4;
                    int64_t k = lane;
                    for (; k + 96 < n16; k += 128) {
                        uint4 v[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) v[u] = ld_stream_16(s4 + k + 32 * u);
#pragma unroll
                        for (int u = 0; u < 4; ++u) st_stream_16(d4 + k + 32 * u, v[u]);
                    }
                    for (; k < n16; k += 32) st_stream_16(d4 + k, ld_stream_16(s4 + k));
                } else {
                    for (int64_t k = lane; k < row_bytes; k += 32) dst[k] = src[k];
                }
                if (lane == 0) atomicAdd(&cnt, 1);
            }
        }
    }
    if (!filled) return;
    __syncthreads();
    if (threadIdx.x == 0 && cnt) atomicAdd(filled, static_cast<unsigned long long>(cnt));
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_store(void *k_pool, void *v_pool, int64_t num_slots, int64_t k_row_stride,
                                int64_t v_row_stride, int32_t kv_heads, int32_t head_dim_k, int32_t head_dim_v,
                                const void *k_new, const void *v_new, const int32_t *slot_mapping,
                                int32_t n_tokens, int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (n_tokens < 0 || num_slots < 0 || kv_heads < 1 || head_dim_k < 1 || (v_pool && head_dim_v < 1))
        return fail(PKV_ERR_INVALID_ARG, "pkv_store: bad sizes");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_store: err_flags is required");
    if (n_tokens == 0) return ok();
    if (!k_pool || !k_new || !slot_mapping) return fail(PKV_ERR_INVALID_ARG, "pkv_store: null pointer");
    if ((v_pool == nullptr) != (v_new == nullptr))
        return fail(PKV_ERR_INVALID_ARG, "pkv_store: v_pool and v_new must both be set or both be NULL");
    const int64_t k_elems = static_cast<int64_t>(kv_heads) * head_dim_k;
    const int64_t v_elems = v_pool ? static_cast<int64_t>(kv_heads) * head_dim_v : 0;
    if (k_row_stride < k_elems || (v_pool && v_row_stride < v_elems))
        return fail(PKV_ERR_INVALID_ARG, "pkv_store: row stride smaller than a row");
    const bool vec = aligned(k_pool, 16) && aligned(k_new, 16) && k_elems % 8 == 0 && k_row_stride % 8 == 0 &&
                     (!v_pool || (aligned(v_pool, 16) && aligned(v_new, 16) && v_elems % 8 == 0 &&
                                  v_row_stride % 8 == 0));
    const int64_t warps = static_cast<int64_t>(n_tokens) * (v_pool ? 2 : 1);
    const int64_t blocks = (warps * 32 + kStoreThreads - 1) / kStoreThreads;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    auto kp = static_cast<uint16_t *>(k_pool), vp = static_cast<uint16_t *>(v_pool);
    auto kn = static_cast<const uint16_t *>(k_new), vn = static_cast<const uint16_t *>(v_new);
    if (vec)
        return launch_status(launch_chained(store_kernel<true>, dim3(blocks), dim3(kStoreThreads), 0, s, kp, vp,
                                            num_slots, k_row_stride, v_row_stride, k_elems, v_elems, kn, vn,
                                            slot_mapping, n_tokens, err_flags),
                             "pkv_store");
    return launch_status(launch_chained(store_kernel<false>, dim3(blocks), dim3(kStoreThreads), 0, s, kp, vp, num_slots,
                                        k_row_stride, v_row_stride, k_elems, v_elems, kn, vn, slot_mapping, n_tokens,
                                        err_flags),
                         "pkv_store");
}

extern "C" pkv_status pkv_ragged_gather(const void *k_pool, const void *v_pool, int64_t num_slots,
                                        int64_t pool_row_stride, int64_t row_elems, const int32_t *req_to_token,
                                        int64_t r2t_rows, int64_t r2t_row_stride, int64_t r2t_width,
                                        const int32_t *req_pool_idx, const int32_t *kv_start,
                                        const int32_t *seq_lens, int32_t batch, int32_t max_seq_len, void *k_out,
                                        void *v_out, int64_t out_rows_cap, int32_t *cu_seqlens,
                                        int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (batch < 0 || num_slots < 0 || row_elems < 1 || pool_row_stride < row_elems || r2t_rows < 0 ||
        r2t_width < 0 || r2t_row_stride < r2t_width || out_rows_cap < 0 || max_seq_len < 0)
        return fail(PKV_ERR_INVALID_ARG, "pkv_ragged_gather: bad sizes");
    if (!err_flags || !cu_seqlens) return fail(PKV_ERR_INVALID_ARG, "pkv_ragged_gather: null err_flags/cu_seqlens");
    if (batch > 0 && (!k_pool || !k_out || !req_to_token || !req_pool_idx || !seq_lens))
        return fail(PKV_ERR_INVALID_ARG, "pkv_ragged_gather: null pointer");
    if ((v_pool == nullptr) != (v_out == nullptr))
        return fail(PKV_ERR_INVALID_ARG, "pkv_ragged_gather: v_pool and v_out must both be set or both be NULL");
    const bool vec = aligned(k_pool, 16) && aligned(k_out, 16) && row_elems % 8 == 0 && pool_row_stride % 8 == 0 &&
                     (!v_pool || (aligned(v_pool, 16) && aligned(v_out, 16)));
    // Enough CTAs to cover ~2 waves of the device even for a handful of long requests.
    const int warps_per_cta = kGatherThreads / 32;
    int64_t splits = (static_cast<int64_t>(max_seq_len) + warps_per_cta * 4 - 1) / (warps_per_cta * 4);
    const int64_t want = 2ll * sm_count() * (2048 / kGatherThreads);
    if (batch > 0) splits = std::min<int64_t>(splits, std::max<int64_t>(1, (want + batch - 1) / batch));
    splits = std::max<int64_t>(1, std::min<int64_t>(splits, 65535));
    const int64_t items = static_cast<int64_t>(std::max(batch, 1)) * splits;
    const dim3 grid(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(items, 8ll * std::max(1, sm_count())))));
    auto s = reinterpret_cast<cudaStream_t>(stream);
    auto kp = static_cast<const uint16_t *>(k_pool), vp = static_cast<const uint16_t *>(v_pool);
    auto ko = static_cast<uint16_t *>(k_out), vo = static_cast<uint16_t *>(v_out);
    if (vec)
        return launch_status(launch_chained(ragged_gather_kernel<true>, dim3(grid), dim3(kGatherThreads), 0, s, kp, vp,
                                            num_slots, pool_row_stride, row_elems, req_to_token, r2t_rows,
                                            r2t_row_stride, r2t_width, req_pool_idx, kv_start, seq_lens, batch, splits,
                                            ko, vo, out_rows_cap, cu_seqlens, err_flags),
                             "pkv_ragged_gather");
    return launch_status(launch_chained(ragged_gather_kernel<false>, dim3(grid), dim3(kGatherThreads), 0, s, kp, vp,
                                        num_slots, pool_row_stride, row_elems, req_to_token, r2t_rows, r2t_row_stride,
                                        r2t_width, req_pool_idx, kv_start, seq_lens, batch, splits, ko, vo, out_rows_cap,
                                        cu_seqlens, err_flags),
                         "pkv_ragged_gather");
}

extern "C" pkv_status pkv_encoder_merge(const void *buffer, int64_t num_blocks, int64_t block_size, int64_t row_bytes,
                                        const int32_t *block_ids, const int64_t *positions, int64_t max_blocks,
                                        void *hidden, int64_t num_tokens, int64_t hidden_row_stride_bytes,
                                        uint64_t *filled, int32_t *err_flags, pkv_stream_t stream) {
    using namespace pkv;
    if (num_blocks < 0 || block_size < 0 || row_bytes < 0 || max_blocks < 0 || num_tokens < 0 ||
        hidden_row_stride_bytes < row_bytes)
        return fail(PKV_ERR_INVALID_ARG, "pkv_encoder_merge: negative or inconsistent size");
    if (!err_flags) return fail(PKV_ERR_INVALID_ARG, "pkv_encoder_merge: err_flags is required");
    const int64_t entries = max_blocks * block_size;
    if (entries == 0 || row_bytes == 0) return ok();
    if (!buffer || !block_ids || !positions || (num_tokens > 0 && !hidden))
        return fail(PKV_ERR_INVALID_ARG, "pkv_encoder_merge: null input");
    const int64_t grid = (entries + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
    if (grid > INT32_MAX) return fail(PKV_ERR_UNSUPPORTED, "pkv_encoder_merge: position map too large");
    const bool vec = aligned(buffer, 16) && aligned(hidden, 16) && row_bytes % 16 == 0 && hidden_row_stride_bytes % 16 == 0;
    auto s = reinterpret_cast<cudaStream_t>(stream);
    auto *cnt = reinterpret_cast<unsigned long long *>(filled);
    if (vec)
        return launch_status(launch_chained(encoder_merge_kernel<true>, dim3(static_cast<unsigned>(grid)),
                                            dim3(kMergeThreads), 0, s, static_cast<const uint8_t *>(buffer),
                                            num_blocks, block_size, row_bytes, block_ids, positions, entries,
                                            static_cast<uint8_t *>(hidden), num_tokens, hidden_row_stride_bytes, cnt,
                                            err_flags),
                             "pkv_encoder_merge");
    return launch_status(launch_chained(encoder_merge_kernel<false>, dim3(static_cast<unsigned>(grid)),
                                        dim3(kMergeThreads), 0, s, static_cast<const uint8_t *>(buffer), num_blocks,
                                        block_size, row_bytes, block_ids, positions, entries,
                                        static_cast<uint8_t *>(hidden), num_tokens, hidden_row_stride_bytes, cnt,
                                        err_flags),
                         "pkv_encoder_merge");
}
