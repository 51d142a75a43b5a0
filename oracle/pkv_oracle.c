/*
 * pkv_oracle.c -- plain, slow, CPU definition of attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference the CUDA
 * library is checked against; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * Every routine walks the token-granular req_to_token table directly, one
 * request and one position at a time, and computes in fp64 (bf16 inputs are
 * widened exactly).  There is no blocking, no fusion and no reordering beyond
 * the plain definitions cited on each function.
 *
 * Sources (web pages describing the method):
 *  [P1] "Enabling Encoder-Decoder Models on Intel XPU in SGLang: A KV-Cache
 *       Story": sections "two pools and a page size", "From slots to a page
 *       table", "Encoder-decoder models", "Approach 1", "Approach 2".
 *  [P4] mini-sglang handbook, "The KV pool, the page table and the token pool":
 *       sections "The KV pool", "The page table", "Tests", "Exercises".
 *  [P5] "AttentionBackend" (SGLang FlashInfer-MLA / FlashMLA notes): sections
 *       "init_forward_metadata", "kv_indptr and kv_indices", worked example.
 *
 * Parity status: every function here is pinned by the not-gpu tests
 * (worked examples printed on the pages, closed forms, invariants, and
 * library routines on special cases).  No function is parity-unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PKVO_OK 0
#define PKVO_ERR_RANGE 1      /* slot/page outside the pool, row or column outside the table */
#define PKVO_ERR_CONTIG 2     /* a page's tokens are not page-aligned and contiguous */
#define PKVO_ERR_CAPACITY 3   /* an output buffer is too small */
#define PKVO_ERR_ARG 4        /* inconsistent sizes */

/* bf16 is the top half of an IEEE-754 binary32; widening is exact. */
static double widen_bf16(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Page lists from the token table.  [P1 "From slots to a page table"]: the
 * page of logical position t is req_to_token[row, t - t % ps] / ps, which is
 * valid because a paged allocator keeps a request's tokens contiguous inside a
 * page ([P1 "two pools and a page size", PagedTokenToKVPoolAllocator]).  The
 * CSR form is [P5 "kv_indptr and kv_indices"]: kv_indptr is the running sum of
 * per-request page counts and kv_indices the pages in order; kv_last_page_len
 * is the number of keys on the last page (L - (n-1)*ps, 0 when L = 0).  The
 * padded table is [P5 "init_forward_metadata"]: [B, cdiv(max L, ps)] filled
 * with -1 past each request's last page.  A request's region starts at column
 * kv_start (the decoder offset of [P1 "Approach 1"]); NULL means 0.
 *
 * Every position is checked: the first slot of a page must be a multiple of ps
 * and the following ones must continue it.  Returns the first error met.
 */
int pkvo_build_indices(const int32_t *r2t, int64_t num_rows, int64_t row_stride, int64_t row_width,
                       const int32_t *req_pool_idx, const int32_t *seq_lens, const int32_t *kv_start,
                       int32_t batch, int32_t page_size, int64_t num_pool_pages,
                       int32_t *kv_indptr, int32_t *kv_indices, int64_t kv_indices_cap,
                       int32_t *kv_last_page_len, int32_t *block_table, int32_t bt_width) {
    if (page_size <= 0 || batch < 0) return PKVO_ERR_ARG;
    if (kv_indptr) kv_indptr[0] = 0;
    int64_t running = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t row = req_pool_idx[b];
        const int64_t start = kv_start ? kv_start[b] : 0;
        const int64_t len = seq_lens[b];
        if (row < 0 || row >= num_rows || start < 0 || len < 0 || start + len > row_width)
            return PKVO_ERR_RANGE;
        const int64_t npages = (len + page_size - 1) / page_size;
        if (block_table && npages > bt_width) return PKVO_ERR_CAPACITY;
        if (kv_indices && running + npages > kv_indices_cap) return PKVO_ERR_CAPACITY;
        for (int64_t p = 0; p < npages; ++p) {
            const int64_t col = start + p * page_size;
            const int64_t first = r2t[row * row_stride + col];
            if (first < 0 || first >= num_pool_pages * (int64_t)page_size) return PKVO_ERR_RANGE;
            if (first % page_size != 0) return PKVO_ERR_CONTIG;
            int64_t on_page = len - p * page_size;
            if (on_page > page_size) on_page = page_size;
            for (int64_t j = 1; j < on_page; ++j)
                if (r2t[row * row_stride + col + j] != first + j) return PKVO_ERR_CONTIG;
            const int32_t page = (int32_t)(first / page_size);
            if (kv_indices) kv_indices[running + p] = page;
            if (block_table) block_table[(int64_t)b * bt_width + p] = page;
        }
        if (block_table)
            for (int64_t p = npages; p < bt_width; ++p) block_table[(int64_t)b * bt_width + p] = -1;
        running += npages;
        if (kv_indptr) kv_indptr[b + 1] = (int32_t)running;
        if (kv_last_page_len) kv_last_page_len[b] = len > 0 ? (int32_t)(len - (npages - 1) * page_size) : 0;
    }
    return PKVO_OK;
}

/*
 * Store of new K/V rows.  [P4 "The KV pool", store_kv/store_cache]:
 * cache[out_loc[i]] = new[i], a bitwise row copy; rows are opaque bytes here.
 * A negative slot is a padded entry and is skipped.
 */
int pkvo_store(uint8_t *pool, int64_t num_slots, int64_t pool_row_stride_bytes, int64_t row_bytes,
               const uint8_t *rows, int64_t src_row_stride_bytes, const int32_t *slot_mapping,
               int32_t n) {
    int status = PKVO_OK;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= num_slots) { status = PKVO_ERR_RANGE; continue; }
        memcpy(pool + slot * pool_row_stride_bytes, rows + (int64_t)i * src_row_stride_bytes,
               (size_t)row_bytes);
    }
    return status;
}

/*
 * Decode attention, one query token per request.
 *
 * For request b and query head h, with g = Hq / Hkv and kv head kh = h / g
 * (consecutive query heads share a kv head), the keys are the positions
 * t in [t_begin, t_end) of the request (clamped to [0, L)), each read from pool
 * slot req_to_token[row, kv_start + t] ([P1 "From slots to a page table": the
 * kernel reads K/V through the per-request map]):
 *     x_t = scale * sum_d q[b,h,d] * K[slot_t, kh, d]
 *     out[b,h,:] = sum_t exp(x_t - m) V[slot_t, kh, :] / sum_t exp(x_t - m),  m = max_t x_t
 *     lse[b,h]   = m + ln(sum_t exp(x_t - m))
 * An empty key set gives out = 0 and lse = -inf ([P1 "Approach 2"]: an empty
 * KV returns a zero context).
 *
 * MLA (latent) attention is the same definition with Hkv = 1, K the full
 * latent row (kv_lora_rank + rope dims) and V its first head_dim_v entries:
 * pass the latent pool as both k_pool and v_pool.
 *
 * t_begin/t_end select a key sub-range (t_end < 0 means L) so that split
 * partials can be formed for the log-sum-exp merge.  req_mask (nullable)
 * skips requests whose entry is 0 (their outputs are left untouched).
 */
int pkvo_decode(const uint16_t *q, int32_t batch, int32_t hq, int32_t hkv, int32_t dqk, int32_t dv,
                const uint16_t *k_pool, int64_t k_row_stride, const uint16_t *v_pool,
                int64_t v_row_stride, int64_t num_slots,
                const int32_t *r2t, int64_t num_rows, int64_t row_stride, int64_t row_width,
                const int32_t *req_pool_idx, const int32_t *kv_start, const int32_t *seq_lens,
                double scale, int32_t t_begin, int32_t t_end, const uint8_t *req_mask,
                double *out, double *lse, int32_t num_threads) {
    if (hkv <= 0 || hq % hkv != 0) return PKVO_ERR_ARG;
    const int32_t g = hq / hkv;
    int status = PKVO_OK;
    const int64_t pairs = (int64_t)batch * hq;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(max : status)
#endif
    for (int64_t bh = 0; bh < pairs; ++bh) {
        const int64_t b = bh / hq, h = bh % hq, kh = h / g;
        if (req_mask && !req_mask[b]) continue;
        double *o = out + bh * dv;
        const int64_t row = req_pool_idx[b];
        const int64_t start = kv_start ? kv_start[b] : 0;
        const int64_t len = seq_lens[b];
        if (row < 0 || row >= num_rows || start < 0 || len < 0 || start + len > row_width) {
            status = PKVO_ERR_RANGE;
            continue;
        }
        int64_t t0 = t_begin < 0 ? 0 : t_begin;
        int64_t t1 = (t_end < 0 || t_end > len) ? len : t_end;
        for (int32_t d = 0; d < dv; ++d) o[d] = 0.0;
        if (t1 <= t0) {
            if (lse) lse[bh] = -INFINITY;
            continue;
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
        const uint16_t *qv = q + bh * dqk;
        int bad = 0;
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t slot = r2t[row * row_stride + start + t];
            if (slot < 0 || slot >= num_slots) { bad = 1; break; }
            const uint16_t *kr = k_pool + slot * k_row_stride + kh * dqk;
            double acc = 0.0;
            for (int32_t d = 0; d < dqk; ++d) acc += widen_bf16(qv[d]) * widen_bf16(kr[d]);
            x[t - t0] = scale * acc;
        }
        if (bad) {
            free(x);
            status = PKVO_ERR_RANGE;
            continue;
        }
        double m = -INFINITY;
        for (int64_t t = t0; t < t1; ++t) m = x[t - t0] > m ? x[t - t0] : m;
        double den = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            const double w = exp(x[t - t0] - m);
            const int64_t slot = r2t[row * row_stride + start + t];
            const uint16_t *vr = v_pool + slot * v_row_stride + kh * dv;
            for (int32_t d = 0; d < dv; ++d) o[d] += w * widen_bf16(vr[d]);
            den += w;
        }
        for (int32_t d = 0; d < dv; ++d) o[d] /= den;
        if (lse) lse[bh] = m + log(den);
        free(x);
    }
    return status;
}

/*
 * Log-sum-exp merge of split partials (the combine step implied by the
 * num_splits a split-KV decode plans, [P5 "init_forward_metadata"]).  Each
 * part i holds a normalised output o_i over a disjoint key subset and that
 * subset's lse_i.  With lse* = max_i lse_i and w_i = exp(lse_i - lse*):
 *     out = sum_i w_i o_i / sum_i w_i,   lse = lse* + ln(sum_i w_i).
 * Parts with lse = -inf (empty subsets) carry no weight; all empty gives 0, -inf.
 * Layout: o_parts [n_parts][rows][dv], lse_parts [n_parts][rows].
 */
void pkvo_lse_merge(int32_t n_parts, int64_t rows, int32_t dv, const double *o_parts,
                    const double *lse_parts, double *out, double *lse) {
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int32_t i = 0; i < n_parts; ++i) {
            const double l = lse_parts[(int64_t)i * rows + r];
            m = l > m ? l : m;
        }
        double *o = out + r * dv;
        for (int32_t d = 0; d < dv; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int32_t i = 0; i < n_parts; ++i) {
            const double l = lse_parts[(int64_t)i * rows + r];
            if (l == -INFINITY) continue;
            const double w = exp(l - m);
            const double *oi = o_parts + ((int64_t)i * rows + r) * dv;
            for (int32_t d = 0; d < dv; ++d) o[d] += w * oi[d];
            wsum += w;
        }
        for (int32_t d = 0; d < dv; ++d) o[d] /= wsum;
        lse[r] = m + log(wsum);
    }
}

/*
 * Ragged gather.  [P1 "Approach 2"]: the valid columns of each request's row
 * (t < L_b), taken in request order, give the flat slot list; K and V rows at
 * those slots are copied into contiguous buffers, and cu_seqlens holds the
 * request boundaries (cu[0] = 0, cu[b+1] = cu[b] + L_b).  Rows are opaque bytes.
 */
int pkvo_ragged_gather(const uint8_t *k_pool, const uint8_t *v_pool, int64_t num_slots,
                       int64_t pool_row_stride_bytes, int64_t row_bytes,
                       const int32_t *r2t, int64_t num_rows, int64_t row_stride, int64_t row_width,
                       const int32_t *req_pool_idx, const int32_t *kv_start, const int32_t *seq_lens,
                       int32_t batch, uint8_t *k_out, uint8_t *v_out, int64_t out_rows_cap,
                       int32_t *cu_seqlens) {
    cu_seqlens[0] = 0;
    int64_t running = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t row = req_pool_idx[b];
        const int64_t start = kv_start ? kv_start[b] : 0;
        const int64_t len = seq_lens[b];
        if (row < 0 || row >= num_rows || start < 0 || len < 0 || start + len > row_width)
            return PKVO_ERR_RANGE;
        if (running + len > out_rows_cap) return PKVO_ERR_CAPACITY;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t slot = r2t[row * row_stride + start + t];
            if (slot < 0 || slot >= num_slots) return PKVO_ERR_RANGE;
            memcpy(k_out + (running + t) * row_bytes, k_pool + slot * pool_row_stride_bytes,
                   (size_t)row_bytes);
            if (v_pool && v_out)
                memcpy(v_out + (running + t) * row_bytes, v_pool + slot * pool_row_stride_bytes,
                       (size_t)row_bytes);
        }
        running += len;
        cu_seqlens[b + 1] = (int32_t)running;
    }
    return PKVO_OK;
}

/*
 * Page allocation for one batch step.  [P1 "two pools and a page size",
 * PagedTokenToKVPoolAllocator alloc_extend / alloc_decode]: the new positions
 * [prefix_len, seq_len) of a request first continue its partly used last page
 * (the slots after last_loc, the slot of position prefix_len - 1), then take
 * whole new pages from the front of the free list, requests in order; page p
 * covers slots p*ps .. p*ps + ps - 1.  At page_size 1 each new position takes
 * one entry (TokenToKVPoolAllocator.alloc pops the first need_size slots).
 * The free list is free_pages[head .. head + count) with free_state = {head,
 * count}; on success head grows and count shrinks by the pages taken.  A step
 * needing more pages than count, or more output slots than out_cap, writes
 * nothing and changes nothing (the allocator's None).  Slots go to
 * out_cache_loc in request order, positions ascending.
 */
int pkvo_alloc_extend(const int32_t *prefix_lens, const int32_t *seq_lens, const int32_t *last_loc, int32_t batch,
                      int32_t page_size, int64_t num_pool_pages, const int32_t *free_pages, int64_t free_pages_len,
                      int32_t *free_state, int32_t *out_cache_loc, int64_t out_cap) {
    if (page_size <= 0 || batch < 0) return PKVO_ERR_ARG;
    const int64_t ps = page_size;
    int64_t pages = 0, toks = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t p = prefix_lens[b], s = seq_lens[b];
        if (p < 0 || s < p) return PKVO_ERR_RANGE;
        if (p % ps != 0) {   /* the partly used page must hold position p - 1 at its offset */
            const int64_t ll = last_loc[b];
            if (ll < 0 || ll >= num_pool_pages * ps) return PKVO_ERR_RANGE;
            if (ll % ps != (p - 1) % ps) return PKVO_ERR_CONTIG;
        }
        pages += (s + ps - 1) / ps - (p + ps - 1) / ps;
        toks += s - p;
    }
    const int64_t head = free_state[0], count = free_state[1];
    if (toks > out_cap || pages > count || head < 0 || head + pages > free_pages_len) return PKVO_ERR_CAPACITY;
    for (int64_t k = 0; k < pages; ++k)
        if (free_pages[head + k] < 0 || free_pages[head + k] >= num_pool_pages) return PKVO_ERR_RANGE;
    int64_t pg = head, o = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t p = prefix_lens[b], s = seq_lens[b];
        const int64_t aligned = (p + ps - 1) / ps * ps;   /* first position on a new page */
        for (int64_t t = p; t < s; ++t) {
            int64_t slot;
            if (t < aligned) slot = last_loc[b] + (t - p + 1);
            else slot = (int64_t)free_pages[pg + (t - aligned) / ps] * ps + t % ps;
            out_cache_loc[o++] = (int32_t)slot;
        }
        pg += (s + ps - 1) / ps - (p + ps - 1) / ps;
    }
    free_state[0] = (int32_t)(head + pages);
    free_state[1] = (int32_t)(count - pages);
    return PKVO_OK;
}

/*
 * Row writer.  [P1 write_cache_indices / write_req_to_token_pool]: for request
 * b, columns kv_start + [0, prefix_len) of row req_pool_idx[b] receive the
 * reused prefix slots prefix_slots[b][0 .. prefix_len) (skipped when that
 * pointer is NULL: they are already in place), and columns kv_start +
 * [prefix_len, seq_len) the freshly allocated slots out_cache_loc[e_b ..), e_b
 * being the extend lengths (seq_len - prefix_len) of the requests before b.
 * A request whose row or columns fall outside the table is skipped with
 * PKVO_ERR_RANGE (the others are written).
 */
int pkvo_write_req_to_token(int32_t *r2t, int64_t num_rows, int64_t row_stride, int64_t row_width,
                            const int32_t *req_pool_idx, const int32_t *kv_start, const int32_t *prefix_lens,
                            const int32_t *seq_lens, const int32_t *const *prefix_slots,
                            const int32_t *out_cache_loc, int32_t batch) {
    int status = PKVO_OK;
    int64_t e = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t row = req_pool_idx[b], st = kv_start ? kv_start[b] : 0;
        const int64_t p = prefix_lens[b], s = seq_lens[b];
        const int64_t ext = s > p ? s - p : 0;
        if (row < 0 || row >= num_rows || st < 0 || p < 0 || s < p || st + s > row_width) {
            status = PKVO_ERR_RANGE;
            e += ext;
            continue;
        }
        int32_t *r = r2t + row * row_stride + st;
        if (prefix_slots && prefix_slots[b])
            for (int64_t t = 0; t < p; ++t) r[t] = prefix_slots[b][t];
        for (int64_t t = p; t < s; ++t) r[t] = out_cache_loc[e + (t - p)];
        e += ext;
    }
    return status;
}

/*
 * Encoder-cache merge (Neuron encoder cache, "Merge Inside Compiled Graph" and
 * "Read Path"): the blocks block_ids[i] of buffer [num_blocks, block_size, row]
 * are stacked and flattened, and token j of block i lands in hidden row
 * positions[i][j] when that position lies in [0, num_tokens); a position at or
 * past num_tokens (the sentinel) writes nothing (the discarded dummy row).  A
 * negative position or a block id outside the buffer is PKVO_ERR_RANGE and that
 * entry is skipped.  *filled counts the rows written, for the check that every
 * scheduled position was filled.  Rows are opaque bytes.
 */
int pkvo_encoder_merge(const uint8_t *buffer, int64_t num_blocks, int64_t block_size, int64_t row_bytes,
                       const int32_t *block_ids, const int64_t *positions, int64_t max_blocks, uint8_t *hidden,
                       int64_t num_tokens, int64_t hidden_row_stride_bytes, int64_t *filled) {
    int status = PKVO_OK;
    int64_t n = 0;
    for (int64_t i = 0; i < max_blocks; ++i) {
        const int64_t blk = block_ids[i];
        for (int64_t j = 0; j < block_size; ++j) {
            const int64_t pos = positions[i * block_size + j];
            if (pos >= num_tokens) continue;
            if (pos < 0 || blk < 0 || blk >= num_blocks) {
                status = PKVO_ERR_RANGE;
                continue;
            }
            memcpy(hidden + pos * hidden_row_stride_bytes, buffer + (blk * block_size + j) * row_bytes,
                   (size_t)row_bytes);
            ++n;
        }
    }
    if (filled) *filled = n;
    return status;
}

/*
 * Multi-query attention through the page table (extend / chunked prefill,
 * speculative target-verify, and the mixed causal/full segments of the
 * diffusion KV path).  Query row j (qo_indptr[b] <= j < qo_indptr[b+1]) belongs
 * to request b and sees the keys t in [0, kv_end[j]) of that request's row,
 * slot req_to_token[row, kv_start + t] ([P1 "From slots to a page table"]);
 * for query head h, with kh = h / (Hq / Hkv):
 *     x_t = scale * q[j,h,:] . K[slot_t, kh, :]
 *     out[j,h,:] = sum_t exp(x_t - m) V[slot_t, kh, :] / sum_t exp(x_t - m),  lse = m + ln sum
 * A causal extend over the last n positions of an L-key request has
 * kv_end = L - n + i + 1 for its i-th query row (AttentionBackend notes: extend
 * with qo_indptr, target-verify with draft tokens); a full segment [a, b) gives
 * its rows kv_end = b (vllm-omni "Attention execution").  kv_end outside
 * [0, L] is PKVO_ERR_RANGE; kv_end = 0 gives out = 0, lse = -inf.
 */
int pkvo_extend(const uint16_t *q, int64_t total_q, int32_t batch, const int32_t *qo_indptr, const int32_t *kv_end,
                int32_t hq, int32_t hkv, int32_t dqk, int32_t dv, const uint16_t *k_pool, int64_t k_row_stride,
                const uint16_t *v_pool, int64_t v_row_stride, int64_t num_slots, const int32_t *r2t, int64_t num_rows,
                int64_t row_stride, int64_t row_width, const int32_t *req_pool_idx, const int32_t *kv_start,
                const int32_t *seq_lens, double scale, double *out, double *lse, int32_t num_threads) {
    if (hkv <= 0 || hq % hkv != 0 || batch < 0) return PKVO_ERR_ARG;
    if (batch > 0 && (qo_indptr[0] != 0 || qo_indptr[batch] != total_q)) return PKVO_ERR_ARG;
    const int32_t g = hq / hkv;
    int status = PKVO_OK;
    const int64_t pairs = total_q * hq;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(max : status)
#endif
    for (int64_t jh = 0; jh < pairs; ++jh) {
        const int64_t j = jh / hq, h = jh % hq, kh = h / g;
        int32_t b = 0;   /* the request owning query row j */
        while (b + 1 < batch && qo_indptr[b + 1] <= j) ++b;
        double *o = out + jh * dv;
        for (int32_t d = 0; d < dv; ++d) o[d] = 0.0;
        const int64_t row = req_pool_idx[b], start = kv_start ? kv_start[b] : 0, len = seq_lens[b];
        const int64_t te = kv_end[j];
        if (row < 0 || row >= num_rows || start < 0 || len < 0 || start + len > row_width || te < 0 || te > len) {
            status = PKVO_ERR_RANGE;
            if (lse) lse[jh] = -INFINITY;
            continue;
        }
        if (te == 0) {
            if (lse) lse[jh] = -INFINITY;
            continue;
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)te);
        const uint16_t *qv = q + jh * dqk;
        int bad = 0;
        for (int64_t t = 0; t < te; ++t) {
            const int64_t slot = r2t[row * row_stride + start + t];
            if (slot < 0 || slot >= num_slots) { bad = 1; break; }
            const uint16_t *kr = k_pool + slot * k_row_stride + kh * dqk;
            double acc = 0.0;
            for (int32_t d = 0; d < dqk; ++d) acc += widen_bf16(qv[d]) * widen_bf16(kr[d]);
            x[t] = scale * acc;
        }
        if (bad) {
            free(x);
            status = PKVO_ERR_RANGE;
            continue;
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < te; ++t) m = x[t] > m ? x[t] : m;
        double den = 0.0;
        for (int64_t t = 0; t < te; ++t) {
            const double w = exp(x[t] - m);
            const int64_t slot = r2t[row * row_stride + start + t];
            const uint16_t *vr = v_pool + slot * v_row_stride + kh * dv;
            for (int32_t d = 0; d < dv; ++d) o[d] += w * widen_bf16(vr[d]);
            den += w;
        }
        for (int32_t d = 0; d < dv; ++d) o[d] /= den;
        if (lse) lse[jh] = m + log(den);
        free(x);
    }
    return status;
}

/*
 * Query rows and key bounds of a row's attention segments (vllm-omni diffusion
 * KV, "Attention execution"): request b's segments seg_indptr[b] ..
 * seg_indptr[b+1]-1, each (kind, start, end) over positions [start, end) of
 * its sequence: a causal segment's position p sees keys [0, p + 1), a full
 * segment's positions see [0, end).  The query rows of b are its segments'
 * positions in order: q_pos[j] = p, kv_end[j] = the bound above, rows counted
 * from qo_indptr[b] (qo_indptr[0] = 0, qo_indptr[b+1] = qo_indptr[b] + the
 * lengths of b's segments).  end < start, start < 0 or more rows than cap is an
 * error.
 */
int pkvo_span_plan(int32_t batch, const int32_t *seg_indptr, const int32_t *seg_kind, const int32_t *seg_start,
                   const int32_t *seg_end, int32_t *qo_indptr, int32_t *q_pos, int32_t *kv_end, int64_t cap) {
    int64_t j = 0;
    qo_indptr[0] = 0;
    for (int32_t b = 0; b < batch; ++b) {
        for (int32_t s = seg_indptr[b]; s < seg_indptr[b + 1]; ++s) {
            const int64_t a = seg_start[s], e = seg_end[s];
            if (a < 0 || e < a || (seg_kind[s] != 0 && seg_kind[s] != 1)) return PKVO_ERR_RANGE;
            if (j + (e - a) > cap) return PKVO_ERR_CAPACITY;
            for (int64_t p = a; p < e; ++p, ++j) {
                q_pos[j] = (int32_t)p;
                kv_end[j] = (int32_t)(seg_kind[s] == 0 ? p + 1 : e);
            }
        }
        qo_indptr[b + 1] = (int32_t)j;
    }
    return PKVO_OK;
}

/* Threads the decode would use (reported beside CPU-baseline timings). */
int32_t pkvo_max_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}
