/*
 * pkv.h -- C ABI of libpkv: attention over a paged KV cache on one GB300 GPU (sm_103a).
 *
 * The KV cache of every in-flight request lives in one preallocated pool of
 * fixed-size pages; a request's token positions map to pool slots through the
 * token-granular table req_to_token[row, position] ("Enabling Encoder-Decoder
 * Models on Intel XPU in SGLang: A KV-Cache Story", section "How SGLang stores
 * the KV cache: two pools and a page size").  The library offers the four
 * steps of a decode layer over that cache:
 *
 *   pkv_build_indices  req_to_token -> per-request page lists (CSR and/or a -1 padded table)
 *   pkv_store          scatter this step's new K/V rows into their pool slots
 *   pkv_decode         one query token per request attending through the page table
 *                      (GQA/MHA, or MLA over a latent pool), split-KV + log-sum-exp merge
 *   pkv_ragged_gather  pack a request's token-granular K/V into a contiguous varlen buffer
 *
 * Conventions shared by every call
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise.  The
 *     library allocates nothing and keeps no state between calls except a
 *     per-device cache of the SM count.
 *   - Every call is asynchronous on the caller's stream and never synchronizes.
 *     Kernels are launched as programmatic dependents of the kernel before them in
 *     the stream: they may be scheduled while it drains, but each waits for its
 *     completion (and the visibility of its writes) before touching memory, so
 *     stream order holds exactly as for ordinary launches.
 *   - Tensors are row-major with the last dimension contiguous.  K/V/q/out are
 *     bf16; tables are int32; lse is fp32.
 *   - Errors the host can see (null pointers, bad sizes, unsupported shapes,
 *     misalignment) return a status before anything is launched;
 *     pkv_last_error() then gives a one-line reason (thread-local).
 *   - Errors only the device can see (a slot or page outside the pool, a page
 *     whose tokens are not contiguous, an output too small) are OR-ed into the
 *     caller's int32 *err_flags on the device as PKV_DEVERR_* bits.  The kernel
 *     never reads or writes outside the buffers it was given: the offending
 *     row or page is skipped (reads of it return zeros) and nothing traps.
 *     The outputs of a request that raised a flag are unspecified.
 *     err_flags is never cleared by the library.
 *   - A request with no keys (L = 0) produces out = 0 and lse = -inf rather
 *     than a launch failure (the guard of "Approach 2: gather and go ragged").
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shapes, misaligned buffer */
    PKV_ERR_UNSUPPORTED = 2, /* a shape the kernels are not built for (see each call) */
    PKV_ERR_CAPACITY = 3,    /* a buffer the host can size is too small (workspace) */
    PKV_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
} pkv_status;

/* Device-side error bits OR-ed into *err_flags. */
#define PKV_DEVERR_RANGE 1    /* slot, page, row or position outside its pool or table */
#define PKV_DEVERR_CONTIG 2   /* a page's tokens are not page-aligned and contiguous */
#define PKV_DEVERR_CAPACITY 4 /* an output had too little room; the excess was not written */
#define PKV_DEVERR_TIMEOUT 8  /* a device-side wait ran past its limit (pkv_set_wait_limit, ~2 s by
                                 default); outputs of the launch unspecified */

/* 3: pkv_extend_args gained the token-table fields (req_to_token ... kv_start) at its end */
#define PKV_ABI_VERSION 3

/*
 * pkv_build_indices -- page lists from the token-granular table.
 *
 * Defined by "From slots to a page table: how attention reads the cache" (the
 * page of position t is req_to_token[row, t - t % ps] / ps, valid because the
 * paged allocator keeps a request's tokens contiguous inside each page) and by
 * the AttentionBackend notes, sections "kv_indptr and kv_indices" (CSR) and
 * "init_forward_metadata" (the FlashMLA table [B, cdiv(max L, ps)] filled with
 * -1 past each request's last page).
 *
 * For request b (row r = req_pool_idx[b], start s = kv_start ? kv_start[b] : 0,
 * L = seq_lens[b] keys, n = ceil(L / ps) pages):
 *   kv_indptr[b+1]              = kv_indptr[b] + n,   kv_indptr[0] = 0
 *   kv_indices[kv_indptr[b]+p]  = req_to_token[r, s + p*ps] / ps          (p < n)
 *   kv_last_page_len[b]         = L - (n-1)*ps, or 0 when L = 0
 *   block_table[b, p]           = the same page for p < n, -1 for n <= p < block_table_width
 * Each CTA streams the page counts of all requests once to find its offsets,
 * so the work is linear in the batch.
 * Every position is checked: each page's first slot must be a multiple of ps,
 * the following ones must continue it (PKV_DEVERR_CONTIG otherwise) and every
 * page must lie in [0, num_pool_pages) (PKV_DEVERR_RANGE).  A row or region
 * outside the table raises PKV_DEVERR_RANGE and the request gets n = 0.  Pages
 * beyond kv_indices_cap or block_table_width raise PKV_DEVERR_CAPACITY and are
 * not written.
 *
 * req_to_token  int32 [r2t_rows, r2t_row_stride], r2t_width valid columns per row
 * req_pool_idx, seq_lens  int32 [batch];  kv_start  int32 [batch] or NULL
 * page_size     >= 1 (any value)
 * Outputs (each group nullable, not both): kv_indptr [batch+1], kv_indices
 * [kv_indices_cap], kv_last_page_len [batch]; block_table [batch, block_table_width].
 * err_flags     int32 on the device, required.
 */
pkv_status pkv_build_indices(const int32_t *req_to_token, int64_t r2t_rows, int64_t r2t_row_stride,
                             int64_t r2t_width, const int32_t *req_pool_idx, const int32_t *seq_lens,
                             const int32_t *kv_start, int32_t batch, int32_t page_size,
                             int64_t num_pool_pages, int32_t *kv_indptr, int32_t *kv_indices,
                             int64_t kv_indices_cap, int32_t *kv_last_page_len, int32_t *block_table,
                             int32_t block_table_width, int32_t *err_flags, pkv_stream_t stream);

/*
 * pkv_store -- write this step's new K/V rows into their pool slots.
 *
 * Defined by the mini-sglang handbook, "The KV pool" (store_kv / store_cache:
 * k_cache[out_loc[i]] = k[i], the same for v; pure indexed movement, one warp
 * per token and 16 bytes per move).  The copy is bitwise.
 *
 * k_pool        bf16 rows of kv_heads*head_dim_k elements, k_row_stride elements apart,
 *               num_slots rows (an MLA latent pool: kv_heads = 1, head_dim_k = 576)
 * v_pool        bf16 rows of kv_heads*head_dim_v elements, v_row_stride apart; NULL for
 *               a latent pool (then v_new must be NULL too)
 * k_new, v_new  bf16 [n_tokens, kv_heads, head_dim] contiguous
 * slot_mapping  int32 [n_tokens]; a negative entry is a padded token and is skipped;
 *               an entry >= num_slots raises PKV_DEVERR_RANGE and is skipped.
 * Duplicate slots in one call give an unspecified winner.
 */
pkv_status pkv_store(void *k_pool, void *v_pool, int64_t num_slots, int64_t k_row_stride,
                     int64_t v_row_stride, int32_t kv_heads, int32_t head_dim_k, int32_t head_dim_v,
                     const void *k_new, const void *v_new, const int32_t *slot_mapping,
                     int32_t n_tokens, int32_t *err_flags, pkv_stream_t stream);

/* pkv_decode: which attention and which page-table form. */
typedef enum pkv_kind {
    PKV_KIND_GQA = 0, /* Hq query heads over Hkv kv heads; kv head of query head h is h / (Hq/Hkv) */
    PKV_KIND_MLA = 1  /* one latent kv head: K = the whole latent row, V = its first head_dim_v entries */
} pkv_kind;

typedef enum pkv_layout {
    PKV_LAYOUT_CSR = 0,         /* kv_indptr / kv_indices / kv_last_page_len */
    PKV_LAYOUT_BLOCK_TABLE = 1, /* block_table [B, block_table_width] + seq_lens */
    PKV_LAYOUT_VARLEN = 2,      /* contiguous rows: keys of b are rows cu_seqlens[b] .. cu_seqlens[b+1]-1 */
    PKV_LAYOUT_REQ_TO_TOKEN = 3 /* the token table itself: req_to_token + req_pool_idx (+ kv_start) + seq_lens;
                                   page of key t = req_to_token[row, s + t - t % ps] / ps (GQA only) */
} pkv_layout;

typedef struct pkv_decode_args {
    int32_t kind;              /* pkv_kind */
    int32_t layout;            /* pkv_layout */
    int32_t batch;             /* B >= 0 */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hkv (must be 1 for MLA) */
    int32_t head_dim_qk;       /* GQA: 64 or 128; MLA: 576 */
    int32_t head_dim_v;        /* GQA: equal to head_dim_qk; MLA: 512 */
    int32_t page_size;         /* power of two, 1..1024 (CSR / block table); ignored for VARLEN */
    float sm_scale;            /* softmax scale, e.g. 1/sqrt(head_dim) */
    int32_t max_seq_len;       /* host upper bound on every request's key count; sizes the split plan */
    int32_t kv_chunk;          /* keys per split, a multiple of 64; 0 lets the library choose (for GQA
                                  and small batches, equal spans; see pkv_decode).  MLA: keys per span
                                  of all requests' keys taken in order */
    int32_t block_table_width; /* columns of block_table (BLOCK_TABLE) */
    int64_t num_slots;         /* rows of the pool(s) (VARLEN: rows of the contiguous buffer) */
    int64_t k_row_stride;      /* elements between consecutive rows of k_pool */
    int64_t v_row_stride;      /* elements between consecutive rows of v_pool (ignored for MLA) */
    int64_t kv_indices_len;    /* CSR: entries of kv_indices (a kv_indptr value beyond it is an error) */
    const void *q;             /* bf16 [B, Hq, head_dim_qk] contiguous */
    const void *k_pool;        /* bf16 rows [Hkv, head_dim_qk] (MLA: the latent row) */
    const void *v_pool;        /* bf16 rows [Hkv, head_dim_v]; NULL for MLA */
    const int32_t *kv_indptr;        /* CSR [B+1] */
    const int32_t *kv_indices;       /* CSR pages */
    const int32_t *kv_last_page_len; /* CSR [B] */
    const int32_t *block_table;      /* BLOCK_TABLE [B, block_table_width], -1 padded */
    const int32_t *seq_lens;         /* BLOCK_TABLE [B] */
    const int32_t *cu_seqlens;       /* VARLEN [B+1] */
    void *out;                 /* bf16 [B, Hq, head_dim_v] */
    float *lse;                /* fp32 [B, Hq], natural log of the softmax denominator; nullable */
    /* PKV_LAYOUT_REQ_TO_TOKEN (added in ABI version 2) */
    const int32_t *req_to_token;     /* int32 [r2t_rows, r2t_row_stride] */
    int64_t r2t_rows;
    int64_t r2t_row_stride;
    int64_t r2t_width;               /* valid columns of a row */
    const int32_t *req_pool_idx;     /* [B] row of request b */
    const int32_t *kv_start;         /* [B] column of b's first key (a multiple of page_size), or NULL for 0 */
    /* fused store (added in ABI version 2; GQA, any layout but VARLEN): both NULL, or both set */
    const void *k_new;               /* bf16 [B, Hkv, head_dim]: the new token's K */
    const void *v_new;               /* bf16 [B, Hkv, head_dim]: the new token's V */
} pkv_decode_args;

/*
 * pkv_decode -- decode attention through the page table.
 *
 * For each request b with L keys (CSR: (n-1)*ps + kv_last_page_len[b] for n
 * pages, BLOCK_TABLE: seq_lens[b], VARLEN: cu_seqlens[b+1]-cu_seqlens[b]) and
 * query head h, key t lives at slot page_table[b][t / ps] * ps + t % ps
 * ("From slots to a page table: how attention reads the cache"; AttentionBackend
 * notes, "kv_indptr and kv_indices": base = page_id * page_size, address = base
 * + offset) and
 *     out[b,h,:] = softmax_t(sm_scale * q[b,h,:] . K[slot_t, kh, :]) V[slot_t, kh, :]
 *     lse[b,h]   = ln sum_t exp(sm_scale * q[b,h,:] . K[slot_t, kh, :])
 * with kh = h / (Hq/Hkv) for GQA and kh = 0 for MLA.  L = 0 gives out = 0,
 * lse = -inf.  Long requests are cut into splits of kv_chunk keys whose
 * partial results are combined by a log-sum-exp merge (the num_splits of the
 * FlashMLA metadata, AttentionBackend notes, "init_forward_metadata").  For
 * MLA the keys of all requests, taken in request order in tiles of 64, are cut
 * into equal spans (kv_chunk keys each, or one span per pair of SMs when
 * kv_chunk is 0); a request that a span boundary cuts is merged the same way.
 * For GQA with kv_chunk 0, pages of >= 8 keys (or VARLEN) and a batch so small
 * that even max_seq_len keys per request would give each of about two spans per
 * SM (three at head_dim 64) at most 128 tiles of 64 keys, the keys of each kv head's requests are cut
 * the same way into equal spans (the same number for every kv head); the
 * workspace size then depends on the SM count, not on the batch.
 * Arithmetic: bf16 inputs, fp32 accumulation and softmax, bf16 output rounded
 * to nearest even.
 *
 * workspace     device scratch of at least pkv_decode_workspace_size(args) bytes,
 *               256-byte aligned; its contents need no initialisation.
 * Supported:    GQA head_dim 64 or 128 with Hq/Hkv in {1,2,4,8,16};
 *               MLA head_dim_qk 576, head_dim_v 512, Hq a multiple of 128.
 * A page id outside the pool or a -1 inside a request's page range raises
 * PKV_DEVERR_RANGE; that key reads as zeros.  A kv_indptr range outside
 * [0, kv_indices_len], a kv_last_page_len outside [1, page_size] or a negative
 * length raises PKV_DEVERR_RANGE and the request is treated as empty.  A
 * request longer than max_seq_len raises PKV_DEVERR_CAPACITY and only its
 * first keys (up to the split plan's reach) are attended.
 *
 * PKV_LAYOUT_REQ_TO_TOKEN (GQA) reads the pages straight from the token table,
 * with no pkv_build_indices launch and no page list in between ("From slots to
 * a page table": the page of position t is req_to_token[row, t - t % ps] / ps):
 * request b has L = seq_lens[b] keys at columns s .. s + L - 1 of row
 * req_pool_idx[b] (s = kv_start[b], or 0), and key t lives at slot
 * req_to_token[row, s + t - t % ps] + t % ps.  A row or region outside the
 * table (or s not a multiple of ps) raises PKV_DEVERR_RANGE and the request is
 * treated as empty; a page's first slot outside the pool raises
 * PKV_DEVERR_RANGE and one that is not a multiple of ps PKV_DEVERR_CONTIG, and
 * its keys read as zeros.  Unlike pkv_build_indices it reads only each page's
 * first position, so it does not check that the other positions continue it.
 *
 * Fused store (k_new and v_new set; GQA; not with VARLEN): the step's new token
 * is request b's last key, t = L - 1.  Before attending, the call writes
 * k_new[b] and v_new[b] into the pools at that key's slot (pkv_store's write,
 * mini-sglang handbook "The KV pool": store_kv before attention), and the
 * attention uses those values for the key.  k_pool and v_pool must then be
 * writable.  A request that raises PKV_DEVERR_CAPACITY (longer than
 * max_seq_len) is not stored.
 */
pkv_status pkv_decode(const pkv_decode_args *args, void *workspace, size_t workspace_bytes,
                      int32_t *err_flags, pkv_stream_t stream);

/* Workspace bytes pkv_decode needs for these arguments (0 on invalid arguments). */
size_t pkv_decode_workspace_size(const pkv_decode_args *args);

/*
 * pkv_decode_no_alloc -- pkv_decode for GQA/MHA without a caller workspace.
 *
 * The pages describe no counterpart of this call; it exists for callers that
 * cannot call cudaMalloc: a plug-in inside a process whose device memory is
 * all owned by another allocator (for instance a serving engine that reserved
 * the rest of HBM for its KV pool at start-up), or a latency-critical loop in
 * which an allocation could block.  It computes exactly what pkv_decode
 * computes (same split plan, same kernels, bitwise the same outputs) but keeps
 * the split partials in a 32 MiB array compiled into the library, which every
 * GPU that loads the library holds until the process exits.  The library
 * still allocates nothing; q, the pools, the page table, out and lse stay
 * caller-owned as for pkv_decode.
 *
 * - Only PKV_KIND_GQA is accepted (PKV_ERR_UNSUPPORTED otherwise).
 * - A split plan needing more than 32 MiB of scratch (pkv_decode_workspace_size
 *   of the same arguments) returns PKV_ERR_CAPACITY before launching; a larger
 *   kv_chunk or a smaller batch brings it under the limit.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is cached for the life of the
 *   process: after cudaDeviceReset (or any teardown of the device's primary
 *   context) the array may move, so do not call this entry point again on
 *   that device until the library has been unloaded and loaded again.
 * - All calls share the one array and it keeps the last call's contents.  No
 *   part of it needs to start at zero (every partial is written before it is
 *   read), but calls whose kernels overlap on the GPU (other streams, other
 *   host threads) race on it: serialise them.
 */
pkv_status pkv_decode_no_alloc(const pkv_decode_args *args, int32_t *err_flags, pkv_stream_t stream);

/*
 * pkv_ragged_gather -- pack token-granular K/V into contiguous varlen buffers.
 *
 * Defined by "Approach 2: gather and go ragged (variable-length
 * FlashAttention)": the valid columns of each row (t < L_b), in request order,
 * give the flat slot list; the K and V rows at those slots are copied into
 * contiguous buffers addressed by cumulative lengths.
 *   cu_seqlens[0] = 0,  cu_seqlens[b+1] = cu_seqlens[b] + seq_lens[b]
 *   k_out[cu_seqlens[b] + t] = k_pool[req_to_token[req_pool_idx[b], s_b + t]]   (t < seq_lens[b])
 * and the same for v.  Rows are row_elems bf16 elements (Hkv * head_dim),
 * pool rows pool_row_stride elements apart, output rows packed.  Rows beyond
 * out_rows_cap raise PKV_DEVERR_CAPACITY and are not written.  A request whose
 * row or region lies outside the table, and a slot outside [0, num_slots),
 * raise PKV_DEVERR_RANGE; the output rows reserved for them are zero-filled
 * (so a following VARLEN pkv_decode reads zeros there, as it does for a bad
 * page).  max_seq_len is a host upper bound on seq_lens (grid sizing only;
 * longer requests are still copied whole).  v_pool / v_out may both be NULL
 * (latent pool).  Each CTA scans the lengths of all requests once, so the
 * work is linear in the batch.
 */
pkv_status pkv_ragged_gather(const void *k_pool, const void *v_pool, int64_t num_slots,
                             int64_t pool_row_stride, int64_t row_elems, const int32_t *req_to_token,
                             int64_t r2t_rows, int64_t r2t_row_stride, int64_t r2t_width,
                             const int32_t *req_pool_idx, const int32_t *kv_start,
                             const int32_t *seq_lens, int32_t batch, int32_t max_seq_len, void *k_out,
                             void *v_out, int64_t out_rows_cap, int32_t *cu_seqlens,
                             int32_t *err_flags, pkv_stream_t stream);

/*
 * Arguments of pkv_extend (multi-query attention through the page table).
 * Pools and layouts as for pkv_decode (CSR or BLOCK_TABLE; page_size a power
 * of two in [1, 1024]; pages under 8 keys are gathered row by row).
 */
typedef struct pkv_extend_args {
    int32_t layout;            /* PKV_LAYOUT_CSR, PKV_LAYOUT_BLOCK_TABLE or PKV_LAYOUT_REQ_TO_TOKEN */
    int32_t batch;             /* B >= 0 */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hkv; Hq / Hkv in {1, 2, 4, 8, 16} */
    int32_t head_dim;          /* 64 or 128 (K and V) */
    int32_t page_size;
    float sm_scale;
    int32_t max_seq_len;       /* host upper bound on every request's key count */
    int32_t kv_chunk;          /* keys per split (multiple of 64, rounded up to whole 128-key tiles);
                                  0 lets the library choose */
    int32_t block_table_width;
    int64_t total_q;           /* query rows: qo_indptr[B] */
    int64_t num_slots;         /* pool rows */
    int64_t k_row_stride;      /* elements between pool rows */
    int64_t v_row_stride;
    int64_t kv_indices_len;    /* CSR: entries of kv_indices */
    const void *q;             /* bf16 [total_q, Hq, head_dim] */
    const void *k_pool;        /* bf16 rows [Hkv, head_dim] */
    const void *v_pool;
    const int32_t *qo_indptr;  /* [B+1]: query rows of request b are qo_indptr[b] .. qo_indptr[b+1]-1 */
    const int32_t *kv_end;     /* [total_q] key bound of each query row, or NULL: causal over the last positions */
    const int32_t *kv_indptr;        /* CSR [B+1] */
    const int32_t *kv_indices;       /* CSR pages */
    const int32_t *kv_last_page_len; /* CSR [B] */
    const int32_t *block_table;      /* BLOCK_TABLE [B, block_table_width] */
    const int32_t *seq_lens;         /* BLOCK_TABLE and REQ_TO_TOKEN [B] */
    void *out;                 /* bf16 [total_q, Hq, head_dim] */
    float *lse;                /* fp32 [total_q, Hq] natural-log softmax denominators; nullable */
    /* REQ_TO_TOKEN (added in ABI version 3; the same fields as pkv_decode_args) */
    const int32_t *req_to_token;     /* int32 [r2t_rows, r2t_row_stride] */
    int64_t r2t_rows;
    int64_t r2t_row_stride;
    int64_t r2t_width;               /* valid columns of a row */
    const int32_t *req_pool_idx;     /* [B] row of request b */
    const int32_t *kv_start;         /* [B] column of b's first key (a multiple of page_size), or NULL for 0 */
} pkv_extend_args;

/*
 * pkv_extend -- attention of many query tokens per request through the page table.
 *
 * Extend / chunked prefill and speculative target-verify (AttentionBackend
 * notes: qo_indptr from seq_lens - prefix_lens; target-verify over draft
 * tokens), and the mixed causal/full segments of a diffusion row (vllm-omni,
 * "Attention execution").  Query row j of request b (qo_indptr[b] <= j <
 * qo_indptr[b+1]) sees the keys t < kv_end[j] of request b, read through its
 * page list exactly as pkv_decode reads them; kv_end NULL means the causal
 * bound of the request's last n_b positions: kv_end = L_b - n_b + i + 1 for its
 * i-th row (n_b <= L_b required).  For query head h, kh = h / (Hq / Hkv):
 *     out[j,h,:] = softmax_{t < kv_end[j]}(sm_scale * q[j,h,:] . K[t, kh, :]) V[t, kh, :]
 * kv_end[j] = 0 gives out = 0, lse = -inf; kv_end outside [0, L_b] raises
 * PKV_DEVERR_RANGE and the row is treated as empty.  The new tokens' K/V must
 * already be in the pool (pkv_store first).  PKV_LAYOUT_REQ_TO_TOKEN reads the
 * pages straight from the token table as pkv_decode does (L_b = seq_lens[b], key
 * t at slot req_to_token[row, s + t - t % ps] + t % ps with row =
 * req_pool_idx[b] and s = kv_start[b] or 0; the same range and alignment
 * checks), so no pkv_build_indices launch is needed.  Arithmetic: bf16 inputs, fp32
 * accumulation and softmax, bf16 output.  The key range of a block of rows may
 * be split into kv_chunk chunks whose partials are merged by log-sum-exp.
 * workspace: at least pkv_extend_workspace_size(args) bytes, 256-byte aligned,
 * non-null, caller-owned, not shared with a concurrent call: it holds the split
 * partials and a work counter that the call resets on the stream before use.
 */
pkv_status pkv_extend(const pkv_extend_args *args, void *workspace, size_t workspace_bytes,
                      int32_t *err_flags, pkv_stream_t stream);

/* Workspace bytes pkv_extend needs for these arguments (at least 256; 0 on invalid arguments). */
size_t pkv_extend_workspace_size(const pkv_extend_args *args);

/*
 * pkv_span_plan -- query rows and key bounds of attention segments.
 *
 * The diffusion KV path's segments (vllm-omni, "Attention execution"): request
 * b has segments seg_indptr[b] .. seg_indptr[b+1]-1, each (kind, start, end)
 * over positions [start, end) of its sequence; kind 0 is causal (position p
 * sees keys [0, p + 1)), kind 1 is full (every position sees [0, end)).  The
 * query rows of b are its segments' positions in order:
 *     q_pos[j] = p,  kv_end[j] = the bound above,  qo_indptr[b+1] = qo_indptr[b] + sum of b's segment lengths
 * (qo_indptr[0] = 0) -- the inputs pkv_extend takes, with q gathered at q_pos.
 * A segment with end < start, start < 0 or another kind raises
 * PKV_DEVERR_RANGE and is skipped; rows past cap raise PKV_DEVERR_CAPACITY and
 * are not written.  One CTA per request.
 */
pkv_status pkv_span_plan(int32_t batch, const int32_t *seg_indptr, const int32_t *seg_kind,
                         const int32_t *seg_start, const int32_t *seg_end, int32_t *qo_indptr,
                         int32_t *q_pos, int32_t *kv_end, int64_t cap, int32_t *err_flags,
                         pkv_stream_t stream);

/*
 * pkv_alloc_extend -- page allocation for one batch step, on the device.
 *
 * The paged allocator's growth path ("Enabling Encoder-Decoder Models on Intel
 * XPU in SGLang", "two pools and a page size": PagedTokenToKVPoolAllocator
 * alloc_extend / alloc_decode): request b grows from prefix_lens[b] to
 * seq_lens[b] tokens.  Its new positions first continue its partly used last
 * page, on the slots after last_loc[b] (the slot of position prefix_lens[b] - 1;
 * read only when prefix_lens[b] % page_size != 0), then take whole new pages
 * from the front of the free list, requests in order; page p covers slots
 * p*page_size .. p*page_size + page_size - 1.  At page_size 1 every new position
 * takes one entry (TokenToKVPoolAllocator.alloc).  This keeps every request's
 * tokens contiguous inside each page, as pkv_build_indices requires.
 *
 * free_pages     device int32 [free_pages_len]; the free list is
 *                free_pages[head .. head + count).
 * free_state     device int32 [2] = {head, count}, read and, on success,
 *                advanced by the pages taken (head += n, count -= n).
 * out_cache_loc  device int32 [out_cap]: the new slots, request order,
 *                positions ascending (sum of seq_lens - prefix_lens entries).
 * A step that needs more pages than count or more slots than out_cap raises
 * PKV_DEVERR_CAPACITY and writes nothing (the allocator returning None); a
 * negative or shrinking length, a last_loc outside the pool or a free page id
 * outside [0, num_pool_pages) raises PKV_DEVERR_RANGE, a last_loc at the wrong
 * page offset PKV_DEVERR_CONTIG, and nothing is written either.
 * Supported: batch <= 8192.  Asynchronous on `stream`.
 */
pkv_status pkv_alloc_extend(const int32_t *prefix_lens, const int32_t *seq_lens, const int32_t *last_loc,
                            int32_t batch, int32_t page_size, int64_t num_pool_pages,
                            const int32_t *free_pages, int64_t free_pages_len, int32_t *free_state,
                            int32_t *out_cache_loc, int64_t out_cap, int32_t *err_flags,
                            pkv_stream_t stream);

/*
 * pkv_write_req_to_token -- lay a step's slots into the requests' rows.
 *
 * write_cache_indices / write_req_to_token_pool (same page, "how those slot
 * numbers are handed out"): for request b, columns kv_start[b] + [0,
 * prefix_lens[b]) of row req_pool_idx[b] receive prefix_slots[b][0 ..
 * prefix_lens[b]) (the reused prefix; a NULL entry, or prefix_slots NULL, leaves
 * those columns as they are), and columns kv_start[b] + [prefix_lens[b],
 * seq_lens[b]) receive out_cache_loc[e_b ..], e_b being the sum of
 * seq_lens - prefix_lens over the requests before b.  prefix_slots is a device
 * array of device pointers.  kv_start may be NULL (0).  A request whose row or
 * columns fall outside the table raises PKV_DEVERR_RANGE and is skipped.
 */
pkv_status pkv_write_req_to_token(int32_t *req_to_token, int64_t r2t_rows, int64_t r2t_row_stride,
                                  int64_t r2t_width, const int32_t *req_pool_idx, const int32_t *kv_start,
                                  const int32_t *prefix_lens, const int32_t *seq_lens,
                                  const int32_t *const *prefix_slots, const int32_t *out_cache_loc,
                                  int32_t batch, int32_t *err_flags, pkv_stream_t stream);

/*
 * pkv_encoder_merge -- gather encoder-cache blocks into positioned hidden rows.
 *
 * The Neuron encoder cache ("Read Path", "Merge Inside Compiled Graph"): the
 * buffer holds [num_blocks, block_size] rows of row_bytes bytes (the last
 * block is scratch); block slot i of the step names block block_ids[i], and
 * positions [max_blocks, block_size] (int64) says where each of its tokens
 * lands:
 *     hidden[positions[i][j]] = buffer[block_ids[i]][j]   if 0 <= positions[i][j] < num_tokens
 * A position at or past num_tokens is the sentinel (a don't-care: nothing is
 * written, the pages' discarded dummy row).  A negative position, or a block id
 * outside [0, num_blocks) for a non-sentinel position, raises PKV_DEVERR_RANGE
 * and that entry is skipped.  hidden rows are hidden_row_stride_bytes apart.
 * filled (device uint64, nullable) is incremented by the number of rows
 * written, for the fail-loud check that every scheduled position was filled;
 * zero it before the call.  Positions are expected to be distinct.
 */
pkv_status pkv_encoder_merge(const void *buffer, int64_t num_blocks, int64_t block_size, int64_t row_bytes,
                             const int32_t *block_ids, const int64_t *positions, int64_t max_blocks,
                             void *hidden, int64_t num_tokens, int64_t hidden_row_stride_bytes,
                             uint64_t *filled, int32_t *err_flags, pkv_stream_t stream);

/* Static description of a status code. */
const char *pkv_status_string(pkv_status status);

/* One-line reason for the last non-OK status returned on this host thread ("" if none). */
const char *pkv_last_error(void);

/* PKV_ABI_VERSION of the loaded library. */
int32_t pkv_abi_version(void);

/*
 * pkv_set_wait_limit -- bound of every wait inside the library's kernels.
 *
 * Failure detection without a hang, after the fail-loud checks of the AWS
 * Neuron encoder-cache doc ("Read Path"): the kernels that pipeline through
 * mbarriers (the TMA decode, MLA decode and pkv_extend kernels) wait on them
 * for at most this many nanoseconds.  A wait that runs out raises
 * PKV_DEVERR_TIMEOUT in err_flags and makes its CTA give up: every CTA that
 * sees the flag stops waiting, lets the copies and MMAs it already issued
 * complete, frees its tensor memory and returns, so the launch ends and the
 * context stays usable; the launch's outputs are unspecified.  The limit
 * applies to launches issued after the call, from any host thread.
 * nanoseconds = 0 restores the default (about 2 s, far above any legitimate
 * wait); a limit of a few nanoseconds makes the first wait that is not already
 * satisfied give up, which is how the give-up path is exercised in tests.
 * Always returns PKV_OK.
 */
pkv_status pkv_set_wait_limit(uint64_t nanoseconds);

/* The current wait limit in nanoseconds. */
uint64_t pkv_wait_limit(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
