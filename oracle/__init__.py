"""CPU oracle for paged-KV attention (fp64, plain C) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does, and the two
share no code.  ``build()`` compiles ``pkv_oracle.c`` with gcc (OpenMP over
(request, head) pairs; each reduction stays sequential, so results do not
depend on the thread count).

All functions take numpy arrays; bf16 tensors are passed as their uint16 bit
patterns.  Each mirrors a function of ``pkv_oracle.c``, whose comments cite the
passages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")

OK, ERR_RANGE, ERR_CONTIG, ERR_CAPACITY, ERR_ARG = 0, 1, 2, 3, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (portable flags: runs on x86 and Arm)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # The mutation tests point this at a deliberately broken copy of the
        # oracle to show that the pins catch it; nothing else sets it.
        override = os.environ.get("PKV_ORACLE_LIB")
        if override:
            lib = ctypes.CDLL(override)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.pkvo_build_indices.argtypes = [P, I64, I64, I64, P, P, P, I32, I32, I64, P, P, I64, P, P, I32]
        lib.pkvo_build_indices.restype = ctypes.c_int
        lib.pkvo_store.argtypes = [P, I64, I64, I64, P, I64, P, I32]
        lib.pkvo_store.restype = ctypes.c_int
        lib.pkvo_decode.argtypes = [P, I32, I32, I32, I32, I32, P, I64, P, I64, I64,
                                    P, I64, I64, I64, P, P, P, D, I32, I32, P, P, P, I32]
        lib.pkvo_decode.restype = ctypes.c_int
        lib.pkvo_lse_merge.argtypes = [I32, I64, I32, P, P, P, P]
        lib.pkvo_lse_merge.restype = None
        lib.pkvo_ragged_gather.argtypes = [P, P, I64, I64, I64, P, I64, I64, I64, P, P, P, I32,
                                           P, P, I64, P]
        lib.pkvo_ragged_gather.restype = ctypes.c_int
        lib.pkvo_alloc_extend.argtypes = [P, P, P, I32, I32, I64, P, I64, P, P, I64]
        lib.pkvo_alloc_extend.restype = ctypes.c_int
        lib.pkvo_write_req_to_token.argtypes = [P, I64, I64, I64, P, P, P, P, P, P, I32]
        lib.pkvo_write_req_to_token.restype = ctypes.c_int
        lib.pkvo_encoder_merge.argtypes = [P, I64, I64, I64, P, P, I64, P, I64, I64, P]
        lib.pkvo_encoder_merge.restype = ctypes.c_int
        lib.pkvo_extend.argtypes = [P, I64, I32, P, P, I32, I32, I32, I32, P, I64, P, I64, I64, P, I64, I64, I64,
                                    P, P, P, D, P, P, I32]
        lib.pkvo_extend.restype = ctypes.c_int
        lib.pkvo_span_plan.argtypes = [I32, P, P, P, P, P, P, P, I64]
        lib.pkvo_span_plan.restype = ctypes.c_int
        lib.pkvo_max_threads.argtypes = []
        lib.pkvo_max_threads.restype = ctypes.c_int32
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def max_threads() -> int:
    return int(_load().pkvo_max_threads())


def build_indices(req_to_token, req_pool_idx, seq_lens, page_size, num_pool_pages, kv_start=None,
                  kv_indices_cap=None, bt_width=None):
    """Returns (status, kv_indptr, kv_indices, kv_last_page_len, block_table)."""
    r2t = _i32(req_to_token)
    rpi, sl, ks = _i32(req_pool_idx), _i32(seq_lens), _i32(kv_start)
    B = len(sl)
    npages = -(-sl.astype(np.int64) // page_size)
    cap = int(npages.sum()) if kv_indices_cap is None else int(kv_indices_cap)
    width = int(npages.max()) if (bt_width is None and B) else int(bt_width or 0)
    indptr = np.zeros(B + 1, dtype=np.int32)
    indices = np.zeros(max(cap, 1), dtype=np.int32)
    last = np.zeros(B, dtype=np.int32)
    bt = np.zeros((B, max(width, 1)), dtype=np.int32)
    st = _load().pkvo_build_indices(_ptr(r2t), r2t.shape[0], r2t.shape[1], r2t.shape[1], _ptr(rpi),
                                    _ptr(sl), _ptr(ks), B, page_size, num_pool_pages, _ptr(indptr),
                                    _ptr(indices), cap, _ptr(last), _ptr(bt), width)
    return st, indptr, indices[:cap], last, bt[:, :width]


def store(pool: np.ndarray, new_rows: np.ndarray, slot_mapping) -> int:
    """In-place bitwise row store ``pool[slot_mapping[i]] = new_rows[i]`` (any dtype)."""
    sm = _i32(slot_mapping)
    assert pool.flags["C_CONTIGUOUS"] and new_rows.flags["C_CONTIGUOUS"]
    row_bytes = new_rows[0].nbytes if len(new_rows) else 0
    pool_row = pool.strides[0]
    assert row_bytes <= pool_row
    return _load().pkvo_store(_ptr(pool), pool.shape[0], pool_row, row_bytes, _ptr(new_rows),
                              new_rows.strides[0] if len(new_rows) else 0, _ptr(sm), len(sm))


def decode(q, k_pool, v_pool, req_to_token, req_pool_idx, seq_lens, scale, kv_start=None,
           head_dim_v=None, t_begin=0, t_end=-1, req_mask=None, num_threads=0):
    """fp64 decode attention.  q [B, Hq, Dqk] uint16 (bf16 bits); k_pool [slots, Hkv, Dqk]
    (or [slots, Dqk] latent); v_pool [slots, Hkv, Dv] (or the latent pool again with
    ``head_dim_v`` set).  Returns (status, out [B, Hq, Dv] float64, lse [B, Hq])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k_pool, dtype=np.uint16)
    v = np.ascontiguousarray(v_pool, dtype=np.uint16)
    B, hq, dqk = q.shape
    if k.ndim == 2:       # latent pool: one kv head
        hkv = 1
        k_row = k.shape[1]
    else:
        hkv = k.shape[1]
        k_row = k.shape[1] * k.shape[2]
        assert k.shape[2] == dqk
    if v.ndim == 2:
        v_row = v.shape[1]
        dv = int(head_dim_v) if head_dim_v is not None else v.shape[1]
    else:
        v_row = v.shape[1] * v.shape[2]
        dv = v.shape[2]
    r2t = _i32(req_to_token)
    rpi, sl, ks = _i32(req_pool_idx), _i32(seq_lens), _i32(kv_start)
    mask = None if req_mask is None else np.ascontiguousarray(req_mask, dtype=np.uint8)
    out = np.zeros((B, hq, dv), dtype=np.float64)
    lse = np.zeros((B, hq), dtype=np.float64)
    st = _load().pkvo_decode(_ptr(q), B, hq, hkv, dqk, dv, _ptr(k), k_row, _ptr(v), v_row, k.shape[0],
                             _ptr(r2t), r2t.shape[0], r2t.shape[1], r2t.shape[1], _ptr(rpi), _ptr(ks),
                             _ptr(sl), float(scale), int(t_begin), int(t_end), _ptr(mask), _ptr(out),
                             _ptr(lse), int(num_threads))
    return st, out, lse


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """o_parts [n, rows, dv], lse_parts [n, rows] (float64) -> (out [rows, dv], lse [rows])."""
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    l = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, rows, dv = o.shape
    out = np.zeros((rows, dv), dtype=np.float64)
    lse = np.zeros(rows, dtype=np.float64)
    _load().pkvo_lse_merge(n, rows, dv, _ptr(o), _ptr(l), _ptr(out), _ptr(lse))
    return out, lse


def ragged_gather(k_pool: np.ndarray, v_pool: Optional[np.ndarray], req_to_token, req_pool_idx,
                  seq_lens, kv_start=None, out_rows_cap=None):
    """Returns (status, k_out, v_out, cu_seqlens); rows keep the pool's trailing shape."""
    k = np.ascontiguousarray(k_pool)
    v = None if v_pool is None else np.ascontiguousarray(v_pool)
    r2t = _i32(req_to_token)
    rpi, sl, ks = _i32(req_pool_idx), _i32(seq_lens), _i32(kv_start)
    B = len(sl)
    cap = int(sl.astype(np.int64).sum()) if out_rows_cap is None else int(out_rows_cap)
    k_out = np.zeros((max(cap, 1),) + k.shape[1:], dtype=k.dtype)
    v_out = None if v is None else np.zeros((max(cap, 1),) + v.shape[1:], dtype=v.dtype)
    cu = np.zeros(B + 1, dtype=np.int32)
    st = _load().pkvo_ragged_gather(_ptr(k), _ptr(v), k.shape[0], k.strides[0], k[0].nbytes,
                                    _ptr(r2t), r2t.shape[0], r2t.shape[1], r2t.shape[1], _ptr(rpi),
                                    _ptr(ks), _ptr(sl), B, _ptr(k_out), _ptr(v_out), cap, _ptr(cu))
    return st, k_out[:cap], (None if v_out is None else v_out[:cap]), cu


def alloc_extend(prefix_lens, seq_lens, last_loc, page_size, num_pool_pages, free_pages, free_state, out_cap=None):
    """Page allocation for a batch step.  free_state = [head, count] (updated in place on success).
    Returns (status, out_cache_loc)."""
    pl, sl, ll = _i32(prefix_lens), _i32(seq_lens), _i32(last_loc)
    fp = _i32(free_pages)
    assert isinstance(free_state, np.ndarray) and free_state.dtype == np.int32 and free_state.flags["C_CONTIGUOUS"]
    need = int(np.maximum(sl.astype(np.int64) - pl, 0).sum()) if len(sl) else 0
    cap = need if out_cap is None else int(out_cap)
    out = np.full(max(cap, 1), -1, dtype=np.int32)
    st = _load().pkvo_alloc_extend(_ptr(pl), _ptr(sl), _ptr(ll), len(sl), page_size, num_pool_pages, _ptr(fp),
                                   len(fp), _ptr(free_state), _ptr(out), cap)
    return st, out[:need]


def write_req_to_token(req_to_token, req_pool_idx, prefix_lens, seq_lens, prefix_slots, out_cache_loc,
                       kv_start=None):
    """In-place row writer.  prefix_slots: a list with, per request, an int32 array of
    its reused prefix slots or None (already in place).  Returns the status."""
    r2t = req_to_token
    assert r2t.dtype == np.int32 and r2t.flags["C_CONTIGUOUS"]
    rpi, ks, pl, sl = _i32(req_pool_idx), _i32(kv_start), _i32(prefix_lens), _i32(seq_lens)
    B = len(sl)
    keep = [None if a is None else np.ascontiguousarray(a, dtype=np.int32) for a in prefix_slots]
    ptrs = (ctypes.c_void_p * max(B, 1))(*[(None if a is None else a.ctypes.data) for a in keep] + [None] * (max(B, 1) - B))
    loc = _i32(out_cache_loc) if out_cache_loc is not None and len(out_cache_loc) else np.zeros(1, np.int32)
    return _load().pkvo_write_req_to_token(_ptr(r2t), r2t.shape[0], r2t.shape[1], r2t.shape[1], _ptr(rpi), _ptr(ks),
                                           _ptr(pl), _ptr(sl), ctypes.cast(ptrs, ctypes.c_void_p), _ptr(loc), B)


def encoder_merge(buffer: np.ndarray, block_ids, positions, hidden: np.ndarray):
    """In-place merge of encoder-cache blocks into hidden rows.  buffer [num_blocks, block_size, ...],
    positions [max_blocks, block_size] int64, hidden [num_tokens, ...] (same row bytes).
    Returns (status, rows written)."""
    assert buffer.flags["C_CONTIGUOUS"] and hidden.flags["C_CONTIGUOUS"]
    nb, bs = buffer.shape[0], buffer.shape[1]
    row_bytes = buffer[0, 0].nbytes
    assert hidden[0].nbytes == row_bytes
    bid = _i32(block_ids)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    assert pos.shape == (len(bid), bs)
    filled = np.zeros(1, dtype=np.int64)
    st = _load().pkvo_encoder_merge(_ptr(buffer), nb, bs, row_bytes, _ptr(bid), _ptr(pos), len(bid), _ptr(hidden),
                                    hidden.shape[0], hidden.strides[0], _ptr(filled))
    return st, int(filled[0])


def extend(q, k_pool, v_pool, req_to_token, req_pool_idx, seq_lens, qo_indptr, kv_end, scale, kv_start=None,
           num_threads=0):
    """fp64 multi-query attention: q [total_q, Hq, D] uint16 (bf16 bits), query row j of request b
    (qo_indptr[b] <= j < qo_indptr[b+1]) sees keys [0, kv_end[j]).  Returns (status, out, lse)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k_pool, dtype=np.uint16)
    v = np.ascontiguousarray(v_pool, dtype=np.uint16)
    T, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    r2t = _i32(req_to_token)
    rpi, sl, ks, qi, ke = _i32(req_pool_idx), _i32(seq_lens), _i32(kv_start), _i32(qo_indptr), _i32(kv_end)
    out = np.zeros((T, hq, dv), dtype=np.float64)
    lse = np.zeros((T, hq), dtype=np.float64)
    st = _load().pkvo_extend(_ptr(q), T, len(sl), _ptr(qi), _ptr(ke), hq, hkv, dqk, dv, _ptr(k), k.shape[1] * k.shape[2],
                             _ptr(v), v.shape[1] * v.shape[2], k.shape[0], _ptr(r2t), r2t.shape[0], r2t.shape[1],
                             r2t.shape[1], _ptr(rpi), _ptr(ks), _ptr(sl), float(scale), _ptr(out), _ptr(lse),
                             int(num_threads))
    return st, out, lse


def span_plan(segments, cap=None):
    """segments: per request a list of (kind, start, end), kind 0 = causal, 1 = full.
    Returns (status, qo_indptr, q_pos, kv_end)."""
    B = len(segments)
    ind = np.zeros(B + 1, dtype=np.int32)
    kinds, starts, ends = [], [], []
    for b, segs in enumerate(segments):
        for kd, a, e in segs:
            kinds.append(kd)
            starts.append(a)
            ends.append(e)
        ind[b + 1] = len(kinds)
    total = sum(max(e - a, 0) for segs in segments for _, a, e in segs)
    cap = total if cap is None else int(cap)
    qo = np.zeros(B + 1, dtype=np.int32)
    qp = np.zeros(max(cap, 1), dtype=np.int32)
    ke = np.zeros(max(cap, 1), dtype=np.int32)
    st = _load().pkvo_span_plan(B, _ptr(ind), _ptr(_i32(kinds or [0])), _ptr(_i32(starts or [0])),
                                _ptr(_i32(ends or [0])), _ptr(qo), _ptr(qp), _ptr(ke), cap)
    return st, qo, qp[:total], ke[:total]
