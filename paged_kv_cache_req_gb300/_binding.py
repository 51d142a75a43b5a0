"""Thin ctypes binding over libpkv.so: argument marshalling only.

Every function has the name of the C entry point it calls (see include/pkv.h),
takes torch tensors that already live on the GPU, passes their data pointers,
sizes and the current CUDA stream, and raises :class:`PkvError` on a non-OK
status.  No step of the computation runs here: there is no CPU fallback, and a
missing or unloadable libpkv.so raises at import time.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CAPACITY, PKV_ERR_CUDA = range(5)
PKV_DEVERR_RANGE, PKV_DEVERR_CONTIG, PKV_DEVERR_CAPACITY, PKV_DEVERR_TIMEOUT = 1, 2, 4, 8
PKV_KIND_GQA, PKV_KIND_MLA = 0, 1
PKV_LAYOUT_CSR, PKV_LAYOUT_BLOCK_TABLE, PKV_LAYOUT_VARLEN, PKV_LAYOUT_REQ_TO_TOKEN = 0, 1, 2, 3

EXPORTED_SYMBOLS = ("pkv_build_indices", "pkv_store", "pkv_decode", "pkv_decode_workspace_size",
                    "pkv_decode_no_alloc", "pkv_ragged_gather", "pkv_alloc_extend", "pkv_write_req_to_token",
                    "pkv_encoder_merge", "pkv_extend", "pkv_extend_workspace_size", "pkv_span_plan",
                    "pkv_status_string", "pkv_last_error", "pkv_abi_version", "pkv_set_wait_limit",
                    "pkv_wait_limit")


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__("%s failed: %s (%s)" % (where, _status_name(status), detail))
        self.status = status


def _status_name(st: int) -> str:
    return {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "buffer too small",
            4: "CUDA error"}.get(st, "status %d" % st)


class DecodeArgs(ctypes.Structure):
    """Mirror of ``pkv_decode_args`` (field order and types must match include/pkv.h)."""
    _fields_ = [
        ("kind", ctypes.c_int32), ("layout", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("max_seq_len", ctypes.c_int32), ("kv_chunk", ctypes.c_int32),
        ("block_table_width", ctypes.c_int32), ("num_slots", ctypes.c_int64),
        ("k_row_stride", ctypes.c_int64), ("v_row_stride", ctypes.c_int64),
        ("kv_indices_len", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
        ("kv_last_page_len", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("req_to_token", ctypes.c_void_p), ("r2t_rows", ctypes.c_int64), ("r2t_row_stride", ctypes.c_int64),
        ("r2t_width", ctypes.c_int64), ("req_pool_idx", ctypes.c_void_p), ("kv_start", ctypes.c_void_p),
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
    ]


class ExtendArgs(ctypes.Structure):
    """Mirror of ``pkv_extend_args`` (field order and types must match include/pkv.h)."""
    _fields_ = [
        ("layout", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("max_seq_len", ctypes.c_int32), ("kv_chunk", ctypes.c_int32),
        ("block_table_width", ctypes.c_int32), ("total_q", ctypes.c_int64), ("num_slots", ctypes.c_int64),
        ("k_row_stride", ctypes.c_int64), ("v_row_stride", ctypes.c_int64), ("kv_indices_len", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("qo_indptr", ctypes.c_void_p), ("kv_end", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p), ("kv_last_page_len", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("req_to_token", ctypes.c_void_p), ("r2t_rows", ctypes.c_int64), ("r2t_row_stride", ctypes.c_int64),
        ("r2t_width", ctypes.c_int64), ("req_pool_idx", ctypes.c_void_p), ("kv_start", ctypes.c_void_p),
    ]


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError("libpkv.so is not built (%s); run `python -m paged_kv_cache_req_gb300.build`" % path)
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.pkv_build_indices.argtypes = [P, I64, I64, I64, P, P, P, I32, I32, I64, P, P, I64, P, P, I32, P, P]
    lib.pkv_store.argtypes = [P, P, I64, I64, I64, I32, I32, I32, P, P, P, I32, P, P]
    lib.pkv_decode.argtypes = [ctypes.POINTER(DecodeArgs), P, SZ, P, P]
    lib.pkv_decode_no_alloc.argtypes = [ctypes.POINTER(DecodeArgs), P, P]
    lib.pkv_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs)]
    lib.pkv_decode_workspace_size.restype = SZ
    lib.pkv_ragged_gather.argtypes = [P, P, I64, I64, I64, P, I64, I64, I64, P, P, P, I32, I32, P, P, I64, P, P, P]
    for f in ("pkv_build_indices", "pkv_store", "pkv_decode", "pkv_decode_no_alloc", "pkv_ragged_gather"):
        getattr(lib, f).restype = ctypes.c_int
    lib.pkv_alloc_extend.argtypes = [P, P, P, I32, I32, I64, P, I64, P, P, I64, P, P]
    lib.pkv_write_req_to_token.argtypes = [P, I64, I64, I64, P, P, P, P, P, P, I32, P, P]
    lib.pkv_encoder_merge.argtypes = [P, I64, I64, I64, P, P, I64, P, I64, I64, P, P, P]
    lib.pkv_extend.argtypes = [ctypes.POINTER(ExtendArgs), P, SZ, P, P]
    lib.pkv_extend_workspace_size.argtypes = [ctypes.POINTER(ExtendArgs)]
    lib.pkv_extend_workspace_size.restype = SZ
    lib.pkv_span_plan.argtypes = [I32, P, P, P, P, P, P, P, I64, P, P]
    for fn in (lib.pkv_alloc_extend, lib.pkv_write_req_to_token, lib.pkv_encoder_merge, lib.pkv_extend,
               lib.pkv_span_plan):
        fn.restype = ctypes.c_int
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_last_error.argtypes = []
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_abi_version.argtypes = []
    lib.pkv_abi_version.restype = ctypes.c_int32
    lib.pkv_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.pkv_set_wait_limit.restype = ctypes.c_int
    lib.pkv_wait_limit.argtypes = []
    lib.pkv_wait_limit.restype = ctypes.c_uint64
    return lib


_lib = load_library()


def _check(st: int, where: str):
    if st != PKV_OK:
        raise PkvError(st, where, _lib.pkv_last_error().decode())


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libpkv takes device tensors only (got a %s tensor)" % t.device)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _i32(t: Optional[torch.Tensor], name: str):
    if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
        raise ValueError("%s must be a contiguous int32 tensor" % name)
    return t


def pkv_build_indices(req_to_token, req_pool_idx, seq_lens, page_size, num_pool_pages, err_flags,
                      kv_start=None, kv_indptr=None, kv_indices=None, kv_last_page_len=None,
                      block_table=None, stream=None):
    _i32(req_to_token, "req_to_token")
    B = seq_lens.numel()
    cap = kv_indices.numel() if kv_indices is not None else 0
    bt_w = block_table.shape[1] if block_table is not None else 0
    st = _lib.pkv_build_indices(_p(req_to_token), req_to_token.shape[0], req_to_token.stride(0),
                                req_to_token.shape[1], _p(_i32(req_pool_idx, "req_pool_idx")),
                                _p(_i32(seq_lens, "seq_lens")), _p(_i32(kv_start, "kv_start")), B,
                                int(page_size), int(num_pool_pages), _p(kv_indptr), _p(kv_indices), cap,
                                _p(kv_last_page_len), _p(block_table), bt_w, _p(err_flags), _stream(stream))
    _check(st, "pkv_build_indices")


def pkv_store(k_pool, v_pool, k_new, v_new, slot_mapping, err_flags, stream=None):
    """k_pool [slots, Hkv, D] (or latent [slots, Dl]); k_new [n, Hkv, D] (or [n, Dl])."""
    n = slot_mapping.numel()
    if k_pool.dim() == 2:
        hkv, dk = 1, k_pool.shape[1]
    else:
        hkv, dk = k_pool.shape[1], k_pool.shape[2]
    dv = v_pool.shape[-1] if v_pool is not None else 0
    st = _lib.pkv_store(_p(k_pool), _p(v_pool), k_pool.shape[0], k_pool.stride(0),
                        v_pool.stride(0) if v_pool is not None else 0, hkv, dk, dv, _p(k_new.contiguous()),
                        _p(v_new.contiguous() if v_new is not None else None),
                        _p(_i32(slot_mapping, "slot_mapping")), n, _p(err_flags), _stream(stream))
    _check(st, "pkv_store")


def make_decode_args(kind, layout, q, k_pool, v_pool, out, *, page_size=1, sm_scale, max_seq_len,
                     num_kv_heads=None, head_dim_v=None, kv_indptr=None, kv_indices=None,
                     kv_last_page_len=None, block_table=None, seq_lens=None, cu_seqlens=None, lse=None,
                     kv_chunk=0, req_to_token=None, req_pool_idx=None, kv_start=None, k_new=None,
                     v_new=None) -> DecodeArgs:
    B, hq, dqk = q.shape
    if kind == PKV_KIND_MLA:
        hkv = 1
        dv = int(head_dim_v)
        v_stride = k_pool.stride(0)
    else:
        hkv = int(num_kv_heads if num_kv_heads is not None else k_pool.shape[1])
        dv = v_pool.shape[-1]
        v_stride = v_pool.stride(0)
    a = DecodeArgs()
    a.kind, a.layout, a.batch = kind, layout, B
    a.num_q_heads, a.num_kv_heads, a.head_dim_qk, a.head_dim_v = hq, hkv, dqk, dv
    a.page_size, a.sm_scale, a.max_seq_len, a.kv_chunk = int(page_size), float(sm_scale), int(max_seq_len), int(kv_chunk)
    a.block_table_width = block_table.shape[1] if block_table is not None else 0
    a.num_slots = k_pool.shape[0]
    a.k_row_stride, a.v_row_stride = k_pool.stride(0), v_stride
    a.kv_indices_len = kv_indices.numel() if kv_indices is not None else 0
    if req_to_token is not None:
        _i32(req_to_token, "req_to_token")
        a.r2t_rows, a.r2t_row_stride, a.r2t_width = req_to_token.shape[0], req_to_token.stride(0), req_to_token.shape[1]
    tensors = (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("kv_indptr", kv_indptr),
               ("kv_indices", kv_indices), ("kv_last_page_len", kv_last_page_len),
               ("block_table", block_table), ("seq_lens", seq_lens), ("cu_seqlens", cu_seqlens),
               ("out", out), ("lse", lse), ("req_to_token", req_to_token),
               ("req_pool_idx", _i32(req_pool_idx, "req_pool_idx")), ("kv_start", _i32(kv_start, "kv_start")),
               ("k_new", k_new), ("v_new", v_new))
    for name, t in tensors:
        setattr(a, name, None if t is None else _p(t).value)
    # the struct holds raw pointers: keep the tensors alive as long as it lives
    a._keep = tuple(t for _, t in tensors if t is not None)
    return a


def pkv_decode_workspace_size(args: DecodeArgs) -> int:
    return int(_lib.pkv_decode_workspace_size(ctypes.byref(args)))


def pkv_decode(args: DecodeArgs, workspace: Optional[torch.Tensor], err_flags, stream=None):
    ws_ptr = _p(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.pkv_decode(ctypes.byref(args), ws_ptr, ws_bytes, _p(err_flags), _stream(stream))
    _check(st, "pkv_decode")


def pkv_decode_no_alloc(args: DecodeArgs, err_flags, stream=None):
    """pkv_decode with the library's built-in scratch array instead of a caller workspace."""
    st = _lib.pkv_decode_no_alloc(ctypes.byref(args), _p(err_flags), _stream(stream))
    _check(st, "pkv_decode_no_alloc")


def pkv_ragged_gather(k_pool, v_pool, req_to_token, req_pool_idx, seq_lens, max_seq_len, k_out, v_out,
                      cu_seqlens, err_flags, kv_start=None, stream=None):
    row_elems = k_pool[0].numel()
    st = _lib.pkv_ragged_gather(_p(k_pool), _p(v_pool), k_pool.shape[0], k_pool.stride(0), row_elems,
                                _p(_i32(req_to_token, "req_to_token")), req_to_token.shape[0],
                                req_to_token.stride(0), req_to_token.shape[1],
                                _p(_i32(req_pool_idx, "req_pool_idx")), _p(_i32(kv_start, "kv_start")),
                                _p(_i32(seq_lens, "seq_lens")), seq_lens.numel(), int(max_seq_len), _p(k_out),
                                _p(v_out), k_out.shape[0], _p(_i32(cu_seqlens, "cu_seqlens")), _p(err_flags),
                                _stream(stream))
    _check(st, "pkv_ragged_gather")


def pkv_alloc_extend(prefix_lens, seq_lens, last_loc, page_size, num_pool_pages, free_pages, free_state,
                     out_cache_loc, err_flags, stream=None):
    """Device page allocation for one step; free_state is a device int32 [2] = {head, count}."""
    B = seq_lens.numel()
    st = _lib.pkv_alloc_extend(_p(_i32(prefix_lens, "prefix_lens")), _p(_i32(seq_lens, "seq_lens")),
                               _p(_i32(last_loc, "last_loc")), B, int(page_size), int(num_pool_pages),
                               _p(_i32(free_pages, "free_pages")), free_pages.numel(),
                               _p(_i32(free_state, "free_state")), _p(_i32(out_cache_loc, "out_cache_loc")),
                               out_cache_loc.numel(), _p(err_flags), _stream(stream))
    _check(st, "pkv_alloc_extend")


def pkv_write_req_to_token(req_to_token, req_pool_idx, prefix_lens, seq_lens, out_cache_loc, err_flags,
                           prefix_slots=None, kv_start=None, stream=None):
    """prefix_slots: None, or a device int64 tensor [B] of device pointers (0 = leave the prefix as is)."""
    B = seq_lens.numel()
    if prefix_slots is not None and (prefix_slots.dtype != torch.int64 or prefix_slots.numel() != B):
        raise ValueError("prefix_slots must be an int64 tensor of B device pointers")
    st = _lib.pkv_write_req_to_token(_p(_i32(req_to_token, "req_to_token")), req_to_token.shape[0],
                                     req_to_token.stride(0), req_to_token.shape[1],
                                     _p(_i32(req_pool_idx, "req_pool_idx")), _p(_i32(kv_start, "kv_start")),
                                     _p(_i32(prefix_lens, "prefix_lens")), _p(_i32(seq_lens, "seq_lens")),
                                     _p(prefix_slots), _p(_i32(out_cache_loc, "out_cache_loc")), B, _p(err_flags),
                                     _stream(stream))
    _check(st, "pkv_write_req_to_token")


def pkv_encoder_merge(buffer, block_ids, positions, hidden, err_flags, filled=None, stream=None):
    """buffer [num_blocks, block_size, ...], positions int64 [max_blocks, block_size], hidden [num_tokens, ...]."""
    if positions.dtype != torch.int64 or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous int64 tensor")
    if not buffer.is_contiguous():
        raise ValueError("buffer must be contiguous")
    nb, bs = buffer.shape[0], buffer.shape[1]
    row_bytes = buffer[0, 0].numel() * buffer.element_size()
    if hidden[0].numel() * hidden.element_size() != row_bytes or hidden.stride(-1) != 1:
        raise ValueError("hidden rows must match the buffer's rows")
    st = _lib.pkv_encoder_merge(_p(buffer), nb, bs, row_bytes, _p(_i32(block_ids, "block_ids")), _p(positions),
                                block_ids.numel(), _p(hidden), hidden.shape[0], hidden.stride(0) * hidden.element_size(),
                                _p(filled), _p(err_flags), _stream(stream))
    _check(st, "pkv_encoder_merge")


def make_extend_args(layout, q, k_pool, v_pool, out, qo_indptr, *, page_size, sm_scale, max_seq_len,
                     kv_end=None, kv_indptr=None, kv_indices=None, kv_last_page_len=None, block_table=None,
                     seq_lens=None, lse=None, kv_chunk=0, req_to_token=None, req_pool_idx=None,
                     kv_start=None) -> ExtendArgs:
    """q [total_q, Hq, D]; pools [slots, Hkv, D]; req_to_token [rows, width] (token-table layout)."""
    T, hq, d = q.shape
    a = ExtendArgs()
    a.layout, a.batch = layout, qo_indptr.numel() - 1
    a.num_q_heads, a.num_kv_heads, a.head_dim = hq, k_pool.shape[1], d
    a.page_size, a.sm_scale, a.max_seq_len, a.kv_chunk = int(page_size), float(sm_scale), int(max_seq_len), int(kv_chunk)
    a.block_table_width = block_table.shape[1] if block_table is not None else 0
    a.total_q, a.num_slots = T, k_pool.shape[0]
    a.k_row_stride, a.v_row_stride = k_pool.stride(0), v_pool.stride(0)
    a.kv_indices_len = kv_indices.numel() if kv_indices is not None else 0
    if req_to_token is not None:
        a.r2t_rows, a.r2t_width = req_to_token.shape
        a.r2t_row_stride = req_to_token.stride(0)
    tensors = (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("qo_indptr", qo_indptr), ("kv_end", kv_end),
               ("kv_indptr", kv_indptr), ("kv_indices", kv_indices), ("kv_last_page_len", kv_last_page_len),
               ("block_table", block_table), ("seq_lens", seq_lens), ("out", out), ("lse", lse),
               ("req_to_token", req_to_token), ("req_pool_idx", req_pool_idx), ("kv_start", kv_start))
    for name, t in tensors:
        setattr(a, name, None if t is None else _p(t).value)
    # the struct holds raw pointers: keep the tensors alive as long as it lives
    a._keep = tuple(t for _, t in tensors if t is not None)
    return a


def pkv_extend_workspace_size(args: ExtendArgs) -> int:
    return int(_lib.pkv_extend_workspace_size(ctypes.byref(args)))


def pkv_extend(args: ExtendArgs, workspace: Optional[torch.Tensor], err_flags, stream=None):
    ws_ptr = _p(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.pkv_extend(ctypes.byref(args), ws_ptr, ws_bytes, _p(err_flags), _stream(stream))
    _check(st, "pkv_extend")


def pkv_span_plan(seg_indptr, seg_kind, seg_start, seg_end, qo_indptr, q_pos, kv_end, err_flags, stream=None):
    B = seg_indptr.numel() - 1
    st = _lib.pkv_span_plan(B, _p(_i32(seg_indptr, "seg_indptr")), _p(_i32(seg_kind, "seg_kind")),
                            _p(_i32(seg_start, "seg_start")), _p(_i32(seg_end, "seg_end")),
                            _p(_i32(qo_indptr, "qo_indptr")), _p(_i32(q_pos, "q_pos")), _p(_i32(kv_end, "kv_end")),
                            q_pos.numel(), _p(err_flags), _stream(stream))
    _check(st, "pkv_span_plan")


def pkv_status_string(status: int) -> str:
    return _lib.pkv_status_string(status).decode()


def pkv_abi_version() -> int:
    return int(_lib.pkv_abi_version())


def pkv_set_wait_limit(nanoseconds: int = 0):
    """Bound of every in-kernel wait for launches issued from now on (0: the default, about 2 s)."""
    _check(_lib.pkv_set_wait_limit(int(nanoseconds)), "pkv_set_wait_limit")


def pkv_wait_limit() -> int:
    return int(_lib.pkv_wait_limit())
