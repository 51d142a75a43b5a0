"""The C ABI: libpkv.so loads, exports every function include/pkv.h declares, the
ctypes mirror of pkv_decode_args has the C layout, and host-side argument checks
return a status before anything touches a GPU (no compute calls here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def binding():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def test_every_declared_symbol_is_exported(binding):
    lib = ctypes.CDLL(binding._LIB_PATH)
    names = declared_functions()
    assert set(binding.EXPORTED_SYMBOLS) <= set(names)
    for name in names:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding._LIB_PATH], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r"\bT (pkv_\w+)", out.stdout))
        assert set(names) <= exported


def test_decode_args_layout_matches_c(binding, tmp_path):
    fields = [f[0] for f in binding.DecodeArgs._fields_]
    src = tmp_path / "layout.c"
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "pkv.h"', "int main(void){",
             'printf("%zu\\n", sizeof(pkv_decode_args));']
    lines += ['printf("%%zu\\n", offsetof(pkv_decode_args, %s));' % f for f in fields]
    lines += ["return 0;}"]
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    vals = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert vals[0] == ctypes.sizeof(binding.DecodeArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(binding.DecodeArgs, f).offset == off, f


def test_extend_args_layout_matches_c(binding, tmp_path):
    fields = [f[0] for f in binding.ExtendArgs._fields_]
    src = tmp_path / "layout_ext.c"
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "pkv.h"', "int main(void){",
             'printf("%zu\\n", sizeof(pkv_extend_args));']
    lines += ['printf("%%zu\\n", offsetof(pkv_extend_args, %s));' % f for f in fields]
    lines += ["return 0;}"]
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout_ext"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    vals = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert vals[0] == ctypes.sizeof(binding.ExtendArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(binding.ExtendArgs, f).offset == off, f
    # host-side validation before any launch
    a = binding.ExtendArgs()
    flag = ctypes.c_int32(0)
    a.batch, a.num_q_heads, a.num_kv_heads, a.head_dim, a.page_size = 1, 12, 4, 128, 16
    assert binding._lib.pkv_extend(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_UNSUPPORTED
    a.num_q_heads, a.head_dim = 16, 96
    assert binding._lib.pkv_extend(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_UNSUPPORTED
    a.head_dim, a.page_size = 128, 24                  # not a power of two
    assert binding._lib.pkv_extend(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_UNSUPPORTED
    assert binding._lib.pkv_extend_workspace_size(ctypes.byref(a)) == 0
    # token-table layout: the table's shape and pointers are checked before any launch
    dummy = ctypes.c_void_p(256).value
    a.page_size, a.layout, a.total_q, a.num_slots = 16, binding.PKV_LAYOUT_REQ_TO_TOKEN, 4, 64
    a.k_row_stride = a.v_row_stride = 4 * 128
    a.q = a.k_pool = a.v_pool = a.out = a.qo_indptr = dummy
    a.r2t_rows, a.r2t_width, a.r2t_row_stride = 2, 64, 32    # stride narrower than the rows
    assert binding._lib.pkv_extend(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    assert b"req_to_token" in binding._lib.pkv_last_error()
    a.r2t_row_stride = 64
    a.req_to_token = a.req_pool_idx = a.seq_lens = None       # the table itself missing
    assert binding._lib.pkv_extend(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    assert b"token-table" in binding._lib.pkv_last_error()
    a.req_to_token = a.req_pool_idx = a.seq_lens = dummy      # valid: the plan has a size
    a.max_seq_len = 64
    assert binding._lib.pkv_extend_workspace_size(ctypes.byref(a)) >= 256
    assert flag.value == 0


def test_status_strings_and_version(binding):
    assert binding.pkv_abi_version() == 3
    assert binding.pkv_status_string(0) == "ok"
    assert binding.pkv_status_string(2) == "unsupported shape"


def test_host_side_validation_needs_no_gpu(binding):
    lib = binding._lib
    # null args / missing err_flags are rejected before any CUDA call
    assert lib.pkv_decode(None, None, 0, None, None) == binding.PKV_ERR_INVALID_ARG
    a = binding.DecodeArgs()
    assert lib.pkv_decode(ctypes.byref(a), None, 0, None, None) == binding.PKV_ERR_INVALID_ARG
    assert b"err_flags" in lib.pkv_last_error()
    flag = ctypes.c_int32(0)
    # unsupported head dim
    a.kind, a.layout, a.batch, a.num_q_heads, a.num_kv_heads = 0, 0, 1, 8, 2
    a.head_dim_qk = a.head_dim_v = 96
    a.page_size = 16
    assert lib.pkv_decode(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_UNSUPPORTED
    # non power-of-two page size for a paged layout
    a.head_dim_qk = a.head_dim_v = 128
    a.page_size = 12
    assert lib.pkv_decode(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_UNSUPPORTED
    # query heads not a multiple of kv heads
    a.page_size, a.num_q_heads = 16, 7
    assert lib.pkv_decode(ctypes.byref(a), None, 0, ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.pkv_decode_workspace_size(ctypes.byref(a)) == 0
    # build_indices: negative batch, no outputs
    assert lib.pkv_build_indices(None, 0, 0, 0, None, None, None, -1, 1, 0, None, None, 0, None, None, 0,
                                 ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.pkv_build_indices(None, 0, 0, 0, None, None, None, 0, 1, 0, None, None, 0, None, None, 0,
                                 ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    # store: v_pool without v_new
    assert lib.pkv_store(ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 8, 8, 1, 8, 8, ctypes.c_void_p(16), None,
                         ctypes.c_void_p(16), 1, ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    # gather: row stride smaller than a row
    assert lib.pkv_ragged_gather(None, None, 4, 4, 8, None, 1, 1, 1, None, None, None, 0, 0, None, None, 0,
                                 ctypes.byref(flag), ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    # allocator: page size 0, missing free_state, too many requests; an empty step is a no-op
    state = (ctypes.c_int32 * 2)(0, 0)
    dummy = ctypes.c_void_p(16)
    assert lib.pkv_alloc_extend(dummy, dummy, dummy, 1, 0, 8, dummy, 1, state, dummy, 1, ctypes.byref(flag),
                                None) == binding.PKV_ERR_INVALID_ARG
    assert lib.pkv_alloc_extend(dummy, dummy, dummy, 1, 16, 8, dummy, 1, None, dummy, 1, ctypes.byref(flag),
                                None) == binding.PKV_ERR_INVALID_ARG
    assert lib.pkv_alloc_extend(dummy, dummy, dummy, 9000, 16, 8, dummy, 1, state, dummy, 1, ctypes.byref(flag),
                                None) == binding.PKV_ERR_UNSUPPORTED
    assert lib.pkv_alloc_extend(None, None, None, 0, 16, 8, None, 0, state, None, 0, ctypes.byref(flag),
                                None) == binding.PKV_OK
    # row writer: stride narrower than the rows; encoder merge: hidden rows narrower than buffer rows
    assert lib.pkv_write_req_to_token(dummy, 4, 8, 16, dummy, None, dummy, dummy, None, dummy, 1,
                                      ctypes.byref(flag), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.pkv_encoder_merge(dummy, 4, 8, 64, dummy, dummy, 2, dummy, 10, 32, None, ctypes.byref(flag),
                                 None) == binding.PKV_ERR_INVALID_ARG
    assert lib.pkv_encoder_merge(None, 4, 8, 64, None, None, 0, None, 10, 64, None, ctypes.byref(flag),
                                 None) == binding.PKV_OK
    assert flag.value == 0


def test_workspace_size_follows_split_plan(binding):
    a = binding.DecodeArgs()
    a.kind, a.layout, a.batch, a.num_q_heads, a.num_kv_heads = 0, 0, 4, 16, 8
    a.head_dim_qk = a.head_dim_v = 128
    a.page_size, a.sm_scale = 16, 0.088
    a.k_row_stride = a.v_row_stride = 8 * 128
    a.max_seq_len, a.kv_chunk = 64, 64          # one chunk per request: no partials
    assert lib_ws(binding, a) == 0
    a.max_seq_len = 256                           # four chunks of 64 keys
    parts = 4 * 8 * 1 * 4 * 2                     # B * Hkv * hsplit * chunks * heads-per-CTA
    expect = -(-parts * 128 * 4 // 256) * 256 + -(-parts * 4 // 256) * 256
    assert lib_ws(binding, a) == expect


def lib_ws(binding, a):
    return int(binding._lib.pkv_decode_workspace_size(ctypes.byref(a)))


def test_wait_limit_round_trip(binding):
    """pkv_set_wait_limit is host state only; 0 restores the ~2 s default."""
    default = binding.pkv_wait_limit()
    assert default == 2_000_000_000
    binding.pkv_set_wait_limit(12345)
    assert binding.pkv_wait_limit() == 12345
    binding.pkv_set_wait_limit(0)
    assert binding.pkv_wait_limit() == default
