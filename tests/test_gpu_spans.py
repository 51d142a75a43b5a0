"""GQA decode with equal spans of tiles (the split for small batches) against the oracle.

When the library chooses the split (kv_chunk = 0) and even the longest requests
would give each of about 2 x SMs spans (3 x SMs at head_dim 64) only a few items, pkv_decode concatenates the
requests' rows of each kv head as tiles of 64 keys and cuts that sequence into equal
spans;
a row cut by a span boundary writes partials that a log-sum-exp merge combines,
exactly as the pieces of a long request are combined ("init_forward_metadata":
num_splits and the merge of split results).  The result is the same softmax
attention as the oracle's fp64 walk of req_to_token, within |err| <= 2e-2 +
2e-2 |ref|.  The workspace size tells which split the library chose.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from _harness import assert_close, bf16_to_f64, bits, paged_table
from test_gpu_parity import _direct_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _r256(x):
    return (x + 255) // 256 * 256


def _span_ws(hq, hkv, d):
    """Workspace of the span split: two partial slots per span, the same whole number of spans
    per kv head (2 x SMs at most, 3 x SMs at head_dim 64: one per CTA the SMs hold), and the
    span records."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    gc = min(hq // hkv, 16)
    units = hkv * (hq // hkv // gc)
    spans = units * ((3 if d == 64 else 2) * sm // units)
    return _r256(2 * spans * gc * d * 4) + _r256(2 * spans * gc * 4) + _r256((spans + 1) * 16)


def _ws(B, lens, ps, hq, hkv, d, chunk):
    dev = torch.device("cuda")
    n = len(lens)
    args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_BLOCK_TABLE,
                              torch.empty((n, hq, d), dtype=torch.bfloat16, device=dev),
                              torch.empty((64, hkv, d), dtype=torch.bfloat16, device=dev),
                              torch.empty((64, hkv, d), dtype=torch.bfloat16, device=dev),
                              torch.empty((n, hq, d), dtype=torch.bfloat16, device=dev), page_size=ps,
                              sm_scale=0.1, max_seq_len=max(lens),
                              block_table=torch.zeros((n, 1), dtype=torch.int32, device=dev),
                              seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev), kv_chunk=chunk)
    return B.pkv_decode_workspace_size(args)


def test_small_batches_take_spans_and_large_ones_pieces(B):
    # batch 32 x 8 kv heads x 4096 keys: a few items per CTA -> spans
    assert _ws(B, [4096] * 32, 16, 16, 8, 128, 0) == _span_ws(16, 8, 128)
    # an explicit kv_chunk keeps the pieces
    assert _ws(B, [4096] * 32, 16, 16, 8, 128, 1024) != _span_ws(16, 8, 128)
    # batch 256 x 32k keys: many items per CTA -> pieces (round-robin)
    assert _ws(B, [32768] * 256, 64, 32, 8, 128, 0) != _span_ws(32, 8, 128)
    # pages of < 8 keys go to the cp.async kernel, which cuts pieces
    assert _ws(B, [4096] * 4, 4, 16, 8, 128, 0) != _span_ws(16, 8, 128)


@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 128), (32, 2, 128), (20, 20, 64), (64, 4, 64)])
def test_one_long_request_cut_by_many_spans(B, hq, hkv, d):
    """One request whose rows each cross dozens of span boundaries."""
    lens = [20000]
    assert _ws(B, lens, 16, hq, hkv, d, 0) == _span_ws(hq, hkv, d)
    gpu, g_lse, ref, ref_lse = _direct_decode(B, lens, 16, hq, hkv, d, seed=hq + d)
    assert_close(gpu, ref, "one long request hq=%d hkv=%d d=%d" % (hq, hkv, d))
    assert_close(g_lse, ref_lse, "one long request (lse)")


def test_spans_with_mostly_empty_requests(B):
    rng = np.random.default_rng(11)
    lens = [0] * 40 + [int(x) for x in rng.integers(1, 3000, 10)]
    rng.shuffle(lens)
    assert _ws(B, lens, 64, 16, 8, 128, 0) == _span_ws(16, 8, 128)
    gpu, g_lse, ref, ref_lse = _direct_decode(B, lens, 64, 16, 8, 128, seed=12)
    assert_close(gpu, ref, "mostly empty")
    for b, L in enumerate(lens):
        if L == 0:
            assert (gpu[b] == 0).all() and np.isneginf(g_lse[b]).all()
        else:
            assert_close(g_lse[b], ref_lse[b], "lse of request %d" % b)


@pytest.mark.parametrize("layout", [None, "block_table"])
def test_spans_agree_with_pieces(B, layout):
    """The same inputs split both ways (spans by default, pieces with kv_chunk 256)."""
    rng = np.random.default_rng(21)
    lens = [int(x) for x in rng.integers(1, 4097, 32)]
    a = _direct_decode(B, lens, 16, 16, 8, 128, chunk=0, layout=layout, seed=22)
    b = _direct_decode(B, lens, 16, 16, 8, 128, chunk=256, layout=layout, seed=22)
    assert_close(a[0], a[2], "spans vs oracle")
    assert_close(b[0], b[2], "pieces vs oracle")
    assert_close(a[0], b[0], "spans vs pieces")


def test_varlen_layout_in_spans(B):
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(31)
    lens = [1500] * 24 + [0, 1, 63, 64, 65]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n, rows, hkv, hq, d = len(lens), int(cu[-1]), 20, 20, 64
    k = torch.randn((rows, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((rows, hkv, d), generator=gen).to(torch.bfloat16)
    q = torch.randn((n, hq, d), generator=gen).to(torch.bfloat16)
    r2t = np.zeros((n + 1, max(lens)), dtype=np.int32)
    for b, L in enumerate(lens):
        r2t[b + 1, :L] = np.arange(cu[b], cu[b] + L)
    scale = 1 / math.sqrt(d)
    st, ref, ref_lse = oracle.decode(bits(q), bits(k), bits(v), r2t, np.arange(1, n + 1), lens, scale)
    assert st == oracle.OK
    out = torch.empty((n, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((n, hq), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_VARLEN, q.to(dev), k.to(dev), v.to(dev), out,
                              sm_scale=scale, max_seq_len=max(lens), cu_seqlens=torch.from_numpy(cu).to(dev), lse=lse)
    assert B.pkv_decode_workspace_size(args) == _span_ws(hq, hkv, d)
    ws = torch.empty(B.pkv_decode_workspace_size(args), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_close(bf16_to_f64(out), ref, "varlen spans")
    live = [b for b, L in enumerate(lens) if L > 0]
    assert_close(lse.double().cpu().numpy()[live], ref_lse[live], "varlen spans (lse)")


def test_spans_report_requests_past_max_seq_len(B):
    """A request longer than max_seq_len raises CAPACITY and attends its first keys up to
    the plan's reach, as with pieces: max_seq_len 200 gives pieces of 64 keys (too few
    items for longer ones) and four of them, so the 300-key request attends 256."""
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(41)
    rng = np.random.default_rng(41)
    lens, ps, hq, hkv, d = [100, 300, 50], 16, 16, 8, 128
    num_pages = 4 + sum(-(-L // ps) for L in lens)
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    k = torch.randn((num_pages * ps, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((num_pages * ps, hkv, d), generator=gen).to(torch.bfloat16)
    q = torch.randn((3, hq, d), generator=gen).to(torch.bfloat16)
    st, ref, _ = oracle.decode(bits(q), bits(k), bits(v), r2t, rpi, [100, 256, 50], 0.1)
    assert st == oracle.OK
    for chunk in (0, 64):
        out = torch.empty((3, hq, d), dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_REQ_TO_TOKEN, q.to(dev), k.to(dev), v.to(dev), out,
                                  page_size=ps, sm_scale=0.1, max_seq_len=200,
                                  seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev), kv_chunk=chunk,
                                  req_to_token=torch.from_numpy(r2t).to(dev), req_pool_idx=torch.from_numpy(rpi).to(dev))
        assert (B.pkv_decode_workspace_size(args) == _span_ws(hq, hkv, d)) == (chunk == 0)
        ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
        B.pkv_decode(args, ws, err)
        torch.cuda.synchronize()
        assert err.item() == B.PKV_DEVERR_CAPACITY
        assert_close(bf16_to_f64(out), ref, "past max_seq_len, kv_chunk %d" % chunk)
