"""GPU parity of pkv_extend (multi-query paged attention) and pkv_span_plan against the oracle.

Outputs are compared with the fp64 oracle elementwise within
|gpu - oracle| <= 2e-2 + 2e-2 |oracle| (bf16 output, fp32 accumulation); the
span planner's rows and bounds bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from _harness import assert_close, bf16_to_f64, bits, paged_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.asarray(a)).to(dtype).cuda()


def _case(seed, lens, nq, hq, hkv, d, ps):
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    num_pages = sum(-(-L // ps) for L in lens) + 8
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    k = torch.randn((num_pages * ps, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((num_pages * ps, hkv, d), generator=gen).to(torch.bfloat16)
    qo = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = torch.randn((int(qo[-1]), hq, d), generator=gen).to(torch.bfloat16)
    return r2t, rpi, num_pages, k, v, q, qo


def _run(B, r2t, rpi, num_pages, k, v, q, qo, lens, ps, kv_end=None, chunk=0, layout="csr"):
    dev = torch.device("cuda")
    hq, d = q.shape[1], q.shape[2]
    scale = 1 / math.sqrt(d)
    st, indptr, indices, last, bt = oracle.build_indices(r2t, rpi, lens, ps, num_pages)
    assert st == oracle.OK
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((q.shape[0], hq), dtype=torch.float32, device=dev)
    kw = dict(page_size=ps, sm_scale=scale, max_seq_len=max(max(lens), 1), lse=lse, kv_chunk=chunk,
              kv_end=None if kv_end is None else _dev(kv_end))
    kd, vd, qd = k.to(dev), v.to(dev), q.to(dev)
    if layout == "csr":
        args = B.make_extend_args(B.PKV_LAYOUT_CSR, qd, kd, vd, out, _dev(qo), kv_indptr=_dev(indptr),
                                  kv_indices=_dev(indices if len(indices) else [0]), kv_last_page_len=_dev(last), **kw)
    elif layout == "token":
        args = B.make_extend_args(B.PKV_LAYOUT_REQ_TO_TOKEN, qd, kd, vd, out, _dev(qo), seq_lens=_dev(lens),
                                  req_to_token=_dev(r2t), req_pool_idx=_dev(rpi), **kw)
    else:
        args = B.make_extend_args(B.PKV_LAYOUT_BLOCK_TABLE, qd, kd, vd, out, _dev(qo), block_table=_dev(bt),
                                  seq_lens=_dev(lens), **kw)
    ws = torch.empty(max(B.pkv_extend_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    B.pkv_extend(args, ws, err)
    torch.cuda.synchronize()
    if kv_end is None:
        kv_end = np.concatenate([np.arange(L - n, L) + 1 for L, n in zip(lens, np.diff(qo))]).astype(np.int32)
    st, ref, ref_lse = oracle.extend(bits(q), bits(k), bits(v), r2t, rpi, lens, qo, kv_end, scale)
    return err.item(), bf16_to_f64(out), lse.double().cpu().numpy(), st, ref, ref_lse


@pytest.mark.parametrize("layout", ["csr", "token"])
@pytest.mark.parametrize("hq,hkv,d,ps", [(32, 8, 128, 64), (16, 16, 128, 16), (8, 1, 64, 8), (32, 4, 128, 32),
                                         (16, 1, 128, 64)])
def test_extend_causal_mix(B, hq, hkv, d, ps, layout):
    # prefill (n = L), chunked prefill (n < L), one new token, 4 draft tokens, long prefix;
    # through the page list and straight through the token table
    lens = [300, 517, 129, 1000, 64, 3001]
    nq = [300, 200, 1, 4, 64, 37]
    case = _case(hq + d + ps, lens, nq, hq, hkv, d, ps)
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, ps, layout=layout)
    assert e == 0 and st == oracle.OK
    assert_close(gpu, ref, "extend out hq=%d hkv=%d d=%d ps=%d %s" % (hq, hkv, d, ps, layout))
    assert_close(g_lse, ref_lse, "extend lse")


@pytest.mark.parametrize("ps", [1, 2, 4])
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 2, 64)])
def test_extend_small_pages_gathered_by_rows(B, ps, hq, hkv, d):
    # pages under 8 keys: the producer gathers rows with cp.async instead of TMA boxes
    lens = [300, 77, 1000, 1, 129]
    nq = [300, 5, 64, 1, 16]
    for chunk, layout in ((0, "csr"), (64, "csr"), (64, "token")):
        case = _case(ps * 10 + d + chunk, lens, nq, hq, hkv, d, ps)
        e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, ps, chunk=chunk, layout=layout)
        assert e == 0 and st == oracle.OK
        assert_close(gpu, ref, "extend ps=%d d=%d chunk=%d %s" % (ps, d, chunk, layout))
        assert_close(g_lse, ref_lse, "extend lse ps=%d" % ps)


@pytest.mark.parametrize("chunk", [64, 192, 1024])
@pytest.mark.parametrize("layout", ["csr", "block_table", "token"])
def test_extend_split_keys_and_layouts(B, chunk, layout):
    lens = [2000, 77, 900, 4100]
    nq = [4, 77, 16, 9]
    case = _case(chunk, lens, nq, 32, 8, 128, 16)
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, 16, chunk=chunk, layout=layout)
    assert e == 0 and st == oracle.OK
    assert_close(gpu, ref, "extend split %d %s" % (chunk, layout))
    assert_close(g_lse, ref_lse, "extend split lse")


def test_span_plan_and_span_attention(B):
    # a diffusion row: causal text prefix then a full image span, and a later step
    # that queries only the image span against prefix + image
    segs = [[(0, 0, 100), (1, 100, 356)], [(1, 100, 356)], [(0, 0, 40)], []]
    ind, kinds, starts, ends = [0], [], [], []
    for row in segs:
        for kd, a, e in row:
            kinds.append(kd)
            starts.append(a)
            ends.append(e)
        ind.append(len(kinds))
    st, qo_ref, qpos_ref, kend_ref = oracle.span_plan(segs)
    assert st == oracle.OK
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qo = torch.empty(len(segs) + 1, dtype=torch.int32, device="cuda")
    qpos = torch.empty(len(qpos_ref), dtype=torch.int32, device="cuda")
    kend = torch.empty(len(qpos_ref), dtype=torch.int32, device="cuda")
    B.pkv_span_plan(_dev(ind), _dev(kinds), _dev(starts), _dev(ends), qo, qpos, kend, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert qo.cpu().numpy().tolist() == qo_ref.tolist()
    assert np.array_equal(qpos.cpu().numpy(), qpos_ref) and np.array_equal(kend.cpu().numpy(), kend_ref)
    lens = [356, 356, 40, 10]
    case = list(_case(11, lens, np.diff(qo_ref).tolist(), 16, 4, 128, 16))
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, 16, kv_end=kend_ref)
    assert e == 0 and st == oracle.OK
    assert_close(gpu, ref, "span attention")
    assert_close(g_lse, ref_lse, "span attention lse")


def test_extend_edges(B):
    # a request with no query rows, an empty request with kv_end 0, a row whose bound is 1
    lens = [50, 0, 20, 33]
    nq = [0, 2, 3, 1]
    case = list(_case(5, lens, nq, 8, 2, 64, 8))
    kv_end = np.array([0, 0, 1, 5, 20, 33], np.int32)
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, 8, kv_end=kv_end)
    assert e == 0 and st == oracle.OK
    assert (gpu[:2] == 0).all() and np.isneginf(g_lse[:2]).all()
    assert_close(gpu, ref, "extend edges")
    # a bound past the request's keys is a range error; that row reads as empty
    bad = kv_end.copy()
    bad[3] = 21
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, 8, kv_end=bad)
    assert e == B.PKV_DEVERR_RANGE and st == oracle.ERR_RANGE
    assert (gpu[3] == 0).all()


def test_extend_verify_long_rows(B):
    # few live rows per block (4 draft tokens x 4 heads of 128) over long key ranges, many
    # items per CTA: the idle row groups must stay in step with the live one
    rng = np.random.default_rng(21)
    lens = rng.integers(6000, 20000, 24).tolist()
    nq = [4] * 24
    case = _case(21, lens, nq, 32, 8, 128, 64)
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, 64)
    assert e == 0 and st == oracle.OK
    assert_close(gpu, ref, "verify long rows")
    assert_close(g_lse, ref_lse, "verify long rows lse")


def test_args_structs_keep_their_tensors_alive(B):
    # the structs hold raw pointers: a temporary passed in must outlive the call that built
    # them (a freed q whose memory the next allocation reuses reads back as that allocation)
    import gc
    import weakref
    dev = torch.device("cuda")
    q = torch.zeros((4, 8, 64), dtype=torch.bfloat16, device=dev)
    ref = weakref.ref(q)
    a = B.make_extend_args(B.PKV_LAYOUT_CSR, q, torch.zeros((16, 2, 64), dtype=torch.bfloat16, device=dev),
                           torch.zeros((16, 2, 64), dtype=torch.bfloat16, device=dev),
                           torch.zeros((4, 8, 64), dtype=torch.bfloat16, device=dev),
                           torch.zeros(2, dtype=torch.int32, device=dev), page_size=8, sm_scale=0.125, max_seq_len=16)
    del q
    gc.collect()
    assert ref() is not None and a.q == ref().data_ptr()
    lat = torch.zeros((64, 576), dtype=torch.bfloat16, device=dev)
    lref = weakref.ref(lat)
    d = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_BLOCK_TABLE,
                           torch.zeros((2, 128, 576), dtype=torch.bfloat16, device=dev), lat, None,
                           torch.zeros((2, 128, 512), dtype=torch.bfloat16, device=dev), page_size=64, sm_scale=0.07,
                           max_seq_len=64, head_dim_v=512, block_table=torch.zeros((2, 1), dtype=torch.int32, device=dev),
                           seq_lens=torch.zeros(2, dtype=torch.int32, device=dev))
    del lat
    gc.collect()
    assert lref() is not None and d.k_pool == lref().data_ptr()


@pytest.mark.parametrize("ps", [2, 16])
def test_extend_flags_out_of_pool_pages(B, ps):
    """A page id outside the pool raises PKV_DEVERR_RANGE and reads as zeros, in both producers
    (row gather for pages under 8 keys, TMA boxes otherwise); other requests stay exact."""
    dev = torch.device("cuda")
    lens, nq = [40, 24], [4, 3]
    case = _case(ps, lens, nq, 16, 4, 128, ps)
    r2t, rpi, num_pages, k, v, q, qo = case
    st, indptr, indices, last, bt = oracle.build_indices(r2t, rpi, lens, ps, num_pages)
    assert st == oracle.OK
    bad = np.array(indices, dtype=np.int32)
    bad[0] = num_pages + 5                       # first page of request 0: outside the pool
    out = torch.zeros(tuple(q.shape), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = B.make_extend_args(B.PKV_LAYOUT_CSR, q.to(dev), k.to(dev), v.to(dev), out, _dev(qo), page_size=ps,
                              sm_scale=1 / math.sqrt(128), max_seq_len=max(lens), kv_indptr=_dev(indptr),
                              kv_indices=_dev(bad), kv_last_page_len=_dev(last))
    ws = torch.empty(max(B.pkv_extend_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_extend(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() & B.PKV_DEVERR_RANGE
    assert torch.isfinite(out.float()).all()
    kv_end = np.concatenate([np.arange(L - n, L) + 1 for L, n in zip(lens, nq)]).astype(np.int32)
    st, ref, _ = oracle.extend(bits(q), bits(k), bits(v), r2t, rpi, lens, qo, kv_end, 1 / math.sqrt(128))
    assert st == oracle.OK
    assert_close(bf16_to_f64(out)[qo[1]:], ref[qo[1]:], "valid request next to a bad one, ps=%d" % ps)
    # the bad page reads as zeros: the oracle over a pool whose rows of that page are zero
    page = int(indices[0])
    kz, vz = k.clone(), v.clone()
    kz[page * ps:(page + 1) * ps] = 0
    vz[page * ps:(page + 1) * ps] = 0
    st, refz, _ = oracle.extend(bits(q), bits(kz), bits(vz), r2t, rpi, lens, qo, kv_end, 1 / math.sqrt(128))
    assert st == oracle.OK
    assert_close(bf16_to_f64(out)[:qo[1]], refz[:qo[1]], "out-of-pool page reads as zeros, ps=%d" % ps)


def test_extend_token_table_matches_the_page_list_bit_for_bit(B):
    """The token-table layout reads the same pool rows in the same order as the page list, so
    the two give the same bits (each is also checked against the oracle above)."""
    lens = [700, 65, 2049, 300]
    nq = [128, 65, 7, 300]
    case = _case(77, lens, nq, 32, 8, 128, 16)
    outs = [_run(B, *case, lens, 16, chunk=256, layout=lay) for lay in ("csr", "token")]
    assert outs[0][0] == 0 and outs[1][0] == 0
    assert np.array_equal(outs[0][1], outs[1][1]) and np.array_equal(outs[0][2], outs[1][2])


@pytest.mark.parametrize("ps", [2, 16])
def test_extend_token_table_flags_bad_rows_and_page_starts(B, ps):
    """Token-table layout: a page start that is not a multiple of the page size raises
    PKV_DEVERR_CONTIG and its keys read as zeros (both producers); a request row outside the
    table raises PKV_DEVERR_RANGE and the request is empty; the other requests stay exact."""
    dev = torch.device("cuda")
    lens, nq = [40, 24, 30], [4, 3, 5]
    r2t, rpi, num_pages, k, v, q, qo = _case(ps + 1, lens, nq, 16, 4, 128, ps)
    scale = 1 / math.sqrt(128)
    kv_end = np.concatenate([np.arange(L - n, L) + 1 for L, n in zip(lens, nq)]).astype(np.int32)
    st, ref, _ = oracle.extend(bits(q), bits(k), bits(v), r2t, rpi, lens, qo, kv_end, scale)
    assert st == oracle.OK

    def call(r2t_d, rpi_d):
        out = torch.zeros(tuple(q.shape), dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        args = B.make_extend_args(B.PKV_LAYOUT_REQ_TO_TOKEN, q.to(dev), k.to(dev), v.to(dev), out, _dev(qo),
                                  page_size=ps, sm_scale=scale, max_seq_len=max(lens), seq_lens=_dev(lens),
                                  req_to_token=r2t_d, req_pool_idx=rpi_d)
        ws = torch.empty(max(B.pkv_extend_workspace_size(args), 256), dtype=torch.uint8, device=dev)
        B.pkv_extend(args, ws, err)
        torch.cuda.synchronize()
        return int(err.item()), bf16_to_f64(out)

    # request 0's first page start moved off the page grid: its keys there read as zeros
    bad = np.array(r2t, dtype=np.int32, copy=True)
    row0 = int(rpi[0])
    page = int(bad[row0, 0]) // ps
    bad[row0, 0] += 1
    e, gpu = call(_dev(bad), _dev(rpi))
    assert e & B.PKV_DEVERR_CONTIG and not e & B.PKV_DEVERR_RANGE
    assert_close(gpu[qo[1]:], ref[qo[1]:], "requests next to a misaligned page start, ps=%d" % ps)
    kz, vz = k.clone(), v.clone()
    kz[page * ps:(page + 1) * ps] = 0
    vz[page * ps:(page + 1) * ps] = 0
    st, refz, _ = oracle.extend(bits(q), bits(kz), bits(vz), r2t, rpi, lens, qo, kv_end, scale)
    assert st == oracle.OK
    assert_close(gpu[:qo[1]], refz[:qo[1]], "misaligned page start reads as zeros, ps=%d" % ps)
    # request 1's row outside the table: a range error, the others exact
    rpi_bad = np.array(rpi, dtype=np.int32, copy=True)
    rpi_bad[1] = r2t.shape[0] + 3
    e, gpu = call(_dev(r2t), _dev(rpi_bad))
    assert e & B.PKV_DEVERR_RANGE
    assert_close(gpu[:qo[1]], ref[:qo[1]], "request before a bad row, ps=%d" % ps)
    assert_close(gpu[qo[2]:], ref[qo[2]:], "request after a bad row, ps=%d" % ps)


def test_extend_token_table_with_start_columns(B):
    """Token-table layout with kv_start: request b's keys are columns s_b .. s_b + L_b - 1 of its
    row. The oracle runs on the same slots moved to column 0; a start that is not a multiple of
    the page size raises PKV_DEVERR_RANGE and only that request is left out."""
    dev = torch.device("cuda")
    ps, lens, nq = 16, [200, 77, 130], [16, 5, 130]
    starts = [32, 0, 160]
    rng = np.random.default_rng(19)
    num_pages = sum(-(-L // ps) for L in lens) + 8
    r2t, rpi = paged_table(rng, lens, ps, num_pages, kv_start=starts)
    shifted = np.zeros_like(r2t)
    for b, (L, st_) in enumerate(zip(lens, starts)):
        shifted[rpi[b], :L] = r2t[rpi[b], st_:st_ + L]
    gen = torch.Generator().manual_seed(19)
    k = torch.randn((num_pages * ps, 4, 128), generator=gen).to(torch.bfloat16)
    v = torch.randn((num_pages * ps, 4, 128), generator=gen).to(torch.bfloat16)
    qo = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = torch.randn((int(qo[-1]), 16, 128), generator=gen).to(torch.bfloat16)
    scale = 1 / math.sqrt(128)
    kv_end = np.concatenate([np.arange(L - n, L) + 1 for L, n in zip(lens, nq)]).astype(np.int32)
    st, ref, ref_lse = oracle.extend(bits(q), bits(k), bits(v), shifted, rpi, lens, qo, kv_end, scale)
    assert st == oracle.OK

    def call(start_cols):
        out = torch.zeros(tuple(q.shape), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((q.shape[0], 16), dtype=torch.float32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        args = B.make_extend_args(B.PKV_LAYOUT_REQ_TO_TOKEN, q.to(dev), k.to(dev), v.to(dev), out, _dev(qo),
                                  page_size=ps, sm_scale=scale, max_seq_len=max(lens), seq_lens=_dev(lens),
                                  req_to_token=_dev(r2t), req_pool_idx=_dev(rpi), kv_start=_dev(start_cols),
                                  lse=lse, kv_chunk=64)
        ws = torch.empty(max(B.pkv_extend_workspace_size(args), 256), dtype=torch.uint8, device=dev)
        B.pkv_extend(args, ws, err)
        torch.cuda.synchronize()
        return int(err.item()), bf16_to_f64(out), lse.double().cpu().numpy()

    e, gpu, g_lse = call(starts)
    assert e == 0
    assert_close(gpu, ref, "token table with start columns")
    assert_close(g_lse, ref_lse, "token table with start columns lse")
    bad = list(starts)
    bad[0] = 33                                  # not a multiple of the page size
    e, gpu, _ = call(bad)
    assert e & B.PKV_DEVERR_RANGE
    assert_close(gpu[qo[1]:], ref[qo[1]:], "requests next to a misaligned start")
