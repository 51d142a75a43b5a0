"""GPU parity: libpkv (through its C ABI) against the fp64 CPU oracle.

Index building, store and gather are compared bit for bit; attention within
|gpu - oracle| <= 2e-2 + 2e-2 |oracle| elementwise (bf16 output, fp32
accumulation).  Small configurations are checked on every output; the large
ones run at full size in the benchmark's launch configuration and are checked
on sampled requests that the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from _harness import assert_close, bf16_to_f64, bits, oracle_decode_problem, paged_table

pytestmark = pytest.mark.gpu

GQA_CONFIGS = ["tiny_gqa", "qwen3_0p6b", "llama3_8b", "whisper_encdec"]


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _step(name, **kw):
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    return DecodeStep(make_workload(name, **{k: v for k, v in kw.items() if k == "batch"}),
                      **{k: v for k, v in kw.items() if k != "batch"})


def _sample(Bn, k, seed=0):
    if Bn <= k:
        return list(range(Bn))
    rng = np.random.default_rng(seed)
    return sorted(set([0, Bn - 1] + rng.choice(Bn, size=k - 2, replace=False).tolist()))


# ------------------------------------------------------------------ build_indices
@pytest.mark.parametrize("name", GQA_CONFIGS + ["deepseek_v3_mla"])
def test_build_indices_bit_exact(B, name):
    from paged_kv_cache_req_gb300.workloads import make_workload
    wl = make_workload(name)
    dev = torch.device("cuda")
    r2t = wl.req_to_token.to(dev)
    rpi = wl.req_pool_idx.to(dev)
    for p in wl.problems:
        lens = p.seq_lens.numpy()
        npages = -(-lens.astype(np.int64) // wl.page_size)
        cap = int(npages.sum())
        width = int(npages.max())
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        indptr = torch.full((wl.batch + 1,), -7, dtype=torch.int32, device=dev)
        indices = torch.full((cap,), -7, dtype=torch.int32, device=dev)
        last = torch.full((wl.batch,), -7, dtype=torch.int32, device=dev)
        bt = torch.full((wl.batch, width), -7, dtype=torch.int32, device=dev)
        B.pkv_build_indices(r2t, rpi, p.seq_lens.to(dev), wl.page_size, wl.num_pool_pages, err,
                            kv_start=p.kv_start.to(dev), kv_indptr=indptr, kv_indices=indices,
                            kv_last_page_len=last, block_table=bt)
        st, e_ptr, e_idx, e_last, e_bt = oracle.build_indices(
            wl.req_to_token.numpy(), wl.req_pool_idx.numpy(), lens, wl.page_size, wl.num_pool_pages,
            kv_start=p.kv_start.numpy(), kv_indices_cap=cap, bt_width=width)
        assert st == oracle.OK
        assert err.item() == 0
        np.testing.assert_array_equal(indptr.cpu().numpy(), e_ptr)
        np.testing.assert_array_equal(indices.cpu().numpy(), e_idx)
        np.testing.assert_array_equal(last.cpu().numpy(), e_last)
        np.testing.assert_array_equal(bt.cpu().numpy(), e_bt)


@pytest.mark.parametrize("ps", [1, 3, 64, 4096])
def test_build_indices_long_rows_and_wide_tables(B, ps):
    """Rows spanning many CTA spans, page sizes that do not divide the span (3) or
    exceed it (4096), and a block table wider than any request needs."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(ps)
    lens = [0, 1, 2047, 2048, 2049, 9001, 5 * ps + 1]
    num_pages = sum(-(-L // ps) for L in lens) + 9
    starts = [0, ps, 0, 2 * ps, 0, 0, ps]
    r2t, rpi = paged_table(rng, lens, ps, num_pages, kv_start=starts)
    width_pages = max(-(-L // ps) for L in lens) + 40
    cap = sum(-(-L // ps) for L in lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    indptr = torch.full((len(lens) + 1,), -7, dtype=torch.int32, device=dev)
    idx = torch.full((cap,), -7, dtype=torch.int32, device=dev)
    last = torch.full((len(lens),), -7, dtype=torch.int32, device=dev)
    bt = torch.full((len(lens), width_pages), -7, dtype=torch.int32, device=dev)
    B.pkv_build_indices(torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev),
                        torch.tensor(lens, dtype=torch.int32, device=dev), ps, num_pages, err,
                        kv_start=torch.tensor(starts, dtype=torch.int32, device=dev), kv_indptr=indptr,
                        kv_indices=idx, kv_last_page_len=last, block_table=bt)
    st, e_ptr, e_idx, e_last, e_bt = oracle.build_indices(r2t, rpi, lens, ps, num_pages, kv_start=starts,
                                                          kv_indices_cap=cap, bt_width=width_pages)
    assert st == oracle.OK and err.item() == 0
    np.testing.assert_array_equal(indptr.cpu().numpy(), e_ptr)
    np.testing.assert_array_equal(idx.cpu().numpy(), e_idx)
    np.testing.assert_array_equal(last.cpu().numpy(), e_last)
    np.testing.assert_array_equal(bt.cpu().numpy(), e_bt)
    # a contiguity break deep inside the longest row is still seen (any slot change
    # breaks a page of more than one key)
    if ps > 1:
        bad = r2t.copy()
        bad[rpi[5], 8001] += 1
        err.zero_()
        B.pkv_build_indices(torch.from_numpy(bad).to(dev), torch.from_numpy(rpi).to(dev),
                            torch.tensor(lens, dtype=torch.int32, device=dev), ps, num_pages, err,
                            kv_start=torch.tensor(starts, dtype=torch.int32, device=dev), kv_indptr=indptr,
                            kv_indices=idx, kv_last_page_len=last, block_table=bt)
        assert err.item() == B.PKV_DEVERR_CONTIG


def test_build_indices_flags_bad_tables(B):
    dev = torch.device("cuda")
    rng = np.random.default_rng(1)
    ps, lens = 16, [40, 17, 0, 64]
    r2t, rpi = paged_table(rng, lens, ps, 32)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)

    def run(table, cap=16, bt_width=8, starts=None):
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        indptr = torch.empty(5, dtype=torch.int32, device=dev)
        idx = torch.empty(cap, dtype=torch.int32, device=dev)
        last = torch.empty(4, dtype=torch.int32, device=dev)
        bt = torch.empty((4, bt_width), dtype=torch.int32, device=dev)
        B.pkv_build_indices(torch.from_numpy(table).to(dev), torch.from_numpy(rpi).to(dev), lens_t, ps, 32, err,
                            kv_start=None if starts is None else torch.tensor(starts, dtype=torch.int32, device=dev),
                            kv_indptr=indptr, kv_indices=idx, kv_last_page_len=last, block_table=bt)
        return err.item(), indptr.cpu().numpy()

    e, ptr = run(r2t)
    assert e == 0 and ptr.tolist() == [0, 3, 5, 5, 9]
    bad = r2t.copy()
    bad[rpi[0], 20] += 1
    assert run(bad)[0] == B.PKV_DEVERR_CONTIG
    bad = r2t.copy()
    bad[rpi[1], 0:16] = np.arange(16) + 600          # page 37 of a 32-page pool
    assert run(bad)[0] & B.PKV_DEVERR_RANGE
    assert run(r2t, cap=6)[0] == B.PKV_DEVERR_CAPACITY
    assert run(r2t, bt_width=3)[0] == B.PKV_DEVERR_CAPACITY
    assert run(r2t, starts=[0, 0, 0, 10_000])[0] == B.PKV_DEVERR_RANGE


# ------------------------------------------------------------------ store
@pytest.mark.parametrize("name", ["tiny_gqa", "whisper_encdec", "deepseek_v3_mla"])
def test_store_bit_exact(B, name):
    from paged_kv_cache_req_gb300.workloads import make_workload
    kw = {"batch": 16} if name == "deepseek_v3_mla" else {}
    step = _step(name, **kw)
    before_k = step.k_pool.clone()
    before_v = step.v_pool.clone() if step.v_pool is not None else None
    step.store("self")
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    sm = step.problems["self"].spec.slot_mapping.numpy()
    exp_k = bits(before_k)
    assert oracle.store(exp_k, bits(step.k_new), sm) == oracle.OK
    np.testing.assert_array_equal(bits(step.k_pool), exp_k)
    if before_v is not None:
        exp_v = bits(before_v)
        assert oracle.store(exp_v, bits(step.v_new), sm) == oracle.OK
        np.testing.assert_array_equal(bits(step.v_pool), exp_v)


def test_store_skips_padding_and_flags_out_of_range(B):
    dev = torch.device("cuda")
    k_pool = torch.zeros((32, 2, 64), dtype=torch.bfloat16, device=dev)
    v_pool = torch.zeros_like(k_pool)
    k_new = torch.randn((3, 2, 64), device=dev).to(torch.bfloat16)
    v_new = torch.randn((3, 2, 64), device=dev).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    B.pkv_store(k_pool, v_pool, k_new, v_new, torch.tensor([-1, 5, 99], dtype=torch.int32, device=dev), err)
    assert err.item() == B.PKV_DEVERR_RANGE
    assert torch.equal(k_pool[5], k_new[1]) and torch.equal(v_pool[5], v_new[1])
    k_pool[5] = 0
    v_pool[5] = 0
    assert not k_pool.any() and not v_pool.any()


# ------------------------------------------------------------------ decode
def _check_decode(step, name, sample, pre_k, pre_v):
    out, lse = oracle_decode_problem(step, name, sample, pre_k=pre_k, pre_v=pre_v)
    pb = step.problems[name]
    gpu = bf16_to_f64(pb.out)[sample]
    err = assert_close(gpu, out, "%s/%s out" % (step.wl.name, name))
    g_lse = pb.lse.double().cpu().numpy()[sample]
    assert_close(g_lse, lse, "%s/%s lse" % (step.wl.name, name))
    return err


@pytest.mark.parametrize("name,sample_k", [("tiny_gqa", 4), ("qwen3_0p6b", 32), ("llama3_8b", 10),
                                           ("whisper_encdec", 12)])
def test_decode_step_parity(B, name, sample_k):
    step = _step(name)
    Bn = step.wl.batch
    sample = _sample(Bn, sample_k)
    if name == "llama3_8b":  # a whole shared-prefix group too
        sample = sorted(set(sample + list(range(16, 32))))
    pre_k = step.k_pool.clone()
    pre_v = step.v_pool.clone()
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    for pname in step.problems:
        _check_decode(step, pname, sample, pre_k, pre_v)


@pytest.mark.parametrize("name,sample_k", [("tiny_gqa", 4), ("qwen3_0p6b", 16), ("llama3_8b", 8),
                                           ("whisper_encdec", 8), ("deepseek_v3_mla", 6)])
def test_decode_step_with_device_allocation(B, name, sample_k):
    """alloc_extend + write_req_to_token ahead of the step: slots, free-list state and the
    whole table bit-exact against the oracle's own allocation, then attention against
    the oracle on the oracle's table."""
    kw = {"batch": 32} if name == "deepseek_v3_mla" else {}
    step = _step(name, alloc=True, **kw)
    wl = step.wl
    pb = step.problems[step.alloc_problem]
    prefix = step.prefix_lens.cpu().numpy()
    last = step.last_loc.cpu().numpy()
    free = step.free_pages.cpu().numpy()
    pre_k = step.k_pool.clone()
    pre_v = step.v_pool.clone() if step.v_pool is not None else None
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    state = np.array([0, len(free)], np.int32)
    seq = pb.spec.seq_lens.numpy()
    st, loc = oracle.alloc_extend(prefix, seq, last, wl.page_size, wl.num_pool_pages, free, state)
    assert st == oracle.OK
    assert np.array_equal(step.out_cache_loc.cpu().numpy(), loc)
    assert step.free_state.cpu().numpy().tolist() == state.tolist()
    table = wl.req_to_token.numpy().copy()
    assert oracle.write_req_to_token(table, wl.req_pool_idx.numpy(), prefix, seq, [None] * wl.batch, loc,
                                     kv_start=pb.spec.kv_start.numpy()) == oracle.OK
    assert np.array_equal(step.r2t.cpu().numpy(), table)
    sample = _sample(wl.batch, sample_k, seed=4)
    for pname in step.problems:
        out, lse = oracle_decode_problem(step, pname, sample, pre_k=pre_k, pre_v=pre_v, r2t=table,
                                         slot_mapping=loc if pname == step.alloc_problem else None)
        assert_close(bf16_to_f64(step.problems[pname].out)[sample], out, "%s/%s out (allocated)" % (name, pname))
        assert_close(step.problems[pname].lse.double().cpu().numpy()[sample], lse, "%s/%s lse" % (name, pname))


def test_whisper_cross_attention_gather_mode(B):
    step = _step("whisper_encdec", cross_mode="gather")
    sample = _sample(step.wl.batch, 12, seed=1)
    pre_k, pre_v = step.k_pool.clone(), step.v_pool.clone()
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    _check_decode(step, "cross", sample, pre_k, pre_v)
    _check_decode(step, "self", sample, pre_k, pre_v)
    # the ragged buffer itself is bit-exact against the oracle's gather
    pb = step.problems["cross"]
    wl = step.wl
    st, ko, vo, cu = oracle.ragged_gather(bits(pre_k), bits(pre_v), wl.req_to_token.numpy(),
                                          wl.req_pool_idx.numpy(), pb.spec.seq_lens.numpy(),
                                          kv_start=pb.spec.kv_start.numpy())
    assert st == oracle.OK
    np.testing.assert_array_equal(pb.cu.cpu().numpy(), cu)
    np.testing.assert_array_equal(bits(pb.k_rag), ko)
    np.testing.assert_array_equal(bits(pb.v_rag), vo)


@pytest.mark.parametrize("chunk", [64, 128, 192])
def test_decode_forced_splits_use_the_merge(B, chunk):
    step = _step("qwen3_0p6b", kv_chunk=chunk)
    pre_k, pre_v = step.k_pool.clone(), step.v_pool.clone()
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    _check_decode(step, "self", list(range(0, 32, 3)), pre_k, pre_v)


def _direct_decode(B, lens, ps, hq, hkv, d, chunk=0, layout=None, seed=0):
    """Decode over a small hand-made paged table through the C ABI; returns gpu and oracle outputs."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    num_pages = 4 + sum(-(-L // ps) for L in lens)
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    slots = num_pages * ps
    k = torch.randn((slots, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((slots, hkv, d), generator=gen).to(torch.bfloat16)
    q = torch.randn((len(lens), hq, d), generator=gen).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    st, ref, ref_lse = oracle.decode(bits(q), bits(k), bits(v), r2t, rpi, lens, scale)
    assert st == oracle.OK
    Bn = len(lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    npages = [-(-L // ps) for L in lens]
    out = torch.empty((Bn, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bn, hq), dtype=torch.float32, device=dev)
    kd, vd, qd = k.to(dev), v.to(dev), q.to(dev)
    if layout == "block_table":
        bt = torch.empty((Bn, max(max(npages), 1)), dtype=torch.int32, device=dev)
        B.pkv_build_indices(torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev), lens_t, ps, num_pages,
                            err, block_table=bt)
        args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_BLOCK_TABLE, qd, kd, vd, out, page_size=ps,
                                  sm_scale=scale, max_seq_len=max(lens), block_table=bt, seq_lens=lens_t, lse=lse,
                                  kv_chunk=chunk)
    else:
        indptr = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
        idx = torch.empty(max(sum(npages), 1), dtype=torch.int32, device=dev)
        last = torch.empty(Bn, dtype=torch.int32, device=dev)
        B.pkv_build_indices(torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev), lens_t, ps, num_pages,
                            err, kv_indptr=indptr, kv_indices=idx, kv_last_page_len=last)
        args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_CSR, qd, kd, vd, out, page_size=ps, sm_scale=scale,
                                  max_seq_len=max(lens), kv_indptr=indptr, kv_indices=idx, kv_last_page_len=last,
                                  lse=lse, kv_chunk=chunk)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return bf16_to_f64(out), lse.double().cpu().numpy(), ref, ref_lse


@pytest.mark.parametrize("ps", [1, 16, 64])
@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 64), (16, 8, 128), (32, 8, 128), (16, 2, 128), (32, 2, 64),
                                      (20, 20, 64)])
def test_decode_edge_lengths(B, ps, hq, hkv, d):
    lens = [0, 1, 2, ps, ps + 1, 63, 64, 65, 129, 3 * ps + 5, 700]
    for chunk in (0, 64):
        gpu, g_lse, ref, ref_lse = _direct_decode(B, lens, ps, hq, hkv, d, chunk=chunk, seed=ps + hq)
        assert (gpu[0] == 0).all() and np.isneginf(g_lse[0]).all()      # empty request
        assert_close(gpu, ref, "edge lengths ps=%d g=%d d=%d chunk=%d" % (ps, hq // hkv, d, chunk))
        assert_close(g_lse[1:], ref_lse[1:], "edge lse")


def test_decode_block_table_layout(B):
    lens = [5, 64, 200, 1000]
    gpu, g_lse, ref, ref_lse = _direct_decode(B, lens, 64, 16, 4, 128, layout="block_table")
    assert_close(gpu, ref, "block table layout")


def test_decode_varlen_layout_direct(B):
    """Keys of request b are rows cu[b]..cu[b+1]-1 of a contiguous buffer."""
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(4)
    lens = [3, 0, 1500, 77]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows, hkv, hq, d = int(cu[-1]), 4, 8, 64
    k = torch.randn((rows, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((rows, hkv, d), generator=gen).to(torch.bfloat16)
    q = torch.randn((4, hq, d), generator=gen).to(torch.bfloat16)
    # identity table: position t of request b is row cu[b] + t
    r2t = np.zeros((5, max(lens)), dtype=np.int32)
    for b, L in enumerate(lens):
        r2t[b + 1, :L] = np.arange(cu[b], cu[b] + L)
    st, ref, _ = oracle.decode(bits(q), bits(k), bits(v), r2t, np.arange(1, 5), lens, 0.125)
    out = torch.empty((4, hq, d), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_VARLEN, q.to(dev), k.to(dev), v.to(dev), out,
                              sm_scale=0.125, max_seq_len=max(lens), cu_seqlens=torch.from_numpy(cu).to(dev))
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_close(bf16_to_f64(out), ref, "varlen")


@pytest.mark.parametrize("chunk", [0, 64])
def test_mla_varlen_layout_direct(B, chunk):
    """MLA over a contiguous latent buffer: keys of request b are rows cu[b]..cu[b+1]-1."""
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(5 + chunk)
    lens = [3, 0, 1500, 77, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    lat = torch.randn((int(cu[-1]), 576), generator=gen).to(torch.bfloat16)
    q = torch.randn((len(lens), 128, 576), generator=gen).to(torch.bfloat16)
    r2t = np.zeros((len(lens) + 1, max(lens)), dtype=np.int32)
    for b, L in enumerate(lens):
        r2t[b + 1, :L] = np.arange(cu[b], cu[b] + L)
    scale = 1 / math.sqrt(192)
    st, ref, ref_lse = oracle.decode(bits(q), bits(lat), bits(lat), r2t, np.arange(1, len(lens) + 1), lens, scale,
                                     head_dim_v=512)
    assert st == oracle.OK
    out = torch.empty((len(lens), 128, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((len(lens), 128), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_VARLEN, q.to(dev), lat.to(dev), None, out,
                              sm_scale=scale, max_seq_len=max(lens), head_dim_v=512,
                              cu_seqlens=torch.from_numpy(cu).to(dev), lse=lse, kv_chunk=chunk)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_close(bf16_to_f64(out), ref, "MLA varlen chunk=%d" % chunk)
    live = [b for b, L in enumerate(lens) if L > 0]
    assert_close(lse.double().cpu().numpy()[live], ref_lse[live], "MLA varlen lse")
    assert (bf16_to_f64(out)[1] == 0).all() and np.isneginf(lse[1].cpu().numpy()).all()


def test_decode_flags_out_of_pool_pages(B):
    dev = torch.device("cuda")
    hq, hkv, d, ps = 8, 2, 128, 16
    k = torch.randn((64, hkv, d), device=dev).to(torch.bfloat16)
    v = torch.randn((64, hkv, d), device=dev).to(torch.bfloat16)
    q = torch.randn((2, hq, d), device=dev).to(torch.bfloat16)
    out = torch.empty((2, hq, d), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    indptr = torch.tensor([0, 2, 3], dtype=torch.int32, device=dev)
    idx = torch.tensor([1, 9, 2], dtype=torch.int32, device=dev)     # page 9 is outside a 4-page pool
    last = torch.tensor([16, 5], dtype=torch.int32, device=dev)
    args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_CSR, q, k, v, out, page_size=ps, sm_scale=0.1,
                              max_seq_len=32, kv_indptr=indptr, kv_indices=idx, kv_last_page_len=last)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_RANGE
    assert torch.isfinite(out[1].float()).all()
    # the request whose pages are all valid is still exact
    st, ref, _ = oracle.decode(bits(q[1:].cpu()), bits(k.cpu()), bits(v.cpu()),
                               np.asarray([[0] * 5, [32, 33, 34, 35, 36]], dtype=np.int32), [1], [5], 0.1)
    assert_close(bf16_to_f64(out[1:]), ref, "valid request next to a bad one")
    # the bad page reads as zeros: request 0 over page 1 and a page of zero rows
    kz = torch.cat([k.cpu(), torch.zeros((16, hkv, d), dtype=torch.bfloat16)])
    vz = torch.cat([v.cpu(), torch.zeros((16, hkv, d), dtype=torch.bfloat16)])
    row0 = np.asarray([list(range(16, 32)) + list(range(64, 80))], dtype=np.int32)
    st, refz, _ = oracle.decode(bits(q[:1].cpu()), bits(kz), bits(vz), np.vstack([np.zeros((1, 32), np.int32), row0]),
                                [1], [32], 0.1)
    assert_close(bf16_to_f64(out[:1]), refz, "out-of-pool page reads as zeros")


@pytest.mark.parametrize("ps", [2, 64])
def test_mla_flags_out_of_pool_pages(B, ps):
    """MLA: a page id outside the pool raises PKV_DEVERR_RANGE in both producers; the other request is exact."""
    dev = torch.device("cuda")
    lens = [3 * ps, 70]
    num_pages = 4 + sum(-(-L // ps) for L in lens)
    rng = np.random.default_rng(ps)
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    gen = torch.Generator().manual_seed(ps)
    lat = torch.randn((num_pages * ps, 576), generator=gen).to(torch.bfloat16)
    q = torch.randn((2, 128, 576), generator=gen).to(torch.bfloat16)
    st, indptr, indices, last, bt = oracle.build_indices(r2t, rpi, lens, ps, num_pages)
    assert st == oracle.OK
    bad = np.array(indices, dtype=np.int32)
    bad[1] = num_pages + 3                       # second page of request 0: outside the pool
    out = torch.zeros((2, 128, 512), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    args = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_CSR, q.to(dev), lat.to(dev), None, out, page_size=ps,
                              sm_scale=1 / math.sqrt(192), max_seq_len=max(lens), head_dim_v=512,
                              kv_indptr=t(indptr), kv_indices=t(bad), kv_last_page_len=t(last))
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() & B.PKV_DEVERR_RANGE
    assert torch.isfinite(out.float()).all()
    st, ref, _ = oracle.decode(bits(q), bits(lat), bits(lat), r2t, rpi, lens, 1 / math.sqrt(192), head_dim_v=512)
    assert_close(bf16_to_f64(out)[1:], ref[1:], "MLA valid request next to a bad one, ps=%d" % ps)
    # the bad page reads as zeros: the oracle over a pool whose rows of that page are zero
    page = int(indices[1])
    latz = lat.clone()
    latz[page * ps:(page + 1) * ps] = 0
    st, refz, _ = oracle.decode(bits(q), bits(latz), bits(latz), r2t, rpi, lens, 1 / math.sqrt(192), head_dim_v=512)
    assert_close(bf16_to_f64(out)[:1], refz[:1], "MLA out-of-pool page reads as zeros, ps=%d" % ps)


def test_decode_clamps_requests_past_max_seq_len(B):
    """A request longer than max_seq_len raises PKV_DEVERR_CAPACITY and attends only its first keys:
    up to the split plan's reach for GQA (here 2 chunks of 64 keys), up to max_seq_len for MLA."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(11)
    gen = torch.Generator().manual_seed(11)
    lens, ps = [200, 50], 16
    num_pages = 4 + sum(-(-L // ps) for L in lens)
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    r2t_d, rpi_d = torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    npages = [-(-L // ps) for L in lens]
    # GQA, CSR pages, kv_chunk 64 and max_seq_len 100: the plan reaches 128 keys
    k = torch.randn((num_pages * ps, 2, 128), generator=gen).to(torch.bfloat16)
    v = torch.randn((num_pages * ps, 2, 128), generator=gen).to(torch.bfloat16)
    q = torch.randn((2, 8, 128), generator=gen).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    indptr = torch.empty(3, dtype=torch.int32, device=dev)
    idx = torch.empty(sum(npages), dtype=torch.int32, device=dev)
    last = torch.empty(2, dtype=torch.int32, device=dev)
    B.pkv_build_indices(r2t_d, rpi_d, lens_t, ps, num_pages, err, kv_indptr=indptr, kv_indices=idx, kv_last_page_len=last)
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=dev)
    args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_CSR, q.to(dev), k.to(dev), v.to(dev), out, page_size=ps,
                              sm_scale=0.09, max_seq_len=100, kv_indptr=indptr, kv_indices=idx, kv_last_page_len=last,
                              kv_chunk=64)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_CAPACITY
    st, ref, _ = oracle.decode(bits(q), bits(k), bits(v), r2t, rpi, [128, 50], 0.09)
    assert st == oracle.OK
    assert_close(bf16_to_f64(out), ref, "GQA request clamped to the plan's reach")
    # MLA, block table, max_seq_len 100
    lat = torch.randn((num_pages * ps, 576), generator=gen).to(torch.bfloat16)
    qm = torch.randn((2, 128, 576), generator=gen).to(torch.bfloat16)
    err.zero_()
    bt = torch.empty((2, max(npages)), dtype=torch.int32, device=dev)
    B.pkv_build_indices(r2t_d, rpi_d, lens_t, ps, num_pages, err, block_table=bt)
    outm = torch.empty((2, 128, 512), dtype=torch.bfloat16, device=dev)
    args = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_BLOCK_TABLE, qm.to(dev), lat.to(dev), None, outm,
                              page_size=ps, sm_scale=1 / math.sqrt(192), max_seq_len=100, head_dim_v=512,
                              block_table=bt, seq_lens=lens_t)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_CAPACITY
    st, refm, _ = oracle.decode(bits(qm), bits(lat), bits(lat), r2t, rpi, [100, 50], 1 / math.sqrt(192), head_dim_v=512)
    assert_close(bf16_to_f64(outm), refm, "MLA request clamped to max_seq_len")


def test_decode_rejects_small_workspace(B):
    step = _step("qwen3_0p6b", kv_chunk=64)
    pb = step.problems["self"]
    with pytest.raises(B.PkvError) as e:
        B.pkv_decode(pb.args, pb.workspace[:128], step.err)
    assert e.value.status == B.PKV_ERR_CAPACITY


# ------------------------------------------------------------------ MLA (latent) decode
def test_mla_decode_step_parity(B):
    step = _step("deepseek_v3_mla")
    sample = _sample(step.wl.batch, 8, seed=2)
    pre_k = step.k_pool.clone()
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    _check_decode(step, "self", sample, pre_k, None)


def _direct_mla(B, lens, ps, hq=128, chunk=0, layout="block_table", seed=0):
    dev = torch.device("cuda")
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    num_pages = 4 + sum(-(-L // ps) for L in lens)
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    lat = torch.randn((num_pages * ps, 576), generator=gen).to(torch.bfloat16)
    q = torch.randn((len(lens), hq, 576), generator=gen).to(torch.bfloat16)
    scale = 1 / math.sqrt(192)
    st, ref, ref_lse = oracle.decode(bits(q), bits(lat), bits(lat), r2t, rpi, lens, scale, head_dim_v=512)
    assert st == oracle.OK
    Bn = len(lens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    npages = [-(-L // ps) for L in lens]
    out = torch.empty((Bn, hq, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bn, hq), dtype=torch.float32, device=dev)
    latd, qd = lat.to(dev), q.to(dev)
    r2t_d, rpi_d = torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev)
    if layout == "block_table":
        bt = torch.empty((Bn, max(max(npages), 1)), dtype=torch.int32, device=dev)
        B.pkv_build_indices(r2t_d, rpi_d, lens_t, ps, num_pages, err, block_table=bt)
        args = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_BLOCK_TABLE, qd, latd, None, out, page_size=ps,
                                  sm_scale=scale, max_seq_len=max(lens), head_dim_v=512, block_table=bt,
                                  seq_lens=lens_t, lse=lse, kv_chunk=chunk)
    else:
        indptr = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
        idx = torch.empty(max(sum(npages), 1), dtype=torch.int32, device=dev)
        last = torch.empty(Bn, dtype=torch.int32, device=dev)
        B.pkv_build_indices(r2t_d, rpi_d, lens_t, ps, num_pages, err, kv_indptr=indptr, kv_indices=idx,
                            kv_last_page_len=last)
        args = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_CSR, qd, latd, None, out, page_size=ps,
                                  sm_scale=scale, max_seq_len=max(lens), head_dim_v=512, kv_indptr=indptr,
                                  kv_indices=idx, kv_last_page_len=last, lse=lse, kv_chunk=chunk)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return bf16_to_f64(out), lse.double().cpu().numpy(), ref, ref_lse


@pytest.mark.parametrize("layout", ["block_table", "csr"])
@pytest.mark.parametrize("chunk", [0, 64, 192])
def test_mla_edge_lengths(B, layout, chunk):
    lens = [0, 1, 63, 64, 65, 130, 1000]
    gpu, g_lse, ref, ref_lse = _direct_mla(B, lens, 64, chunk=chunk, layout=layout, seed=7)
    assert (gpu[0] == 0).all() and np.isneginf(g_lse[0]).all()
    assert_close(gpu, ref, "MLA edge lengths %s chunk=%d" % (layout, chunk))
    assert_close(g_lse[1:], ref_lse[1:], "MLA lse")


@pytest.mark.parametrize("ps", [1, 2, 4])
@pytest.mark.parametrize("layout", ["block_table", "csr"])
def test_mla_small_pages_gathered_by_rows(B, ps, layout):
    # pages under 8 keys: the producer gathers the latent rows with cp.async instead of TMA boxes
    lens = [0, 1, 63, 65, 300, 1000]
    for chunk in (0, 64):
        gpu, g_lse, ref, ref_lse = _direct_mla(B, lens, ps, chunk=chunk, layout=layout, seed=ps + chunk)
        assert (gpu[0] == 0).all() and np.isneginf(g_lse[0]).all()
        assert_close(gpu, ref, "MLA ps=%d %s chunk=%d" % (ps, layout, chunk))
        assert_close(g_lse[1:], ref_lse[1:], "MLA lse ps=%d" % ps)


@pytest.mark.parametrize("ps", [16, 128])
def test_mla_other_page_sizes_and_head_groups(B, ps):
    gpu, g_lse, ref, ref_lse = _direct_mla(B, [5, 300, 777], ps, hq=256, seed=ps)
    assert_close(gpu, ref, "MLA ps=%d, 256 heads" % ps)
