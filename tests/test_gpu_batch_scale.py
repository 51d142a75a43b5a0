"""Large batches through the index and gather calls, bit-exact against the oracle.

pkv_build_indices and pkv_ragged_gather find each request's output offset
(kv_indptr, cu_seqlens) as the sum over the requests before it; every CTA streams
the batch's counts once, so the work grows linearly with the batch.  These cases
run 8192 requests of mixed lengths (with empty ones) and report the launch time.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from _harness import bits, paged_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _timed(fn, reps=5):
    fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_build_indices_batch_8192(B, ps):
    dev = torch.device("cuda")
    rng = np.random.default_rng(8192 + ps)
    Bn = 8192
    lens = rng.integers(0, 700, size=Bn)
    lens[rng.choice(Bn, 64, replace=False)] = 0
    starts = np.zeros(Bn, dtype=np.int64)
    starts[::7] = ps * rng.integers(0, 3, size=len(starts[::7]))
    num_pages = int(sum(-(-int(L) // ps) for L in lens)) + 17
    r2t, rpi = paged_table(rng, lens.tolist(), ps, num_pages, kv_start=starts)
    cap = int(sum(-(-int(L) // ps) for L in lens))
    width = int(max(-(-int(L) // ps) for L in lens)) + 2
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    indptr = torch.full((Bn + 1,), -7, dtype=torch.int32, device=dev)
    idx = torch.full((cap,), -7, dtype=torch.int32, device=dev)
    last = torch.full((Bn,), -7, dtype=torch.int32, device=dev)
    bt = torch.full((Bn, width), -7, dtype=torch.int32, device=dev)
    r2t_d, rpi_d = torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev)
    lens_d = torch.from_numpy(lens.astype(np.int32)).to(dev)
    starts_d = torch.from_numpy(starts.astype(np.int32)).to(dev)

    def run():
        B.pkv_build_indices(r2t_d, rpi_d, lens_d, ps, num_pages, err, kv_start=starts_d, kv_indptr=indptr,
                            kv_indices=idx, kv_last_page_len=last, block_table=bt)
    ms = _timed(run)
    st, e_ptr, e_idx, e_last, e_bt = oracle.build_indices(r2t, rpi, lens, ps, num_pages, kv_start=starts,
                                                          kv_indices_cap=cap, bt_width=width)
    assert st == oracle.OK and err.item() == 0
    np.testing.assert_array_equal(indptr.cpu().numpy(), e_ptr)
    np.testing.assert_array_equal(idx.cpu().numpy(), e_idx)
    np.testing.assert_array_equal(last.cpu().numpy(), e_last)
    np.testing.assert_array_equal(bt.cpu().numpy(), e_bt)
    print("\npkv_build_indices batch %d ps %d: %.1f us per launch (%d positions)" % (Bn, ps, ms * 1e3, lens.sum()))


def test_ragged_gather_batch_8192(B):
    dev = torch.device("cuda")
    rng = np.random.default_rng(77)
    Bn, ps, heads, d = 8192, 16, 2, 64
    lens = rng.integers(0, 160, size=Bn)
    num_pages = int(sum(-(-int(L) // ps) for L in lens)) + 5
    r2t, rpi = paged_table(rng, lens.tolist(), ps, num_pages)
    slots = num_pages * ps
    gen = torch.Generator(device=dev).manual_seed(5)
    kp = torch.randn((slots, heads, d), generator=gen, device=dev).to(torch.bfloat16)
    vp = torch.randn((slots, heads, d), generator=gen, device=dev).to(torch.bfloat16)
    total = int(lens.sum())
    ko = torch.empty((total, heads, d), dtype=torch.bfloat16, device=dev)
    vo = torch.empty_like(ko)
    cu = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    r2t_d, rpi_d = torch.from_numpy(r2t).to(dev), torch.from_numpy(rpi).to(dev)
    lens_d = torch.from_numpy(lens.astype(np.int32)).to(dev)

    def run():
        B.pkv_ragged_gather(kp, vp, r2t_d, rpi_d, lens_d, int(lens.max()), ko, vo, cu, err)
    ms = _timed(run)
    st, e_k, e_v, e_cu = oracle.ragged_gather(bits(kp), bits(vp), r2t, rpi, lens)
    assert st == oracle.OK and err.item() == 0
    np.testing.assert_array_equal(cu.cpu().numpy(), e_cu)
    np.testing.assert_array_equal(bits(ko), e_k)
    np.testing.assert_array_equal(bits(vo), e_v)
    print("\npkv_ragged_gather batch %d: %.1f us per launch (%d rows of %d B, K and V)" % (
        Bn, ms * 1e3, total, heads * d * 2))


def test_ragged_gather_zero_fills_rows_of_bad_requests(B):
    """A request whose row lies outside the table and a slot outside the pool raise
    PKV_DEVERR_RANGE; the rows reserved for them read as zeros, the others are exact."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(3)
    ps, lens = 8, [20, 13, 9, 30]
    num_pages = 40
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    slots = num_pages * ps
    kp = torch.randn((slots, 1, 64), device=dev).to(torch.bfloat16)
    vp = torch.randn((slots, 1, 64), device=dev).to(torch.bfloat16)
    st, e_k, e_v, e_cu = oracle.ragged_gather(bits(kp), bits(vp), r2t, rpi, lens)
    assert st == oracle.OK
    bad_table = r2t.copy()
    bad_table[rpi[3], 5] = slots + 100                 # one slot outside the pool
    bad_rpi = rpi.copy()
    bad_rpi[1] = r2t.shape[0] + 3                      # request 1's row outside the table
    total = sum(lens)
    ko = torch.full((total, 1, 64), 7.0, dtype=torch.bfloat16, device=dev)
    vo = torch.full_like(ko, 7.0)
    cu = torch.empty(len(lens) + 1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    B.pkv_ragged_gather(kp, vp, torch.from_numpy(bad_table).to(dev), torch.from_numpy(bad_rpi).to(dev),
                        torch.tensor(lens, dtype=torch.int32, device=dev), max(lens), ko, vo, cu, err)
    assert err.item() == B.PKV_DEVERR_RANGE
    np.testing.assert_array_equal(cu.cpu().numpy(), e_cu)
    k, v = bits(ko), bits(vo)
    zero_rows = list(range(e_cu[1], e_cu[2])) + [e_cu[3] + 5]
    keep = [r for r in range(total) if r not in zero_rows]
    assert (k[zero_rows] == 0).all() and (v[zero_rows] == 0).all()
    np.testing.assert_array_equal(k[keep], e_k[keep])
    np.testing.assert_array_equal(v[keep], e_v[keep])
