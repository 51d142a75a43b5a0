"""The fused decode step (PKV_LAYOUT_REQ_TO_TOKEN + the fused store) against the oracle.

pkv_decode with the token-table layout reads each page's start straight from
req_to_token ("From slots to a page table": page of position t =
req_to_token[row, t - t % ps] / ps) and, with k_new / v_new, first writes the
new token's K/V into its pool slot (the mini-sglang store_kv before attention).
The oracle does the same two steps separately in fp64: store, then decode
walking req_to_token.  Attention is compared within |err| <= 2e-2 + 2e-2 |ref|;
the pool rows the fused store wrote are compared bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from _harness import assert_close, bf16_to_f64, bits, oracle_decode_problem, paged_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _new_slots(wl, pb):
    r2t = wl.req_to_token.numpy()
    rpi = wl.req_pool_idx.numpy().astype(np.int64)
    lens = pb.spec.seq_lens.numpy().astype(np.int64)
    st = pb.spec.kv_start.numpy().astype(np.int64)
    return np.array([r2t[rpi[b], st[b] + lens[b] - 1] for b in range(wl.batch)], dtype=np.int64)


@pytest.mark.parametrize("name,cross,batch", [("qwen3_0p6b", "paged", None), ("whisper_encdec", "paged", None),
                                              ("whisper_encdec", "gather", None), ("llama3_8b", "paged", 64),
                                              ("tiny_gqa", "paged", None)])
def test_fused_step_matches_the_oracle_and_stores(B, name, cross, batch):
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    wl = make_workload(name, batch=batch)
    step = DecodeStep(wl, cross_mode=cross, fused=True)
    pb = step.problems["self"]
    slots = torch.from_numpy(_new_slots(wl, pb)).cuda()
    step.k_pool[slots] = 0                      # the fused store must write these rows
    step.v_pool[slots] = 0
    assert step.launches_per_step() == sum(1 + (1 if p.ws_bytes else 0) + (1 if p.gather else 0)
                                           for p in step.problems.values())
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    np.testing.assert_array_equal(bits(step.k_pool[slots]), bits(step.k_new))
    np.testing.assert_array_equal(bits(step.v_pool[slots]), bits(step.v_new))
    rng = np.random.default_rng(5)
    sample = sorted(set([0, wl.batch - 1] + rng.choice(wl.batch, min(wl.batch, 8), replace=False).tolist()))
    for pname, p in step.problems.items():
        ref, ref_lse = oracle_decode_problem(step, pname, sample)
        assert_close(bf16_to_f64(p.out)[sample], ref, "%s %s fused out" % (name, pname))
        assert_close(p.lse.double().cpu().numpy()[sample], ref_lse, "%s %s fused lse" % (name, pname))


def test_fused_step_agrees_with_the_unfused_step(B):
    """Same split plan and kernels; the fused step adds the new key to the softmax state
    after its tile instead of inside it, so the two agree to rounding."""
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    wl = make_workload("qwen3_0p6b")
    a = DecodeStep(wl)
    b = DecodeStep(wl, fused=True, pools=(a.k_pool, a.v_pool))
    a.run()
    torch.cuda.synchronize()
    b.run()
    torch.cuda.synchronize()
    assert a.check_errors() == 0 and b.check_errors() == 0
    assert_close(bf16_to_f64(b.problems["self"].out), bf16_to_f64(a.problems["self"].out), "fused vs unfused")


def _direct(B, lens, ps, hq, hkv, d, starts=None, chunk=0, seed=0, store=True, r2t_edit=None, rpi_edit=None):
    dev = torch.device("cuda")
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    num_pages = 4 + sum(-(-L // ps) for L in lens) + (sum(starts) // ps if starts else 0)
    r2t, rpi = paged_table(rng, lens, ps, num_pages, kv_start=starts)
    slots = num_pages * ps
    k = torch.randn((slots, hkv, d), generator=gen).to(torch.bfloat16)
    v = torch.randn((slots, hkv, d), generator=gen).to(torch.bfloat16)
    q = torch.randn((len(lens), hq, d), generator=gen).to(torch.bfloat16)
    k_new = torch.randn((len(lens), hkv, d), generator=gen).to(torch.bfloat16)
    v_new = torch.randn((len(lens), hkv, d), generator=gen).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    st_ = np.zeros(len(lens), dtype=np.int64) if starts is None else np.asarray(starts, dtype=np.int64)
    # oracle: store (the new token is each non-empty request's last key), then decode
    kh, vh = bits(k), bits(v)
    live = [b for b, L in enumerate(lens) if L > 0]
    if store and live:
        sm = np.array([r2t[rpi[b], st_[b] + lens[b] - 1] for b in live], dtype=np.int32)
        assert oracle.store(kh, bits(k_new)[live], sm) == oracle.OK
        assert oracle.store(vh, bits(v_new)[live], sm) == oracle.OK
    st, ref, ref_lse = oracle.decode(bits(q), kh, vh, r2t, rpi, lens, scale, kv_start=st_)
    assert st == oracle.OK
    table, rpi_g = r2t.copy(), rpi.copy()
    if r2t_edit:
        r2t_edit(table, rpi_g)
    if rpi_edit:
        rpi_edit(rpi_g)
    kd, vd, qd = k.to(dev), v.to(dev), q.to(dev)
    out = torch.empty((len(lens), hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((len(lens), hq), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_REQ_TO_TOKEN, qd, kd, vd, out, page_size=ps,
                              sm_scale=scale, max_seq_len=max(max(lens), 1),
                              seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev), lse=lse, kv_chunk=chunk,
                              req_to_token=torch.from_numpy(table).to(dev), req_pool_idx=torch.from_numpy(rpi_g).to(dev),
                              kv_start=None if starts is None else torch.tensor(starts, dtype=torch.int32, device=dev),
                              k_new=k_new.to(dev) if store else None, v_new=v_new.to(dev) if store else None)
    ws = torch.empty(max(B.pkv_decode_workspace_size(args), 256), dtype=torch.uint8, device=dev)
    B.pkv_decode(args, ws, err)
    torch.cuda.synchronize()
    return err.item(), bf16_to_f64(out), lse.double().cpu().numpy(), ref, ref_lse, bits(kd), bits(vd), kh, vh


@pytest.mark.parametrize("ps", [1, 2, 16, 64, 128])
@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 128), (32, 2, 64), (20, 20, 64), (8, 8, 128)])
def test_fused_edge_lengths_and_page_sizes(B, ps, hq, hkv, d):
    lens = [1, 2, ps, ps + 1, 63, 64, 65, 129, 3 * ps + 5, 700]
    starts = [0, ps, 0, 2 * ps, 0, 0, ps, 0, 3 * ps, 0]
    for chunk in (0, 64):
        e, gpu, g_lse, ref, ref_lse, kp, vp, kh, vh = _direct(B, lens, ps, hq, hkv, d, starts=starts, chunk=chunk,
                                                             seed=ps * 7 + hq + chunk)
        assert e == 0
        assert_close(gpu, ref, "fused ps=%d hq=%d hkv=%d d=%d chunk=%d" % (ps, hq, hkv, d, chunk))
        assert_close(g_lse, ref_lse, "fused lse")
        np.testing.assert_array_equal(kp, kh)     # the pool after the fused store, bit for bit
        np.testing.assert_array_equal(vp, vh)


def test_token_table_layout_without_store(B):
    lens = [0, 1, 77, 500, 1025]
    e, gpu, g_lse, ref, ref_lse, kp, vp, kh, vh = _direct(B, lens, 16, 16, 8, 128, store=False, seed=3)
    assert e == 0
    assert_close(gpu, ref, "token-table layout")
    assert (gpu[0] == 0).all() and np.isneginf(g_lse[0]).all()      # L = 0: out = 0, lse = -inf
    np.testing.assert_array_equal(kp, kh)


def test_token_table_flags(B):
    lens = [40, 70, 33]

    def misalign(table, rpi):
        table[rpi[1], 16:32] += 1                 # a page start that is not a multiple of 16
    e, *_ = _direct(B, lens, 16, 16, 8, 128, store=False, r2t_edit=misalign, seed=4)
    assert e == B.PKV_DEVERR_CONTIG

    def outside(table, rpi):
        table[rpi[2], 0:16] = 10_000 * 16 + np.arange(16)   # a page past the pool
    e, *_ = _direct(B, lens, 16, 16, 8, 128, store=False, r2t_edit=outside, seed=4)
    assert e == B.PKV_DEVERR_RANGE

    def bad_row(rpi):
        rpi[0] = 999
    e, gpu, g_lse, *_ = _direct(B, lens, 16, 16, 8, 128, store=False, rpi_edit=bad_row, seed=4)
    assert e == B.PKV_DEVERR_RANGE
    assert (gpu[0] == 0).all()                    # treated as empty


def test_token_table_layout_is_gqa_only(B):
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    with pytest.raises(ValueError):
        DecodeStep(make_workload("deepseek_v3_mla", batch=2), fused=True)
