"""Pins for the CPU oracle: each test checks it against something other than itself.

* values printed on the pages (fixtures under tests/golden, each citing its source),
* closed forms (one key gives V; identical keys or q = 0 give mean(V)),
* invariants (placement of pages in the pool does not change attention),
* library routines on special cases (torch's scaled_dot_product_attention in
  float64 on contiguous copies made with numpy indexing; numpy cumsum),
* brute force on tiny tables (search over every pool page).

Together these fail on a dropped scale, a wrong kv-head mapping, a wrong
row / column / kv_start, an off-by-one key range, a transposed operand, a
wrong V stride for the latent pool, or a wrong page/offset split.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from _harness import paged_table

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(torch.float64)


# ---------------------------------------------------------------- index building
def test_p5_csr_worked_example():
    g = golden("p5_csr_page_lists.json")
    ps = g["page_size"]
    for lens_key, last_key in (("seq_lens_full", "expected_last_page_len_full"),
                               ("seq_lens_partial", "expected_last_page_len_partial")):
        lens = g[lens_key]
        r2t = np.zeros((4, 512), dtype=np.int32)
        for b, (pages, L) in enumerate(zip(g["page_lists"], lens)):
            slots = (np.asarray(pages)[:, None] * ps + np.arange(ps)).reshape(-1)[:L]
            r2t[b + 1, :L] = slots
        st, indptr, indices, last, bt = oracle.build_indices(r2t, [1, 2, 3], lens, ps, 32)
        assert st == oracle.OK
        assert indices.tolist() == g["expected_kv_indices"]
        assert indptr.tolist() == g["expected_kv_indptr"]
        assert last.tolist() == g[last_key]
        # padded block table: the same pages, -1 past each request's last page
        assert bt.tolist() == [[5, 6, 8, -1], [2, 3, -1, -1], [10, 11, 15, 18]]


def test_p5_indptr_worked_example():
    g = golden("p5_indptr_seq_lens.json")
    lens = g["seq_lens"]
    rng = np.random.default_rng(3)
    r2t, rpi = paged_table(rng, lens, 1, 64)
    st, indptr, indices, last, _ = oracle.build_indices(r2t, rpi, lens, 1, 64)
    assert st == oracle.OK
    assert indptr.tolist() == g["expected_kv_indptr"]
    # at page_size 1 the page list is the token-slot row itself
    assert indices.tolist() == np.concatenate([r2t[rpi[b], :L] for b, L in enumerate(lens)]).tolist()
    assert last.tolist() == [1, 1, 1]


def test_p4_page_table_rows():
    g = golden("p4_page_table_rows.json")
    ps = g["page_size"]
    r2t = np.zeros((3, 64), dtype=np.int32)
    for i, row in enumerate(g["rows"]):
        r2t[i, :len(row)] = row
    lens = [len(r) for r in g["rows"]]
    st, indptr, indices, last, bt = oracle.build_indices(r2t, [0, 1], lens, ps, g["pool_pages"])
    assert st == oracle.OK
    assert [indices[indptr[b]:indptr[b + 1]].tolist() for b in range(2)] == g["expected_pages"]
    assert last.tolist() == g["expected_last_page_len"]


@pytest.mark.parametrize("ps", [1, 2, 4, 16, 64])
def test_build_indices_roundtrip_and_brute_force(ps):
    rng = np.random.default_rng(ps)
    lens = [0, 1, ps, ps + 1, 3 * ps, 5 * ps - 1, 77]
    starts = [0, ps, 0, 2 * ps, 0, ps, 4 * ps]
    num_pages = 4 + sum(-(-L // ps) for L in lens)
    r2t, rpi = paged_table(rng, lens, ps, num_pages, kv_start=starts)
    st, indptr, indices, last, bt = oracle.build_indices(r2t, rpi, lens, ps, num_pages, kv_start=starts)
    assert st == oracle.OK
    for b, L in enumerate(lens):
        row = r2t[rpi[b], starts[b]:starts[b] + L].astype(np.int64)
        pages = indices[indptr[b]:indptr[b + 1]]
        # round trip: page_table[t // ps] * ps + t % ps reproduces every slot
        t = np.arange(L)
        assert np.array_equal(pages[t // ps].astype(np.int64) * ps + t % ps, row)
        # brute force: for each chunk of ps positions, the one pool page holding all its slots
        for p in range(-(-L // ps)):
            chunk = row[p * ps:(p + 1) * ps]
            holders = [pg for pg in range(num_pages) if all(pg * ps <= s < pg * ps + ps for s in chunk)]
            assert holders == [pages[p]]
        assert last[b] == (L - (len(pages) - 1) * ps if L else 0)
        assert bt[b, :len(pages)].tolist() == pages.tolist()
        assert (bt[b, len(pages):] == -1).all()


def test_build_indices_rejects_bad_tables():
    rng = np.random.default_rng(7)
    ps, lens = 4, [9, 6]
    r2t, rpi = paged_table(rng, lens, ps, 16)
    good = r2t.copy()
    assert oracle.build_indices(good, rpi, lens, ps, 16)[0] == oracle.OK
    bad = good.copy()
    bad[rpi[0], 5] += 1                      # breaks contiguity inside page 1
    assert oracle.build_indices(bad, rpi, lens, ps, 16)[0] == oracle.ERR_CONTIG
    bad = good.copy()
    bad[rpi[1], 0:4] = [5, 6, 7, 8]          # page not aligned to a page boundary
    assert oracle.build_indices(bad, rpi, lens, ps, 16)[0] == oracle.ERR_CONTIG
    bad = good.copy()
    bad[rpi[1], 0:4] = np.arange(64, 68)     # page 16 is outside a 16-page pool
    assert oracle.build_indices(bad, rpi, lens, ps, 16)[0] == oracle.ERR_RANGE
    assert oracle.build_indices(good, rpi, lens, ps, 16, kv_indices_cap=4)[0] == oracle.ERR_CAPACITY
    assert oracle.build_indices(good, [99, 1], lens, ps, 16)[0] == oracle.ERR_RANGE
    # a page size that does not divide the decoder offset breaks alignment
    assert oracle.build_indices(good, rpi, [4, 4], ps, 16, kv_start=[2, 0])[0] == oracle.ERR_CONTIG


def test_arithmetic_on_the_pages():
    from paged_kv_cache_req_gb300.workloads import make_workload, round_up
    g = golden("p1_p4_arithmetic.json")
    assert g["whisper_enc_len"] % 128 == g["enc_len_mod_128"]
    assert round_up(g["whisper_enc_len"], 128) == g["ceil_align_1500_128"]
    wl = make_workload("whisper_encdec", batch=4)
    assert wl.meta["enc_reserve"] == round_up(1500, 16) == 1504
    assert (wl.problem("self").kv_start.numpy() == 1504).all()
    # 17 tokens at page size 16 occupy two pages
    st, indptr, *_ = oracle.build_indices(np.arange(32, dtype=np.int32)[None, :] + 16, [0], [17], 16, 4)
    assert st == oracle.OK and indptr.tolist() == [0, 2] == [0, g["pages_for_17_tokens_at_ps16"]]


def test_kv_bytes_per_token_against_pool_allocation():
    """2 x layers x kv_heads x head_dim x 2 B, measured on the pools the generator builds."""
    from paged_kv_cache_req_gb300.workloads import fill_pool, make_workload
    g = golden("p1_p4_arithmetic.json")
    for wname, key in (("qwen3_0p6b", "qwen3_0p6b"), ("llama3_8b", "llama31_8b")):
        wl = make_workload(wname, batch=2)
        wl.num_slots = 64 * wl.page_size        # a small pool of the same row layout
        k, v = fill_pool(wl)
        per_layer = (k.stride(0) * k.element_size()) + (v.stride(0) * v.element_size())
        assert per_layer * g[key]["layers"] == g[key]["kv_bytes_per_token"]
    q = g["qwen3_0p6b"]
    assert 40 * 2**30 // q["kv_bytes_per_token"] == q["tokens_in_40GiB"]
    assert 4 * 2**30 // q["kv_bytes_per_token"] == q["tokens_in_4GiB"]


# ---------------------------------------------------------------- store
def test_p4_store_worked_example():
    g = golden("p4_store_layout.json")
    n_slots = g["num_pages"] * g["page_size"]
    shape = (n_slots, g["kv_heads"], g["head_dim"])
    k_pool = np.zeros(shape, dtype=np.float32)
    v_pool = np.zeros(shape, dtype=np.float32)
    k = np.asarray(g["token_values"], dtype=np.float32).reshape(3, g["kv_heads"], g["head_dim"])
    assert oracle.store(k_pool, k, g["out_loc"]) == oracle.OK
    assert oracle.store(v_pool, np.ascontiguousarray(-k), g["out_loc"]) == oracle.OK
    for slot, tok in g["expect_k_slot"].items():
        assert np.array_equal(k_pool[int(slot)], k[tok])
    e = g["expect_v_page_offset"]
    v_paged = v_pool.reshape(g["num_pages"], g["page_size"], g["kv_heads"], g["head_dim"])
    assert np.array_equal(v_paged[e["page"], e["offset"]], e["sign"] * k[e["token"]])
    untouched = [s for s in range(n_slots) if str(s) not in g["expect_k_slot"]]
    assert not k_pool[untouched].any()


def test_store_skips_negative_and_flags_out_of_range():
    # guard rows on both sides of the pool catch a write through a padded (-1)
    # or out-of-range slot
    buf = np.zeros((10, 4), dtype=np.uint16)
    pool = buf[1:9]
    rows = np.arange(12, dtype=np.uint16).reshape(3, 4) + 1
    assert oracle.store(pool, rows, [-1, 3, 9]) == oracle.ERR_RANGE
    assert np.array_equal(pool[3], rows[1])
    assert buf.sum() == rows[1].sum()


# ---------------------------------------------------------------- decode
def _sdpa_reference(q_bits, k_bits, v_bits, r2t, rpi, lens, scale, kv_start=None, dv=None):
    """Library attention on contiguous K/V copied out with numpy indexing."""
    B, hq, dqk = q_bits.shape
    outs = []
    for b in range(B):
        s = 0 if kv_start is None else int(kv_start[b])
        slots = r2t[rpi[b], s:s + lens[b]].astype(np.int64)
        q = bits_to_f64(q_bits[b])[None, :, None, :]                 # [1, Hq, 1, D]
        if k_bits.ndim == 2:                                          # latent pool
            k = bits_to_f64(k_bits[slots])[None, None]                # [1, 1, L, 576]
            v = bits_to_f64(k_bits[slots][:, :dv])[None, None]
        else:
            k = bits_to_f64(k_bits[slots]).permute(1, 0, 2)[None]     # [1, Hkv, L, D]
            v = bits_to_f64(v_bits[slots]).permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale, enable_gqa=True)
        outs.append(o[0, :, 0, :].numpy())
    return np.stack(outs)


def _rand_bits(gen, shape):
    return bf16_bits(torch.randn(shape, generator=gen).to(torch.bfloat16))


@pytest.mark.parametrize("hq,hkv,d,dv,ps", [(4, 4, 64, 64, 1), (8, 4, 128, 128, 16), (16, 4, 32, 32, 4),
                                           (6, 2, 16, 16, 64), (4, 2, 32, 16, 4)])
def test_decode_matches_library_attention(hq, hkv, d, dv, ps):
    rng = np.random.default_rng(hq * 131 + ps)
    gen = torch.Generator().manual_seed(hq + d)
    lens = [1, 5, ps + 3, 70]
    starts = [0, ps, 2 * ps, 0]
    num_pages = 2 + sum(-(-L // ps) for L in lens)
    r2t, rpi = paged_table(rng, lens, ps, num_pages, kv_start=starts)
    slots = num_pages * ps
    k = _rand_bits(gen, (slots, hkv, d))
    v = _rand_bits(gen, (slots, hkv, dv))
    q = _rand_bits(gen, (len(lens), hq, d))
    scale = 1.0 / math.sqrt(d)
    st, out, lse = oracle.decode(q, k, v, r2t, rpi, lens, scale, kv_start=starts)
    assert st == oracle.OK
    ref = _sdpa_reference(q, k, v, r2t, rpi, lens, scale, kv_start=starts)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # lse = ln sum exp(scale q.k) computed by a library logsumexp
    for b in range(len(lens)):
        sl = r2t[rpi[b], starts[b]:starts[b] + lens[b]]
        for h in range(hq):
            kk = bits_to_f64(k[sl][:, h // (hq // hkv)])
            x = scale * (kk @ bits_to_f64(q[b, h]))
            assert abs(torch.logsumexp(x, 0).item() - lse[b, h]) < 1e-10


def test_decode_closed_forms():
    rng = np.random.default_rng(11)
    gen = torch.Generator().manual_seed(11)
    hq, hkv, d, ps = 8, 2, 32, 4
    lens = [1, 9, 16]
    r2t, rpi = paged_table(rng, lens, ps, 16)
    k = _rand_bits(gen, (64, hkv, d))
    v = _rand_bits(gen, (64, hkv, d))
    q = _rand_bits(gen, (3, hq, d))
    g = hq // hkv
    # one cached key: out = V of that key (for every query head of the group)
    st, out, lse = oracle.decode(q, k, v, r2t, rpi, lens, 0.125)
    slot = r2t[rpi[0], 0]
    for h in range(hq):
        np.testing.assert_array_equal(out[0, h], bits_to_f64(v[slot, h // g]).numpy())
    # identical keys: out = mean of V over the keys
    k_same = k.copy()
    for b, L in enumerate(lens):
        for s in r2t[rpi[b], :L]:
            k_same[s] = k[r2t[rpi[b], 0]]
    st, out, lse = oracle.decode(q, k_same, v, r2t, rpi, lens, 0.125)
    for b, L in enumerate(lens):
        vb = bits_to_f64(v[r2t[rpi[b], :L]]).numpy()          # [L, Hkv, D]
        for h in range(hq):
            np.testing.assert_allclose(out[b, h], vb[:, h // g].mean(0), atol=1e-12)
    # q = 0: uniform weights, out = mean(V), lse = ln L
    st, out, lse = oracle.decode(np.zeros_like(q), k, v, r2t, rpi, lens, 0.125)
    for b, L in enumerate(lens):
        vb = bits_to_f64(v[r2t[rpi[b], :L]]).numpy()
        for h in range(hq):
            np.testing.assert_allclose(out[b, h], vb[:, h // g].mean(0), atol=1e-12)
            assert abs(lse[b, h] - math.log(L)) < 1e-12


def test_decode_empty_key_set():
    rng = np.random.default_rng(2)
    gen = torch.Generator().manual_seed(2)
    r2t, rpi = paged_table(rng, [0, 3], 1, 16)
    k = _rand_bits(gen, (16, 1, 8))
    q = _rand_bits(gen, (2, 2, 8))
    st, out, lse = oracle.decode(q, k, k, r2t, rpi, [0, 3], 0.3)
    assert st == oracle.OK
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1]).all()


def test_decode_invariant_under_page_placement():
    """Moving pages to other pool locations (and rewriting the rows) changes nothing."""
    rng = np.random.default_rng(5)
    gen = torch.Generator().manual_seed(5)
    ps, hq, hkv, d = 8, 4, 2, 64
    lens = [8, 17, 40]
    num_pages = 16
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    k = _rand_bits(gen, (num_pages * ps, hkv, d))
    v = _rand_bits(gen, (num_pages * ps, hkv, d))
    q = _rand_bits(gen, (3, hq, d))
    st, out0, lse0 = oracle.decode(q, k, v, r2t, rpi, lens, 0.1)
    perm = np.concatenate([[0], rng.permutation(np.arange(1, num_pages))])   # old page -> new page
    k2 = np.zeros_like(k)
    v2 = np.zeros_like(v)
    for old, new in enumerate(perm):
        k2[new * ps:(new + 1) * ps] = k[old * ps:(old + 1) * ps]
        v2[new * ps:(new + 1) * ps] = v[old * ps:(old + 1) * ps]
    r2t2 = (perm[r2t // ps] * ps + r2t % ps).astype(np.int32)
    st, out1, lse1 = oracle.decode(q, k2, v2, r2t2, rpi, lens, 0.1)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


def test_decode_mla_latent():
    """Latent pool: K = full 576-dim row, V = its first 512 dims, one kv head."""
    rng = np.random.default_rng(9)
    gen = torch.Generator().manual_seed(9)
    ps, hq, dqk, dv = 64, 16, 576, 512
    lens = [3, 64, 130]
    num_pages = 8
    r2t, rpi = paged_table(rng, lens, ps, num_pages)
    lat = _rand_bits(gen, (num_pages * ps, dqk))
    q = _rand_bits(gen, (3, hq, dqk))
    scale = 1 / math.sqrt(192)
    st, out, lse = oracle.decode(q, lat, lat, r2t, rpi, lens, scale, head_dim_v=dv)
    assert st == oracle.OK
    ref = _sdpa_reference(q, lat, None, r2t, rpi, lens, scale, dv=dv)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # the same numbers from the GQA form with separate K and V copies and Hkv = 1
    k_sep = np.ascontiguousarray(lat[:, None, :])
    v_sep = np.ascontiguousarray(lat[:, None, :dv])
    st, out2, lse2 = oracle.decode(q, k_sep, v_sep, r2t, rpi, lens, scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_lse_merge_of_splits_equals_unsplit():
    rng = np.random.default_rng(13)
    gen = torch.Generator().manual_seed(13)
    ps, hq, hkv, d = 4, 4, 2, 32
    lens = [1, 30, 57, 64]
    r2t, rpi = paged_table(rng, lens, ps, 64)
    k = _rand_bits(gen, (256, hkv, d))
    v = _rand_bits(gen, (256, hkv, d))
    q = _rand_bits(gen, (4, hq, d))
    st, ref, ref_lse = oracle.decode(q, k, v, r2t, rpi, lens, 0.2)
    for cuts in ([0, 16, 32, 48, 64], [0, 1, 2, 64], [0, 40, 64]):
        parts = [oracle.decode(q, k, v, r2t, rpi, lens, 0.2, t_begin=a, t_end=b)[1:]
                 for a, b in zip(cuts[:-1], cuts[1:])]
        o = np.stack([p[0].reshape(-1, d) for p in parts])
        l = np.stack([p[1].reshape(-1) for p in parts])
        out, lse = oracle.lse_merge(o, l)
        np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse.reshape(ref_lse.shape), ref_lse, rtol=1e-13)


# ---------------------------------------------------------------- ragged gather
def test_ragged_gather_contiguous_and_cu_seqlens():
    rng = np.random.default_rng(17)
    lens = [0, 5, 1, 12]
    starts = [0, 3, 1, 2]
    pool_k = rng.integers(0, 2**16, size=(64, 3, 8), dtype=np.uint16)
    pool_v = rng.integers(0, 2**16, size=(64, 3, 8), dtype=np.uint16)
    # an identity (arange) table: the gather is a contiguous slice of the pool
    r2t = np.tile(np.arange(40, dtype=np.int32), (5, 1))
    st, ko, vo, cu = oracle.ragged_gather(pool_k, pool_v, r2t, [1, 2, 3, 4], lens, kv_start=starts)
    assert st == oracle.OK
    assert cu.tolist() == [0] + np.cumsum(lens).tolist()
    for b, L in enumerate(lens):
        np.testing.assert_array_equal(ko[cu[b]:cu[b + 1]], pool_k[starts[b]:starts[b] + L])
        np.testing.assert_array_equal(vo[cu[b]:cu[b + 1]], pool_v[starts[b]:starts[b] + L])
    # a shuffled paged table: each packed row is the pool row the table names
    r2t2, rpi = paged_table(rng, lens, 4, 16)
    st, ko, vo, cu = oracle.ragged_gather(pool_k, pool_v, r2t2, rpi, lens)
    flat = np.concatenate([r2t2[rpi[b], :L] for b, L in enumerate(lens)])
    np.testing.assert_array_equal(ko, pool_k[flat])
    np.testing.assert_array_equal(vo, pool_v[flat])
    assert oracle.ragged_gather(pool_k, pool_v, r2t2, rpi, lens, out_rows_cap=10)[0] == oracle.ERR_CAPACITY


# ---------------------------------------------------------------- allocator and row writer
def _rows_after_prefix(rng, lens, ps, num_pages, width):
    """Rows already holding `lens` tokens each (whole shuffled pages), the rest of the
    pool as the free list; returns (r2t, rpi, free_pages)."""
    r2t, rpi = paged_table(rng, lens, ps, num_pages, width=width)
    used = set()
    for b, L in enumerate(lens):
        used.update((r2t[rpi[b], :L] // ps).tolist())
    free = np.array([p for p in rng.permutation(np.arange(1, num_pages)) if p not in used], dtype=np.int32)
    return r2t, rpi, free


def test_alloc_page_size_one_pops_the_front_of_the_free_list():
    # TokenToKVPoolAllocator: alloc(need) returns the first `need` free slots
    free = np.array([7, 3, 9, 1, 12, 5], dtype=np.int32)
    state = np.array([0, 6], dtype=np.int32)
    st, out = oracle.alloc_extend([0, 2], [2, 5], [-1, 4], 1, 16, free, state)
    assert st == oracle.OK and out.tolist() == [7, 3, 9, 1, 12] and state.tolist() == [5, 1]


def test_alloc_extend_equals_one_token_at_a_time_for_one_request():
    # alloc_extend of positions [p, s) equals s - p alloc_decode steps of one request
    ps, p, s = 8, 13, 42
    rng = np.random.default_rng(3)
    free = rng.permutation(np.arange(2, 40)).astype(np.int32)
    last = 5 * ps + (p - 1) % ps
    st, out = oracle.alloc_extend([p], [s], [last], ps, 40, free, np.array([0, len(free)], np.int32))
    assert st == oracle.OK
    state = np.array([0, len(free)], np.int32)
    step, prev = [], last
    for t in range(p, s):
        st, o = oracle.alloc_extend([t], [t + 1], [prev], ps, 40, free, state)
        assert st == oracle.OK
        step.append(int(o[0]))
        prev = int(o[0])
    assert out.tolist() == step


@pytest.mark.parametrize("ps", [1, 4, 16])
def test_alloc_then_write_keeps_pages_contiguous(ps):
    # the allocator's invariant ("keeps a sequence's tokens contiguous within each
    # page"): after alloc_extend + write_req_to_token every row passes build_indices,
    # the new pages are the front of the free list, each owned by one request
    rng = np.random.default_rng(ps)
    num_pages = 400 // ps + 40
    prefix = [0, 1, ps, 3 * ps + 1, 5]
    seq = [3, 1 + 2 * ps, 4 * ps, 3 * ps + 2, 5 + 7 * ps]
    r2t, rpi, free = _rows_after_prefix(rng, prefix, ps, num_pages, max(seq) + 8)
    last = [int(r2t[rpi[b], p - 1]) if p else -1 for b, p in enumerate(prefix)]
    state = np.array([2, len(free) - 2], np.int32)
    st, out = oracle.alloc_extend(prefix, seq, last, ps, num_pages, free, state)
    assert st == oracle.OK
    taken = sum(-(-s // ps) - (-(-p // ps)) for p, s in zip(prefix, seq))
    assert state.tolist() == [2 + taken, len(free) - 2 - taken]
    new_pages = sorted(set((out // ps).tolist()) - set(last_p // ps for last_p in last if last_p >= 0))
    assert new_pages == sorted(free[2:2 + taken].tolist())
    assert len(set(out.tolist())) == len(out)
    assert oracle.write_req_to_token(r2t, rpi, prefix, seq, [None] * len(seq), out) == oracle.OK
    st, *_ = oracle.build_indices(r2t, rpi, seq, ps, num_pages)
    assert st == oracle.OK
    e = 0
    for b, (p, s) in enumerate(zip(prefix, seq)):   # brute force: the row is prefix then the new slots
        assert r2t[rpi[b], p:s].tolist() == out[e:e + s - p].tolist()
        e += s - p


def test_alloc_out_of_pages_changes_nothing():
    free = np.arange(10, 20, dtype=np.int32)                                         # entries past the count
    state = np.array([1, 2], np.int32)                                               # are not free
    st, out = oracle.alloc_extend([0, 0], [16, 20], [-1, -1], 16, 64, free, state)   # needs 3 pages, 2 free
    assert st == oracle.ERR_CAPACITY and state.tolist() == [1, 2] and (out == -1).all()
    st, _ = oracle.alloc_extend([5], [6], [2 * 16 + 3], 16, 64, free, state)        # last_loc at the wrong offset
    assert st == oracle.ERR_CONTIG and state.tolist() == [1, 2]


def test_write_req_to_token_prefix_and_new_slots():
    r2t = np.full((4, 12), -5, dtype=np.int32)
    pre = [np.array([40, 41, 42], np.int32), None, np.array([9], np.int32)]
    st = oracle.write_req_to_token(r2t, [2, 1, 3], [3, 2, 1], [5, 4, 2], pre, np.array([7, 8, 100, 101, 55]),
                                   kv_start=[0, 4, 8])
    assert st == oracle.OK
    assert r2t[2].tolist() == [40, 41, 42, 7, 8] + [-5] * 7
    assert r2t[1].tolist() == [-5] * 4 + [-5, -5, 100, 101] + [-5] * 4      # NULL prefix: columns 4, 5 untouched
    assert r2t[3].tolist() == [-5] * 8 + [9, 55, -5, -5]
    assert (r2t[0] == -5).all()
    assert oracle.write_req_to_token(r2t, [2], [0], [13], [None], np.arange(13)) == oracle.ERR_RANGE


# ---------------------------------------------------------------- encoder-cache merge
def test_encoder_merge_matches_numpy_indexing():
    rng = np.random.default_rng(11)
    nb, bs, d, ntok = 6, 8, 5, 30
    buf = rng.integers(-1000, 1000, size=(nb, bs, d)).astype(np.int32)
    block_ids = np.array([0, 2, 3, 4, 5], np.int32)                 # an image, a 3-block video, the scratch block
    pos = np.full((5, bs), ntok, dtype=np.int64)                    # sentinel everywhere ...
    perm = rng.permutation(ntok)
    pos[0, :6] = perm[:6]                                           # ... but 6 image tokens,
    pos[1:4, :] = perm[6:30].reshape(3, 8)                          # 24 video tokens
    pos[4, 3] = ntok + 7                                            # past the end: also a don't-care
    hidden = np.full((ntok, d), -1, np.int32)
    st, filled = oracle.encoder_merge(buf, block_ids, pos, hidden)
    assert st == oracle.OK and filled == 30
    ref = np.full((ntok, d), -1, np.int32)
    flat = buf[block_ids].reshape(-1, d)
    valid = (pos.reshape(-1) < ntok)
    ref[pos.reshape(-1)[valid]] = flat[valid]
    assert np.array_equal(hidden, ref)
    bad = pos.copy()
    bad[0, 6] = -1
    assert oracle.encoder_merge(buf, block_ids, bad, hidden.copy())[0] == oracle.ERR_RANGE
    assert oracle.encoder_merge(buf, np.array([0, 2, 3, 4, 9], np.int32), pos, hidden.copy())[0] == oracle.OK  # all sentinel


# ---------------------------------------------------------------- multi-query (extend / verify / spans)
def _sdpa_masked(q_bits, k_bits, v_bits, r2t, rpi, lens, qo, kv_end, scale):
    """Library attention with an explicit boolean mask from the key bounds."""
    outs = []
    for b in range(len(lens)):
        slots = r2t[rpi[b], :lens[b]].astype(np.int64)
        q = bits_to_f64(q_bits[qo[b]:qo[b + 1]]).permute(1, 0, 2)[None]          # [1, Hq, n, D]
        k = bits_to_f64(k_bits[slots]).permute(1, 0, 2)[None]                     # [1, Hkv, L, D]
        v = bits_to_f64(v_bits[slots]).permute(1, 0, 2)[None]
        mask = torch.arange(lens[b])[None, :] < torch.as_tensor(kv_end[qo[b]:qo[b + 1]])[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask[None, None], scale=scale,
                                                             enable_gqa=True)
        outs.append(o[0].permute(1, 0, 2).numpy())
    return np.concatenate(outs)


@pytest.mark.parametrize("hq,hkv,d,ps,kind", [(8, 2, 32, 4, "extend"), (4, 4, 16, 1, "verify"), (8, 2, 32, 16, "spans"),
                                             (6, 3, 16, 8, "extend")])
def test_extend_matches_masked_library_attention(hq, hkv, d, ps, kind):
    rng = np.random.default_rng(hq * 10 + ps)
    gen = torch.Generator().manual_seed(ps)
    lens = [37, 64, 9, 120]
    r2t, rpi = paged_table(rng, lens, ps, 200 // ps + 40)
    slots = (200 // ps + 40) * ps
    k = _rand_bits(gen, (slots, hkv, d))
    v = _rand_bits(gen, (slots, hkv, d))
    if kind == "extend":        # the last n positions are new, causal
        n = [5, 64, 1, 17]
        kv_end = np.concatenate([np.arange(L - m, L) + 1 for L, m in zip(lens, n)])
    elif kind == "verify":      # 4 draft tokens each
        n = [4] * 4
        kv_end = np.concatenate([np.arange(L - 4, L) + 1 for L in lens])
    else:                       # causal prefix then a full span (a diffusion row), through the planner
        segs = [[(0, 0, 20), (1, 20, 37)], [(1, 32, 64)], [(0, 0, 9)], [(1, 100, 120)]]
        st, qo, q_pos, kv_end = oracle.span_plan(segs)
        assert st == oracle.OK
        n = np.diff(qo).tolist()
    qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    q = _rand_bits(gen, (int(qo[-1]), hq, d))
    st, out, lse = oracle.extend(q, k, v, r2t, rpi, lens, qo, kv_end, 1 / math.sqrt(d))
    assert st == oracle.OK
    ref = _sdpa_masked(q, k, v, r2t, rpi, lens, qo, kv_end, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    # lse against the log-sum-exp of the same scores
    j, h = int(qo[1]) + 3, hq - 1
    b = 1
    slots_b = r2t[rpi[b], :kv_end[j]].astype(np.int64)
    sc = (bits_to_f64(k[slots_b][:, h // (hq // hkv)]) @ bits_to_f64(q[j, h])) / math.sqrt(d)
    assert abs(lse[j, h] - float(torch.logsumexp(sc, 0))) < 1e-10


def test_extend_prefill_is_library_causal_attention():
    # prefix 0: every position is new, the mask is the ordinary causal one
    rng = np.random.default_rng(2)
    gen = torch.Generator().manual_seed(2)
    L, hq, hkv, d = 50, 4, 2, 16
    r2t, rpi = paged_table(rng, [L], 1, 80)
    k = _rand_bits(gen, (80, hkv, d))
    v = _rand_bits(gen, (80, hkv, d))
    q = _rand_bits(gen, (L, hq, d))
    st, out, _ = oracle.extend(q, k, v, r2t, rpi, [L], [0, L], np.arange(1, L + 1), 0.25)
    assert st == oracle.OK
    slots = r2t[rpi[0], :L].astype(np.int64)
    ref = torch.nn.functional.scaled_dot_product_attention(
        bits_to_f64(q).permute(1, 0, 2)[None], bits_to_f64(k[slots]).permute(1, 0, 2)[None],
        bits_to_f64(v[slots]).permute(1, 0, 2)[None], is_causal=True, scale=0.25, enable_gqa=True)
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_extend_closed_forms():
    rng = np.random.default_rng(4)
    gen = torch.Generator().manual_seed(4)
    r2t, rpi = paged_table(rng, [10, 10], 2, 20)
    k = _rand_bits(gen, (40, 2, 8))
    v = _rand_bits(gen, (40, 2, 8))
    q = _rand_bits(gen, (3, 4, 8))
    st, out, lse = oracle.extend(q, k, v, r2t, rpi, [10, 10], [0, 2, 3], [1, 0, 10], 0.3)
    assert st == oracle.OK
    first = r2t[rpi[0], 0]
    np.testing.assert_array_equal(out[0, :2], bits_to_f64(v[first][0:1]).numpy().repeat(2, 0))   # one key: V
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()                                     # no keys
    assert oracle.extend(q, k, v, r2t, rpi, [10, 10], [0, 2, 3], [1, 11, 10], 0.3)[0] == oracle.ERR_RANGE


def test_span_plan_follows_the_segment_table():
    g = golden("span_segments.json")
    st, qo, q_pos, kv_end = oracle.span_plan([[tuple(s) for s in g["first_step"]["segments"]],
                                              [tuple(s) for s in g["later_step"]["segments"]]])
    assert st == oracle.OK
    assert qo.tolist() == [0, 7, 10]
    assert q_pos.tolist() == g["first_step"]["q_pos"] + g["later_step"]["q_pos"]
    assert kv_end.tolist() == g["first_step"]["kv_end"] + g["later_step"]["kv_end"]
    assert g["later_step"]["kv_end"][0] == g["later_step"]["prefix_len"] + g["later_step"]["target_len"]
    assert oracle.span_plan([[(1, 5, 3)]])[0] == oracle.ERR_RANGE
