"""GPU parity of the slot bookkeeping and the encoder-cache merge against the CPU oracle.

pkv_alloc_extend, pkv_write_req_to_token and pkv_encoder_merge are integer or
byte work: every output is compared bit for bit (slots, free-list state, whole
tables, hidden rows), including the all-or-nothing failure of a step that does
not fit and the sentinel positions of the merge.
"""
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


def _dev(a, dtype=torch.int32):
    return torch.as_tensor(np.asarray(a)).to(dtype).cuda()


def _step_case(rng, ps, batch, max_prefix, max_extend, num_pages):
    """Rows holding `prefix` tokens (whole shuffled pages), a free list of the other pages,
    and a growth to `seq`: a mix of decode (+1), extends and fresh requests."""
    prefix = rng.integers(0, max_prefix + 1, batch)
    prefix[rng.random(batch) < 0.2] = 0
    grow = np.where(rng.random(batch) < 0.5, 1, rng.integers(1, max_extend + 1, batch))
    seq = prefix + grow
    width = int(seq.max()) + 32
    r2t, rpi = paged_table(rng, prefix.tolist(), ps, num_pages, width=width, rows=batch + 5)
    used = set()
    for b, L in enumerate(prefix):
        used.update((r2t[rpi[b], :L] // ps).tolist())
    free = np.array([p for p in rng.permutation(np.arange(1, num_pages)) if p not in used], dtype=np.int32)
    last = np.array([r2t[rpi[b], p - 1] if p else -1 for b, p in enumerate(prefix)], dtype=np.int32)
    return prefix.astype(np.int32), seq.astype(np.int32), last, r2t, rpi, free


@pytest.mark.parametrize("ps,batch", [(1, 37), (16, 256), (64, 1000), (64, 4096)])
def test_alloc_and_row_writer_bit_exact(B, ps, batch):
    rng = np.random.default_rng(ps * 7 + batch)
    num_pages = (batch * 600) // ps + 64
    prefix, seq, last, r2t, rpi, free = _step_case(rng, ps, batch, 400, 300, num_pages)
    head = 3
    state_ref = np.array([head, len(free) - head], np.int32)
    st, loc_ref = oracle.alloc_extend(prefix, seq, last, ps, num_pages, free, state_ref)
    assert st == oracle.OK
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = _dev([head, len(free) - head])
    loc = torch.full((len(loc_ref) + 5,), -7, dtype=torch.int32, device="cuda")
    B.pkv_alloc_extend(_dev(prefix), _dev(seq), _dev(last), ps, num_pages, _dev(free), state, loc, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(loc[:len(loc_ref)].cpu().numpy(), loc_ref)
    assert (loc[len(loc_ref):] == -7).all()
    assert state.cpu().numpy().tolist() == state_ref.tolist()

    # rows: reused prefixes for a third of the requests (fresh copies elsewhere in the table
    # beforehand would be overwritten), the others already in place
    reuse = rng.random(batch) < 0.33
    pref_arrays = [r2t[rpi[b], :prefix[b]].copy() if reuse[b] and prefix[b] else None for b in range(batch)]
    table = r2t.copy()
    for b in range(batch):
        if pref_arrays[b] is not None:
            table[rpi[b], :prefix[b]] = -1          # the writer must restore them from the pointer
    ref = table.copy()
    assert oracle.write_req_to_token(ref, rpi, prefix, seq, pref_arrays, loc_ref) == oracle.OK
    keep = [_dev(a) if a is not None else None for a in pref_arrays]
    ptrs = _dev([t.data_ptr() if t is not None else 0 for t in keep], torch.int64)
    tab_d = _dev(table)
    B.pkv_write_req_to_token(tab_d, _dev(rpi), _dev(prefix), _dev(seq), loc[:len(loc_ref)], err, prefix_slots=ptrs)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(tab_d.cpu().numpy(), ref)
    # the allocator's invariant: the new rows pass the contiguity check of build_indices
    indptr = torch.empty(batch + 1, dtype=torch.int32, device="cuda")
    idx = torch.empty(int((-(-seq.astype(np.int64) // ps)).sum()), dtype=torch.int32, device="cuda")
    lastp = torch.empty(batch, dtype=torch.int32, device="cuda")
    B.pkv_build_indices(tab_d, _dev(rpi), _dev(seq), ps, num_pages, err, kv_indptr=indptr, kv_indices=idx,
                        kv_last_page_len=lastp)
    torch.cuda.synchronize()
    assert err.item() == 0


def test_alloc_step_that_does_not_fit_changes_nothing(B):
    rng = np.random.default_rng(5)
    ps, batch, num_pages = 16, 64, 3000
    prefix, seq, last, r2t, rpi, free = _step_case(rng, ps, batch, 200, 200, num_pages)
    need = int(((-(-seq.astype(np.int64) // ps)) - (-(-prefix.astype(np.int64) // ps))).sum())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    state = _dev([0, need - 1])                         # one page short
    loc = torch.full((int((seq - prefix).sum()),), -7, dtype=torch.int32, device="cuda")
    B.pkv_alloc_extend(_dev(prefix), _dev(seq), _dev(last), ps, num_pages, _dev(free), state, loc, err)
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_CAPACITY
    assert (loc == -7).all() and state.cpu().tolist() == [0, need - 1]
    # last_loc at the wrong page offset: a contiguity error, nothing written
    bad = last.copy()
    assert (prefix % ps != 0).any()
    j = int(np.argmax(prefix % ps != 0))
    bad[j] = (bad[j] // ps) * ps + ((bad[j] % ps) + 1) % ps
    err.zero_()
    state = _dev([0, len(free)])
    B.pkv_alloc_extend(_dev(prefix), _dev(seq), _dev(bad), ps, num_pages, _dev(free), state, loc, err)
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_CONTIG and (loc == -7).all() and state.cpu().tolist() == [0, len(free)]


def test_row_writer_long_rows_and_range(B):
    rng = np.random.default_rng(9)
    rows, width = 6, 20000
    table = np.full((rows, width), -3, np.int32)
    prefix = np.array([0, 9000, 5, 12000], np.int32)
    seq = np.array([13000, 9001, 17000, 12000], np.int32)
    rpi = np.array([4, 1, 2, 5], np.int32)
    starts = np.array([100, 0, 2000, 8], np.int32)
    loc = rng.integers(0, 1 << 30, int((seq - prefix).sum())).astype(np.int32)
    pref = [None, rng.integers(0, 1000, 9000).astype(np.int32), None, rng.integers(0, 9, 12000).astype(np.int32)]
    ref = table.copy()
    assert oracle.write_req_to_token(ref, rpi, prefix, seq, pref, loc, kv_start=starts) == oracle.OK
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    keep = [_dev(a) if a is not None else None for a in pref]
    ptrs = _dev([t.data_ptr() if t is not None else 0 for t in keep], torch.int64)
    tab_d = _dev(table)
    B.pkv_write_req_to_token(tab_d, _dev(rpi), _dev(prefix), _dev(seq), _dev(loc), err, prefix_slots=ptrs,
                             kv_start=_dev(starts))
    torch.cuda.synchronize()
    assert err.item() == 0 and np.array_equal(tab_d.cpu().numpy(), ref)
    # a request past the table's width is skipped with a range error; the others are written
    starts2 = starts.copy()
    starts2[2] = width - 100
    ref2 = table.copy()
    assert oracle.write_req_to_token(ref2, rpi, prefix, seq, pref, loc, kv_start=starts2) == oracle.ERR_RANGE
    tab_d = _dev(table)
    B.pkv_write_req_to_token(tab_d, _dev(rpi), _dev(prefix), _dev(seq), _dev(loc), err, prefix_slots=ptrs,
                             kv_start=_dev(starts2))
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_RANGE and np.array_equal(tab_d.cpu().numpy(), ref2)


def _merge_case(rng, nb, bs, d, n_items, tokens_per_item, num_tokens, dtype=torch.bfloat16):
    gen = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
    buf = torch.randn((nb, bs, d), generator=gen).to(dtype)
    max_blocks = n_items + 2
    block_ids = np.full(max_blocks, nb - 1, np.int32)          # unused slots name the scratch block
    block_ids[:n_items] = rng.permutation(nb - 1)[:n_items]
    pos = np.full((max_blocks, bs), num_tokens, np.int64)      # sentinel
    dest = rng.permutation(num_tokens)[:n_items * tokens_per_item].reshape(n_items, tokens_per_item)
    pos[:n_items, :tokens_per_item] = dest
    return buf, block_ids, pos


@pytest.mark.parametrize("d,dtype", [(20480, torch.bfloat16), (1024, torch.bfloat16), (7, torch.bfloat16)])
def test_encoder_merge_bit_exact(B, d, dtype):
    rng = np.random.default_rng(d)
    nb, bs = 12, 512 if d > 1000 else 64
    num_tokens = 9 * 256 + 300
    buf, block_ids, pos = _merge_case(rng, nb, bs, d, 9, 256 if bs == 512 else 40, num_tokens, dtype)
    gen = torch.Generator().manual_seed(1)
    hidden = torch.randn((num_tokens, d), generator=gen).to(dtype)
    ref = bits(hidden).copy()
    st, filled_ref = oracle.encoder_merge(bits(buf), block_ids, pos, ref)
    assert st == oracle.OK
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    filled = torch.zeros(1, dtype=torch.int64, device="cuda")
    hid_d = hidden.cuda()
    B.pkv_encoder_merge(buf.cuda(), _dev(block_ids), _dev(pos, torch.int64), hid_d, err, filled=filled)
    torch.cuda.synchronize()
    assert err.item() == 0 and filled.item() == filled_ref
    assert np.array_equal(bits(hid_d), ref)


def test_encoder_merge_range_errors(B):
    rng = np.random.default_rng(3)
    buf, block_ids, pos = _merge_case(rng, 6, 64, 128, 3, 30, 200)
    pos[1, 3] = -4
    block_ids[2] = 40
    hidden = torch.zeros((200, 128), dtype=torch.bfloat16)
    ref = bits(hidden).copy()
    st, filled_ref = oracle.encoder_merge(bits(buf), block_ids, pos, ref)
    assert st == oracle.ERR_RANGE
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    filled = torch.zeros(1, dtype=torch.int64, device="cuda")
    hid_d = hidden.cuda()
    B.pkv_encoder_merge(buf.cuda(), _dev(block_ids), _dev(pos, torch.int64), hid_d, err, filled=filled)
    torch.cuda.synchronize()
    assert err.item() == B.PKV_DEVERR_RANGE and filled.item() == filled_ref
    assert np.array_equal(bits(hid_d), ref)
