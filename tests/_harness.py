"""Test-side glue between the CUDA path and the CPU oracle.

Nothing here computes attention, page lists or gathers: it moves tensors to
numpy, compacts a sampled set of requests into a small host pool (slot
numbers are relabelled, which the oracle's page-placement invariance pin shows
does not change results), and applies the tolerance.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL = 2e-2
RTOL = 2e-2


def paged_table(rng, lens, ps, num_pages, kv_start=None, width=None, rows=None):
    """Tiny paged layout: shuffled whole pages per request; returns (r2t, rpi)."""
    B = len(lens)
    starts = np.zeros(B, dtype=np.int64) if kv_start is None else np.asarray(kv_start)
    width = width or int((starts + np.asarray(lens)).max()) + 3
    rows = rows or B + 1
    r2t = np.zeros((rows, width), dtype=np.int32)
    rpi = (rng.permutation(rows - 1)[:B] + 1).astype(np.int32)
    free = list(rng.permutation(np.arange(1, num_pages)))
    for b, L in enumerate(lens):
        s = int(starts[b])
        assert s % ps == 0
        n = -(-L // ps)
        pages, free = free[:n], free[n:]
        slots = (np.asarray(pages, dtype=np.int64)[:, None] * ps + np.arange(ps)).reshape(-1)[:L]
        r2t[rpi[b], s:s + L] = slots
    return r2t, rpi


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 bit patterns on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError("%s: %d / %d elements outside |err| <= %.0e + %.0e|ref|; first at %s: gpu %r ref %r "
                             "(max abs err %.3e)" % (what, bad.sum(), bad.size, ATOL, RTOL, tuple(idx),
                                                     gpu[tuple(idx)], ref[tuple(idx)], err.max()))
    return float(err.max())


def compact(r2t: np.ndarray, rpi: np.ndarray, lens: np.ndarray, starts: np.ndarray, sample, extra_slots=()):
    """Slots the sampled requests touch, relabelled 0..n-1 in a one-row-per-request table."""
    rows = [r2t[rpi[b], starts[b]:starts[b] + lens[b]].astype(np.int64) for b in sample]
    allslots = np.unique(np.concatenate(rows + [np.asarray(list(extra_slots), dtype=np.int64)]))
    relabel = {int(s): i for i, s in enumerate(allslots)}
    width = int(max([len(r) for r in rows] + [1]))
    t = np.zeros((len(sample) + 1, width), dtype=np.int32)
    for i, r in enumerate(rows):
        t[i + 1, :len(r)] = np.searchsorted(allslots, r)
    return allslots, t, np.arange(1, len(sample) + 1, dtype=np.int32), relabel


def oracle_decode_problem(step, name, sample, pre_k=None, pre_v=None, store=True, r2t=None, slot_mapping=None):
    """fp64 oracle output of one problem of a DecodeStep for the sampled requests.

    pre_k / pre_v: the pool rows as they were before the GPU step ran (host
    tensors indexed by slot), or None to read them now from the device (valid
    when the step does not store into this problem's rows, or before it runs).
    The oracle applies the store itself, then decodes.  r2t / slot_mapping
    replace the workload's table and new-token slots (the oracle's own
    allocation, for steps that allocate on the device).
    """
    wl = step.wl
    pb = step.problems[name]
    r2t = wl.req_to_token.numpy() if r2t is None else r2t
    rpi = wl.req_pool_idx.numpy()
    lens = pb.spec.seq_lens.numpy()
    starts = pb.spec.kv_start.numpy()
    sample = list(sample)
    new_slots = []
    if store and pb.spec.stores:
        sm_all = pb.spec.slot_mapping.numpy() if slot_mapping is None else np.asarray(slot_mapping)
        new_slots = sm_all[sample]
    allslots, t, rpi_c, relabel = compact(r2t, rpi, lens, starts, sample, extra_slots=new_slots)
    idx = torch.from_numpy(allslots)
    src_k = pre_k if pre_k is not None else step.k_pool
    k_host = bits(src_k[idx.to(src_k.device)])
    v_host = None
    if step.v_pool is not None:
        src_v = pre_v if pre_v is not None else step.v_pool
        v_host = bits(src_v[idx.to(src_v.device)])
    if store and pb.spec.stores:
        sm = np.asarray([relabel[int(s)] for s in new_slots], dtype=np.int32)
        assert oracle.store(k_host, bits(step.k_new)[sample], sm) == oracle.OK
        if v_host is not None:
            assert oracle.store(v_host, bits(step.v_new)[sample], sm) == oracle.OK
    q = bits(pb.q)[sample]
    if wl.kind == "mla":
        st, out, lse = oracle.decode(q, k_host, k_host, t, rpi_c, lens[sample], wl.sm_scale,
                                     head_dim_v=wl.head_dim_v)
    else:
        st, out, lse = oracle.decode(q, k_host, v_host, t, rpi_c, lens[sample], wl.sm_scale)
    assert st == oracle.OK
    return out, lse
