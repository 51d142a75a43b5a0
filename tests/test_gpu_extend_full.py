"""Full-size parity of the three benchmarked multi-query recipes.

Each recipe runs through ExtendStep at its benchmark size and launch configuration
(pkv_build_indices, pkv_store, pkv_span_plan where the rows have segments,
pkv_extend with the library's own split plan), and sampled query rows of sampled
requests are checked against the fp64 oracle within |gpu - oracle| <= 2e-2 +
2e-2 |oracle|: every row of a target-verify request, and for the long prefill
and span rows a spread of rows that includes each request's first and last rows
and, for spans, the rows on both sides of the causal/full boundary.
"""
import numpy as np
import pytest
import torch

import oracle
from _harness import assert_close, bf16_to_f64, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _row_bounds(ew):
    """Per request: its query rows' key bounds (causal over the last positions, or the span plan)."""
    lens = ew.seq_lens.numpy().astype(np.int64)
    qo = ew.qo_lens.numpy().astype(np.int64)
    if ew.segments is not None:
        st, ind, _, kend = oracle.span_plan(ew.segments)
        assert st == oracle.OK
        return [kend[ind[b]:ind[b + 1]].astype(np.int64) for b in range(ew.batch)]
    return [np.arange(L - n, L) + 1 for L, n in zip(lens, qo)]


def _check(step, requests, rows_of):
    ew = step.ew
    bounds = _row_bounds(ew)
    r2t = ew.req_to_token.numpy()
    rpi = ew.req_pool_idx.numpy().astype(np.int64)
    lens = ew.seq_lens.numpy().astype(np.int64)
    qo_all = np.concatenate([[0], np.cumsum(ew.qo_lens.numpy().astype(np.int64))])
    out = bf16_to_f64(step.out)
    lse = step.lse.double().cpu().numpy()
    q_bits = bits(step.q)
    for b in requests:
        rows = np.asarray(rows_of(b, len(bounds[b])), dtype=np.int64)
        slots = r2t[rpi[b], :lens[b]].astype(np.int64)
        uniq = np.unique(slots)
        idx = torch.from_numpy(uniq).to(step.k_pool.device)
        k = bits(step.k_pool[idx])
        v = bits(step.v_pool[idx])
        table = np.zeros((2, max(int(lens[b]), 1)), dtype=np.int32)
        table[1, :lens[b]] = np.searchsorted(uniq, slots)
        glob = qo_all[b] + rows
        st, ref, ref_lse = oracle.extend(q_bits[glob], k, v, table, np.array([1], dtype=np.int32),
                                         [int(lens[b])], np.array([0, len(rows)], dtype=np.int32),
                                         bounds[b][rows].astype(np.int32), ew.sm_scale)
        assert st == oracle.OK
        assert_close(out[glob], ref, "%s request %d out" % (ew.name, b))
        assert_close(lse[glob], ref_lse, "%s request %d lse" % (ew.name, b))


def _spread(n, k, extra=()):
    return sorted(set(np.linspace(0, n - 1, num=min(n, k)).astype(np.int64).tolist() + [r for r in extra if r < n]))


@pytest.mark.parametrize("name,token_table", [("llama3_8b_verify", False), ("qwen3_0p6b_prefill", False),
                                              ("hunyuan_image_spans", False), ("qwen3_0p6b_prefill", True)])
def test_extend_recipe_at_full_size(B, name, token_table):
    """The benchmarked steps at full size; prefill also with the pages read straight from
    req_to_token (no pkv_build_indices launch)."""
    from paged_kv_cache_req_gb300.engine import ExtendStep
    from paged_kv_cache_req_gb300.workloads import make_extend_workload
    ew = make_extend_workload(name)
    step = ExtendStep(ew, device="cuda", token_table=token_table)
    assert step.launches_per_step() == (2 if token_table else 3) + (1 if ew.segments is not None else 0) + \
        (1 if step.ws_bytes > 0 else 0)
    step.run()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    rng = np.random.default_rng(11)
    if name == "llama3_8b_verify":
        lens = ew.seq_lens.numpy()
        requests = sorted(set([int(np.argmax(lens)), int(np.argmin(lens))] +
                              rng.choice(ew.batch, 6, replace=False).tolist()))
        _check(step, requests, lambda b, n: range(n))
    elif name == "qwen3_0p6b_prefill":
        requests = sorted(rng.choice(ew.batch, 3, replace=False).tolist())
        _check(step, requests, lambda b, n: _spread(n, 24, extra=(1, n - 2)))
    else:
        requests = [0, ew.batch - 1]
        _check(step, requests, lambda b, n: _spread(n, 24, extra=(1023, 1024, 1025)))
