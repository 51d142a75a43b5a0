"""pkv_decode_no_alloc: decode for callers that cannot call cudaMalloc.

Such callers (a plug-in whose host process gives all device memory to another
allocator, or a loop that must never block on an allocation) cannot provide
pkv_decode's workspace, so this entry point keeps the split partials in a
fixed array inside the library.  The test calls it through the C ABI twice in
a row, on a workload whose requests split into several chunks (so the scratch
and the merge are really used), and checks each result against pkv_decode with
a caller workspace, within the parity tolerance (in practice the two are
bitwise equal: same plan, same kernels), and against the fp64 oracle on
sampled requests.  It also checks that a plan larger
than the array is refused before launching.  This file sorts last so that a
run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2


def _close(a, b):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    assert (np.abs(a - b) <= ATOL + RTOL * np.abs(b)).all(), float(np.abs(a - b).max())


def test_no_alloc_decode_matches_workspace_decode_twice():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding as B
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload

    step = DecodeStep(make_workload("qwen3_0p6b"), kv_chunk=128)
    pb = step.problems["self"]
    assert pb.ws_bytes > 0, "the case must use split scratch"
    step.build_indices("self")
    step.store("self")
    step.decode("self")
    torch.cuda.synchronize()
    ref_out, ref_lse = pb.out.clone(), pb.lse.clone()
    # the fp64 oracle of the same step, on sampled requests (the store is idempotent,
    # so the pool as it is now gives the pre-step rows once the oracle re-applies it)
    from _harness import oracle_decode_problem
    sample = list(range(0, step.wl.batch, 5))
    oracle_out, oracle_lse = oracle_decode_problem(step, "self", sample)
    for _ in range(2):
        pb.out.fill_(0)
        pb.lse.fill_(0)
        B.pkv_decode_no_alloc(pb.args, step.err)
        torch.cuda.synchronize()
        assert step.check_errors() == 0
        _close(pb.out, ref_out)
        _close(pb.lse, ref_lse)
        got = pb.out.float().cpu().double().numpy()[sample]
        assert (np.abs(got - oracle_out) <= ATOL + RTOL * np.abs(oracle_out)).all(), \
            float(np.abs(got - oracle_out).max())

    # a plan that needs more scratch than the built-in array is refused up front
    big = DecodeStep(make_workload("llama3_8b", batch=64), kv_chunk=64)
    with pytest.raises(B.PkvError) as e:
        B.pkv_decode_no_alloc(big.problems["self"].args, big.err)
    assert e.value.status == B.PKV_ERR_CAPACITY
