"""The bounded-wait give-up path of the pipelined kernels, exercised on the GPU.

Every mbarrier wait inside the TMA/tcgen05 kernels is bounded (pkv_set_wait_limit).
With a limit of one nanosecond the first wait that is not already satisfied gives
up: the CTA raises PKV_DEVERR_TIMEOUT, stops waiting, lets the copies it issued
land and returns.  The test checks that such a launch ends (the synchronize
returns), that the flag is raised, and that the next launch with the default limit
on the same stream is again correct against the fp64 oracle.  Nothing here faults,
traps or hangs: the failure is a wait that runs out of time by design.
"""
import numpy as np
import pytest
import torch

from _harness import assert_close, bf16_to_f64, oracle_decode_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    yield _binding
    _binding.pkv_set_wait_limit(0)


def _give_up_then_recover(B, step, name, sample):
    pb = step.problems[name]
    step.build_indices(name)
    if pb.spec.stores:
        step.store(name)
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    B.pkv_set_wait_limit(1)
    try:
        step.decode(name)
        torch.cuda.synchronize()          # the abandoned launch ends
    finally:
        B.pkv_set_wait_limit(0)
    assert B.pkv_wait_limit() == 2_000_000_000
    assert step.check_errors() & B.PKV_DEVERR_TIMEOUT
    step.err.zero_()
    pb.out.fill_(0)
    step.decode(name)                     # default limit, same stream
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    ref, _ = oracle_decode_problem(step, name, sample)
    assert_close(bf16_to_f64(pb.out)[sample], ref, "decode after a timed-out launch")


@pytest.mark.parametrize("kv_chunk", [256, 0])
def test_gqa_tma_decode_gives_up_and_the_next_call_is_correct(B, kv_chunk):
    """decode_tma_kernel (page_size 16, GQA groups of 2 on the tensor-core path), with
    the work cut into pieces of 256 keys and into equal spans (the library's choice
    at this batch): the span merge reads only records the split kernel writes before
    its first wait."""
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    step = DecodeStep(make_workload("qwen3_0p6b", batch=16), kv_chunk=kv_chunk)
    _give_up_then_recover(B, step, "self", list(range(0, 16, 3)))


def test_mla_decode_gives_up_and_the_next_call_is_correct(B):
    """mla_decode_kernel: a 2-CTA cluster that swaps partial scores; a CTA that gives up
    stops sending, its peer's waits run out too, and both let what was sent land
    before releasing shared memory."""
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    step = DecodeStep(make_workload("deepseek_v3_mla", batch=6), kv_chunk=1024)
    _give_up_then_recover(B, step, "self", [0, 2, 5])


def test_extend_gives_up_and_the_next_call_is_correct(B):
    """ext_kernel (tcgen05, the item queue between warps, a global work counter)."""
    from test_gpu_extend_full import _check
    from paged_kv_cache_req_gb300.engine import ExtendStep
    from paged_kv_cache_req_gb300.workloads import make_extend_workload
    ew = make_extend_workload("qwen3_0p6b_prefill", batch=3)
    step = ExtendStep(ew, device="cuda")
    step.build_indices()
    step.store()
    step.plan()
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    B.pkv_set_wait_limit(1)
    try:
        step.attend()
        torch.cuda.synchronize()          # the abandoned launch ends
    finally:
        B.pkv_set_wait_limit(0)
    assert step.check_errors() & B.PKV_DEVERR_TIMEOUT
    step.err.zero_()
    step.out.fill_(0)
    step.attend()                         # default limit, same stream
    torch.cuda.synchronize()
    assert step.check_errors() == 0
    _check(step, [0, 2], lambda b, n: sorted(set([0, 1, n // 2, n - 1])))
