"""Whole steps captured in a CUDA graph.

A serving loop captures its decode step once and replays it.  Every libpkv call is
asynchronous, allocates nothing and launches its kernels as programmatic dependents of
the previous kernel, so a captured step must replay with the same results as eager
launches.  The kernels are deterministic (no atomics feed the arithmetic), so the
replayed outputs are compared bit for bit with an eager run of the same step, and the
eager run itself is checked against the fp64 oracle by the parity tests.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _replay_matches_eager(run, outputs, err):
    """Run eagerly, capture, zero the outputs, replay twice; compare the bits."""
    run()                                   # first calls set kernel attributes outside the capture
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = [t.clone() for t in outputs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for t in outputs:
        t.zero_()
    torch.cuda.synchronize()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error flags 0x%x after replay" % int(err.item())
    for r, t in zip(ref, outputs):
        assert torch.equal(r.view(torch.uint8) if r.dtype == torch.bfloat16 else r,
                           t.view(torch.uint8) if t.dtype == torch.bfloat16 else t)


@pytest.mark.parametrize("name,kw", [
    ("tiny_gqa", {}),
    ("qwen3_0p6b", {"batch": 8}),
    ("llama3_8b", {"batch": 16, "alloc": True}),
    ("whisper_encdec", {"batch": 8, "cross_mode": "gather"}),
    ("deepseek_v3_mla", {"batch": 8}),
])
def test_decode_step_graph_replay_matches_eager(B, name, kw):
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    step = DecodeStep(make_workload(name, batch=kw.get("batch")),
                      **{k: v for k, v in kw.items() if k != "batch"})
    outs = []
    for pb in step.problems.values():
        outs += [pb.out, pb.lse]
    _replay_matches_eager(step.run, outs, step.err)


@pytest.mark.parametrize("name,batch", [("llama3_8b_verify", 8), ("qwen3_0p6b_prefill", 2), ("hunyuan_image_spans", 1)])
def test_extend_step_graph_replay_matches_eager(B, name, batch):
    from paged_kv_cache_req_gb300.engine import ExtendStep
    from paged_kv_cache_req_gb300.workloads import make_extend_workload
    step = ExtendStep(make_extend_workload(name, batch=batch))
    _replay_matches_eager(step.run, [step.out, step.lse], step.err)
