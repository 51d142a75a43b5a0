"""Seeded random configurations against the fp64 oracle.

The parity tests pin the benchmark recipes and chosen edge cases; these draw the
remaining knobs at random (batch, lengths including 0 and 1, page size, head
grouping, head_dim, split size, layout, explicit key bounds) so that combinations
nobody picked by hand are exercised too.  Each case is small enough for the oracle
to finish in well under a second; the seeds are fixed, so a failure reproduces.
"""
import numpy as np
import pytest

import oracle
from _harness import assert_close
from test_gpu_extend import _case, _run
from test_gpu_parity import _direct_decode, _direct_mla

pytestmark = pytest.mark.gpu

GQA_SHAPES = [(8, 8, 64), (20, 20, 64), (16, 8, 128), (32, 8, 128), (16, 2, 128), (32, 2, 64), (16, 4, 64),
              (64, 4, 128), (8, 1, 128), (4, 2, 64)]
PAGE_SIZES = [1, 2, 4, 8, 16, 32, 64, 128, 256]


@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_req_gb300 import build
    build.build()
    from paged_kv_cache_req_gb300 import _binding
    return _binding


def _lengths(rng, n, hi):
    lens = rng.integers(0, hi, size=n)
    lens[rng.random(n) < 0.15] = 0
    lens[rng.random(n) < 0.15] = 1
    if lens.max() == 0:
        lens[0] = 1
    return [int(x) for x in lens]


@pytest.mark.parametrize("seed", range(12))
def test_gqa_decode_random_configs(B, seed):
    rng = np.random.default_rng(1000 + seed)
    hq, hkv, d = GQA_SHAPES[seed % len(GQA_SHAPES)]
    ps = int(rng.choice(PAGE_SIZES))
    lens = _lengths(rng, int(rng.integers(1, 9)), int(rng.choice([70, 700, 3000])))
    chunk = int(rng.choice([0, 64, 128, 192, 512]))
    layout = "block_table" if rng.random() < 0.3 else None
    gpu, g_lse, ref, ref_lse = _direct_decode(B, lens, ps, hq, hkv, d, chunk=chunk, layout=layout, seed=seed)
    what = "seed %d: hq %d hkv %d d %d ps %d chunk %d %s lens %s" % (seed, hq, hkv, d, ps, chunk, layout, lens)
    assert_close(gpu, ref, what)
    live = [b for b, L in enumerate(lens) if L > 0]
    assert_close(g_lse[live], ref_lse[live], what + " (lse)")
    for b, L in enumerate(lens):
        if L == 0:
            assert (gpu[b] == 0).all() and np.isneginf(g_lse[b]).all(), what


@pytest.mark.parametrize("seed", range(6))
def test_mla_decode_random_configs(B, seed):
    rng = np.random.default_rng(2000 + seed)
    ps = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256]))
    lens = _lengths(rng, int(rng.integers(1, 6)), int(rng.choice([100, 1500, 3000])))
    chunk = int(rng.choice([0, 64, 128, 320]))
    layout = "csr" if rng.random() < 0.5 else "block_table"
    hq = 256 if seed % 3 == 2 else 128
    gpu, g_lse, ref, ref_lse = _direct_mla(B, lens, ps, hq=hq, chunk=chunk, layout=layout, seed=seed)
    what = "seed %d: ps %d chunk %d %s hq %d lens %s" % (seed, ps, chunk, layout, hq, lens)
    assert_close(gpu, ref, what)
    live = [b for b, L in enumerate(lens) if L > 0]
    assert_close(g_lse[live], ref_lse[live], what + " (lse)")


@pytest.mark.parametrize("seed", range(12))
def test_extend_random_configs(B, seed):
    rng = np.random.default_rng(3000 + seed)
    hq, hkv, d = [(32, 8, 128), (16, 16, 128), (8, 1, 64), (32, 4, 128), (16, 2, 64), (16, 1, 64)][seed % 6]
    ps = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256]))
    nb = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(1, 1200, size=nb)]
    nq = [int(rng.integers(1, min(L, 128) + 1)) for L in lens]
    chunk = int(rng.choice([0, 64, 192, 512]))
    layout = "csr" if rng.random() < 0.6 else "block_table"
    kv_end = None
    if seed % 3 == 1:   # explicit key bounds, zeros and full rows included
        kv_end = np.concatenate([rng.integers(0, L + 1, size=n) for L, n in zip(lens, nq)]).astype(np.int32)
    case = _case(4000 + seed, lens, nq, hq, hkv, d, ps)
    e, gpu, g_lse, st, ref, ref_lse = _run(B, *case, lens, ps, kv_end=kv_end, chunk=chunk, layout=layout)
    what = "seed %d: hq %d hkv %d d %d ps %d chunk %d %s lens %s nq %s bounds %s" % (
        seed, hq, hkv, d, ps, chunk, layout, lens, nq, "explicit" if kv_end is not None else "causal")
    assert e == 0 and st == oracle.OK, what
    assert_close(gpu, ref, what)
    finite = np.isfinite(ref_lse)
    assert_close(np.where(finite, g_lse, 0), np.where(finite, ref_lse, 0), what + " (lse)")
    assert np.isneginf(g_lse[~finite]).all(), what
