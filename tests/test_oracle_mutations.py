"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a copy of the oracle's C source (on the
CPU, in a temporary directory), compiles it, and runs the pin suite against
the broken library.  The suite must fail for every one of them: a dropped
term, a wrong sign or index, a swapped operand or stride, a missing offset.
The committed oracle itself is never modified.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

# (name, text in the source, replacement, how many occurrences to replace; 0 = all).
# A deleted statement is replaced by ";" so that the surrounding code keeps its shape.
MUTANTS = [
    ("interleaved_kv_head", "const int64_t b = bh / hq, h = bh % hq, kh = h / g;",
     "const int64_t b = bh / hq, h = bh % hq, kh = h % hkv;", 1),
    ("dropped_scale", "x[t - t0] = scale * acc;", "x[t - t0] = acc;", 1),
    ("shared_query_row", "q + bh * dqk", "q + b * dqk", 1),
    ("v_offset_uses_dqk", "v_pool + slot * v_row_stride + kh * dv", "v_pool + slot * v_row_stride + kh * dqk", 0),
    ("decode_ignores_kv_start", "for (int64_t t = t0; t < t1; ++t) {\n            const int64_t slot = r2t[row * row_stride + start + t];",
     "for (int64_t t = t0; t < t1; ++t) {\n            const int64_t slot = r2t[row * row_stride + t];", 1),
    ("lse_without_max", "if (lse) lse[bh] = m + log(den);", "if (lse) lse[bh] = log(den);", 1),
    ("empty_lse_zero", "if (lse) lse[bh] = -INFINITY;", "if (lse) lse[bh] = 0.0;", 1),
    ("merge_sign", "const double w = exp(l - m);", "const double w = exp(m - l);", 1),
    ("merge_unnormalised", "for (int32_t d = 0; d < dv; ++d) o[d] /= wsum;", ";", 1),
    ("indices_ignore_kv_start", "const int64_t col = start + p * page_size;", "const int64_t col = p * page_size;", 1),
    ("last_page_len_mod", "(int32_t)(len - (npages - 1) * page_size)", "(int32_t)(len % page_size)", 1),
    ("no_alignment_check", "if (first % page_size != 0) return PKVO_ERR_CONTIG;", ";", 1),
    ("no_contiguity_check", "if (r2t[row * row_stride + col + j] != first + j) return PKVO_ERR_CONTIG;", ";", 1),
    ("block_table_pad_zero", "block_table[(int64_t)b * bt_width + p] = -1;", "block_table[(int64_t)b * bt_width + p] = 0;", 1),
    ("indptr_not_cumulative", "if (kv_indptr) kv_indptr[b + 1] = (int32_t)running;",
     "if (kv_indptr) kv_indptr[b + 1] = (int32_t)npages;", 1),
    ("store_indexes_source_by_slot", "rows + (int64_t)i * src_row_stride_bytes", "rows + slot * src_row_stride_bytes", 1),
    ("store_ignores_padding", "if (slot < 0) continue;", ";", 1),
    ("cu_seqlens_not_cumulative", "cu_seqlens[b + 1] = (int32_t)running;", "cu_seqlens[b + 1] = (int32_t)len;", 1),
    ("alloc_partial_page_off_by_one", "if (t < aligned) slot = last_loc[b] + (t - p + 1);",
     "if (t < aligned) slot = last_loc[b] + (t - p);", 1),
    ("alloc_no_partial_page", "const int64_t aligned = (p + ps - 1) / ps * ps;", "const int64_t aligned = p;", 1),
    ("alloc_pages_not_advanced", "        pg += (s + ps - 1) / ps - (p + ps - 1) / ps;", "        pg += 0;", 1),
    ("alloc_state_not_updated", "free_state[0] = (int32_t)(head + pages);", "free_state[0] = (int32_t)head;", 1),
    ("alloc_no_capacity_check", "if (toks > out_cap || pages > count ||", "if (toks > out_cap ||", 1),
    ("write_skips_prefix", "for (int64_t t = 0; t < p; ++t) r[t] = prefix_slots[b][t];", ";", 1),
    ("write_new_slots_not_offset", "for (int64_t t = p; t < s; ++t) r[t] = out_cache_loc[e + (t - p)];",
     "for (int64_t t = p; t < s; ++t) r[t] = out_cache_loc[t - p];", 1),
    ("merge_ignores_block_ids", "buffer + (blk * block_size + j) * row_bytes", "buffer + (i * block_size + j) * row_bytes", 1),
    ("extend_bound_off_by_one", "        for (int64_t t = 0; t < te; ++t) {\n            const int64_t slot = r2t[row * row_stride + start + t];\n            if (slot < 0 || slot >= num_slots) { bad = 1; break; }",
     "        for (int64_t t = 0; t < te - (te > 1); ++t) {\n            const int64_t slot = r2t[row * row_stride + start + t];\n            if (slot < 0 || slot >= num_slots) { bad = 1; break; }", 1),
    ("extend_head_mapping", "const int64_t j = jh / hq, h = jh % hq, kh = h / g;", "const int64_t j = jh / hq, h = jh % hq, kh = h % hkv;", 1),
    ("span_causal_bound", "kv_end[j] = (int32_t)(seg_kind[s] == 0 ? p + 1 : e);", "kv_end[j] = (int32_t)(seg_kind[s] == 0 ? p : e);", 1),
    ("span_full_bound", "kv_end[j] = (int32_t)(seg_kind[s] == 0 ? p + 1 : e);", "kv_end[j] = (int32_t)(seg_kind[s] == 0 ? p + 1 : p + 1);", 1),
    ("gather_ignores_kv_start",
     "const int64_t slot = r2t[row * row_stride + start + t];\n            if (slot < 0 || slot >= num_slots) return",
     "const int64_t slot = r2t[row * row_stride + t];\n            if (slot < 0 || slot >= num_slots) return", 1),
]


def _mutate(src: str, old: str, new: str, count: int) -> str:
    n = src.count(old)
    assert n >= 1, "mutation anchor not found: %r" % old
    if count:
        assert n == count, "mutation anchor %r occurs %d times" % (old, n)
    return src.replace(old, new)


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, count):
    with open(SRC) as f:
        src = f.read()
    mutated = _mutate(src, old, new, count)
    c = tmp_path / ("mutant_%s.c" % name)
    c.write_text(mutated)
    lib = tmp_path / ("libmutant_%s.so" % name)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(c), "-lm"])
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, "pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
