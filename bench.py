"""Benchmark: paged decode attention over a paged KV cache on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one decode layer step of the whole hot path over one batch of the
workload: pkv_build_indices (req_to_token -> page lists), pkv_store (one new
K/V row per request), pkv_decode (split-KV attention + log-sum-exp merge); the
encoder-decoder workload adds its cross-attention (page-aligned, or
pkv_ragged_gather + varlen decode with --cross-mode gather).

Prints ONE JSON line.  ``value`` is the step's algorithmic bytes (unique KV
bytes read, q/out, page-table reads, stored rows; a shared prefix page counts
once) per second of device time, with every input resident in HBM;
``decode_steps_per_s`` the matching step rate.  ``roofline`` reports the decode
launch (split kernel + merge) against the measured HBM copy bandwidth,
``e2e`` the same metric through the host-buffer API (pinned h2d of the step
inputs and d2h of the outputs inside the timed region), ``cpu_baseline`` the
fp64 CPU oracle timed on a bounded sample of the same workload on this host.

With N > 1 (torchrun), every rank runs its own replica of the workload on its
own GPU: requests are independent, so the work shards with no collective on
the data path (weak scaling); the barrier and max-over-ranks timing use
torch.distributed only for timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read GB/s (frac of HBM peak) and decode steps/s"
DEFAULT_WORKLOAD = "llama3_8b"
L2_BYTES = 129 * 10**6
WORKLOAD_TEXT = {
    "tiny_gqa": "tiny GQA decode: 4 requests, cached lengths {17,64,100,255}, 16 q / 8 kv heads x 128, page_size 1",
    "qwen3_0p6b": "Qwen3-0.6B-shaped decode: batch 32, cached lengths U[1,4096], 16 q / 8 kv heads x 128, page_size 16, 200k-token pool",
    "llama3_8b": "Llama-3-8B-shaped large-batch decode: batch 256, cached lengths log-U[128,32768], 32 q / 8 kv heads x 128, page_size 64, groups of 16 share a 2048-token prefix",
    "whisper_encdec": "Whisper-large-shaped encoder-decoder step: batch 64, decoder lengths U[1,448] + cross-attention over 1500 encoder tokens, 20 heads x 64, page_size 16",
    "deepseek_v3_mla": "DeepSeek-V3-shaped MLA decode: batch 128, cached lengths U[512,16384], 128 q heads over a 512+64 latent, page_size 64",
    "encoder_merge": "Qwen3-VL-32B-shaped encoder-cache read path: 30 cached 512x512 images (256 tokens each, one 512-row block each) of fat_dim 20480 bf16 gathered into an 8672-row prefill sequence",
}
MERGE_METRIC = "encoder-cache merge GB/s (bytes read + written)"
WORKLOAD_TEXT.update({
    "llama3_8b_verify": "Llama-3-8B-shaped speculative target-verify: batch 128, cached lengths log-U[128,32768] + 4 draft tokens per request (causal), 32 q / 8 kv heads x 128, page_size 64",
    "qwen3_0p6b_prefill": "Qwen3-0.6B-shaped chunked prefill: 8 requests, cached prefix U[0,4096] + a 1024-token chunk each (causal), 16 q / 8 kv heads x 128, page_size 16",
    "hunyuan_image_spans": "HunyuanImage-shaped first denoising step: 4 rows (2 requests x 2 CFG branches) of a 1024-token causal text segment + a 4096-token full image segment, all 5120 positions queried, 32 q / 8 kv heads x 128, page_size 64",
})
EXTEND_WORKLOADS = ("llama3_8b_verify", "qwen3_0p6b_prefill", "hunyuan_image_spans")
EXTEND_METRIC = {"llama3_8b_verify": ("paged multi-query attention KV-read GB/s (target-verify)", "GB/s", "hbm"),
                 "qwen3_0p6b_prefill": ("paged multi-query attention TFLOP/s (chunked prefill)", "TFLOP/s", "tensor"),
                 "hunyuan_image_spans": ("paged multi-query attention TFLOP/s (causal + full spans)", "TFLOP/s", "tensor")}


# ---------------------------------------------------------------- accounting
def step_bytes(wl, cross_mode="paged", alloc=False, fused=False):
    """Algorithmic bytes of one step and of its decode launches (unique slots once).
    With device allocation: per request its lengths and last slot read, one slot
    written to the output and one to its row, and the free-list pages taken.
    Fused (the decode reads the page starts from req_to_token and stores the new
    rows itself): no full-row table read and no page-list write."""
    r2t = wl.req_to_token.numpy()
    rpi = wl.req_pool_idx.numpy().astype(np.int64)
    if wl.kind == "mla":
        kv_row = wl.head_dim_qk * 2                     # one latent row serves K and V
        store_row = kv_row
    else:
        kv_row = 2 * wl.num_kv_heads * wl.head_dim_qk * 2
        store_row = kv_row
    total = 0
    decode = 0
    for p in wl.problems:
        lens = p.seq_lens.numpy().astype(np.int64)
        starts = p.kv_start.numpy().astype(np.int64)
        slots = np.concatenate([r2t[rpi[b], starts[b]:starts[b] + lens[b]] for b in range(wl.batch)]) \
            if wl.batch else np.zeros(0, np.int64)
        uniq = np.unique(slots).size
        q_out = wl.batch * wl.num_q_heads * (wl.head_dim_qk + wl.head_dim_v) * 2
        pages = int((-(-lens // wl.page_size)).sum())
        dec = uniq * kv_row + q_out + pages * 4
        decode += dec
        if p.name == "cross" and cross_mode == "gather":
            total += dec + 2 * int(lens.sum()) * kv_row + int(lens.sum()) * 4
        elif fused:
            total += dec                                        # page starts: the 4 B per page in dec
        else:
            total += dec + int(lens.sum()) * 4 + pages * 4        # table read + page-list write
        if p.stores:
            total += 2 * wl.batch * store_row                   # read new rows + write pool rows
            if alloc:
                new_pages = int((lens % wl.page_size == 1).sum()) if wl.page_size > 1 else wl.batch
                total += wl.batch * (3 * 4 + 4 + 4) + new_pages * 4
    return total, decode


def unique_keys(wl):
    r2t = wl.req_to_token.numpy()
    rpi = wl.req_pool_idx.numpy().astype(np.int64)
    out = {}
    for p in wl.problems:
        lens = p.seq_lens.numpy().astype(np.int64)
        starts = p.kv_start.numpy().astype(np.int64)
        slots = np.concatenate([r2t[rpi[b], starts[b]:starts[b] + lens[b]] for b in range(wl.batch)])
        out[p.name] = (int(lens.sum()), int(np.unique(slots).size))
    return out


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1961.1)), float(d.get("bf16_tflops_sustained", 1733.8)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def decode_traffic(workload):
    """Per-launch DRAM bytes of the workload's dominant kernel from a committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get("workloads", {}).get(workload)
    if not ent:
        return None
    src = os.path.join(ROOT, "paged_kv_cache_req_gb300", "csrc", ent.get("source", d.get("source", "decode_gqa.cu")))
    if ent.get("source_sha") != hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]:
        return None
    return ent.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.proc = None
        self.gpu = gpu_index
        self.start_count = 0
        if not enabled:
            return
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.count() == 0:   # sampler is live before timing starts
            time.sleep(0.02)
        self.start_count = self.count()

    def count(self):
        try:
            with open(self.tmp.name) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for i, line in enumerate(f):
                if i < self.start_count:
                    continue
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


# ---------------------------------------------------------------- CPU oracle leg
def oracle_sample_run(wl, budget_key_heads, seed=0, num_threads=0, fetch_rows=None):
    """Times the fp64 oracle (store + decode) on a sample of the workload's requests.

    The sampled requests keep the recipe's lengths and page layout; their slots
    are relabelled into a compact host pool.  ``fetch_rows(slots)`` returns the
    pool rows of those slots as bf16 bit patterns (K, V); without it the values
    are drawn on the CPU from the same N(0,1) recipe.
    Returns (seconds, algorithmic bytes of the sample, description, threads).
    """
    import oracle
    rng = np.random.default_rng(seed)
    order = rng.permutation(wl.batch)
    r2t = wl.req_to_token.numpy()
    rpi = wl.req_pool_idx.numpy().astype(np.int64)
    per_req = np.zeros(wl.batch, dtype=np.int64)
    for p in wl.problems:
        per_req += p.seq_lens.numpy().astype(np.int64) * wl.num_q_heads
    sample, acc = [], 0
    for b in order:
        sample.append(int(b))
        acc += int(per_req[b])
        if acc >= budget_key_heads:
            break
    sample.sort()
    gen = torch.Generator().manual_seed(7 + seed)
    secs = 0.0
    nbytes = 0
    kv_row = (wl.head_dim_qk * 2) if wl.kind == "mla" else 2 * wl.num_kv_heads * wl.head_dim_qk * 2
    for p in wl.problems:
        lens = p.seq_lens.numpy().astype(np.int64)[sample]
        starts = p.kv_start.numpy().astype(np.int64)[sample]
        rows = [r2t[rpi[b], s:s + L].astype(np.int64) for b, s, L in zip(sample, starts, lens)]
        allslots = np.unique(np.concatenate(rows))
        table = np.zeros((len(sample) + 1, max(int(lens.max()), 1)), dtype=np.int32)
        for i, r in enumerate(rows):
            table[i + 1, :len(r)] = np.searchsorted(allslots, r)
        shape = (len(allslots), wl.head_dim_qk) if wl.kind == "mla" else (len(allslots), wl.num_kv_heads, wl.head_dim_qk)
        if fetch_rows is not None:
            k, v = fetch_rows(allslots)
            if v is None:
                v = k
        else:
            nrng = np.random.default_rng(11 + seed)

            def draw():
                x = nrng.standard_normal(size=shape, dtype=np.float32)
                return (x.view(np.uint32) >> 16).astype(np.uint16)
            k = draw()
            v = k if wl.kind == "mla" else draw()
        q = torch.randn((len(sample), wl.num_q_heads, wl.head_dim_qk), generator=gen).to(torch.bfloat16) \
            .view(torch.int16).numpy().view(np.uint16)
        rpi_c = np.arange(1, len(sample) + 1, dtype=np.int32)
        t0 = time.perf_counter()
        if p.stores:
            new_rows = k[:len(sample)].copy()
            oracle.store(k, new_rows, np.searchsorted(allslots, [r[-1] for r in rows]).astype(np.int32))
        st, out, lse = oracle.decode(q, k, v, table, rpi_c, lens, wl.sm_scale,
                                     head_dim_v=wl.head_dim_v if wl.kind == "mla" else None,
                                     num_threads=num_threads)
        secs += time.perf_counter() - t0
        nbytes += len(allslots) * kv_row + len(sample) * wl.num_q_heads * (wl.head_dim_qk + wl.head_dim_v) * 2
    desc = "%d of %d requests (%d key x q-head pairs), compact host pool" % (len(sample), wl.batch, int(per_req[sample].sum()))
    if len(sample) == wl.batch:
        desc = "whole step: all %d requests (%d key x q-head pairs), compact host pool" % (wl.batch, int(per_req.sum()))
    return secs, nbytes, desc, oracle.max_threads() if num_threads <= 0 else num_threads


# ---------------------------------------------------------------- multi-process plumbing
def reduce_max(x, dist=None, device="cpu"):
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_gbs(world, bytes_per_step, steps, max_ms):
    """Whole-job GB/s: every rank processed its own replica of the step in max_ms (slowest rank)."""
    return world * bytes_per_step * steps / (max_ms / 1e3) / 1e9


# ---------------------------------------------------------------- configs (shared by both arms)
def parallelism(world):
    return "replicas" if world > 1 else "single GPU"


def l2_note(nbytes):
    return "flushed between steps (2x L2 write)" if nbytes < 4 * L2_BYTES else "inputs larger than L2"


def decode_config(wl, cross_mode, alloc, world, fused=False):
    """The `config` object of a decode line: the same dict in both arms."""
    keys = unique_keys(wl)
    total_bytes, _ = step_bytes(wl, cross_mode, alloc=alloc, fused=fused)
    return {"workload": WORKLOAD_TEXT[wl.name], "name": wl.name, "batch": wl.batch,
            "cross_mode": cross_mode if wl.kind == "gqa" and len(wl.problems) > 1 else None,
            "page_table": "req_to_token read by pkv_decode, new rows stored by it (fused)" if fused
            else "pkv_build_indices page lists, then pkv_store and pkv_decode",
            "new_slots": "allocated on the device each step (pkv_alloc_extend + pkv_write_req_to_token)"
            if alloc else "given by the workload",
            "keys_per_step": {k: v[0] for k, v in keys.items()},
            "unique_keys_per_step": {k: v[1] for k, v in keys.items()},
            "algorithmic_bytes_per_step": total_bytes,
            "l2": l2_note(total_bytes), "parallelism": parallelism(world)}


def extend_config(ew, world, token_table=False):
    flops, step_bytes_, _ = extend_amounts(ew)
    return {"workload": WORKLOAD_TEXT[ew.name], "name": ew.name, "batch": ew.batch,
            "query_rows": int(ew.qo_lens.sum()), "keys": int(ew.seq_lens.sum()),
            "pages": "read from req_to_token (no pkv_build_indices)" if token_table else "kv_indptr / kv_indices",
            "attention_flops_per_step": flops, "algorithmic_bytes_per_step": step_bytes_,
            "l2": l2_note(step_bytes_), "parallelism": parallelism(world)}


def merge_config(mw, world):
    nbytes = merge_bytes(mw)
    return {"workload": WORKLOAD_TEXT["encoder_merge"], "name": "encoder_merge", "items": mw.items,
            "rows_moved": mw.rows_moved, "row_bytes": mw.row_bytes, "num_blocks": mw.num_blocks,
            "num_tokens": mw.num_tokens, "algorithmic_bytes_per_step": nbytes,
            "l2": l2_note(nbytes), "parallelism": parallelism(world)}


def finish_clocks(clocks, opts, soak_step):
    """Stops the sampler; a region shorter than a few samples is extended, untimed, by the same load."""
    soak = 0
    if clocks.proc is not None and not opts.profile_run and clocks.count() - clocks.start_count < 5:
        t_soak = time.perf_counter()
        while clocks.count() - clocks.start_count < 5 and time.perf_counter() - t_soak < 3.0:
            for _ in range(max(1, opts.steps)):
                soak_step()
                soak += 1
            torch.cuda.synchronize()
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = "timed region" + (" + %d untimed steps of the same load" % soak if soak else "")
    return clk


def with_cycles(clk, ms_per_step):
    """Adds the step's length in SM cycles at the sampled median clock (time x MHz)."""
    if clk is not None and clk.get("sm_mhz"):
        clk["sm_cycles_per_step"] = int(round(ms_per_step * 1e3 * clk["sm_mhz"]))
    return clk


# ---------------------------------------------------------------- encoder-cache merge
def merge_oracle_pass(mw, buf_bits, hidden_bits):
    """One oracle merge of the whole step on host copies; returns (seconds, rows)."""
    import oracle
    t0 = time.perf_counter()
    st, filled = oracle.encoder_merge(buf_bits, mw.block_ids, mw.positions, hidden_bits)
    secs = time.perf_counter() - t0
    if st != oracle.OK or filled != mw.rows_moved:
        raise SystemExit("oracle merge failed: status %d, %d rows" % (st, filled))
    return secs, filled


def merge_bytes(mw):
    return mw.rows_moved * mw.row_bytes * 2 + mw.positions.nbytes + mw.block_ids.nbytes


def reference_merge(args, world):
    from paged_kv_cache_req_gb300.workloads import fill_merge_buffers, make_encoder_merge
    import oracle
    oracle.build()
    mw = make_encoder_merge(seed=args.seed)
    buf, hidden = fill_merge_buffers(mw)
    bb = buf.view(torch.int16).numpy().view(np.uint16)
    hb = hidden.view(torch.int16).numpy().view(np.uint16)
    for _ in range(args.warmup):
        merge_oracle_pass(mw, bb, hb)
    times = [merge_oracle_pass(mw, bb, hb)[0] for _ in range(args.steps)]
    value = merge_bytes(mw) * len(times) / sum(times) / 1e9
    desc = "whole step: %d rows of %d B gathered by the byte-copy oracle on 1 host thread" % (
        mw.rows_moved, mw.row_bytes)
    return {"impl": "reference", "metric": MERGE_METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": merge_config(mw, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def measure_merge(opts, world, rank, local, dist):
    """One step = one pkv_encoder_merge of the whole prefill's cached images."""
    from paged_kv_cache_req_gb300 import _binding as B
    from paged_kv_cache_req_gb300.workloads import fill_merge_buffers, make_encoder_merge
    mw = make_encoder_merge(seed=opts.seed)
    dev = torch.device("cuda", local)
    buf, hidden = fill_merge_buffers(mw, device=dev)
    bid = torch.from_numpy(mw.block_ids).to(dev)
    pos = torch.from_numpy(mw.positions).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    filled = torch.zeros(1, dtype=torch.int64, device=dev)
    nbytes = merge_bytes(mw)
    flush = nbytes < 4 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    stream = torch.cuda.current_stream()

    def step():
        B.pkv_encoder_merge(buf, bid, pos, hidden, err, filled=filled)

    for _ in range(opts.warmup):
        step()
    torch.cuda.synchronize()
    if err.item() or filled.item() != opts.warmup * mw.rows_moved:
        raise SystemExit("merge check failed: err %d, filled %d" % (err.item(), filled.item()))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, enabled=not opts.profile_run)
    wall0 = time.perf_counter()
    for i in range(opts.steps):
        if flush:
            flush_buf.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = finish_clocks(clocks, opts, step)
    tot_ms = reduce_max(sum(a.elapsed_time(b) for a, b in ev), dist, "cuda")
    value = weak_scaling_gbs(world, nbytes, opts.steps, tot_ms)
    if opts.profile_run:
        if rank == 0:
            print(json.dumps({"profile_run": True, "workload": "encoder_merge", "ms_per_step": round(tot_ms / opts.steps, 4)}))
        return None
    # end to end: the step's index inputs from pinned host memory, the filled count back
    h_bid, h_pos = torch.from_numpy(mw.block_ids).pin_memory(), torch.from_numpy(mw.positions).pin_memory()
    h_filled = torch.zeros(1, dtype=torch.int64).pin_memory()
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    for i in range(opts.steps):
        if flush:
            flush_buf.zero_()
        e_ev[i][0].record(stream)
        bid.copy_(h_bid, non_blocking=True)
        pos.copy_(h_pos, non_blocking=True)
        filled.zero_()
        step()
        h_filled.copy_(filled, non_blocking=True)
        e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    if int(h_filled.item()) != mw.rows_moved or err.item():
        raise SystemExit("merge check failed in the end-to-end pass")
    e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e_ev), dist, "cuda")
    if rank != 0:
        return None
    hbm, _, _, peak_kind = measured_peaks()
    avg_ms = tot_ms / opts.steps
    achieved = nbytes / (avg_ms / 1e3) / 1e9
    cpu = None
    if world == 1 and not opts.no_cpu_baseline:
        import oracle
        oracle.build()
        bb = buf.cpu().view(torch.int16).numpy().view(np.uint16)
        hb = hidden.cpu().view(torch.int16).numpy().view(np.uint16)
        tot_s, passes = 0.0, 0
        while passes < 20 and (tot_s < 3.0 or passes == 0):
            tot_s += merge_oracle_pass(mw, bb, hb)[0]
            passes += 1
        cpu = {"value": round(nbytes * passes / tot_s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "whole step (%d rows of %d B); %d pass(es), %.1f s on 1 host thread" % (
                   mw.rows_moved, mw.row_bytes, passes, tot_s), "host_cpus": os.cpu_count()}
    return {
        "metric": MERGE_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": opts.steps,
        "warmup": opts.warmup, "ms_per_step": round(avg_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": merge_config(mw, world),
        "roofline": {"bound": "hbm", "kernel": "pkv_encoder_merge", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": round(avg_ms, 4),
                     "traffic": decode_traffic("encoder_merge")},
        "cpu_baseline": cpu,
        "e2e": {"value": round(weak_scaling_gbs(world, nbytes, opts.steps, e_ms), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(mw.block_ids.nbytes + mw.positions.nbytes), "d2h_bytes_per_step": 8,
                "ms_per_step": round(e_ms / opts.steps, 4)},
        "gpu_launches": opts.steps,
        "clocks": with_cycles(clk, avg_ms),
        "wall_s_timed_region": round(wall, 3),
    }


# ---------------------------------------------------------------- multi-query steps
def extend_rows(ew):
    """Per request: its query rows' key bounds (numpy int64)."""
    import oracle
    lens = ew.seq_lens.numpy().astype(np.int64)
    qo = ew.qo_lens.numpy().astype(np.int64)
    if ew.segments is not None:
        st, _, _, kend = oracle.span_plan(ew.segments)
        assert st == oracle.OK
        ind = np.concatenate([[0], np.cumsum(qo)])
        return [kend[ind[b]:ind[b + 1]].astype(np.int64) for b in range(ew.batch)]
    return [np.arange(L - n, L) + 1 for L, n in zip(lens, qo)]


def extend_amounts(ew):
    """(attention flops of the step, algorithmic bytes of the step, bytes of the extend launch)."""
    kv_row = 2 * ew.num_kv_heads * ew.head_dim * 2
    rows = extend_rows(ew)
    flops = sum(4.0 * ew.num_q_heads * ew.head_dim * float(r.sum()) for r in rows)
    lens = ew.seq_lens.numpy().astype(np.int64)
    keys = int(sum(int(r.max()) if len(r) else 0 for r in rows))       # keys a block of the request reads
    total_q = int(ew.qo_lens.sum())
    pages = int((-(-lens // ew.page_size)).sum())
    launch = keys * kv_row + total_q * ew.num_q_heads * ew.head_dim * 2 * 2 + pages * 4
    step = launch + int(lens.sum()) * 4 + pages * 4 + 2 * int(ew.new_lens.sum()) * kv_row   # + table, page list, store
    return flops, step, launch


def extend_oracle_sample(ew, budget_pairs, fetch_kv=None, seed=0, num_threads=0):
    """fp64 oracle on a bounded sample: whole requests while they fit the budget in
    (row, head, visible key) units, else evenly spaced rows of one request.
    Returns (seconds, flops, bytes, description, threads)."""
    import oracle
    rng = np.random.default_rng(seed)
    rows = extend_rows(ew)
    r2t = ew.req_to_token.numpy()
    rpi = ew.req_pool_idx.numpy().astype(np.int64)
    lens = ew.seq_lens.numpy().astype(np.int64)
    sel = []
    acc = 0
    for b in rng.permutation(ew.batch):
        cost = int(rows[b].sum()) * ew.num_q_heads
        if acc + cost <= budget_pairs:
            sel.append((int(b), np.arange(len(rows[b]))))
            acc += cost
        else:
            room = max(1, (budget_pairs - acc) // max(1, int(rows[b].mean()) * ew.num_q_heads))
            pick = np.linspace(0, len(rows[b]) - 1, num=min(len(rows[b]), room)).astype(np.int64)
            sel.append((int(b), pick))
            acc += int(rows[b][pick].sum()) * ew.num_q_heads
            break
    used = [r2t[rpi[b], :lens[b]].astype(np.int64) for b, _ in sel]
    allslots = np.unique(np.concatenate(used))
    table = np.zeros((len(sel) + 1, max(int(lens.max()), 1)), dtype=np.int32)
    for i, (b, _) in enumerate(sel):
        table[i + 1, :lens[b]] = np.searchsorted(allslots, used[i])
    if fetch_kv is not None:
        k, v = fetch_kv(allslots)
    else:
        nrng = np.random.default_rng(17 + seed)
        shape = (len(allslots), ew.num_kv_heads, ew.head_dim)
        k = (nrng.standard_normal(size=shape, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
        v = (nrng.standard_normal(size=shape, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kend = np.concatenate([rows[b][pick] for b, pick in sel]).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum([len(pick) for _, pick in sel])]).astype(np.int32)
    gen = torch.Generator().manual_seed(23 + seed)
    q = torch.randn((int(qo[-1]), ew.num_q_heads, ew.head_dim), generator=gen).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    st, out, lse = oracle.extend(q, k, v, table, np.arange(1, len(sel) + 1, dtype=np.int32),
                                 [int(lens[b]) for b, _ in sel], qo, kend, ew.sm_scale, num_threads=num_threads)
    secs = time.perf_counter() - t0
    assert st == oracle.OK
    flops = 4.0 * ew.num_q_heads * ew.head_dim * float(kend.sum())
    kv_row = 2 * ew.num_kv_heads * ew.head_dim * 2
    nbytes = len(allslots) * kv_row + int(qo[-1]) * ew.num_q_heads * ew.head_dim * 4
    desc = "%d query rows of %d request(s) (%d row x head x key triples), compact host pool" % (
        int(qo[-1]), len(sel), int(kend.sum()) * ew.num_q_heads)
    return secs, flops, nbytes, desc, (oracle.max_threads() if num_threads <= 0 else num_threads)


def reference_extend(args, world):
    from paged_kv_cache_req_gb300.workloads import make_extend_workload
    import oracle
    oracle.build()
    ew = make_extend_workload(args.workload, seed=args.seed, batch=args.batch)
    metric, unit, _ = EXTEND_METRIC[args.workload]
    for _ in range(args.warmup):
        extend_oracle_sample(ew, args.ref_key_heads // 8, seed=0)
    secs = flops = nbytes = 0.0
    desc, threads = "", 0
    for i in range(args.steps):
        s_, f_, b_, desc, threads = extend_oracle_sample(ew, args.ref_key_heads // 2, seed=i)
        secs += s_
        flops += f_
        nbytes += b_
    value = (flops / secs / 1e12) if unit == "TFLOP/s" else (nbytes / secs / 1e9)
    return {"impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": extend_config(ew, world, token_table=args.fused),
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": threads, "kind": "oracle",
                             "sample": "each step: " + desc},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def measure_extend(opts, world, rank, local, dist):
    from paged_kv_cache_req_gb300.engine import DecodeStep, ExtendStep
    from paged_kv_cache_req_gb300.workloads import make_extend_workload
    import oracle
    oracle.build()
    ew = make_extend_workload(opts.workload, seed=opts.seed, batch=opts.batch)
    metric, unit, bound = EXTEND_METRIC[opts.workload]
    step = ExtendStep(ew, device="cuda", kv_chunk=opts.kv_chunk, seed=opts.seed, token_table=opts.fused)
    flops, step_bytes_, launch_bytes = extend_amounts(ew)
    amount = flops / 1e12 if unit == "TFLOP/s" else step_bytes_ / 1e9
    launch_amount = flops / 1e12 if unit == "TFLOP/s" else launch_bytes / 1e9
    flush = step_bytes_ < 4 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    stream = torch.cuda.current_stream()
    for _ in range(opts.warmup):
        step.run()
    torch.cuda.synchronize()
    if step.check_errors():
        raise SystemExit("device error flags raised: %d" % step.check_errors())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, enabled=not opts.profile_run)
    wall0 = time.perf_counter()
    for i in range(opts.steps):
        if flush:
            flush_buf.zero_()
        ev[i][0].record(stream)
        step.build_indices()
        step.store()
        step.plan()
        kev[i][0].record(stream)
        step.attend()
        kev[i][1].record(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = finish_clocks(clocks, opts, step.run)
    if step.check_errors():
        raise SystemExit("device error flags raised: %d" % step.check_errors())
    tot_ms = reduce_max(sum(a.elapsed_time(b) for a, b in ev), dist, "cuda")
    k_ms = sum(a.elapsed_time(b) for a, b in kev) / opts.steps
    value = world * amount * opts.steps / (tot_ms / 1e3)
    if opts.profile_run:
        if rank == 0:
            print(json.dumps({"profile_run": True, "workload": opts.workload, "ms_per_step": round(tot_ms / opts.steps, 4),
                              "extend_ms": round(k_ms, 4)}))
        return None
    h_in, h_out = step.host_step_tensors()
    h2d, d2h = DecodeStep.bytes_of(h_in), DecodeStep.bytes_of(h_out)
    for _ in range(2):
        step.run_from_host(h_in, h_out)
    torch.cuda.synchronize()
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    for i in range(opts.steps):
        if flush:
            flush_buf.zero_()
        e_ev[i][0].record(stream)
        step.run_from_host(h_in, h_out)
        e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e_ev), dist, "cuda")
    if rank != 0:
        return None
    hbm, bf16, bf16_sus, peak_kind = measured_peaks()
    peak = hbm if bound == "hbm" else bf16
    achieved = launch_amount / (k_ms / 1e3)
    cpu = None
    if world == 1 and not opts.no_cpu_baseline:
        def fetch(slots):
            idx = torch.from_numpy(slots).cuda()
            return (step.k_pool[idx].cpu().view(torch.int16).numpy().view(np.uint16),
                    step.v_pool[idx].cpu().view(torch.int16).numpy().view(np.uint16))
        tot_s = tot_f = tot_b = 0.0
        passes, desc, threads = 0, "", 0
        while passes < 10 and (tot_s < 3.0 or passes == 0):
            s_, f_, b_, desc, threads = extend_oracle_sample(ew, opts.cpu_key_heads // 4, fetch_kv=fetch, seed=passes)
            tot_s += s_
            tot_f += f_
            tot_b += b_
            passes += 1
        cv = tot_f / tot_s / 1e12 if unit == "TFLOP/s" else tot_b / tot_s / 1e9
        cpu = {"value": round(cv, 6), "unit": unit, "cores": threads, "kind": "oracle",
               "sample": desc + "; %d pass(es), %.1f s of fp64 attention on %d host threads" % (passes, tot_s, threads),
               "host_cpus": os.cpu_count()}
    roof = {"bound": bound, "kernel": "pkv_extend (attention kernel + merge)", "achieved": round(achieved, 3),
            "peak": peak, "unit": unit, "frac": round(achieved / peak, 4),
            "peak_kind": peak_kind + (" (bf16 dense, burst)" if bound == "tensor" else ""),
            "avg_launch_ms": round(k_ms, 4), "traffic": decode_traffic(opts.workload)}
    if bound == "tensor":
        roof["frac_of_sustained"] = round(achieved / bf16_sus, 4)
    return {
        "metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": opts.steps,
        "warmup": opts.warmup, "ms_per_step": round(tot_ms / opts.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "fp32", "data": "synthetic",
        "config": extend_config(ew, world, token_table=opts.fused),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * amount * opts.steps / (e_ms / 1e3), 3), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms / opts.steps, 4)},
        "gpu_launches": step.launches_per_step() * opts.steps,
        "clocks": with_cycles(clk, tot_ms / opts.steps),
        "wall_s_timed_region": round(wall, 3),
    }


# ---------------------------------------------------------------- decode steps
def decode_cpu_baseline(wl, budget, fetch, threads=0):
    """The oracle (store + decode) on bounded samples of the workload, repeated for at least 3 s."""
    tot_s, tot_b, passes = 0.0, 0, 0
    desc, used = "", 0
    while passes < 10 and (tot_s < 3.0 or passes == 0):
        secs, nb, desc, used = oracle_sample_run(wl, budget, seed=passes, fetch_rows=fetch, num_threads=threads)
        tot_s += secs
        tot_b += nb
        passes += 1
    return {"value": round(tot_b / tot_s / 1e9, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": desc + "; %d pass(es), %.1f s of fp64 store+decode on %d host thread(s)" % (passes, tot_s, used),
            "host_cpus": os.cpu_count()}


def measure_decode(opts, world, rank, local, dist, one_thread_baseline=False):
    from paged_kv_cache_req_gb300.engine import DecodeStep
    from paged_kv_cache_req_gb300.workloads import make_workload
    wl = make_workload(opts.workload, seed=opts.seed, batch=opts.batch)
    step = DecodeStep(wl, device="cuda", cross_mode=opts.cross_mode, kv_chunk=opts.kv_chunk, seed=opts.seed,
                      alloc=opts.alloc, fused=opts.fused)
    total_bytes, decode_bytes = step_bytes(wl, opts.cross_mode, alloc=opts.alloc, fused=opts.fused)
    flush = total_bytes < 4 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None
    stream = torch.cuda.current_stream()

    for _ in range(opts.warmup):
        step.run()
    torch.cuda.synchronize()
    if step.check_errors():
        raise SystemExit("device error flags raised: %d" % step.check_errors())

    # ---- device-timed steps (inputs resident) ----
    n_dec = len(step.problems)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    dev_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dec)]
              for _ in range(opts.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local, enabled=not opts.profile_run)
    wall0 = time.perf_counter()
    for i in range(opts.steps):
        if flush:
            flush_buf.zero_()
        ev[i][0].record(stream)
        if step.alloc:
            step.allocate()
        for j, (name, pb) in enumerate(step.problems.items()):
            if pb.gather:
                step.gather(name)
            else:
                step.build_indices(name)
            if pb.spec.stores:
                step.store(name)
            dev_ev[i][j][0].record(stream)
            step.decode(name)
            dev_ev[i][j][1].record(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = finish_clocks(clocks, opts, step.run)
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [sum(a.elapsed_time(b) for a, b in row) for row in dev_ev]
    tot_ms = reduce_max(sum(step_ms), dist, "cuda")
    ms_per_step = tot_ms / opts.steps
    value = weak_scaling_gbs(world, total_bytes, opts.steps, tot_ms)
    if step.check_errors():
        raise SystemExit("device error flags raised: %d" % step.check_errors())

    if opts.profile_run:
        if rank == 0:
            print(json.dumps({"profile_run": True, "workload": opts.workload, "batch": wl.batch,
                              "ms_per_step": round(tot_ms / opts.steps, 4),
                              "decode_ms": round(sum(dec_ms) / len(dec_ms), 4)}), flush=True)
        return None

    # ---- end to end through the host-buffer API ----
    h_in, h_out = step.host_step_tensors()
    h2d = DecodeStep.bytes_of(h_in)
    d2h = DecodeStep.bytes_of(h_out)
    for _ in range(2):
        step.run_from_host(h_in, h_out)
    torch.cuda.synchronize()
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(opts.steps)]
    for i in range(opts.steps):
        if flush:
            flush_buf.zero_()
        e_ev[i][0].record(stream)
        step.run_from_host(h_in, h_out)
        e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e_ev), dist, "cuda")
    e2e_value = weak_scaling_gbs(world, total_bytes, opts.steps, e_ms)
    if rank != 0:
        return None

    hbm, bf16, bf16_sus, peak_kind = measured_peaks()
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    achieved = decode_bytes / (dec_avg_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": "pkv_decode (split kernel + merge)",
            "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_kind": peak_kind,
            "frac_of_8TBs": round(achieved / 8000.0, 4),
            "algorithmic_bytes_per_launch": decode_bytes, "avg_launch_ms": round(dec_avg_ms, 4),
            "traffic": decode_traffic(opts.workload)}
    if wl.kind == "mla":
        # near the ridge: the tensor pipe's share too (q.k over 576 dims + P.V over 512 per key and head)
        keys = sum(int(p.seq_lens.sum()) for p in wl.problems)
        flops = 2.0 * keys * wl.num_q_heads * (wl.head_dim_qk + wl.head_dim_v)
        tfs = flops / (dec_avg_ms / 1e3) / 1e12
        roof["tensor"] = {"achieved": round(tfs, 2), "unit": "TFLOP/s", "flops_per_launch": flops,
                          "peak": bf16, "frac": round(tfs / bf16, 4), "peak_sustained": bf16_sus,
                          "frac_of_sustained": round(tfs / bf16_sus, 4)}

    cpu = cpu1 = None
    if world == 1 and not opts.no_cpu_baseline:
        import oracle
        oracle.build()

        def fetch(slots):
            idx = torch.from_numpy(slots).cuda()
            kb = step.k_pool[idx].cpu().view(torch.int16).numpy().view(np.uint16)
            vb = None if step.v_pool is None else step.v_pool[idx].cpu().view(torch.int16).numpy().view(np.uint16)
            return kb, vb
        cpu = decode_cpu_baseline(wl, opts.cpu_key_heads, fetch)
        if one_thread_baseline:
            cpu1 = decode_cpu_baseline(wl, max(1, opts.cpu_key_heads // 16), fetch, threads=1)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": opts.steps,
        "warmup": opts.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "fp32", "data": "synthetic",
        "decode_steps_per_s": round(world * 1e3 / ms_per_step, 2),
        "config": decode_config(wl, opts.cross_mode, opts.alloc, world, fused=opts.fused),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e_ms / opts.steps, 4)},
        "gpu_launches": step.launches_per_step() * opts.steps,
        "clocks": with_cycles(clk, ms_per_step),
        "wall_s_timed_region": round(wall, 3),
    }
    if cpu1 is not None:
        line["cpu_baseline_1thread"] = cpu1
    return line


# ---------------------------------------------------------------- arms
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measure(opts, world, rank, local, dist, one_thread_baseline=False):
    if opts.workload == "encoder_merge":
        return measure_merge(opts, world, rank, local, dist)
    if opts.workload in EXTEND_WORKLOADS:
        return measure_extend(opts, world, rank, local, dist)
    return measure_decode(opts, world, rank, local, dist, one_thread_baseline=one_thread_baseline)


# Every other recipe, measured after the headline on the same GPU (N = 1): workload,
# cross-attention mode, timed steps.  Each entry carries its own clocks, roofline,
# traffic and CPU baseline; the configurations the oracle runs in seconds also carry
# a 1-thread oracle time.
PER_CONFIG = (
    ("tiny_gqa", "paged", 200, False),
    ("qwen3_0p6b", "paged", 200, False),
    ("qwen3_0p6b", "paged", 200, True),
    ("whisper_encdec", "paged", 200, False),
    ("whisper_encdec", "paged", 200, True),
    ("whisper_encdec", "gather", 200, False),
    ("whisper_encdec", "gather", 200, True),
    ("llama3_8b", "paged", 100, True),
    ("deepseek_v3_mla", "paged", 100, False),
    ("llama3_8b_verify", "paged", 100, False),
    ("llama3_8b_verify", "paged", 100, True),
    ("qwen3_0p6b_prefill", "paged", 100, False),
    ("qwen3_0p6b_prefill", "paged", 100, True),
    ("hunyuan_image_spans", "paged", 50, False),
    ("hunyuan_image_spans", "paged", 50, True),
    ("encoder_merge", "paged", 200, False),
)
ONE_THREAD_BASELINE = ("tiny_gqa", "qwen3_0p6b")


def per_config_entries(args, world, rank, local, dist):
    out = {}
    for name, cross, steps, fused in PER_CONFIG:
        if name == args.workload and cross == args.cross_mode and fused == args.fused:
            continue
        opts = argparse.Namespace(**vars(args))
        opts.workload, opts.cross_mode, opts.steps, opts.fused = name, cross, steps, fused
        opts.alloc, opts.kv_chunk, opts.batch = False, 0, None
        opts.cpu_key_heads = args.cpu_key_heads // 3
        line = measure(opts, world, rank, local, dist, one_thread_baseline=name in ONE_THREAD_BASELINE)
        torch.cuda.empty_cache()
        if line is None:
            continue
        for k in ("n_gpus", "higher_is_better", "scaling", "vs_baseline", "data", "warmup"):
            line.pop(k, None)
        key = name if name != "whisper_encdec" else "whisper_encdec_" + cross
        out[key + ("_fused" if fused else "")] = line
    return out


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload == "encoder_merge":
        line = reference_merge(args, world)
    elif args.workload in EXTEND_WORKLOADS:
        line = reference_extend(args, world)
    else:
        from paged_kv_cache_req_gb300.workloads import make_workload
        wl = make_workload(args.workload, seed=args.seed, batch=args.batch)
        import oracle
        oracle.build()
        budget = args.ref_key_heads
        for _ in range(args.warmup):
            oracle_sample_run(wl, budget // 4, seed=0)
        times, total_bytes, desc, threads = [], 0, "", 0
        for i in range(args.steps):
            secs, nb, desc, threads = oracle_sample_run(wl, budget, seed=i)
            times.append(secs)
            total_bytes += nb
        value = total_bytes / sum(times) / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": decode_config(wl, args.cross_mode, args.alloc, world, fused=args.fused),
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                 "sample": "each step: " + desc},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from paged_kv_cache_req_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if dist is not None:
        dist.barrier()
    line = measure(args, world, rank, local, dist)
    if line is not None and world == 1 and not args.profile_run and not args.no_per_config \
            and args.batch is None and args.workload == DEFAULT_WORKLOAD and not args.alloc:
        line["per_config"] = per_config_entries(args, world, rank, local, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--cross-mode", default="paged", choices=["paged", "gather"])
    ap.add_argument("--kv-chunk", type=int, default=0)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="headline workload only (no per_config entries for the other recipes)")
    ap.add_argument("--fused", action="store_true",
                    help="GQA decode reads its pages from req_to_token and stores the new rows itself "
                         "(one launch per attention problem, no pkv_build_indices / pkv_store); "
                         "the multi-query steps read their pages from req_to_token (no pkv_build_indices)")
    ap.add_argument("--alloc", action="store_true",
                    help="allocate each step's new slots on the device (pkv_alloc_extend + pkv_write_req_to_token)")
    ap.add_argument("--profile-run", action="store_true",
                    help="only warm-up + timed steps (for ncu); prints a short line")
    ap.add_argument("--batch", type=int, default=None, help="smaller batch of the same recipe (profiling)")
    ap.add_argument("--cpu-key-heads", type=int, default=300_000_000,
                    help="cap on the CPU-oracle sample in (key, query head) pairs (~5 s on 16 Grace cores)")
    ap.add_argument("--ref-key-heads", type=int, default=150_000_000,
                    help="cap on each reference-arm step in (key, query head) pairs")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
