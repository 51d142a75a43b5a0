"""Seeded synthetic workloads for paged-KV decode attention.

This module only *produces inputs*: pool geometry, page placement, the
token-granular ``req_to_token`` table, lengths, the new token's slot and the
bf16 q / k / v values.  It holds none of the method's arithmetic (no page-table
derivation, no attention, no gather): both the CUDA path and the CPU oracle
consume what it produces.

Layout conventions follow the pages' description of an SGLang-style engine
("Enabling Encoder-Decoder Models on Intel XPU in SGLang", section "How SGLang
stores the KV cache: two pools and a page size"; mini-sglang handbook, "The KV
pool, the page table and the token pool"):

* ``req_to_token`` is int32 ``[rows, W]``; row 0 is a padding row that no real
  request uses, and ``W`` is the longest position rounded up to 32 columns
  (128-byte aligned rows, as the mini-sglang page table does).
* K and V pools are per-layer ``[num_slots, num_kv_heads, head_dim]`` bf16
  (MLA: one latent pool ``[num_slots, kv_lora_rank + rope_dim]``).  Slot 0
  (page 0) is the padding page and is never handed to a request.
* A paged allocator hands out whole pages, so a request's tokens are
  contiguous inside each page (the invariant the stride-and-divide page-table
  derivation relies on); pages themselves are shuffled across the pool.
* Decode step: each request has ``cached_len`` tokens in the cache; the step
  stores one new K/V row at position ``cached_len`` (its slot comes from the
  row, as ``out_loc = page_table[row, cached_len:device_len]``) and attends over
  ``cached_len + 1`` keys.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

__all__ = [
    "CONFIGS",
    "Problem",
    "Workload",
    "make_workload",
    "fill_pool",
    "make_values",
    "round_up",
    "MergeWorkload",
    "make_encoder_merge",
    "fill_merge_buffers",
    "EXTEND_CONFIGS",
    "ExtendWorkload",
    "make_extend_workload",
]


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


# --------------------------------------------------------------------------
# Workload recipes (shapes, length mixes, pool geometry).
# --------------------------------------------------------------------------
CONFIGS: Dict[str, dict] = {
    # 4 requests, cached lengths {17, 64, 100, 255}; 16 q / 8 kv heads x 128;
    # page_size 1; a 2048-slot pool whose slots are handed out in a random
    # permutation (a token allocator's free list after churn).
    "tiny_gqa": dict(kind="gqa", batch=4, lens=[17, 64, 100, 255], hq=16, hkv=8, d=128,
                     ps=1, pool_slots=2048),
    # Qwen3-0.6B attention shapes: batch 32, cached lengths U[1, 4096],
    # 16 q / 8 kv heads x 128, page_size 16, pages shuffled over a 200k-token pool.
    "qwen3_0p6b": dict(kind="gqa", batch=32, len_dist=("uniform", 1, 4096), hq=16, hkv=8, d=128,
                       ps=16, pool_tokens=200_000, num_layers=28),
    # Llama-3-8B attention shapes, large batch: 256 requests, cached lengths
    # log-uniform in [128, 32768], 32 q / 8 kv heads x 128, page_size 64;
    # groups of 16 requests share a 2048-token prefix on the same pages.
    "llama3_8b": dict(kind="gqa", batch=256, len_dist=("loguniform", 128, 32768), hq=32, hkv=8,
                      d=128, ps=64, prefix_group=16, prefix_tokens=2048, pool_factor=1.25,
                      num_layers=32),
    # Whisper-large encoder-decoder step: batch 64, decoder cached lengths
    # U[1, 448], 1500 encoder tokens per request, 20 heads x 64, page_size 16.
    # Row = [encoder 0:1500 | pad to ceil_align(1500, 16) = 1504 | decoder].
    "whisper_encdec": dict(kind="gqa", batch=64, len_dist=("uniform", 1, 448), enc_len=1500, hq=20,
                           hkv=20, d=64, ps=16, pool_factor=1.25),
    # DeepSeek-V3 MLA decode: batch 128, cached lengths U[512, 16384], 128 q
    # heads over one latent KV of 512 + 64 rope dims, softmax scale 1/sqrt(192),
    # page_size 64, a -1 padded block table.
    "deepseek_v3_mla": dict(kind="mla", batch=128, len_dist=("uniform", 512, 16384), hq=128,
                            kv_lora_rank=512, rope_dim=64, qk_nope_dim=128, ps=64, pool_factor=1.25),
}


@dataclass
class Problem:
    """One attention problem over the shared pool (a layer's self- or cross-attention).

    ``seq_lens`` are the key counts the decode attends over, ``kv_start`` the
    column where the problem's region begins in each ``req_to_token`` row.
    ``cached_lens``/``slot_mapping`` are set when the step also stores one new
    K/V row per request (decoder self-attention); cross-attention over a
    finished encoder stores nothing.
    """

    name: str
    seq_lens: torch.Tensor            # int32 [B]
    kv_start: torch.Tensor            # int32 [B]
    stores: bool
    cached_lens: Optional[torch.Tensor] = None   # int32 [B]
    slot_mapping: Optional[torch.Tensor] = None  # int32 [B]
    causal: bool = True


@dataclass
class Workload:
    name: str
    kind: str                 # "gqa" (MHA/GQA) or "mla"
    batch: int
    num_q_heads: int
    num_kv_heads: int         # 1 for MLA
    head_dim_qk: int          # 576 for MLA
    head_dim_v: int           # 512 for MLA
    page_size: int
    sm_scale: float
    num_slots: int            # pool rows (multiple of page_size)
    req_to_token: torch.Tensor     # int32 [rows, W]
    req_pool_idx: torch.Tensor     # int32 [B]
    problems: List[Problem]
    seed: int
    num_layers: Optional[int] = None
    # slots each problem reads, for byte accounting (numpy int64 arrays)
    meta: dict = field(default_factory=dict)

    @property
    def num_pool_pages(self) -> int:
        return self.num_slots // self.page_size

    @property
    def has_v_pool(self) -> bool:
        return self.kind != "mla"

    def problem(self, name: str) -> Problem:
        for p in self.problems:
            if p.name == name:
                return p
        raise KeyError(name)


def _draw_lengths(rng: np.random.Generator, spec, batch: int) -> np.ndarray:
    kind, lo, hi = spec
    if kind == "uniform":
        return rng.integers(lo, hi + 1, size=batch).astype(np.int64)
    if kind == "loguniform":
        x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=batch))
        return np.clip(np.round(x), lo, hi).astype(np.int64)
    raise ValueError(kind)


class _PageAllocator:
    """Hands out pool pages from a shuffled free list (page 0 is padding)."""

    def __init__(self, rng: np.random.Generator, num_pages: int):
        self.free = list(rng.permutation(np.arange(1, num_pages)).tolist())

    def take(self, n: int) -> List[int]:
        if n > len(self.free):
            raise RuntimeError("pool too small for the recipe")
        out, self.free = self.free[:n], self.free[n:]
        return out


def _pages_to_slots(pages: List[int], ps: int, count: int) -> np.ndarray:
    """Token slots of the first ``count`` positions laid over ``pages``."""
    if count == 0:
        return np.zeros(0, dtype=np.int64)
    slots = (np.asarray(pages, dtype=np.int64)[:, None] * ps + np.arange(ps)[None, :]).reshape(-1)
    return slots[:count]


def make_workload(name: str, seed: int = 0, batch: Optional[int] = None) -> Workload:
    """Index structures of a recipe (CPU tensors); values come from ``fill_pool``/``make_values``.

    ``batch`` overrides the recipe's batch size (smaller parity cases of the
    same shape).
    """
    cfg = dict(CONFIGS[name])
    B = int(batch if batch is not None else cfg["batch"])
    rng = np.random.default_rng(seed)
    ps = int(cfg["ps"])

    if "lens" in cfg:
        lens = np.asarray(cfg["lens"][:B], dtype=np.int64)
        if len(lens) < B:
            lens = np.concatenate([lens, rng.integers(1, 256, size=B - len(lens))])
    else:
        lens = _draw_lengths(rng, cfg["len_dist"], B)
    new_lens = lens + 1                   # keys after storing this step's token

    enc_len = int(cfg.get("enc_len", 0))
    enc_reserve = round_up(enc_len, ps) if enc_len else 0   # ceil_align(enc_len, page_size)
    dec_start = enc_reserve

    # ---- pages each request needs -------------------------------------------
    group = int(cfg.get("prefix_group", 0))
    prefix_tokens = int(cfg.get("prefix_tokens", 0))
    shared_tok = np.zeros(B, dtype=np.int64)
    if group:
        # The prefix cache holds whole pages only: request j maps its first
        # min(prefix_tokens, ps * floor(L_j / ps)) positions onto the group's
        # shared pages; the rest, and the new token, go on private pages.
        shared_tok = np.minimum(prefix_tokens, (lens // ps) * ps)
    private_tok = new_lens - shared_tok
    private_pages = -(-private_tok // ps)
    enc_pages = enc_reserve // ps
    n_groups = -(-B // group) if group else 0
    shared_pages_per_group = prefix_tokens // ps if group else 0
    need_pages = int(private_pages.sum() + B * enc_pages + n_groups * shared_pages_per_group)

    if "pool_slots" in cfg:
        num_pages = int(cfg["pool_slots"]) // ps
    elif "pool_tokens" in cfg:
        num_pages = int(cfg["pool_tokens"]) // ps
    else:
        num_pages = int(math.ceil(need_pages * float(cfg.get("pool_factor", 1.25)))) + 1
    num_slots = num_pages * ps
    alloc = _PageAllocator(rng, num_pages)

    width = round_up(int(dec_start + new_lens.max()) + 1, 32)
    rows = B + 1                                   # row 0 is the padding row
    r2t = np.zeros((rows, width), dtype=np.int32)
    req_pool_idx = (rng.permutation(B) + 1).astype(np.int32)

    group_pages = [alloc.take(shared_pages_per_group) for _ in range(n_groups)]
    for b in range(B):
        row = req_pool_idx[b]
        col = 0
        if enc_len:
            pages = alloc.take(enc_pages)
            r2t[row, 0:enc_reserve] = _pages_to_slots(pages, ps, enc_reserve)
            col = dec_start
        if group and shared_tok[b]:
            gp = group_pages[b // group][: shared_tok[b] // ps]
            r2t[row, col:col + shared_tok[b]] = _pages_to_slots(gp, ps, int(shared_tok[b]))
        pages = alloc.take(int(private_pages[b]))
        c0 = col + int(shared_tok[b])
        r2t[row, c0:c0 + int(private_tok[b])] = _pages_to_slots(pages, ps, int(private_tok[b]))

    r2t_t = torch.from_numpy(r2t)
    rpi = torch.from_numpy(req_pool_idx)
    cached = torch.from_numpy(lens.astype(np.int32))
    dec_start_t = torch.full((B,), dec_start, dtype=torch.int32)
    # out_loc of the new token = req_to_token[row, kv_start + cached_len]
    slot_new = torch.from_numpy(
        r2t[req_pool_idx.astype(np.int64), dec_start + lens].astype(np.int32))

    problems = [Problem(name="self", seq_lens=torch.from_numpy(new_lens.astype(np.int32)),
                        kv_start=dec_start_t, stores=True, cached_lens=cached,
                        slot_mapping=slot_new, causal=True)]
    if enc_len:
        problems.append(Problem(name="cross", seq_lens=torch.full((B,), enc_len, dtype=torch.int32),
                                kv_start=torch.zeros(B, dtype=torch.int32), stores=False,
                                causal=False))

    if cfg["kind"] == "mla":
        hq, hkv = int(cfg["hq"]), 1
        dqk = int(cfg["kv_lora_rank"]) + int(cfg["rope_dim"])
        dv = int(cfg["kv_lora_rank"])
        scale = 1.0 / math.sqrt(int(cfg["qk_nope_dim"]) + int(cfg["rope_dim"]))
    else:
        hq, hkv = int(cfg["hq"]), int(cfg["hkv"])
        dqk = dv = int(cfg["d"])
        scale = 1.0 / math.sqrt(dqk)

    return Workload(name=name, kind=cfg["kind"], batch=B, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim_qk=dqk, head_dim_v=dv, page_size=ps, sm_scale=scale,
                    num_slots=num_slots, req_to_token=r2t_t, req_pool_idx=rpi,
                    problems=problems, seed=seed, num_layers=cfg.get("num_layers"),
                    meta=dict(enc_len=enc_len, enc_reserve=enc_reserve, shared_tok=shared_tok,
                              need_pages=need_pages, num_pages=num_pages))


# --------------------------------------------------------------------------
# Values
# --------------------------------------------------------------------------
def fill_pool(wl: Workload, device="cpu", seed: Optional[int] = None, chunk_elems: int = 1 << 28):
    """bf16 N(0,1) K and V pools (``v`` is None for an MLA latent pool).

    Filled in chunks with a seeded generator on ``device`` so that multi-GB
    pools never need a float32 staging copy.
    """
    seed = wl.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(1_000_003 + seed)
    shape = (wl.num_slots, wl.head_dim_qk) if wl.kind == "mla" else \
        (wl.num_slots, wl.num_kv_heads, wl.head_dim_qk)
    pools = []
    for _ in range(2 if wl.has_v_pool else 1):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        for i in range(0, flat.numel(), chunk_elems):
            flat[i:i + chunk_elems].normal_(generator=gen)
        pools.append(t)
    return pools[0], (pools[1] if wl.has_v_pool else None)


def make_values(wl: Workload, seed: Optional[int] = None) -> dict:
    """bf16 N(0,1) per-step tensors on the CPU: q for every problem, new K/V rows."""
    seed = wl.seed if seed is None else seed
    gen = torch.Generator(device="cpu")
    gen.manual_seed(2_000_029 + seed)
    B = wl.batch
    out = {}
    for p in wl.problems:
        out["q_" + p.name] = torch.randn((B, wl.num_q_heads, wl.head_dim_qk), generator=gen).to(torch.bfloat16)
    if wl.kind == "mla":
        out["k_new"] = torch.randn((B, wl.head_dim_qk), generator=gen).to(torch.bfloat16)
        out["v_new"] = None
    else:
        out["k_new"] = torch.randn((B, wl.num_kv_heads, wl.head_dim_qk), generator=gen).to(torch.bfloat16)
        out["v_new"] = torch.randn((B, wl.num_kv_heads, wl.head_dim_v), generator=gen).to(torch.bfloat16)
    return out


# --------------------------------------------------------------------------
# Encoder-cache merge (the Neuron encoder cache's read path)
# --------------------------------------------------------------------------
@dataclass
class MergeWorkload:
    """A prefill step's encoder-cache gather: `items` cached images, each one block of
    `block_size` rows of `fat_dim` bf16 values, of which `tokens_per_item` are real;
    the position map places them in a sequence of `num_tokens` rows."""
    name: str
    num_blocks: int          # cache blocks, the last one scratch
    block_size: int
    fat_dim: int
    max_blocks: int          # fixed shape of the step's block-id / position inputs
    num_tokens: int
    items: int
    tokens_per_item: int
    block_ids: np.ndarray    # int32 [max_blocks]
    positions: np.ndarray    # int64 [max_blocks, block_size]; num_tokens = sentinel
    seed: int = 0

    @property
    def rows_moved(self) -> int:
        return int((self.positions < self.num_tokens).sum())

    @property
    def row_bytes(self) -> int:
        return self.fat_dim * 2


def make_encoder_merge(seed: int = 0, items: int = 30, tokens_per_item: int = 256, fat_dim: int = 5120 * 4,
                       block_size: int = 2048 // 4, cache_tokens: int = 16384, text_tokens: int = 16,
                       lead_tokens: int = 512) -> MergeWorkload:
    """Qwen3-VL-32B-shaped read path: fat_dim 5120 x (1 + 3 deepstack levels), blocks of
    2048 / 4 = 512 post-merger tokens, one 512x512 image = 256 tokens per block, 30
    images.  The cache holds ceil(cache_tokens / block_size) blocks + 1 scratch; the
    step's fixed shape has room for all of them; unused slots name the scratch block
    with sentinel positions.  The sequence is `lead_tokens` of text, then for every
    image `text_tokens` of text followed by its image tokens."""
    rng = np.random.default_rng(seed)
    num_blocks = -(-cache_tokens // block_size) + 1
    max_blocks = num_blocks - 1
    if items > max_blocks:
        raise ValueError("more items than cache blocks")
    num_tokens = lead_tokens + items * (text_tokens + tokens_per_item)
    block_ids = np.full(max_blocks, num_blocks - 1, dtype=np.int32)
    block_ids[:items] = rng.permutation(num_blocks - 1)[:items]       # cache hits anywhere in the buffer
    positions = np.full((max_blocks, block_size), num_tokens, dtype=np.int64)
    for k in range(items):
        start = lead_tokens + k * (text_tokens + tokens_per_item) + text_tokens
        positions[k, :tokens_per_item] = np.arange(start, start + tokens_per_item)
    return MergeWorkload(name="encoder_merge", num_blocks=num_blocks, block_size=block_size, fat_dim=fat_dim,
                         max_blocks=max_blocks, num_tokens=num_tokens, items=items, tokens_per_item=tokens_per_item,
                         block_ids=block_ids, positions=positions, seed=seed)


def fill_merge_buffers(mw: MergeWorkload, device="cpu", chunk_elems: int = 1 << 28):
    """bf16 N(0,1) cache buffer [num_blocks, block_size, fat_dim] and hidden rows [num_tokens, fat_dim]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(3_000_017 + mw.seed)
    out = []
    for shape in ((mw.num_blocks, mw.block_size, mw.fat_dim), (mw.num_tokens, mw.fat_dim)):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        for i in range(0, flat.numel(), chunk_elems):
            flat[i:i + chunk_elems].normal_(generator=gen)
        out.append(t)
    return out[0], out[1]


# --------------------------------------------------------------------------
# Multi-query steps: target-verify, chunked prefill, diffusion rows with spans
# --------------------------------------------------------------------------
EXTEND_CONFIGS: Dict[str, dict] = {
    # Llama-3-8B shapes, speculative target-verify of 4 draft tokens per request
    # over cached lengths log-U[128, 32768] (the large-batch decode mix), page 64.
    "llama3_8b_verify": dict(batch=128, hq=32, hkv=8, d=128, ps=64, cached=("loguniform", 128, 32768),
                             new=("fixed", 4, 4)),
    # Qwen3-0.6B shapes, chunked prefill: 8 requests with a cached prefix U[0, 4096]
    # and a 1024-token chunk each (causal), page 16.
    "qwen3_0p6b_prefill": dict(batch=8, hq=16, hkv=8, d=128, ps=16, cached=("uniform", 0, 4096),
                               new=("fixed", 1024, 1024)),
    # HunyuanImage-shaped first denoising step: 2 requests x 2 CFG rows, a 1024-token
    # text prefix (causal segment) then 4096 image tokens (one full segment), all
    # positions queried, 32 q / 8 kv heads x 128, page 64.
    "hunyuan_image_spans": dict(batch=4, hq=32, hkv=8, d=128, ps=64, cached=("fixed", 0, 0),
                                new=("fixed", 5120, 5120), spans=((0, 0, 1024), (1, 1024, 5120))),
}


@dataclass
class ExtendWorkload:
    """Index structures of a multi-query step: request b holds seq_lens[b] keys, the
    last new_lens[b] of which are stored this step; its qo_lens[b] query rows are
    its last positions (causal) or, with `segments`, its segments' positions."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    sm_scale: float
    num_slots: int
    req_to_token: torch.Tensor     # int32 [rows, W]
    req_pool_idx: torch.Tensor     # int32 [B]
    seq_lens: torch.Tensor         # int32 [B]
    new_lens: torch.Tensor         # int32 [B]
    qo_lens: torch.Tensor          # int32 [B]
    slot_mapping: torch.Tensor     # int32 [sum new_lens]: slots of the stored positions
    segments: Optional[List[List[tuple]]] = None
    seed: int = 0

    @property
    def num_pool_pages(self) -> int:
        return self.num_slots // self.page_size


def _draw(rng, spec, batch):
    kind, lo, hi = spec
    if kind == "fixed":
        return np.full(batch, lo, dtype=np.int64)
    return _draw_lengths(rng, (kind, lo, hi), batch)


def make_extend_workload(name: str, seed: int = 0, batch: Optional[int] = None) -> ExtendWorkload:
    cfg = dict(EXTEND_CONFIGS[name])
    B = int(batch if batch is not None else cfg["batch"])
    rng = np.random.default_rng(seed)
    ps = int(cfg["ps"])
    cached = _draw(rng, cfg["cached"], B)
    new = _draw(rng, cfg["new"], B)
    lens = cached + new
    need_pages = int((-(-lens // ps)).sum())
    num_pages = int(math.ceil(need_pages * 1.25)) + 8
    width = round_up(int(lens.max()) + 1, 32)
    r2t = np.zeros((B + 1, width), dtype=np.int32)
    rpi = (rng.permutation(B) + 1).astype(np.int32)
    alloc = _PageAllocator(rng, num_pages)
    slots_new = []
    for b in range(B):
        pages = alloc.take(int(-(-lens[b] // ps)))
        row = _pages_to_slots(pages, ps, int(lens[b]))
        r2t[rpi[b], :lens[b]] = row
        slots_new.append(row[cached[b]:])
    segments = None
    if "spans" in cfg:
        segments = [[tuple(sp) for sp in cfg["spans"]] for _ in range(B)]
        qo = np.array([sum(e - a for _, a, e in segs) for segs in segments], dtype=np.int64)
    else:
        qo = new
    return ExtendWorkload(name=name, batch=B, num_q_heads=cfg["hq"], num_kv_heads=cfg["hkv"], head_dim=cfg["d"],
                          page_size=ps, sm_scale=1.0 / math.sqrt(cfg["d"]), num_slots=num_pages * ps,
                          req_to_token=torch.from_numpy(r2t), req_pool_idx=torch.from_numpy(rpi),
                          seq_lens=torch.from_numpy(lens.astype(np.int32)),
                          new_lens=torch.from_numpy(new.astype(np.int32)),
                          qo_lens=torch.from_numpy(qo.astype(np.int32)),
                          slot_mapping=torch.from_numpy(np.concatenate(slots_new).astype(np.int32)),
                          segments=segments, seed=seed)
