"""Decode step over a paged KV cache: the library's public, per-step API.

``DecodeStep`` keeps a workload's req_to_token table, pools and step buffers
resident on one GPU and runs one decode layer step as a sequence of libpkv
calls on the current stream:

    pkv_build_indices   req_to_token -> kv_indptr / kv_indices (or the -1 padded table)
    pkv_store           this step's new K/V rows -> their pool slots
    pkv_decode          attention of every request's new token over its pages

With ``alloc=True`` the new token's slot is not taken from the workload but
allocated on the device first, as a serving loop would:

    pkv_alloc_extend        each request grows by one position: the slot after
                            its last one, or a fresh page from the free list
    pkv_write_req_to_token  that slot into the request's row of req_to_token

(the free list is restored before every step, so steps stay idempotent).

With ``fused=True`` (GQA) the decode call reads its pages straight from
req_to_token (PKV_LAYOUT_REQ_TO_TOKEN: no pkv_build_indices launch, no page list
in between) and, for the problem that stores, writes the new token's K/V into
the pool itself before attending (the fused store): a step is then one decode
launch (+ its merge) per problem.

For an encoder-decoder workload the cross-attention over the encoder region
runs either through its own page list ("paged": the page-aligned encoder of
"Approach 1") or through pkv_ragged_gather into a contiguous varlen buffer
followed by a varlen decode ("gather": "Approach 2").

Nothing here computes: every step runs in libpkv's kernels.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from . import _binding as B
from .workloads import Workload, fill_pool, make_values

__all__ = ["DecodeStep", "ExtendStep"]


class _ProblemBuffers:
    pass


def _pack(owners, device):
    """Moves tensors into consecutive 256-byte aligned slices of one new device buffer.

    ``owners`` lists (object, attribute) pairs; each attribute is replaced by a view of
    the buffer holding the same values, so one copy of the buffer fills them all (the
    per-step inputs come from the host in a single transfer, the outputs go back in one).
    Returns the buffer.
    """
    sizes = [getattr(o, a).numel() * getattr(o, a).element_size() for o, a in owners]
    offs, total = [], 0
    for nb in sizes:
        offs.append(total)
        total += (nb + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
    for (o, a), off, nb in zip(owners, offs, sizes):
        t = getattr(o, a)
        v = buf[off:off + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        setattr(o, a, v)
    return buf


class DecodeStep:
    def __init__(self, wl: Workload, device="cuda", cross_mode: str = "paged", kv_chunk: int = 0,
                 pools=None, values: Optional[Dict[str, torch.Tensor]] = None, seed: Optional[int] = None,
                 alloc: bool = False, fused: bool = False):
        if cross_mode not in ("paged", "gather"):
            raise ValueError(cross_mode)
        if fused and wl.kind != "gqa":
            raise ValueError("the token-table layout and the fused store are GQA only")
        self.fused = bool(fused)
        self.wl = wl
        self.device = torch.device(device)
        self.cross_mode = cross_mode
        self.kv_chunk = int(kv_chunk)
        dev = self.device
        ps = wl.page_size
        self.r2t = wl.req_to_token.to(dev)
        self.req_pool_idx = wl.req_pool_idx.to(dev)
        if pools is None:
            pools = fill_pool(wl, device=dev, seed=seed)
        self.k_pool, self.v_pool = pools
        vals = make_values(wl, seed=seed) if values is None else values
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        Bn = wl.batch
        self.k_new = vals["k_new"].to(dev)
        self.v_new = vals["v_new"].to(dev) if vals["v_new"] is not None else None
        self.problems: Dict[str, _ProblemBuffers] = {}
        for p in wl.problems:
            pb = _ProblemBuffers()
            pb.spec = p
            pb.seq_lens = p.seq_lens.to(dev)
            pb.kv_start = p.kv_start.to(dev)
            pb.slot_mapping = p.slot_mapping.to(dev) if p.stores else None
            pb.max_len = int(p.seq_lens.max()) if Bn else 0
            pb.q = vals["q_" + p.name].to(dev)
            pb.out = torch.empty((Bn, wl.num_q_heads, wl.head_dim_v), dtype=torch.bfloat16, device=dev)
            pb.lse = torch.empty((Bn, wl.num_q_heads), dtype=torch.float32, device=dev)
            pb.gather = (p.name == "cross" and cross_mode == "gather")
            self.problems[p.name] = pb
        self.alloc = bool(alloc)
        if self.alloc:
            self._setup_alloc(seed)
        # the step's host inputs and its outputs each live in one buffer (one copy per direction)
        ins = [(self, "k_new"), (self, "req_pool_idx")] + ([(self, "v_new")] if self.v_new is not None else [])
        for name, pb in self.problems.items():
            ins += [(pb, "q"), (pb, "seq_lens")]
            if pb.slot_mapping is not None and not (self.alloc and name == self.alloc_problem):
                ins.append((pb, "slot_mapping"))
        if self.alloc:
            ins += [(self, "prefix_lens"), (self, "last_loc")]
        self.in_buf = _pack(ins, dev)
        self.out_buf = _pack([(pb, "out") for pb in self.problems.values()], dev)
        for pb in self.problems.values():
            p = pb.spec
            max_pages = -(-pb.max_len // ps) if pb.max_len else 0
            if pb.gather:
                rows = int(p.seq_lens.sum())
                pb.k_rag = torch.empty((max(rows, 1),) + tuple(self.k_pool.shape[1:]), dtype=torch.bfloat16, device=dev)
                pb.v_rag = torch.empty_like(pb.k_rag)
                pb.cu = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
                layout = B.PKV_LAYOUT_VARLEN
                pb.args = B.make_decode_args(B.PKV_KIND_GQA, layout, pb.q, pb.k_rag, pb.v_rag, pb.out,
                                             sm_scale=wl.sm_scale, max_seq_len=pb.max_len,
                                             cu_seqlens=pb.cu, lse=pb.lse, kv_chunk=self.kv_chunk)
            elif self.fused:
                # pages straight from req_to_token; the problem that stores writes its new rows itself
                kn, vn = (self.k_new, self.v_new) if p.stores else (None, None)
                pb.args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_REQ_TO_TOKEN, pb.q, self.k_pool,
                                             self.v_pool, pb.out, page_size=ps, sm_scale=wl.sm_scale,
                                             max_seq_len=pb.max_len, seq_lens=pb.seq_lens, lse=pb.lse,
                                             kv_chunk=self.kv_chunk, req_to_token=self.r2t,
                                             req_pool_idx=self.req_pool_idx, kv_start=pb.kv_start,
                                             k_new=kn, v_new=vn)
            elif wl.kind == "mla":
                pb.block_table = torch.empty((Bn, max(max_pages, 1)), dtype=torch.int32, device=dev)
                pb.args = B.make_decode_args(B.PKV_KIND_MLA, B.PKV_LAYOUT_BLOCK_TABLE, pb.q, self.k_pool, None,
                                             pb.out, page_size=ps, sm_scale=wl.sm_scale, max_seq_len=pb.max_len,
                                             head_dim_v=wl.head_dim_v, block_table=pb.block_table,
                                             seq_lens=pb.seq_lens, lse=pb.lse, kv_chunk=self.kv_chunk)
            else:
                pb.kv_indptr = torch.empty(Bn + 1, dtype=torch.int32, device=dev)
                pb.kv_indices = torch.empty(max(Bn * max_pages, 1), dtype=torch.int32, device=dev)
                pb.kv_last = torch.empty(Bn, dtype=torch.int32, device=dev)
                pb.args = B.make_decode_args(B.PKV_KIND_GQA, B.PKV_LAYOUT_CSR, pb.q, self.k_pool, self.v_pool,
                                             pb.out, page_size=ps, sm_scale=wl.sm_scale, max_seq_len=pb.max_len,
                                             kv_indptr=pb.kv_indptr, kv_indices=pb.kv_indices,
                                             kv_last_page_len=pb.kv_last, lse=pb.lse, kv_chunk=self.kv_chunk)
            nbytes = B.pkv_decode_workspace_size(pb.args)
            pb.ws_bytes = nbytes
            pb.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)

    def _setup_alloc(self, seed):
        """Free list = the pool pages no cached position uses (page 0 is padding), in a
        seeded order; each request grows from its cached length by one position."""
        wl = self.wl
        ps = wl.page_size
        r2t = wl.req_to_token.numpy()
        rpi = wl.req_pool_idx.numpy().astype(np.int64)
        names = [n for n, pb in self.problems.items() if pb.spec.stores]
        if len(names) != 1:
            raise ValueError("device allocation needs exactly one problem that stores new tokens")
        self.alloc_problem = names[0]
        used = [np.zeros(1, dtype=np.int64)]
        for pb in self.problems.values():
            lens = pb.spec.seq_lens.numpy().astype(np.int64)
            starts = pb.spec.kv_start.numpy().astype(np.int64)
            cached = lens - 1 if pb.spec.stores else lens
            for b in range(wl.batch):
                used.append(r2t[rpi[b], starts[b]:starts[b] + cached[b]].astype(np.int64) // ps)
        used_pages = np.unique(np.concatenate(used))
        free = np.setdiff1d(np.arange(wl.num_pool_pages, dtype=np.int64), used_pages)
        free = np.random.default_rng(0 if seed is None else seed).permutation(free).astype(np.int32)
        spec = self.problems[self.alloc_problem].spec
        lens = spec.seq_lens.numpy().astype(np.int64)
        starts = spec.kv_start.numpy().astype(np.int64)
        prefix = lens - 1
        last = np.array([r2t[rpi[b], starts[b] + prefix[b] - 1] if prefix[b] > 0 else -1
                         for b in range(wl.batch)], dtype=np.int32)
        dev = self.device
        self.free_pages = torch.from_numpy(free).to(dev)
        self.free_state0 = torch.tensor([0, len(free)], dtype=torch.int32, device=dev)
        self.free_state = self.free_state0.clone()
        self.prefix_lens = torch.from_numpy(prefix.astype(np.int32)).to(dev)
        self.last_loc = torch.from_numpy(last).to(dev)
        self.out_cache_loc = torch.empty(wl.batch, dtype=torch.int32, device=dev)
        self.problems[self.alloc_problem].slot_mapping = self.out_cache_loc

    def allocate(self):
        """This step's slots on the device: one position per request, then into the rows."""
        wl = self.wl
        pb = self.problems[self.alloc_problem]
        self.free_state.copy_(self.free_state0, non_blocking=True)
        B.pkv_alloc_extend(self.prefix_lens, pb.seq_lens, self.last_loc, wl.page_size, wl.num_pool_pages,
                           self.free_pages, self.free_state, self.out_cache_loc, self.err)
        B.pkv_write_req_to_token(self.r2t, self.req_pool_idx, self.prefix_lens, pb.seq_lens, self.out_cache_loc,
                                 self.err, kv_start=pb.kv_start)

    # ------------------------------------------------------------------ steps
    def build_indices(self, name: str):
        pb = self.problems[name]
        wl = self.wl
        if pb.gather or self.fused:
            return
        if wl.kind == "mla":
            B.pkv_build_indices(self.r2t, self.req_pool_idx, pb.seq_lens, wl.page_size, wl.num_pool_pages,
                                self.err, kv_start=pb.kv_start, block_table=pb.block_table)
        else:
            B.pkv_build_indices(self.r2t, self.req_pool_idx, pb.seq_lens, wl.page_size, wl.num_pool_pages,
                                self.err, kv_start=pb.kv_start, kv_indptr=pb.kv_indptr, kv_indices=pb.kv_indices,
                                kv_last_page_len=pb.kv_last)

    def store(self, name: str = "self"):
        pb = self.problems[name]
        if self.fused and not pb.gather:
            return                                   # the decode call stores the new rows itself
        B.pkv_store(self.k_pool, self.v_pool, self.k_new, self.v_new, pb.slot_mapping, self.err)

    def gather(self, name: str):
        pb = self.problems[name]
        B.pkv_ragged_gather(self.k_pool, self.v_pool, self.r2t, self.req_pool_idx, pb.seq_lens, pb.max_len,
                            pb.k_rag, pb.v_rag, pb.cu, self.err, kv_start=pb.kv_start)

    def decode(self, name: str):
        pb = self.problems[name]
        B.pkv_decode(pb.args, pb.workspace, self.err)

    def run(self):
        """One decode step: (allocation), then for each problem page lists, (store), (gather), attention."""
        if self.alloc:
            self.allocate()
        for name, pb in self.problems.items():
            if pb.gather:
                self.gather(name)
            else:
                self.build_indices(name)
            if pb.spec.stores:
                self.store(name)
            self.decode(name)

    def launches_per_step(self) -> int:
        """libpkv kernel launches one ``run()`` issues."""
        n = 2 if self.alloc else 0                  # alloc_extend + write_req_to_token
        for pb in self.problems.values():
            if not self.fused or pb.gather:
                n += 1                               # gather or build_indices
                n += 1 if pb.spec.stores else 0      # store
            n += 1 + (1 if pb.ws_bytes > 0 else 0)   # split kernel (+ merge when requests can split)
        return n

    def check_errors(self) -> int:
        """Synchronises and returns the device error bits raised so far."""
        return int(self.err.item())

    # ------------------------------------------------------------------ host I/O
    def host_step_tensors(self):
        """Pinned host copies of the step's packed inputs and outputs (for end-to-end timing)."""
        return {"inputs": self.in_buf.cpu().pin_memory()}, {"outputs": torch.empty_like(self.out_buf, device="cpu").pin_memory()}

    def run_from_host(self, h_in, h_out):
        """One host-to-device copy of the step's inputs (new K/V rows, q, lengths, slots, row
        indices: packed in one buffer), the step, one device-to-host copy of the outputs."""
        self.in_buf.copy_(h_in["inputs"], non_blocking=True)
        self.run()
        h_out["outputs"].copy_(self.out_buf, non_blocking=True)

    @staticmethod
    def bytes_of(tensors) -> int:
        return int(sum(t.numel() * t.element_size() for t in tensors.values()))


class ExtendStep:
    """One multi-query step over a paged KV cache (extend / target-verify / span rows):

        pkv_build_indices   req_to_token -> kv_indptr / kv_indices
        pkv_store           this step's new tokens' K/V -> their pool slots
        pkv_span_plan       (rows with segments) segment lists -> query rows and key bounds
        pkv_extend          attention of every query row over its visible keys

    With ``token_table=True`` pkv_extend reads the pages straight from req_to_token
    (PKV_LAYOUT_REQ_TO_TOKEN) and the step has no pkv_build_indices launch.
    """

    def __init__(self, ew, device="cuda", kv_chunk: int = 0, seed: Optional[int] = None, token_table: bool = False):
        self.token_table = bool(token_table)
        self.ew = ew
        dev = self.device = torch.device(device)
        seed = ew.seed if seed is None else seed
        B_ = ew.batch
        self.r2t = ew.req_to_token.to(dev)
        self.req_pool_idx = ew.req_pool_idx.to(dev)
        self.seq_lens = ew.seq_lens.to(dev)
        self.slot_mapping = ew.slot_mapping.to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(4_000_037 + seed)
        shape = (ew.num_slots, ew.num_kv_heads, ew.head_dim)
        self.k_pool = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        self.v_pool = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        for t in (self.k_pool, self.v_pool):
            flat = t.view(-1)
            for i in range(0, flat.numel(), 1 << 28):
                flat[i:i + (1 << 28)].normal_(generator=gen)
        cgen = torch.Generator().manual_seed(5_000_011 + seed)
        total_q = int(ew.qo_lens.sum())
        n_new = int(ew.new_lens.sum())
        self.q = torch.randn((total_q, ew.num_q_heads, ew.head_dim), generator=cgen).to(torch.bfloat16).to(dev)
        self.k_new = torch.randn((n_new, ew.num_kv_heads, ew.head_dim), generator=cgen).to(torch.bfloat16).to(dev)
        self.v_new = torch.randn((n_new, ew.num_kv_heads, ew.head_dim), generator=cgen).to(torch.bfloat16).to(dev)
        qo = np.concatenate([[0], np.cumsum(ew.qo_lens.numpy())]).astype(np.int32)
        self.qo_indptr = torch.from_numpy(qo).to(dev)
        self.kv_end = None
        if ew.segments is not None:
            ind, kinds, starts, ends = [0], [], [], []
            for segs in ew.segments:
                for kd, a, e in segs:
                    kinds.append(kd)
                    starts.append(a)
                    ends.append(e)
                ind.append(len(kinds))
            self.seg = [torch.tensor(x, dtype=torch.int32, device=dev) for x in (ind, kinds, starts, ends)]
            self.plan_qo = torch.empty(B_ + 1, dtype=torch.int32, device=dev)
            self.q_pos = torch.empty(total_q, dtype=torch.int32, device=dev)
            self.kv_end = torch.empty(total_q, dtype=torch.int32, device=dev)
        ps = ew.page_size
        pages = int((-(-ew.seq_lens.numpy().astype(np.int64) // ps)).sum())
        self.kv_indptr = torch.empty(B_ + 1, dtype=torch.int32, device=dev)
        self.kv_indices = torch.empty(max(pages, 1), dtype=torch.int32, device=dev)
        self.kv_last = torch.empty(B_, dtype=torch.int32, device=dev)
        self.out = torch.empty((total_q, ew.num_q_heads, ew.head_dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((total_q, ew.num_q_heads), dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # the step's host inputs in one buffer (one copy per step)
        ins = [(self, "q"), (self, "k_new"), (self, "v_new"), (self, "seq_lens"), (self, "slot_mapping"),
               (self, "qo_indptr"), (self, "req_pool_idx")]
        if self.kv_end is not None:
            self._seg_holder = _ProblemBuffers()
            for i, t in enumerate(self.seg):
                setattr(self._seg_holder, "s%d" % i, t)
            ins += [(self._seg_holder, "s%d" % i) for i in range(len(self.seg))]
        self.in_buf = _pack(ins, dev)
        if self.kv_end is not None:
            self.seg = [getattr(self._seg_holder, "s%d" % i) for i in range(len(self.seg))]
        if self.token_table:
            self.args = B.make_extend_args(B.PKV_LAYOUT_REQ_TO_TOKEN, self.q, self.k_pool, self.v_pool, self.out,
                                           self.qo_indptr, page_size=ps, sm_scale=ew.sm_scale,
                                           max_seq_len=int(ew.seq_lens.max()), kv_end=self.kv_end,
                                           seq_lens=self.seq_lens, req_to_token=self.r2t,
                                           req_pool_idx=self.req_pool_idx, lse=self.lse, kv_chunk=kv_chunk)
        else:
            self.args = B.make_extend_args(B.PKV_LAYOUT_CSR, self.q, self.k_pool, self.v_pool, self.out, self.qo_indptr,
                                           page_size=ps, sm_scale=ew.sm_scale, max_seq_len=int(ew.seq_lens.max()),
                                           kv_end=self.kv_end, kv_indptr=self.kv_indptr, kv_indices=self.kv_indices,
                                           kv_last_page_len=self.kv_last, lse=self.lse, kv_chunk=kv_chunk)
        self.ws_bytes = B.pkv_extend_workspace_size(self.args)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)

    def build_indices(self):
        if self.token_table:
            return                                   # pkv_extend reads req_to_token itself
        ew = self.ew
        B.pkv_build_indices(self.r2t, self.req_pool_idx, self.seq_lens, ew.page_size, ew.num_pool_pages, self.err,
                            kv_indptr=self.kv_indptr, kv_indices=self.kv_indices, kv_last_page_len=self.kv_last)

    def store(self):
        B.pkv_store(self.k_pool, self.v_pool, self.k_new, self.v_new, self.slot_mapping, self.err)

    def plan(self):
        if self.kv_end is not None:
            B.pkv_span_plan(*self.seg, self.plan_qo, self.q_pos, self.kv_end, self.err)

    def attend(self):
        B.pkv_extend(self.args, self.workspace, self.err)

    def run(self):
        self.build_indices()
        self.store()
        self.plan()
        self.attend()

    def launches_per_step(self) -> int:
        return (2 if self.token_table else 3) + (1 if self.kv_end is not None else 0) + (1 if self.ws_bytes > 0 else 0)

    def check_errors(self) -> int:
        return int(self.err.item())

    def host_step_tensors(self):
        """Pinned host copies of the step's packed inputs and of its output (for end-to-end timing)."""
        return {"inputs": self.in_buf.cpu().pin_memory()}, {"out": torch.empty_like(self.out, device="cpu").pin_memory()}

    def run_from_host(self, h_in, h_out):
        """One host-to-device copy of the step's inputs (q, new K/V rows, lengths, slots, query
        offsets, segments: packed in one buffer), the step, one copy of the output back."""
        self.in_buf.copy_(h_in["inputs"], non_blocking=True)
        self.run()
        h_out["out"].copy_(self.out, non_blocking=True)
