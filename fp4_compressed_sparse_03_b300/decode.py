"""Device-resident paged cache and a decode step over a static CSA2 mode schedule.

Thin host-side orchestration of the C ABI (tech-report digest, jiwasawa.github.io,
section "Compressed Sparse Attention 2 (CSA2)": each layer is statically Full,
Reindex or Reuse; the first Full layer of a group picks the candidate pool that the
group's Reindex layers search).  torch only allocates device memory; every step is
a libcsa2 kernel.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import (CSA2_FULL, CSA2_REINDEX, CSA2_REUSE, D_IDX, D_KV, H_IDX, H_Q, PAGE, check,
               csa2_attn_workspace_size, csa2_index, csa2_index_workspace_size,
               csa2_sparse_attn, csa2_sparse_attn_mx, make_index_args, make_pages)


class DecodeCache:
    """Paged FP4 latent (codes + E4M3 scales per 16 channels, or E8M0 scales per 32 for
    the MXFP4 variant) and bf16 indexer keys of `n_groups` Full-layer groups, sharing one
    page table."""

    def __init__(self, seq_lens, page_table, num_pages: int, n_groups: int = 1, device="cuda",
                 mx: bool = False):
        self.device = torch.device(device)
        self.seq_lens = torch.as_tensor(np.asarray(seq_lens, np.int32), device=self.device)
        self.page_table = torch.as_tensor(np.asarray(page_table, np.int32), device=self.device)
        self.num_pages = int(num_pages)
        self.n_groups = int(n_groups)
        self.mx = bool(mx)
        slots = self.num_pages * PAGE
        self.codes = torch.zeros((n_groups, slots, D_KV // 2), dtype=torch.uint8, device=self.device)
        self.scales = torch.zeros((n_groups, slots, D_KV // (32 if mx else 16)), dtype=torch.uint8,
                                  device=self.device)
        self.keys = torch.zeros((n_groups, slots, D_IDX), dtype=torch.int16, device=self.device)
        self.pages = make_pages(self.seq_lens, self.page_table, self.num_pages)

    @property
    def num_slots(self) -> int:
        return self.num_pages * PAGE

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])


class DecodeStep:
    """One decode step of `len(schedule)` layers for a batch of query tokens."""

    def __init__(self, cache: DecodeCache, q_seq, schedule, pool_size: int, topk: int,
                 max_q_per_seq: int = 1, softmax_scale: float | None = None):
        self.cache = cache
        dev = cache.device
        self.schedule = list(schedule)
        self.q_seq = torch.as_tensor(np.asarray(q_seq, np.int32), device=dev)
        self.num_q = int(self.q_seq.numel())
        self.pool_size = int(pool_size)
        self.topk = int(topk)
        self.max_q_per_seq = int(max_q_per_seq)
        self.softmax_scale = float(np.float32(1.0 / math.sqrt(D_KV))) if softmax_scale is None \
            else float(softmax_scale)
        L = len(self.schedule)
        # group of each layer and the layer whose indices it uses
        self.group, self.src = [], []
        g, s = -1, -1
        for l, m in enumerate(self.schedule):
            if m == CSA2_FULL:
                g += 1
            if m in (CSA2_FULL, CSA2_REINDEX):
                s = l
            if g < 0 or s < 0:
                raise ValueError("a schedule must start with a Full layer")
            self.group.append(g)
            self.src.append(s)
        if g + 1 > cache.n_groups:
            raise ValueError("schedule has more Full groups than the cache")
        self.idx = torch.full((L, self.num_q, self.topk), -1, dtype=torch.int32, device=dev)
        self.pool = torch.full((max(g + 1, 1), self.num_q, max(self.pool_size, 1)), -1,
                               dtype=torch.int32, device=dev)
        self.out = torch.zeros((L, self.num_q, H_Q, D_KV), dtype=torch.float32, device=dev)
        self.lse = torch.zeros((L, self.num_q, H_Q), dtype=torch.float32, device=dev)
        ws = max(csa2_index_workspace_size(CSA2_FULL, self.num_q, cache.max_pages, self.pool_size),
                 csa2_index_workspace_size(CSA2_REINDEX, self.num_q, cache.max_pages, self.pool_size),
                 csa2_attn_workspace_size(self.num_q, self.topk), 256)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        # the parallel schedule (run_parallel) gives each attention branch its own workspace
        self.attn_branches = min(L, self.ATTN_BRANCHES)
        ws_a = max(csa2_attn_workspace_size(self.num_q, self.topk), 256)
        self.attn_workspace = [torch.empty(ws_a, dtype=torch.uint8, device=dev)
                               for _ in range(self.attn_branches)]
        self._branches = [torch.cuda.Stream(dev) for _ in range(self.attn_branches)]
        # With several Full groups the index calls gate the later groups' attention, so they
        # run on a stream of higher priority (ragged, 20 layers: 7.71 -> 7.59 ms per step);
        # with one group the caller's stream serves (the decode batch measured 0.3 % slower
        # with the extra stream)
        groups = sum(1 for m in self.schedule if m == CSA2_FULL)
        self._index_stream = torch.cuda.Stream(dev, priority=-1) if groups > 1 else None
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.use_pool = self.pool_size > 0 and any(m == CSA2_REINDEX for m in self.schedule)

    def layer_index(self, l: int, q_idx_l, stream=None) -> None:
        m, g = self.schedule[l], self.group[l]
        c = self.cache
        if m == CSA2_REUSE:
            return  # the attention reads the source layer's indices in place
        args = make_index_args(self.num_q, self.q_seq, self.max_q_per_seq, self.pool_size,
                               None, self.workspace, None, self.dev_status)
        pool = self.pool[g] if (self.use_pool or m == CSA2_REINDEX) else None
        check(csa2_index(m, q_idx_l, c.keys[g], pool, self.topk, self.idx[l], c.pages, args,
                         stream), f"csa2_index(layer {l})")

    def layer_attn(self, l: int, q_l, stream=None, workspace=None) -> None:
        g, s = self.group[l], self.src[l]
        c = self.cache
        attn = csa2_sparse_attn_mx if c.mx else csa2_sparse_attn
        ws = self.workspace if workspace is None else workspace
        check(attn(q_l, c.codes[g], c.scales[g], self.idx[s], c.pages, self.out[l], self.lse[l],
                   self.num_q, self.q_seq, self.topk, self.softmax_scale, ws, None,
                   self.dev_status, stream),
              f"csa2_sparse_attn(layer {l})")

    def run(self, q_idx, q, stream=None) -> None:
        """q_idx: bf16 bits [L, num_q, 4, 128]; q: bf16 bits [L, num_q, 16, 512] (device)."""
        for l in range(len(self.schedule)):
            self.layer_index(l, q_idx[l], stream)
            self.layer_attn(l, q[l], stream)

    def indices(self, l: int):
        return self.idx[self.src[l]]

    # ---- parallel schedule: independent calls on separate streams ----
    # A layer's attention needs only its source layer's indices, and no index call reads
    # an attention's output, so the index calls run in order on one stream (the caller's,
    # or a high-priority one with several Full groups) while the attention calls run on
    # ATTN_BRANCHES side streams (layer l on branch l % B, each branch with its own
    # workspace), each waiting for the event recorded after its source layer's index call.
    # The caller's stream waits for every stream at the end.  The results are those of
    # run(): the same calls on the same buffers.
    ATTN_BRANCHES = 4

    def run_parallel(self, q_idx, q) -> None:
        main = torch.cuda.current_stream(self.cache.device)
        ix = self._index_stream if self._index_stream is not None else main
        start = torch.cuda.Event()
        start.record(main)
        if ix is not main:
            ix.wait_event(start)
        for b in self._branches:
            b.wait_event(start)
        done = {}
        for l, m in enumerate(self.schedule):
            if m != CSA2_REUSE:
                self.layer_index(l, q_idx[l], ix)
                ev = torch.cuda.Event()
                ev.record(ix)
                done[l] = ev
            br = self._branches[l % self.attn_branches]
            br.wait_event(done[self.src[l]])
            with torch.cuda.stream(br):
                self.layer_attn(l, q[l], br, self.attn_workspace[l % self.attn_branches])
        for b in ([ix] if ix is not main else []) + self._branches:
            ev = torch.cuda.Event()
            ev.record(b)
            main.wait_event(ev)

    # ---- CUDA graphs: the same libcsa2 launches, replayed without per-call host work ----
    # Every libcsa2 call is an ordered launch sequence on the given stream, so a captured
    # step replays exactly the kernels of an eager step on the same buffers.  Run the step
    # eagerly once before capturing (first calls set kernel attributes).

    @staticmethod
    def _capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            fn()
        return g

    def capture(self, q_idx, q, parallel: bool = False):
        """Graph of one whole step reading the device buffers q_idx and q; with `parallel`,
        of the parallel schedule (run_parallel)."""
        if parallel:
            return self._capture(lambda: self.run_parallel(q_idx, q))
        return self._capture(lambda: self.run(q_idx, q))

    def capture_calls(self, q_idx, q):
        """Per-call graphs: {(layer, "index")} for index-producing layers and
        {(layer, "attn")} for every layer."""
        graphs = {}
        for l, m in enumerate(self.schedule):
            if m != CSA2_REUSE:
                graphs[(l, "index")] = self._capture(lambda l=l: self.layer_index(l, q_idx[l]))
            graphs[(l, "attn")] = self._capture(lambda l=l: self.layer_attn(l, q[l]))
        return graphs
