"""One attention layer of a continuous-batching engine over a paged KV pool.

Each iteration: the scheduler (host) picks the batch; the host computes the slot
mapping; the step's metadata and new rows go to the device; the copies of shared blocks
that are about to be written (copy-on-write), the KV write and one varlen attention call
run on the GPU through the public API of this package.
"""
from __future__ import annotations

import numpy as np

from . import (BLOCK_SIZE, OP_VARLEN, BlockManager, copy_blocks, paged_attention_varlen,
               reshape_and_cache, slot_mapping, workspace_size)
from .scheduler import IterationBatch, Scheduler, Sequence


class PagedKVEngine:
    def __init__(self, num_blocks: int, num_heads: int, num_kv_heads: int, head_dim: int,
                 max_num_seqs: int = 128, chunk_size: int = 512, device="cuda",
                 max_num_batched_tokens: int | None = None, prefix_cache: bool = False):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        self.num_heads, self.num_kv_heads, self.head_dim = num_heads, num_kv_heads, head_dim
        self.scale = 1.0 / float(np.sqrt(head_dim))
        self.bm = BlockManager(num_blocks)
        self.sched = Scheduler(self.bm, max_num_seqs, chunk_size, BLOCK_SIZE, max_num_batched_tokens,
                               prefix_cache=prefix_cache)
        shape = (num_blocks, BLOCK_SIZE, num_kv_heads, head_dim)
        self.k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        self.v_cache = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
        self._ws = None

    def add(self, seq: Sequence) -> None:
        self.sched.add(seq)

    def schedule(self) -> IterationBatch:
        return self.sched.schedule()

    def complete(self, batch: IterationBatch) -> None:
        self.sched.complete(batch)

    def _workspace(self, num_seqs, total_q):
        n = workspace_size(OP_VARLEN, num_seqs, total_q, self.num_heads, self.num_kv_heads, self.head_dim)
        if self._ws is None or self._ws.numel() < n:
            self._ws = self.torch.empty(n, dtype=self.torch.uint8, device=self.device)
        return self._ws

    def run(self, batch: IterationBatch, q, k, v):
        """q [T, Hq, d], k/v [T, Hkv, d] (bf16 tensors on the device, or uint16 bf16 bit
        patterns on the host) for the batch's T new tokens; returns out [T, Hq, d]."""
        torch = self.torch
        if batch.num_seqs == 0:
            return None

        def dev_bf16(x):
            if isinstance(x, np.ndarray):
                return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(self.device).view(torch.bfloat16)
            return x
        q, k, v = dev_bf16(q), dev_bf16(k), dev_bf16(v)
        slots = slot_mapping(batch.block_tables, batch.token_seq, batch.token_pos, BLOCK_SIZE)
        meta = [torch.from_numpy(a).to(self.device, non_blocking=True)
                for a in (slots, batch.block_tables, batch.context_lens, batch.query_start_loc)]
        sm, bt, cl, qsl = meta
        if batch.copies.shape[0]:  # copy-on-write of shared blocks, before anything writes them
            copy_blocks(self.k_cache, self.v_cache, torch.from_numpy(batch.copies).to(self.device))
        reshape_and_cache(self.k_cache, self.v_cache, k, v, sm)
        out = torch.empty_like(q)
        paged_attention_varlen(out, q, qsl, self.k_cache, self.v_cache, bt, cl, self.scale, causal=True,
                               max_q_len=batch.max_q_len,
                               workspace=self._workspace(batch.num_seqs, batch.num_tokens))
        return out
