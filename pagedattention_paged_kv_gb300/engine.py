"""One attention layer of a continuous-batching engine over a paged KV pool.

Each iteration: the scheduler (host) picks the batch; the host computes the slot
mapping; the step's metadata and new rows go to the device; the copies of shared blocks
that are about to be written (copy-on-write), the KV write and one varlen attention call
run on the GPU through the public API of this package.
"""
from __future__ import annotations

import numpy as np

from . import (BLOCK_SIZE, OP_VARLEN, BlockManager, attention_launches, copy_blocks,
               paged_attention_varlen, reshape_and_cache, slot_mapping, workspace_size)
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

    def prepare(self, batch: IterationBatch, q, k, v) -> dict:
        """Host part of an iteration: the slot mapping of the new tokens and the copies of the
        step's metadata (and of q/k/v given as host arrays) to the device.  q [T, Hq, d],
        k/v [T, Hkv, d]: bf16 tensors on the device, or uint16 bf16 bit patterns on the host."""
        torch = self.torch

        def dev_bf16(x):
            if isinstance(x, np.ndarray):
                return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(self.device).view(torch.bfloat16)
            return x
        slots = slot_mapping(batch.block_tables, batch.token_seq, batch.token_pos, BLOCK_SIZE)
        sm, bt, cl, qsl = [torch.from_numpy(a).to(self.device, non_blocking=True)
                           for a in (slots, batch.block_tables, batch.context_lens, batch.query_start_loc)]
        copies = torch.from_numpy(batch.copies).to(self.device) if batch.copies.shape[0] else None
        return {"q": dev_bf16(q), "k": dev_bf16(k), "v": dev_bf16(v), "slots": sm, "tables": bt,
                "lens": cl, "qsl": qsl, "copies": copies, "max_q_len": batch.max_q_len,
                "num_seqs": batch.num_seqs, "num_tokens": batch.num_tokens}

    def launch(self, p: dict):
        """Device part of an iteration (stream-ordered library calls only): copy-on-write
        block copies, the KV write and one varlen attention call; returns out [T, Hq, d]."""
        if p["copies"] is not None:  # copy-on-write of shared blocks, before anything writes them
            copy_blocks(self.k_cache, self.v_cache, p["copies"])
        reshape_and_cache(self.k_cache, self.v_cache, p["k"], p["v"], p["slots"])
        out = self.torch.empty_like(p["q"])
        paged_attention_varlen(out, p["q"], p["qsl"], self.k_cache, self.v_cache, p["tables"], p["lens"],
                               self.scale, causal=True, max_q_len=p["max_q_len"],
                               workspace=self._workspace(p["num_seqs"], p["num_tokens"]))
        return out

    def run(self, batch: IterationBatch, q, k, v):
        """One iteration: prepare() then launch(); returns out [T, Hq, d] (None for an empty batch)."""
        if batch.num_seqs == 0:
            return None
        return self.launch(self.prepare(batch, q, k, v))

    def launches(self, batch: IterationBatch) -> int:
        """Library kernels one iteration launches: block copies (if any), the KV write, the
        attention kernel and its merge(s)."""
        if batch.num_seqs == 0:
            return 0
        ql = np.diff(batch.query_start_loc)
        return (1 if batch.copies.shape[0] else 0) + 1 + attention_launches(int(ql.max()) if len(ql) else 0)
