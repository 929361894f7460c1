"""Iteration-level (continuous-batching) scheduler over the paged KV pool (host).

Follows the loop that the pages print:

* "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış Prefill"
  (aiengineeringfromscratch.com, Phase 17 - 04), "What the scheduler looks like":
  every iteration (1) drops finished sequences and returns their blocks, (2) admits
  sequences from the head of the waiting queue while there are free blocks for them,
  (3) gives every running sequence either its next prefill chunk (up to 512 tokens,
  "Chunked prefill protects the TTFT tail") or one decode token, and (4) runs one
  fused forward over that batch.
* "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn) §3.1 Scheduler: admission
  allocates ceil(prompt_len / block_size) blocks (a failed allocation puts the
  sequence back at the head of the queue and stops admission); a running sequence that
  grows past its blocks gets one more block, and if none is free it is preempted:
  its blocks are freed, its computed tokens reset to 0 and it goes to the tail of the
  waiting queue (§3.2: recovery by recomputation, not swapping).

Readings where the pages leave a step open (see the design notes): a sequence finishes
when it has produced output_len tokens, one per decode step; the last prefill chunk
produces no token; a preempted sequence recomputes its prompt and the tokens it had
already produced as one longer prefill; the waiting queue is FIFO; running sequences
keep their admission order in the batch.

Token budget (the lesson's "Exercises": add --max-num-batched-tokens to the toy
scheduler).  When max_num_batched_tokens is set, an iteration schedules at most that
many new tokens: every running decode first (one token each, so a long prompt's chunk
never delays the decodes -- the inter-token latency that chunked prefill is there to
protect), then the prefilling sequences in admission order, each taking
min(chunk, tokens it still needs, budget left).  The budget must be at least
max_num_seqs, so the decodes always fit and, whenever a sequence is prefilling, at
least one token is left for it: every sequence keeps making progress.

Fragmentation report (the lesson's fragmentation exercise, measured instead of
computed): after every forward pass the scheduler records the slots its running
sequences hold in their blocks, the tokens whose K/V those slots store, and the slots
reserved for prompt tokens not yet computed; the rest is internal fragmentation, at
most block_size - 1 slots per sequence.  When a sequence finishes, the slots it held
and the tokens it stored are added to run-wide totals.
"""
from __future__ import annotations

import hashlib
from collections import OrderedDict
from dataclasses import dataclass, field

import numpy as np

from . import BLOCK_SIZE, BlockManager, OutOfBlocks


@dataclass
class Sequence:
    seq_id: int
    prompt_len: int
    output_len: int
    arrival: int = 0
    block_table: list = field(default_factory=list)
    prefill_target: int = 0   # tokens to (re)compute before decoding: prompt (+ output so far)
    computed: int = 0         # tokens whose K/V are in the cache
    decoded: int = 0          # output tokens produced
    preemptions: int = 0
    prompt_tokens: np.ndarray | None = None  # token ids (needed for prefix caching only)
    cached_tokens: int = 0    # prompt tokens whose K/V came from the prefix cache

    def __post_init__(self):
        if self.prefill_target == 0:
            self.prefill_target = self.prompt_len

    @property
    def in_prefill(self) -> bool:
        return self.computed < self.prefill_target

    @property
    def finished(self) -> bool:
        return self.decoded >= self.output_len


@dataclass
class ScheduledItem:
    seq: Sequence
    start: int       # first position written this iteration
    q_len: int       # tokens written and attended this iteration

    @property
    def context_len(self) -> int:
        return self.start + self.q_len


@dataclass
class IterationBatch:
    """The metadata of one fused attention call (host arrays)."""
    items: list
    query_start_loc: np.ndarray   # int32 [S+1]
    context_lens: np.ndarray      # int32 [S]
    block_tables: np.ndarray      # int32 [S, MB], unused entries -1
    token_seq: np.ndarray         # int32 [T] batch row of each new token
    token_pos: np.ndarray         # int32 [T] absolute position of each new token
    admitted: int = 0
    finished: int = 0
    preempted: int = 0
    copies: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int32))  # (src, dst) block copies to run first

    @property
    def num_seqs(self) -> int:
        return len(self.items)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1]) if len(self.query_start_loc) else 0

    @property
    def max_q_len(self) -> int:
        return max((it.q_len for it in self.items), default=0)


class PrefixCache:
    """Read-only reuse of a shared prompt prefix's KV blocks ("vLLM推理引擎架构PagedAttention
    机制与高吞吐推理" (lpnh.cn) §4.3: requests with the same system-prompt prefix reuse one
    set of read-only blocks, at the cost of prefix matching in the scheduler).

    Only full blocks are cached.  The key of prompt block i is a SHA-256 chain over the
    token ids of blocks 0..i, so equal keys mean equal prefixes (up to a hash collision).
    The cache holds one reference on every block it lists; blocks that only the cache still
    holds are evicted, least recently matched first, when the pool runs short.
    """

    def __init__(self, block_manager: BlockManager, block_size: int = BLOCK_SIZE):
        self.bm = block_manager
        self.block_size = int(block_size)
        self.blocks: OrderedDict[bytes, int] = OrderedDict()
        self.hits = 0      # blocks reused
        self.inserted = 0
        self.evicted = 0

    def _keys(self, tokens, n_blocks):
        h = b""
        bs = self.block_size
        for i in range(n_blocks):
            blk = np.ascontiguousarray(tokens[i * bs:(i + 1) * bs], dtype=np.int64).tobytes()
            h = hashlib.sha256(h + blk).digest()
            yield h

    def match(self, tokens, max_blocks: int) -> list:
        """Ids of the longest cached run of the prompt's first full blocks (<= max_blocks)."""
        ids = []
        for key in self._keys(tokens, max_blocks):
            b = self.blocks.get(key)
            if b is None:
                break
            self.blocks.move_to_end(key)
            ids.append(b)
        self.hits += len(ids)
        return ids

    def insert(self, tokens, block_table, n_full: int) -> None:
        """Lists the sequence's first n_full blocks (their K/V is computed); the cache takes
        a reference on each block it did not list yet."""
        for i, key in enumerate(self._keys(tokens, n_full)):
            if key not in self.blocks:
                b = block_table[i]
                self.bm.share([b])
                self.blocks[key] = b
                self.inserted += 1

    def evict(self, n: int) -> int:
        """Frees up to n blocks that only the cache holds; returns how many."""
        freed = 0
        for key in list(self.blocks):
            if freed >= n:
                break
            b = self.blocks[key]
            if self.bm.ref_count(b) == 1:
                del self.blocks[key]
                self.bm.free([b])
                freed += 1
        self.evicted += freed
        return freed


@dataclass
class FragmentationSample:
    """KV slot accounting of the running sequences after one forward pass."""
    iteration: int
    slots_held: int       # slots in the blocks the running sequences hold
    tokens_stored: int    # tokens whose K/V are in those slots
    tokens_reserved: int  # slots kept for prompt tokens not computed yet (chunked prefill)
    max_seq_wasted: int   # the largest number of wasted slots of one sequence

    @property
    def wasted(self) -> int:
        return self.slots_held - self.tokens_stored - self.tokens_reserved


class Scheduler:
    def __init__(self, block_manager: BlockManager, max_num_seqs: int = 128, chunk_size: int = 512,
                 block_size: int = BLOCK_SIZE, max_num_batched_tokens: int | None = None,
                 prefix_cache: bool = False):
        if max_num_batched_tokens is not None and max_num_batched_tokens < max_num_seqs:
            raise ValueError("max_num_batched_tokens must be >= max_num_seqs (every running decode "
                             "gets its token before any prefill chunk)")
        self.bm = block_manager
        self.cache = PrefixCache(block_manager, block_size) if prefix_cache else None
        self._copies: list = []
        self.max_num_seqs = int(max_num_seqs)
        self.chunk_size = int(chunk_size)
        self.block_size = int(block_size)
        self.max_num_batched_tokens = max_num_batched_tokens
        self.waiting: list[Sequence] = []
        self.running: list[Sequence] = []
        self.done: list[Sequence] = []
        self.iteration = 0
        self.total_preemptions = 0
        self.fragmentation: list[FragmentationSample] = []
        self.released_slots = 0    # slots held by finished sequences when they were released
        self.released_tokens = 0   # tokens those sequences had stored

    # -- queue -------------------------------------------------------------------
    def add(self, seq: Sequence) -> None:
        self.waiting.append(seq)

    def _blocks_for(self, tokens: int) -> int:
        return -(-tokens // self.block_size)

    def _allocate(self, n: int) -> list:
        """n fresh blocks, evicting cache-only blocks first if the pool is short."""
        if self.cache is not None and self.bm.num_free() < n:
            self.cache.evict(n - self.bm.num_free())
        return self.bm.allocate(n)

    def fork(self, parent: Sequence, seq_id: int, output_len: int) -> Sequence:
        """A new sequence that continues from parent's current state (e.g. another sample
        of the same prompt): it shares all of parent's blocks read-only; whichever of them
        first writes into a shared block gets a private copy (copy-on-write)."""
        child = Sequence(seq_id, parent.prompt_len, output_len, parent.arrival, list(parent.block_table),
                         parent.prefill_target, parent.computed, parent.decoded, 0, parent.prompt_tokens)
        self.bm.share(child.block_table)
        self.running.append(child)
        return child

    def _own_block(self, s: Sequence, pos: int) -> bool:
        """Makes the block holding position pos private to s before it is written."""
        i = pos // self.block_size
        if i >= len(s.block_table):
            return True
        b = s.block_table[i]
        if self.bm.ref_count(b) == 1:
            return True
        if self.cache is not None and self.bm.num_free() == 0:
            self.cache.evict(1)
        try:
            new, copied = self.bm.copy_on_write(b)
        except OutOfBlocks:
            return False
        if copied:
            self._copies.append((b, new))
            s.block_table[i] = new
        return True

    def _preempt(self, seq: Sequence) -> None:
        """Free everything the sequence holds; it recomputes its tokens later."""
        self.bm.free(seq.block_table)
        seq.block_table = []
        seq.prefill_target = seq.prompt_len + seq.decoded
        seq.computed = 0
        seq.cached_tokens = 0
        seq.preemptions += 1
        self.total_preemptions += 1
        self.waiting.append(seq)

    # -- one iteration -------------------------------------------------------------
    def schedule(self) -> IterationBatch:
        finished = preempted = admitted = 0
        # (1) release finished sequences
        keep = []
        for s in self.running:
            if s.finished:
                self.released_slots += len(s.block_table) * self.block_size
                self.released_tokens += s.computed
                self.bm.free(s.block_table)
                s.block_table = []
                self.done.append(s)
                finished += 1
            else:
                keep.append(s)
        self.running = keep
        # (2) growth: a decode step writing position p needs block p // block_size (and
        # needs it to itself: copy-on-write of a block shared by a fork)
        keep = []
        for s in self.running:
            if not s.in_prefill:
                pos = s.computed
                need = self._blocks_for(pos + 1) - len(s.block_table)
                try:
                    if need > 0:
                        s.block_table.extend(self._allocate(need))
                    elif not self._own_block(s, pos):
                        raise OutOfBlocks(-5, "copy_on_write")
                except OutOfBlocks:
                    self._preempt(s)
                    preempted += 1
                    continue
            keep.append(s)
        self.running = keep
        # (3) admission from the head of the waiting queue; with the prefix cache, the
        # longest cached run of the prompt's full blocks is shared instead of recomputed
        # (never the block of the prompt's last token, which must be computed)
        while self.waiting and len(self.running) < self.max_num_seqs:
            s = self.waiting[0]
            hit = []
            if self.cache is not None and s.prompt_tokens is not None:
                usable = min(s.prompt_len, s.prefill_target - 1) // self.block_size
                hit = self.cache.match(s.prompt_tokens, usable)
                self.bm.share(hit)
            try:
                fresh = self._allocate(self._blocks_for(s.prefill_target) - len(hit))
            except OutOfBlocks:
                if hit:
                    self.bm.free(hit)
                break
            s.block_table = hit + fresh
            s.computed = len(hit) * self.block_size
            s.cached_tokens = s.computed
            self.waiting.pop(0)
            self.running.append(s)
            admitted += 1
        # (4) one chunk or one decode token per running sequence; under a token budget the
        # decodes are served first, then the chunks in admission order
        budget = self.max_num_batched_tokens
        take = {}
        if budget is not None:
            for s in self.running:
                if not s.in_prefill:
                    take[id(s)] = 1
                    budget -= 1
            assert budget >= 0  # running <= max_num_seqs <= max_num_batched_tokens
        for s in self.running:
            if s.in_prefill:
                n = min(self.chunk_size, s.prefill_target - s.computed)
                if budget is not None:
                    n = min(n, budget)
                    budget -= n
                if n > 0:
                    take[id(s)] = n
            elif budget is None:
                take[id(s)] = 1
        items = [ScheduledItem(s, s.computed, take[id(s)]) for s in self.running if id(s) in take]
        self.iteration += 1
        batch = self._pack(items, admitted, finished, preempted)
        if self._copies:
            batch.copies = np.array(self._copies, dtype=np.int32).reshape(-1, 2)
            self._copies = []
        return batch

    def complete(self, batch: IterationBatch) -> None:
        """Account for the forward pass of `batch`: cache grows, decodes emit tokens; with
        the prefix cache, the prompt's newly completed full blocks become reusable."""
        for it in batch.items:
            s = it.seq
            was_decode = not s.in_prefill
            s.computed += it.q_len
            if was_decode:
                s.decoded += 1
            if self.cache is not None and s.prompt_tokens is not None and not was_decode:
                self.cache.insert(s.prompt_tokens, s.block_table, min(s.computed, s.prompt_len) // self.block_size)
        held = stored = reserved = worst = 0
        for s in self.running:
            h = len(s.block_table) * self.block_size
            r = max(0, s.prefill_target - s.computed)
            held += h
            stored += s.computed
            reserved += r
            worst = max(worst, h - s.computed - r)
        self.fragmentation.append(FragmentationSample(self.iteration, held, stored, reserved, worst))

    def _pack(self, items, admitted, finished, preempted) -> IterationBatch:
        S = len(items)
        q_lens = np.array([it.q_len for it in items], dtype=np.int32)
        qsl = np.zeros(S + 1, dtype=np.int32)
        if S:
            np.cumsum(q_lens, out=qsl[1:])
        ctx = np.array([it.context_len for it in items], dtype=np.int32)
        mb = max((len(it.seq.block_table) for it in items), default=1)
        tables = np.full((S, max(mb, 1)), -1, dtype=np.int32)
        for i, it in enumerate(items):
            tables[i, :len(it.seq.block_table)] = it.seq.block_table
        tok_seq = np.repeat(np.arange(S, dtype=np.int32), q_lens)
        tok_pos = (np.concatenate([np.arange(it.start, it.start + it.q_len, dtype=np.int32) for it in items])
                   if S else np.zeros(0, np.int32))
        return IterationBatch(items, qsl, ctx, tables, tok_seq, tok_pos, admitted, finished, preempted)

    # -- accounting ----------------------------------------------------------------
    def blocks_in_use(self) -> int:
        return sum(len(s.block_table) for s in self.running)

    def fragmentation_report(self) -> dict:
        """Internal fragmentation measured over the run: per iteration (mean and worst share
        of held slots that store nothing and are reserved for nothing) and at release
        (slots the finished sequences held minus the tokens they stored)."""
        per_iter = [f.wasted / f.slots_held for f in self.fragmentation if f.slots_held]
        return {
            "iterations": len(self.fragmentation),
            "mean_wasted_share": float(np.mean(per_iter)) if per_iter else 0.0,
            "max_wasted_share": float(np.max(per_iter)) if per_iter else 0.0,
            "max_wasted_slots_per_seq": max((f.max_seq_wasted for f in self.fragmentation), default=0),
            "released_slots": self.released_slots,
            "released_tokens": self.released_tokens,
            "released_wasted_share": (1.0 - self.released_tokens / self.released_slots)
            if self.released_slots else 0.0,
        }

    def slot_waste(self) -> list:
        """Per running sequence: slots its blocks hold beyond the tokens they are held
        for (the prompt still being prefilled, else the tokens in the cache).  Measured
        after complete(), each is at most block_size - 1."""
        return [len(s.block_table) * self.block_size - (s.prefill_target if s.in_prefill else s.computed)
                for s in self.running]
