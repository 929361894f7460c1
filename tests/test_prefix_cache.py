"""Host logic of shared prefix blocks ("vLLM推理引擎架构PagedAttention机制与高吞吐推理"
(lpnh.cn) §4.3): reference counts in the C++ block manager, the scheduler's prefix cache
and copy-on-write after a fork.  CPU only (the block manager is host code)."""
import numpy as np
import pytest

import pagedattention_paged_kv_gb300 as pkv
from pagedattention_paged_kv_gb300 import workloads as W
from pagedattention_paged_kv_gb300.scheduler import Scheduler, Sequence


def _seq(i, tokens, out=4):
    return Sequence(i, len(tokens), out, 0, prompt_tokens=np.asarray(tokens, np.int64))


def _run_prefill(sched):
    """Schedules and completes iterations until nothing is in prefill."""
    for _ in range(100):
        b = sched.schedule()
        sched.complete(b)
        if not any(s.in_prefill for s in sched.running) and not sched.waiting:
            return b
    raise AssertionError("prefill did not finish")


def _held_refs(sched):
    """References the sequences and the cache hold on every block."""
    refs = np.zeros(sched.bm.num_blocks, np.int64)
    for s in sched.running:
        for b in s.block_table:
            refs[b] += 1
    if sched.cache is not None:
        for b in sched.cache.blocks.values():
            refs[b] += 1
    return refs


def _check_counts(sched):
    refs = _held_refs(sched)
    for b in range(sched.bm.num_blocks):
        assert sched.bm.ref_count(b) == refs[b], b
    assert sched.bm.num_free() == int((refs == 0).sum())


def test_block_manager_reference_counts():
    bm = pkv.BlockManager(8)
    a = bm.allocate(3)
    bm.share([a[0], a[0], a[1]])
    assert [bm.ref_count(b) for b in a] == [3, 2, 1]
    bm.free([a[0]])
    assert bm.ref_count(a[0]) == 2 and bm.num_free() == 5
    with pytest.raises(pkv.PagedKVError):
        bm.free([a[2], a[2]])          # held once, listed twice: nothing changes
    assert bm.ref_count(a[2]) == 1
    with pytest.raises(pkv.PagedKVError):
        bm.share([7])                  # not held
    bm.free([a[0], a[0], a[1], a[1], a[2]])
    assert bm.num_free() == 8


def test_copy_on_write_moves_the_writers_reference():
    bm = pkv.BlockManager(4)
    (b,) = bm.allocate(1)
    assert bm.copy_on_write(b) == (b, False)     # sole holder writes in place
    bm.share([b])
    new, copied = bm.copy_on_write(b)
    assert copied and new != b and bm.ref_count(b) == 1 and bm.ref_count(new) == 1
    bm.share([b])
    bm.allocate(bm.num_free())
    with pytest.raises(pkv.OutOfBlocks):
        bm.copy_on_write(b)
    assert bm.ref_count(b) == 2


def test_second_request_reuses_the_shared_prefix():
    rng = np.random.Generator(np.random.PCG64(1))
    system = rng.integers(0, 1000, size=40)
    sched = Scheduler(pkv.BlockManager(64), prefix_cache=True)
    s0 = _seq(0, np.r_[system, rng.integers(0, 1000, size=7)])
    sched.add(s0)
    _run_prefill(sched)
    assert s0.cached_tokens == 0
    s1 = _seq(1, np.r_[system, rng.integers(0, 1000, size=20)])
    sched.add(s1)
    b = sched.schedule()
    assert s1.cached_tokens == 32                      # two full blocks of the 40-token prompt
    assert s1.block_table[:2] == s0.block_table[:2]
    assert all(sched.bm.ref_count(x) == 3 for x in s1.block_table[:2])  # cache + 2 sequences
    item = [it for it in b.items if it.seq is s1][0]
    assert item.start == 32 and item.q_len == len(s1.prompt_tokens) - 32
    sched.complete(b)
    _check_counts(sched)


def test_fully_cached_prompt_still_computes_its_last_block():
    tokens = np.arange(48)
    sched = Scheduler(pkv.BlockManager(32), prefix_cache=True)
    sched.add(_seq(0, tokens))
    _run_prefill(sched)
    s1 = _seq(1, tokens)
    sched.add(s1)
    b = sched.schedule()
    assert s1.cached_tokens == 32                       # blocks 0, 1; block 2 holds the last token
    assert [it.q_len for it in b.items if it.seq is s1] == [16]
    sched.complete(b)
    _check_counts(sched)


def test_cache_only_blocks_are_evicted_before_allocation_fails():
    sched = Scheduler(pkv.BlockManager(12), prefix_cache=True, max_num_seqs=4)
    rng = np.random.Generator(np.random.PCG64(3))
    sched.add(_seq(0, rng.integers(0, 1000, size=64), out=1))
    _run_prefill(sched)
    for _ in range(3):                                 # finish it: its blocks stay cached
        sched.complete(sched.schedule())
    assert not sched.running and len(sched.cache.blocks) == 4
    assert sched.bm.num_free() == 8
    sched.add(_seq(1, rng.integers(0, 1000, size=150), out=1))  # needs 10 blocks
    sched.complete(sched.schedule())
    assert sched.cache.evicted == 2 and sched.running
    _check_counts(sched)


def test_fork_shares_blocks_and_copies_the_partial_one_on_write():
    sched = Scheduler(pkv.BlockManager(16), prefix_cache=False)
    p = Sequence(0, 20, 6, 0)
    sched.add(p)
    _run_prefill(sched)                                # 20 tokens: block 1 is partial
    c = sched.fork(p, 1, 6)
    assert c.block_table == p.block_table
    assert all(sched.bm.ref_count(x) == 2 for x in p.block_table)
    shared = p.block_table[1]
    b = sched.schedule()                               # both decode into the shared partial block
    assert b.copies.shape == (1, 2)                    # the first writer copies, the second writes in place
    src, dst = b.copies[0]
    assert src == shared and dst != shared
    assert {p.block_table[1], c.block_table[1]} == {int(src), int(dst)}
    assert sched.bm.ref_count(src) == 1 and sched.bm.ref_count(dst) == 1
    assert p.block_table[0] == c.block_table[0]        # the full block stays shared
    sched.complete(b)
    _check_counts(sched)
    b2 = sched.schedule()
    assert b2.copies.shape == (0, 2)


def test_shared_prefix_stream_accounting_over_many_iterations():
    reqs = W.request_stream_shared_prefix(seed=7, iterations=60, rate=2.0)
    sched = Scheduler(pkv.BlockManager(2000), prefix_cache=True, max_num_seqs=32)
    by = {}
    for r in reqs:
        by.setdefault(r.arrival, []).append(r)
    reused = 0
    for it in range(60):
        for r in by.get(it, []):
            sched.add(_seq(r.req_id, r.tokens, out=r.output_len))
        b = sched.schedule()
        for s in sched.running:
            assert s.cached_tokens % 16 == 0 and s.cached_tokens < s.prompt_len
        sched.complete(b)
        _check_counts(sched)
    reused = sched.cache.hits
    assert reused > 50
