"""GPU parity under preemption ("vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn)
§3.1 `_preempt`, §3.2 recovery by recomputation): the engine runs a request stream
against a pool of only 400 blocks, so decodes regularly fail to grow and their
sequences are preempted, freed, re-admitted later and recomputed (prompt plus the
tokens already produced, as one longer prefill) into whatever blocks are free then.

The oracle keeps its own copy of the pool and applies its own slot mapping and KV write
every iteration; on every iteration in which a preempted sequence recomputes, it checks
every output row of the batch.  At the end the GPU pool equals the oracle's bit for bit.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import bf16_bits_to_f64, bf16_to_np, compare
from pagedattention_paged_kv_gb300 import workloads as W
from pagedattention_paged_kv_gb300.scheduler import Sequence

pytestmark = pytest.mark.gpu

SEED = 5003
NB, HQ, HKV, D = 400, 64, 8, 128


def test_preempted_sequences_recompute_on_new_blocks():
    import pagedattention_paged_kv_gb300 as pkv
    from pagedattention_paged_kv_gb300.engine import PagedKVEngine
    orc = oracle.load()
    eng = PagedKVEngine(NB, HQ, HKV, D, max_num_seqs=32, chunk_size=512)
    host_k = np.zeros((NB, 16, HKV, D), np.uint16)
    host_v = np.zeros((NB, 16, HKV, D), np.uint16)
    reqs = W.request_stream(seed=SEED, iterations=60, rate=2.0, mean_prompt=300.0, std_prompt=100.0,
                            out_lo=50, out_hi=200)
    by_iter = {}
    for r in reqs:
        by_iter.setdefault(r.arrival, []).append(r)
    it = n_checked = n_rows = 0
    moved = 0  # recomputed sequences whose new blocks differ from the ones they held before
    last_table = {}
    while it < 60 or eng.sched.running or eng.sched.waiting:
        for r in by_iter.get(it, []):
            eng.add(Sequence(r.req_id, r.prompt_len, r.output_len, r.arrival))
        batch = eng.schedule()
        if batch.num_seqs:
            q, k, v = W.iteration_values(SEED, it, batch.num_tokens, HQ, HKV, D)
            out = eng.run(batch, q, k, v)
            slots = orc.slot_mapping(batch.block_tables, batch.token_seq, batch.token_pos, 16)
            orc.reshape_and_cache(host_k, host_v, k, v, slots)
            recompute = [x for x in batch.items if x.seq.preemptions > 0 and x.q_len > 1]
            for x in recompute:
                if x.start == 0 and last_table.get(x.seq.seq_id, x.seq.block_table) != x.seq.block_table:
                    moved += 1
            if recompute:
                ref = orc.paged_attention(q, host_k, host_v, batch.block_tables, batch.context_lens,
                                          eng.scale, query_start_loc=batch.query_start_loc, causal=True)
                compare(bf16_bits_to_f64(bf16_to_np(out)), ref)
                n_checked += 1
                n_rows += batch.num_tokens
            for x in batch.items:
                last_table[x.seq.seq_id] = list(x.seq.block_table)
        eng.complete(batch)
        it += 1
        assert it < 5000, "the stream does not drain"
    assert pkv.get_device_error() == 0
    assert eng.sched.total_preemptions >= 10, eng.sched.total_preemptions
    assert n_checked >= 10 and moved > 0
    assert len(eng.sched.done) == len(reqs) and eng.bm.num_free() == NB
    assert np.array_equal(bf16_to_np(eng.k_cache), host_k), "K pool differs from the oracle's"
    assert np.array_equal(bf16_to_np(eng.v_cache), host_v), "V pool differs from the oracle's"
    print(f"preemption: {eng.sched.total_preemptions} preemptions, {n_checked} recompute iterations "
          f"checked ({n_rows} rows), {moved} sequences recomputed on different blocks")
