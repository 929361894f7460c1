"""GPU parity over the continuous-batching trace: 300 iterations of the scheduler loop
(Poisson(4) arrivals per iteration, log-normal prompts with mean 1500 capped at 8192,
outputs uniform in [16, 512], at most 128 running, 512-token prefill chunks, a
65,536-block pool), each iteration running the KV write and one varlen attention call
through the library.

The oracle keeps its own host copy of the pool and applies its own slot mapping and
KV write every iteration; on a seeded subset of iterations it computes the attention
of every decode row and of sampled rows of every prefill chunk.  At the end the whole
GPU pool must equal the oracle's bit for bit.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import ATOL, RTOL, bf16_bits_to_f64, bf16_to_np, compare
from pagedattention_paged_kv_gb300 import workloads as W
from pagedattention_paged_kv_gb300.scheduler import Sequence

pytestmark = pytest.mark.gpu

SEED = 5001
NB, HQ, HKV, D = 65536, 64, 8, 128


def test_continuous_batching_trace():
    import torch
    from pagedattention_paged_kv_gb300.engine import PagedKVEngine
    orc = oracle.load()
    eng = PagedKVEngine(NB, HQ, HKV, D, max_num_seqs=128, chunk_size=512)
    host_k = np.zeros((NB, 16, HKV, D), np.uint16)
    host_v = np.zeros((NB, 16, HKV, D), np.uint16)
    reqs = W.request_stream(seed=SEED, iterations=300)
    by_iter = {}
    for r in reqs:
        by_iter.setdefault(r.arrival, []).append(r)
    rng = np.random.Generator(np.random.PCG64(SEED + 7))
    checked = set(rng.choice(300, size=40, replace=False).tolist())
    n_checked = n_chunk_rows = 0
    worst = 0.0
    for it in range(300):
        for r in by_iter.get(it, []):
            eng.add(Sequence(r.req_id, r.prompt_len, r.output_len, r.arrival))
        batch = eng.schedule()
        if batch.num_seqs == 0:
            eng.complete(batch)
            continue
        q, k, v = W.iteration_values(SEED, it, batch.num_tokens, HQ, HKV, D)
        out = eng.run(batch, q, k, v)
        slots = orc.slot_mapping(batch.block_tables, batch.token_seq, batch.token_pos, 16)
        orc.reshape_and_cache(host_k, host_v, k, v, slots)
        if it in checked:
            qsl = batch.query_start_loc
            mask = np.zeros(batch.num_tokens, np.uint8)
            for s in range(batch.num_seqs):
                n = qsl[s + 1] - qsl[s]
                if n == 1:
                    mask[qsl[s]] = 1
                else:  # first, last and 6 sampled rows of each chunk
                    pick = np.unique(np.r_[0, n - 1, rng.integers(0, n, size=6)])
                    mask[qsl[s] + pick] = 1
                    n_chunk_rows += len(pick)
            ref = orc.paged_attention(q, host_k, host_v, batch.block_tables, batch.context_lens,
                                      eng.scale, query_start_loc=qsl, causal=True, row_mask=mask)
            got = bf16_bits_to_f64(bf16_to_np(out))
            rows = np.nonzero(mask)[0]
            max_abs, _ = compare(got, ref, rows)
            worst = max(worst, max_abs)
            n_checked += 1
        eng.complete(batch)
    import pagedattention_paged_kv_gb300 as pkv
    assert pkv.get_device_error() == 0
    assert n_checked >= 30 and n_chunk_rows > 0
    assert np.array_equal(bf16_to_np(eng.k_cache), host_k), "K pool differs from the oracle's"
    assert np.array_equal(bf16_to_np(eng.v_cache), host_v), "V pool differs from the oracle's"
    print(f"trace: {n_checked} iterations checked, {n_chunk_rows} chunk rows, max_abs {worst:.3g}")
