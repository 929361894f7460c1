"""GPU parity with shared read-only prefix blocks and copy-on-write
("vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn) §4.3): the block copy bit for
bit, attention over block tables that alias the same physical blocks, and a
continuous-batching run with the prefix cache and forked sequences against the oracle."""
import numpy as np
import pytest

import oracle
import pagedattention_paged_kv_gb300 as pkv
from gpu_helpers import bf16_bits_to_f64, bf16_to_np, compare, torch_bf16, torch_u8
from pagedattention_paged_kv_gb300 import workloads as W
from pagedattention_paged_kv_gb300.scheduler import Sequence

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp8", [False, True])
def test_copy_blocks_bit_exact(fp8):
    import torch
    rng = np.random.Generator(np.random.PCG64(61))
    NB, bs, Hkv, d = 40, 16, 8, 128
    if fp8:
        kc0 = rng.integers(0, 256, size=(NB, bs, Hkv, d), dtype=np.uint8)
        vc0 = rng.integers(0, 256, size=(NB, bs, Hkv, d), dtype=np.uint8)
        kc, vc = torch_u8(kc0), torch_u8(vc0)
    else:
        kc0, vc0 = W.normal_bf16(rng, (NB, bs, Hkv, d)), W.normal_bf16(rng, (NB, bs, Hkv, d))
        kc, vc = torch_bf16(kc0), torch_bf16(vc0)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int32)  # dsts distinct from srcs
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    rk, rv = kc0.copy(), vc0.copy()
    oracle.load().copy_blocks(rk, rv, pairs)
    got_k = kc.cpu().numpy() if fp8 else bf16_to_np(kc)
    got_v = vc.cpu().numpy() if fp8 else bf16_to_np(vc)
    assert pkv.get_device_error() == 0
    assert np.array_equal(got_k, rk) and np.array_equal(got_v, rv)


def test_copy_blocks_flags_ids_outside_the_pool():
    import torch
    NB = 4
    kc = torch.zeros(NB, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pkv.copy_blocks(kc, vc, torch.tensor([[0, NB]], dtype=torch.int32, device="cuda"))
    assert pkv.get_device_error() == 0x2


def test_attention_over_aliased_prefix_blocks():
    """Decode and varlen rows of sequences whose tables share their first blocks."""
    import torch
    rng = np.random.Generator(np.random.PCG64(62))
    NB, bs, Hq, Hkv, d = 64, 16, 64, 8, 128
    kc0, vc0 = W.normal_bf16(rng, (NB, bs, Hkv, d)), W.normal_bf16(rng, (NB, bs, Hkv, d))
    shared = [5, 17, 40, 2]
    tables = np.full((4, 8), -1, np.int32)
    tables[0, :6] = shared + [9, 10]
    tables[1, :5] = shared + [11]
    tables[2, :4] = shared
    tables[3, :7] = shared[:2] + [20, 21, 22, 23, 24]
    ctx = np.array([90, 70, 64, 100], np.int32)
    qsl = np.array([0, 1, 2, 34, 35], np.int32)   # sequence 2 is a 32-row chunk
    q = W.normal_bf16(rng, (35, Hq, d))
    out = torch.empty(35, Hq, d, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_varlen(out, torch_bf16(q), torch.from_numpy(qsl).cuda(), torch_bf16(kc0), torch_bf16(vc0),
                               torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), 1 / np.sqrt(d))
    ref = oracle.load().paged_attention(q, kc0, vc0, tables, ctx, 1 / np.sqrt(d), query_start_loc=qsl)
    assert pkv.get_device_error() == 0
    compare(bf16_bits_to_f64(bf16_to_np(out)), ref)


def test_prefix_cache_and_forks_over_a_shared_prompt_stream():
    """120 scheduler iterations over requests that share three system prompts, with the
    prefix cache on and every third request forked once its prompt is in the cache;
    the oracle mirrors the pool (block copies, KV writes) and checks the decode rows and
    sampled chunk rows of 20 seeded iterations and of every iteration that copies a block;
    the pools must match bit for bit at the end."""
    from pagedattention_paged_kv_gb300.engine import PagedKVEngine
    orc = oracle.load()
    NB, HQ, HKV, D, SEED = 4096, 64, 8, 128, 6001
    eng = PagedKVEngine(NB, HQ, HKV, D, max_num_seqs=64, chunk_size=512, prefix_cache=True)
    host_k = np.zeros((NB, 16, HKV, D), np.uint16)
    host_v = np.zeros((NB, 16, HKV, D), np.uint16)
    reqs = W.request_stream_shared_prefix(seed=SEED, iterations=120, rate=2.0)
    by_iter = {}
    for r in reqs:
        by_iter.setdefault(r.arrival, []).append(r)
    rng = np.random.Generator(np.random.PCG64(SEED + 1))
    check_at = set(rng.choice(120, size=20, replace=False).tolist())
    next_id, forked, n_copies, checked = 10 ** 6, set(), 0, 0
    for it in range(120):
        for r in by_iter.get(it, []):
            eng.add(Sequence(r.req_id, r.prompt_len, r.output_len, r.arrival, prompt_tokens=r.tokens))
        for s in list(eng.sched.running):
            if s.seq_id % 3 == 0 and s.seq_id not in forked and not s.in_prefill and s.decoded == 0:
                eng.sched.fork(s, next_id, s.output_len)
                forked.add(s.seq_id)
                next_id += 1
        batch = eng.schedule()
        if batch.num_seqs == 0:
            eng.complete(batch)
            continue
        q, k, v = W.iteration_values(SEED, it, batch.num_tokens, HQ, HKV, D)
        out = eng.run(batch, q, k, v)
        if batch.copies.shape[0]:
            orc.copy_blocks(host_k, host_v, batch.copies)
            n_copies += batch.copies.shape[0]
        slots = orc.slot_mapping(batch.block_tables, batch.token_seq, batch.token_pos, 16)
        orc.reshape_and_cache(host_k, host_v, k, v, slots)
        if it in check_at or batch.copies.shape[0]:
            qsl = batch.query_start_loc
            mask = np.zeros(batch.num_tokens, np.uint8)
            for s in range(batch.num_seqs):
                n = qsl[s + 1] - qsl[s]
                pick = [0] if n == 1 else np.unique(np.r_[0, n - 1, rng.integers(0, n, size=3)])
                mask[qsl[s] + np.asarray(pick)] = 1
            ref = orc.paged_attention(q, host_k, host_v, batch.block_tables, batch.context_lens, eng.scale,
                                      query_start_loc=qsl, causal=True, row_mask=mask)
            compare(bf16_bits_to_f64(bf16_to_np(out)), ref, np.nonzero(mask)[0])
            checked += 1
        eng.complete(batch)
    assert pkv.get_device_error() == 0
    assert eng.sched.cache.hits > 100 and n_copies > 0 and checked >= 20
    assert np.array_equal(bf16_to_np(eng.k_cache), host_k), "K pool differs from the oracle's"
    assert np.array_equal(bf16_to_np(eng.v_cache), host_v), "V pool differs from the oracle's"
