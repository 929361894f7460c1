"""CPU tests of the synthetic input recipe (workloads.py): the layouts every GPU test and
the bench draw from -- seeded and reproducible, block tables that give each sequence its
own distinct pool blocks, contexts and query lengths as each workload states them, bf16
values that are N(0,1) draws, and FP8 pools that are torch's e4m3 cast of value / scale."""
import math

import numpy as np

from pagedattention_paged_kv_gb300 import workloads as W


def _check_layout(b):
    ctx = b.context_lens.astype(np.int64)
    nblk = -(-ctx // b.block_size)
    used = []
    for s in range(b.num_seqs):
        row = b.block_tables[s]
        assert np.all(row[:nblk[s]] >= 0) and np.all(row[:nblk[s]] < b.num_blocks)
        assert np.all(row[nblk[s]:] == -1)
        used.extend(row[:nblk[s]].tolist())
    assert len(used) == len(set(used)), "a pool block is given to two sequences"
    ql = b.q_lens
    assert np.all(ql <= ctx)
    # the new tokens are each sequence's last q_len positions
    assert np.array_equal(b.new_token_seq, np.repeat(np.arange(b.num_seqs), ql))
    assert np.array_equal(b.new_token_pos, np.concatenate([np.arange(c - n, c) for c, n in zip(ctx, ql)]))
    assert b.q.shape == (int(ql.sum()), b.num_heads, b.head_dim)
    assert b.k_new.shape == b.v_new.shape == (int(ql.sum()), b.num_kv_heads, b.head_dim)
    assert math.isclose(b.scale, 1.0 / math.sqrt(b.head_dim))


def test_tiny_decode_recipe():
    b = W.tiny_decode()
    _check_layout(b)
    assert b.num_seqs == 4 and b.num_heads == b.num_kv_heads == 4 and b.head_dim == 64 and b.num_blocks == 64
    assert np.all((b.context_lens >= 1) & (b.context_lens <= 100))
    assert b.query_start_loc is None


def test_gqa_decode_recipe_and_headroom():
    b = W.gqa_decode(num_seqs=24)
    _check_layout(b)
    assert (b.num_heads, b.num_kv_heads, b.head_dim, b.block_size) == (64, 8, 128, 16)
    assert np.all((b.context_lens >= 500) & (b.context_lens <= 2500))
    need = int((-(-b.context_lens.astype(np.int64) // 16)).sum())
    assert b.num_blocks == math.ceil(1.1 * need)


def test_mixed_varlen_recipe():
    b = W.mixed_varlen(num_decodes=7)
    _check_layout(b)
    assert b.context_lens[0] == 16896 and b.q_lens[0] == 512 and np.all(b.q_lens[1:] == 1)
    assert np.array_equal(b.query_start_loc, np.concatenate([[0], np.cumsum(b.q_lens)]))
    assert b.new_token_pos[0] == 16384 and b.new_token_pos[511] == 16895 and b.causal


def test_same_seed_same_batch_and_other_seed_differs():
    a, b, c = W.tiny_decode(seed=7), W.tiny_decode(seed=7), W.tiny_decode(seed=8)
    for f in ("q", "k_cache", "v_cache", "block_tables", "context_lens", "k_new"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.q, c.q)


def test_values_are_bf16_normal_draws():
    b = W.gqa_decode(num_seqs=8)
    x = W.bf16_to_f32(b.k_cache[:64]).astype(np.float64).ravel()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    # bf16: the low 16 bits of the fp32 pattern are zero
    assert np.all((W.bf16_to_f32(b.q).view(np.uint32) & 0xFFFF) == 0)


def test_nan_fill_keeps_context_slots_finite():
    b = W.make_batch("nanfill", context_lens=[3, 17, 40], q_lens=[1, 1, 5], num_heads=4, num_kv_heads=2,
                     head_dim=16, seed=5, pool_fill="nan")
    _check_layout(b)
    kf = W.bf16_to_f32(b.k_cache)
    for s, c in enumerate(b.context_lens):
        for p in range(64):
            blk = b.block_tables[s, p // 16] if p // 16 < b.block_tables.shape[1] else -1
            if p < c:
                assert np.all(np.isfinite(kf[blk, p % 16]))
            elif blk >= 0:
                assert np.all(np.isnan(kf[blk, p % 16]))


def test_fp8_pool_is_the_e4m3_cast_of_value_over_scale():
    import torch
    b = W.tiny_decode()
    f = W.to_fp8_pool(b, k_scale=0.5, v_scale=0.25)
    k = torch.from_numpy(W.bf16_to_f32(b.k_cache) / np.float32(0.5)).to(torch.float8_e4m3fn).view(torch.uint8)
    v = torch.from_numpy(W.bf16_to_f32(b.v_cache) / np.float32(0.25)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(f.k_cache, k.numpy()) and np.array_equal(f.v_cache, v.numpy())
    assert f.meta["k_scale"] == 0.5 and f.meta["v_scale"] == 0.25 and f.meta["kv_dtype"] == "fp8_e4m3"
    assert np.array_equal(f.q, b.q) and np.array_equal(f.k_new, b.k_new)


def test_select_seqs_keeps_each_sequence_as_it_was():
    b = W.mixed_varlen(num_decodes=5)
    for seqs in ([0], [1, 2, 3, 4, 5], [3, 0]):
        s = W.select_seqs(b, seqs)
        assert s.num_seqs == len(seqs)
        assert np.array_equal(s.context_lens, b.context_lens[seqs])
        assert np.array_equal(s.block_tables, b.block_tables[seqs])
        assert np.array_equal(s.q_lens, b.q_lens[seqs])
        assert s.k_cache is b.k_cache and s.v_cache is b.v_cache
        for i, old in enumerate(seqs):
            rows = slice(b.query_start_loc[old], b.query_start_loc[old + 1])
            assert np.array_equal(s.q[s.query_start_loc[i]:s.query_start_loc[i + 1]], b.q[rows])
            assert np.array_equal(s.k_new[s.new_token_seq == i], b.k_new[b.new_token_seq == old])
            assert np.array_equal(s.new_token_pos[s.new_token_seq == i], b.new_token_pos[b.new_token_seq == old])
