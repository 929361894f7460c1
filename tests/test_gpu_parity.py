"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

KV writes must match bit for bit over the whole pool; bf16 attention outputs must
satisfy |gpu - ref| <= 1e-2 + 2e-2 |ref| element-wise (gpu_helpers.ATOL/RTOL).
"""
import math

import numpy as np
import pytest

from gpu_helpers import compare, gpu_step, oracle_step
import pagedattention_paged_kv_gb300 as pkv
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check_step(b, row_mask=None):
    out, kc, vc, err = gpu_step(b)
    ref, rkc, rvc = oracle_step(b, row_mask=row_mask)
    assert err == 0, f"device error flags {err:#x}"
    assert np.array_equal(kc, rkc), "k_cache differs from the oracle's KV write"
    assert np.array_equal(vc, rvc), "v_cache differs from the oracle's KV write"
    rows = None if row_mask is None else np.nonzero(row_mask)[0]
    return compare(out, ref, rows)


# ---- the five workloads' step shapes ------------------------------------------------

def test_tiny_decode():
    _check_step(W.tiny_decode())


def test_gqa_decode_full_size():
    _check_step(W.gqa_decode())


def test_skewed_long_context_decode():
    _check_step(W.skewed_decode())


def test_mixed_varlen_full_size_every_row():
    # workload 4 in one varlen call: the 512-row chunk behind its 16,384-token prefix and the
    # 127 decodes, every output row against the oracle (decode and prefill CTAs of one launch)
    _check_step(W.mixed_varlen())


@pytest.mark.parametrize("chunk_len,chunk_start,num_decodes", [
    (16, 0, 127),        # almost all decode work: the grid gives the chunk one or a few CTAs
    (512, 16384, 1),     # almost all prefill work: one decode CTA
    (512, 4096, 300),    # more sequences than SMs, both sides split
])
def test_mixed_varlen_split_extremes(chunk_len, chunk_start, num_decodes):
    b = W.mixed_varlen(seed=4100 + num_decodes, chunk_start=chunk_start, chunk_len=chunk_len,
                       num_decodes=num_decodes)
    _check_step(b)


# ---- shapes and edge cases ----------------------------------------------------------

@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 64), (8, 1, 128), (32, 8, 128), (16, 2, 64),
                                      (64, 8, 128), (40, 8, 128), (24, 8, 64), (64, 1, 128)])
def test_decode_head_layouts(Hq, Hkv, d):
    ctx = [1, 2, 15, 16, 17, 31, 33, 100, 257, 1000]
    b = W.make_batch("heads", context_lens=ctx, q_lens=np.ones(len(ctx), np.int64), num_heads=Hq,
                     num_kv_heads=Hkv, head_dim=d, seed=7 + Hq + Hkv + d)
    _check_step(b)


def test_decode_empty_contexts_give_zero_rows():
    b = W.make_batch("empty", context_lens=[0, 5, 0, 40], q_lens=[0, 1, 0, 1], num_heads=8,
                     num_kv_heads=2, head_dim=128, seed=3, varlen=False)
    # decode rows for empty sequences still exist in q/out (idle batch slots)
    b.q = W.normal_bf16(np.random.Generator(np.random.PCG64(4)), (4, 8, 128))
    out, kc, vc, err = gpu_step(b)
    ref, _, _ = oracle_step(b)
    assert err == 0
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    compare(out, ref)


def test_unused_slots_are_never_read():
    # Every slot outside a context holds bf16 NaN; a kernel that let one into a
    # score or a weighted sum would produce NaN.
    ctx = [1, 7, 16, 17, 45, 300]
    b = W.make_batch("nanpool", context_lens=ctx, q_lens=np.ones(len(ctx), np.int64), num_heads=16,
                     num_kv_heads=4, head_dim=128, seed=5, pool_fill="nan")
    _check_step(b)


def test_block_permutation_gives_identical_bits():
    b = W.gqa_decode(seed=99, num_seqs=24)
    out1, _, _, _ = gpu_step(b)
    rng = np.random.Generator(np.random.PCG64(100))
    perm = rng.permutation(b.num_blocks)
    kc2, vc2 = np.empty_like(b.k_cache), np.empty_like(b.v_cache)
    kc2[perm], vc2[perm] = b.k_cache, b.v_cache
    b.k_cache, b.v_cache = kc2, vc2
    b.block_tables = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    out2, _, _, _ = gpu_step(b)
    assert np.array_equal(out1, out2)


def test_context_len_one_returns_v_exactly():
    b = W.make_batch("one", context_lens=[1] * 5, q_lens=[1] * 5, num_heads=64, num_kv_heads=8,
                     head_dim=128, seed=11)
    out, _, vc, err = gpu_step(b)
    assert err == 0
    for s in range(5):
        blk = b.block_tables[s, 0]
        v_row = ((vc[blk, 0].astype(np.uint32) << 16).view(np.float32)).astype(np.float64)  # [Hkv, d]
        assert np.array_equal(out[s], np.repeat(v_row, 8, axis=0))


@pytest.mark.parametrize("q_lens,ctx", [
    ([2, 1, 17, 1, 100], [2, 30, 17, 1, 500]),           # whole prompts and decodes
    ([512, 1, 1, 33], [16896, 600, 1, 1000]),            # a chunk with a long prefix
    ([16, 15, 48, 1], [16, 40, 1100, 2]),                # tile-aligned and ragged chunks
    ([5, 300], [5, 300]),                                 # first chunks of prompts
])
def test_varlen_chunks_and_decodes(q_lens, ctx):
    b = W.make_batch("varlen", context_lens=ctx, q_lens=q_lens, num_heads=64, num_kv_heads=8,
                     head_dim=128, seed=sum(q_lens), varlen=True)
    _check_step(b)


def _boost_keys(b, seq, lo, hi, factor):
    """Multiplies the cached K rows of positions [lo, hi) of sequence `seq` by `factor`
    (in the pool, through the block table), so the scores against them jump."""
    for pos in range(lo, hi):
        blk, off = b.block_tables[seq, pos // b.block_size], pos % b.block_size
        b.k_cache[blk, off] = W.bf16_bits(W.bf16_to_f32(b.k_cache[blk, off]) * np.float32(factor))


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("factor", [6.0, 40.0])
def test_prefill_score_jumps(factor, fp8):
    # Keys 900..1000 of a 1500-token context score far above the ones before them: x6 moves
    # the rows' reference maximum by ~10-25 (log2 units), x40 by far more, so the chunked
    # prefill takes both its deferred reference move and its exact recomputation of a chunk.
    b = W.make_batch("jumps", context_lens=[1500, 700, 1200], q_lens=[300, 1, 64], num_heads=64,
                     num_kv_heads=8, head_dim=128, seed=91, varlen=True)
    _boost_keys(b, 0, 900, 1000, factor)
    _boost_keys(b, 2, 300, 310, factor)
    if fp8:
        # K scale 1: the boosted keys (|x| up to ~200) stay inside e4m3's range (+-448)
        from test_gpu_fp8 import _check_fp8
        _check_fp8(W.to_fp8_pool(b, k_scale=1.0))
    else:
        _check_step(b)


@pytest.mark.parametrize("varlen", [False, True])
def test_decode_split_off_computes_items_whole(varlen):
    # The split-K ablation: with the split off every (sequence, KV-head tile) item is
    # computed whole by one CTA and no merge job runs; results stay within tolerance.
    # Short contexts and two long ones (one item then spans several CTA shares); the varlen
    # form adds a prefill chunk, so the decode CTAs of the one-launch kernel take the mode.
    ctx = [300, 17, 1200, 5000, 64, 9000, 700, 1]
    ql = [1] * len(ctx)
    if varlen:
        ctx, ql = ctx + [400], ql + [100]
    b = W.make_batch("split_off", context_lens=ctx, q_lens=ql, num_heads=64, num_kv_heads=8,
                     head_dim=128, seed=95, varlen=varlen, pool_fill="nan")
    pkv.set_decode_split(False)
    try:
        _check_step(b)
    finally:
        pkv.set_decode_split(True)


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_growing_scores(fp8):
    # K rows scaled by 1 + pos / 40: each row's scores climb along the context, so its
    # reference maximum moves again and again, in either 64-key round of a 128-key chunk
    # (a move in the second round rescales the first round's weights in place).
    b = W.make_batch("growing", context_lens=[2000, 900, 40], q_lens=[64, 1, 40], num_heads=64,
                     num_kv_heads=8, head_dim=128, seed=93, varlen=True)
    for seq, ctx in ((0, 2000), (2, 40)):
        for pos in range(ctx):
            blk, off = b.block_tables[seq, pos // b.block_size], pos % b.block_size
            b.k_cache[blk, off] = W.bf16_bits(W.bf16_to_f32(b.k_cache[blk, off]) * np.float32(1 + pos / 40))
    if fp8:
        from test_gpu_fp8 import _check_fp8
        _check_fp8(W.to_fp8_pool(b, k_scale=1.0))  # |K| stays below ~300, inside e4m3's range
    else:
        _check_step(b)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 64), (8, 2, 128), (12, 4, 64), (56, 8, 128)])
def test_varlen_head_layouts(Hq, Hkv, d):
    b = W.make_batch("varlen_heads", context_lens=[70, 3, 129], q_lens=[37, 1, 129], num_heads=Hq,
                     num_kv_heads=Hkv, head_dim=d, seed=Hq * 7 + d, varlen=True)
    _check_step(b)


def test_varlen_non_causal():
    b = W.make_batch("noncausal", context_lens=[40, 9, 200], q_lens=[12, 1, 64], num_heads=16,
                     num_kv_heads=4, head_dim=128, seed=21, varlen=True, causal=False)
    _check_step(b)


def test_varlen_decode_rows_match_decode_kernel():
    b = W.gqa_decode(seed=5, num_seqs=40)
    out_dec, _, _, _ = gpu_step(b)
    b.query_start_loc = np.arange(b.num_seqs + 1, dtype=np.int32)
    out_var, _, _, _ = gpu_step(b)
    assert np.array_equal(out_dec, out_var)


def test_chunked_prompt_matches_whole_prompt():
    # The same prompt once as one varlen item and once as 4 chunks of 128 tokens.
    L = 512
    rng = np.random.Generator(np.random.PCG64(8))
    b = W.make_batch("whole", context_lens=[L], q_lens=[L], num_heads=64, num_kv_heads=8,
                     head_dim=128, seed=8, varlen=True)
    whole, kc, vc, _ = gpu_step(b)
    parts = []
    for lo in range(0, L, 128):
        hi = lo + 128
        c = W.make_batch("part", context_lens=[hi], q_lens=[128], num_heads=64, num_kv_heads=8,
                         head_dim=128, seed=9, varlen=True, num_blocks=b.num_blocks,
                         max_blocks_per_seq=b.max_blocks_per_seq)
        c.k_cache, c.v_cache, c.block_tables = kc, vc, b.block_tables
        c.q = b.q[lo:hi]
        c.k_new, c.v_new = b.k_new[lo:hi], b.v_new[lo:hi]
        c.new_token_pos = np.arange(lo, hi, dtype=np.int32)
        out, _, _, _ = gpu_step(c)
        parts.append(out)
    chunked = np.concatenate(parts)
    assert np.max(np.abs(chunked - whole)) < 2e-2


# ---- device-side checks of bad metadata ---------------------------------------------

def test_bad_block_id_is_flagged_not_read():
    import pagedattention_paged_kv_gb300 as pkv
    b = W.make_batch("badblock", context_lens=[40, 20], q_lens=[1, 1], num_heads=8,
                     num_kv_heads=2, head_dim=128, seed=31)
    b.block_tables[0, 1] = b.num_blocks + 5
    b.new_token_pos[:] = 0  # keep the KV write away from the bad block
    out, _, _, err = gpu_step(b)
    assert err & pkv.DEVERR_BLOCK_ID
    assert np.all(np.isfinite(out))


def test_slot_outside_pool_is_flagged_and_skipped():
    import torch
    import pagedattention_paged_kv_gb300 as pkv
    from gpu_helpers import bf16_to_np, torch_bf16
    rng = np.random.Generator(np.random.PCG64(3))
    kc = torch_bf16(W.normal_bf16(rng, (4, 16, 2, 64)))
    vc = torch_bf16(W.normal_bf16(rng, (4, 16, 2, 64)))
    before_k, before_v = bf16_to_np(kc), bf16_to_np(vc)
    k = torch_bf16(W.normal_bf16(rng, (2, 2, 64)))
    v = torch_bf16(W.normal_bf16(rng, (2, 2, 64)))
    pkv.reshape_and_cache(kc, vc, k, v, torch.tensor([64, -1], dtype=torch.int64, device="cuda"))
    assert pkv.get_device_error() & pkv.DEVERR_SLOT
    assert np.array_equal(bf16_to_np(kc), before_k) and np.array_equal(bf16_to_np(vc), before_v)


def test_workspace_too_small_is_refused():
    import torch
    import pagedattention_paged_kv_gb300 as pkv
    b = W.tiny_decode()
    from gpu_helpers import torch_bf16
    q = torch_bf16(b.q)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode(torch.empty_like(q), q, torch_bf16(b.k_cache), torch_bf16(b.v_cache),
                                   torch.from_numpy(b.block_tables).cuda(),
                                   torch.from_numpy(b.context_lens).cuda(), b.scale,
                                   workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == -3
