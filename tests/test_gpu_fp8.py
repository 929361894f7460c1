"""GPU parity of the FP8 (e4m3) cache path through the C ABI against the fp64 oracle:
the quantising KV write bit for bit over the whole pool, decode and varlen (chunked
prefill + decode) attention within |gpu - ref| <= 1e-2 + 2e-2 |ref| of attention over
the dequantised pool."""
import numpy as np
import pytest

import oracle
import pagedattention_paged_kv_gb300 as pkv
from gpu_helpers import (bf16_bits_to_f64, bf16_to_np, compare, gpu_step_fp8, oracle_step_fp8,
                         torch_bf16, torch_u8)
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check_fp8(b, row_mask=None):
    out, kc, vc, err = gpu_step_fp8(b)
    ref, rkc, rvc = oracle_step_fp8(b, row_mask=row_mask)
    assert err == 0, f"device error flags {err:#x}"
    assert np.array_equal(kc, rkc), f"k_cache differs in {int((kc != rkc).sum())} bytes"
    assert np.array_equal(vc, rvc), f"v_cache differs in {int((vc != rvc).sum())} bytes"
    rows = None if row_mask is None else np.nonzero(row_mask)[0]
    return compare(out, ref, rows)


def test_fp8_gqa_decode_full_size():
    b = W.to_fp8_pool(W.gqa_decode())
    rows = np.zeros(b.q.shape[0], np.uint8)
    rows[np.r_[0:8, 40:48, 120:128]] = 1
    _check_fp8(b, row_mask=rows)


def test_fp8_skewed_long_context_decode():
    """Contexts of 32768 next to short ones: the split-K parts and their merge."""
    b = W.to_fp8_pool(W.skewed_decode())
    rows = np.zeros(b.q.shape[0], np.uint8)
    rows[np.nonzero(b.context_lens == 32768)[0]] = 1
    rows[:6] = 1
    _check_fp8(b, row_mask=rows)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (32, 8), (64, 8), (40, 8), (64, 1), (16, 16)])
def test_fp8_decode_head_layouts(Hq, Hkv):
    ctx = [1, 2, 15, 16, 17, 31, 33, 100, 257, 1000]
    b = W.make_batch("heads", context_lens=ctx, q_lens=np.ones(len(ctx), np.int64), num_heads=Hq,
                     num_kv_heads=Hkv, head_dim=128, seed=11 + Hq + Hkv, pool_fill="nan")
    _check_fp8(W.to_fp8_pool(b))


def test_fp8_scales_other_than_powers_of_two():
    ctx = [3, 50, 200, 513]
    b = W.make_batch("scales", context_lens=ctx, q_lens=np.ones(len(ctx), np.int64), num_heads=16,
                     num_kv_heads=4, head_dim=128, seed=23, pool_fill="nan")
    _check_fp8(W.to_fp8_pool(b, k_scale=0.0123, v_scale=0.0371))


def test_fp8_kv_write_saturates_and_keeps_subnormals():
    """New rows far outside +-448 x scale clamp to +-448; tiny ones land on subnormal
    codes; both exactly as the oracle's nearest-code rule."""
    import torch
    rng = np.random.Generator(np.random.PCG64(31))
    NB, bs, Hkv, d, T = 8, 16, 2, 128, 20
    k = W.normal_bf16(rng, (T, Hkv, d))
    v = W.normal_bf16(rng, (T, Hkv, d))
    mag = np.exp2(rng.uniform(-14, 12, size=(T, Hkv, d))).astype(np.float32)
    k = W.bf16_bits(W.bf16_to_f32(k) * mag)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[5] = -1
    kc0 = np.full((NB, bs, Hkv, d), 0x7F, np.uint8)
    vc0 = kc0.copy()
    ks, vs = 2.0 ** -6, 0.3
    kc, vc = torch_u8(kc0), torch_u8(vc0)
    pkv.reshape_and_cache_fp8(kc, vc, torch_bf16(k), torch_bf16(v), torch.from_numpy(slots).cuda(), ks, vs)
    orc = oracle.load()
    rkc, rvc = kc0.copy(), vc0.copy()
    orc.reshape_and_cache_fp8(rkc, rvc, k, v, slots, ks, vs)
    assert pkv.get_device_error() == 0
    assert np.array_equal(kc.cpu().numpy(), rkc)
    assert np.array_equal(vc.cpu().numpy(), rvc)
    codes = rkc[rkc != 0x7F]
    assert np.any((codes & 0x7F) == 0x7E) and np.any(((codes & 0x78) == 0) & ((codes & 7) != 0))


def test_fp8_empty_contexts_give_zero_rows():
    ctx = [0, 5, 0, 40]
    b = W.to_fp8_pool(W.make_batch("empty", context_lens=[5, 5, 5, 40], q_lens=[1, 1, 1, 1],
                                   num_heads=8, num_kv_heads=2, head_dim=128, seed=5))
    b.context_lens[:] = ctx
    b.new_token_seq = np.array([1, 3], np.int32)
    b.new_token_pos = np.array([4, 39], np.int32)
    b.k_new, b.v_new = b.k_new[[1, 3]], b.v_new[[1, 3]]
    out, _, _, err = gpu_step_fp8(b)
    ref, _, _ = oracle_step_fp8(b)
    assert err == 0
    assert np.all(out[[0, 2]] == 0.0)
    compare(out, ref)


def test_fp8_matches_bf16_path_on_dequantised_pool():
    """With power-of-two scales the dequantised pool is exact in bf16: the FP8 kernel
    and the bf16 kernel over that pool agree within the tolerance (they differ only in
    the fp16 vs bf16 rounding of q and of the weights)."""
    import torch
    b8 = W.to_fp8_pool(W.make_batch("cross", context_lens=[7, 300, 1500], q_lens=[1, 1, 1],
                                    num_heads=64, num_kv_heads=8, head_dim=128, seed=41))
    orc = oracle.load()
    lut = np.array([orc.e4m3_decode(c) for c in range(256)], np.float64)
    kb = W.bf16_bits((lut[b8.k_cache] * b8.meta["k_scale"]).astype(np.float32))
    vb = W.bf16_bits((lut[b8.v_cache] * b8.meta["v_scale"]).astype(np.float32))
    q = torch_bf16(b8.q)
    bt = torch.from_numpy(b8.block_tables).cuda()
    cl = torch.from_numpy(b8.context_lens).cuda()
    o8 = torch.empty_like(q)
    o16 = torch.empty_like(q)
    pkv.paged_attention_decode_fp8(o8, q, torch_u8(b8.k_cache), torch_u8(b8.v_cache), bt, cl, b8.scale,
                                   b8.meta["k_scale"], b8.meta["v_scale"])
    pkv.paged_attention_decode(o16, q, torch_bf16(kb), torch_bf16(vb), bt, cl, b8.scale)
    compare(bf16_bits_to_f64(bf16_to_np(o8)), bf16_bits_to_f64(bf16_to_np(o16)))


def test_fp8_rejects_unsupported_and_bad_scales():
    import torch
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 4, 64, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(2, 1, dtype=torch.int32, device="cuda")
    cl = torch.ones(2, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode_fp8(torch.empty_like(q), q, kc, kc, bt, cl, 0.1, 1.0, 1.0)
    assert e.value.status == -2  # head_dim 64: not built for FP8
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 4, 128, dtype=torch.uint8, device="cuda")
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_attention_decode_fp8(torch.empty_like(q), q, kc, kc, bt, cl, 0.1, ks, vs)
        assert e.value.status == -1


# ---- varlen batches: FP8 prefill chunks next to FP8 decodes ---------------------------

@pytest.mark.parametrize("q_lens,ctx", [
    ([2, 1, 17, 1, 100], [2, 30, 17, 1, 500]),           # whole prompts and decodes
    ([512, 1, 1, 33], [16896, 600, 1, 1000]),            # a chunk with a long prefix
    ([16, 15, 48, 1], [16, 40, 1100, 2]),                # tile-aligned and ragged chunks
    ([5, 300], [5, 300]),                                 # first chunks of prompts
])
def test_fp8_varlen_chunks_and_decodes(q_lens, ctx):
    """Pool rows past every context hold the NaN code: the prefill's converters must zero
    V there and the softmax mask K there."""
    b = W.make_batch("varlen", context_lens=ctx, q_lens=q_lens, num_heads=64, num_kv_heads=8,
                     head_dim=128, seed=sum(q_lens) + 3, varlen=True, pool_fill="nan")
    _check_fp8(W.to_fp8_pool(b))


def test_fp8_mixed_varlen_full_size_sampled_chunk_rows():
    b = W.to_fp8_pool(W.mixed_varlen())
    mask = np.zeros(b.q.shape[0], np.uint8)
    mask[np.r_[0, 1, 2, 15, 16, 17, 31, 32, np.arange(47, 512, 37), 510, 511]] = 1
    mask[np.r_[512:520, 600:608]] = 1  # decode rows
    _check_fp8(b, row_mask=mask)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (56, 8), (16, 16), (64, 8), (32, 4)])
def test_fp8_varlen_head_layouts(Hq, Hkv):
    b = W.make_batch("varlen_heads", context_lens=[70, 3, 129, 260], q_lens=[37, 1, 129, 131],
                     num_heads=Hq, num_kv_heads=Hkv, head_dim=128, seed=Hq * 7 + Hkv,
                     varlen=True, pool_fill="nan")
    _check_fp8(W.to_fp8_pool(b))


def test_fp8_varlen_non_causal_and_scales_other_than_powers_of_two():
    b = W.make_batch("noncausal", context_lens=[40, 9, 200, 700], q_lens=[12, 1, 64, 300],
                     num_heads=16, num_kv_heads=4, head_dim=128, seed=27, varlen=True, causal=False,
                     pool_fill="nan")
    _check_fp8(W.to_fp8_pool(b, k_scale=0.0123, v_scale=0.0371))


def test_fp8_long_prefix_splits_across_ctas():
    """One 256-token chunk behind a 20000-token prefix: its tiles split across CTAs and
    the parts (scaled by v_scale before the merge) are combined."""
    b = W.make_batch("longprefix", context_lens=[20256, 3], q_lens=[256, 1], num_heads=64,
                     num_kv_heads=8, head_dim=128, seed=77, varlen=True, pool_fill="nan")
    _check_fp8(W.to_fp8_pool(b, k_scale=0.02, v_scale=0.05))


def test_fp8_prefill_matches_bf16_prefill_on_dequantised_pool():
    """With power-of-two scales the dequantised pool is exact in bf16: the FP8 and bf16
    prefill kernels over it agree within the tolerance."""
    import torch
    b8 = W.to_fp8_pool(W.make_batch("cross", context_lens=[700, 5, 1500], q_lens=[200, 1, 333],
                                    num_heads=64, num_kv_heads=8, head_dim=128, seed=43, varlen=True))
    orc = oracle.load()
    lut = np.array([orc.e4m3_decode(c) for c in range(256)], np.float64)
    kb = W.bf16_bits((lut[b8.k_cache] * b8.meta["k_scale"]).astype(np.float32))
    vb = W.bf16_bits((lut[b8.v_cache] * b8.meta["v_scale"]).astype(np.float32))
    q = torch_bf16(b8.q)
    qsl = torch.from_numpy(b8.query_start_loc).cuda()
    bt = torch.from_numpy(b8.block_tables).cuda()
    cl = torch.from_numpy(b8.context_lens).cuda()
    o8 = torch.empty_like(q)
    o16 = torch.empty_like(q)
    pkv.paged_attention_varlen(o8, q, qsl, torch_u8(b8.k_cache), torch_u8(b8.v_cache), bt, cl, b8.scale,
                               k_scale=b8.meta["k_scale"], v_scale=b8.meta["v_scale"])
    pkv.paged_attention_varlen(o16, q, qsl, torch_bf16(kb), torch_bf16(vb), bt, cl, b8.scale)
    assert pkv.get_device_error() == 0
    compare(bf16_bits_to_f64(bf16_to_np(o8)), bf16_bits_to_f64(bf16_to_np(o16)))


def test_fp8_varlen_rejects_bad_scales_and_head_dim():
    import torch
    q = torch.zeros(4, 8, 128, dtype=torch.bfloat16, device="cuda")
    qsl = torch.tensor([0, 3, 4], dtype=torch.int32, device="cuda")
    kc = torch.zeros(4, 16, 2, 128, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(2, 1, dtype=torch.int32, device="cuda")
    cl = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
    for ks, vs in ((0.0, 1.0), (1.0, float("nan"))):
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.paged_attention_varlen(torch.empty_like(q), q, qsl, kc, kc, bt, cl, 0.1, k_scale=ks, v_scale=vs)
        assert e.value.status == -1
    with pytest.raises(ValueError):
        pkv.paged_attention_varlen(torch.empty_like(q), q, qsl, kc, kc, bt, cl, 0.1)
    q64 = torch.zeros(4, 8, 64, dtype=torch.bfloat16, device="cuda")
    kc64 = torch.zeros(4, 16, 2, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_varlen(torch.empty_like(q64), q64, qsl, kc64, kc64, bt, cl, 0.1,
                                   k_scale=1.0, v_scale=1.0)
    assert e.value.status == -2
