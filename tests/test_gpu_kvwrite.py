"""The decode step with its KV write fused into the attention launch gives the same
pool bytes and the same outputs as the separate KV write + decode calls, and matches
the oracle (bf16 and FP8 caches, several block sizes, empty and one-token contexts)."""
import numpy as np
import pytest

import pagedattention_paged_kv_gb300 as pkv
from gpu_helpers import (bf16_bits_to_f64, bf16_to_np, compare, gpu_step, gpu_step_fp8, oracle_step,
                         oracle_step_fp8, torch_bf16, torch_u8)
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CTX = [0, 1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 1000, 2047]


def _fused(b, fp8):
    import torch
    kc = torch_u8(b.k_cache) if fp8 else torch_bf16(b.k_cache)
    vc = torch_u8(b.v_cache) if fp8 else torch_bf16(b.v_cache)
    S = b.num_seqs
    # one new row per sequence (zeros for empty contexts, which write nothing)
    k_new = np.zeros((S, b.num_kv_heads, b.head_dim), np.uint16)
    v_new = np.zeros_like(k_new)
    k_new[b.new_token_seq] = b.k_new
    v_new[b.new_token_seq] = b.v_new
    q = torch_bf16(b.q)
    out = torch.full_like(q, float("nan"))
    kw = {"k_scale": b.meta["k_scale"], "v_scale": b.meta["v_scale"]} if fp8 else {}
    pkv.paged_attention_decode_kvwrite(out, q, torch_bf16(k_new), torch_bf16(v_new), kc, vc,
                                       torch.from_numpy(b.block_tables).cuda(),
                                       torch.from_numpy(b.context_lens).cuda(), b.scale, **kw)
    err = pkv.get_device_error()
    kb = kc.cpu().numpy() if fp8 else bf16_to_np(kc)
    vb = vc.cpu().numpy() if fp8 else bf16_to_np(vc)
    return bf16_bits_to_f64(bf16_to_np(out)), kb, vb, err


def _batch(bs, seed, Hq=64, Hkv=8, d=128):
    ctx = np.array(CTX)
    b = W.make_batch("fused", context_lens=np.maximum(ctx, 1), q_lens=np.ones(len(ctx), np.int64),
                     num_heads=Hq, num_kv_heads=Hkv, head_dim=d, seed=seed, block_size=bs, pool_fill="nan")
    # empty contexts: no new token, zero output
    keep = ctx > 0
    b.context_lens[:] = ctx
    b.new_token_seq = b.new_token_seq[keep]
    b.new_token_pos = b.new_token_pos[keep]
    b.k_new, b.v_new = b.k_new[keep], b.v_new[keep]
    return b


@pytest.mark.parametrize("bs", [16, 8, 64])
def test_fused_kv_write_bf16(bs):
    b = _batch(bs, 300 + bs)
    out, kc, vc, err = _fused(b, False)
    sep, skc, svc, serr = gpu_step(b)
    ref, rkc, rvc = oracle_step(b)
    assert err == 0 and serr == 0
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc)
    assert np.array_equal(out, sep)
    compare(out, ref)


@pytest.mark.parametrize("bs", [16, 32])
def test_fused_kv_write_fp8(bs):
    b = W.to_fp8_pool(_batch(bs, 400 + bs))
    out, kc, vc, err = _fused(b, True)
    sep, skc, svc, serr = gpu_step_fp8(b)
    ref, rkc, rvc = oracle_step_fp8(b)
    assert err == 0 and serr == 0
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc)
    assert np.array_equal(out, sep)
    compare(out, ref)


def test_fused_kv_write_full_size_gqa():
    b = W.gqa_decode()
    out, kc, vc, err = _fused(b, False)
    sep, _, _, _ = gpu_step(b)
    _, rkc, rvc = oracle_step(b, row_mask=np.zeros(b.q.shape[0], np.uint8))
    assert err == 0
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc)
    assert np.array_equal(out, sep)
