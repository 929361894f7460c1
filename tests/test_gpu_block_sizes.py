"""Decode with pool blocks of 8, 32 and 64 tokens ("vLLM推理引擎架构PagedAttention机制与高吞吐
推理" (lpnh.cn) §4.1: the block size trades block-table overhead and kernel access
efficiency against slot waste; 16 is the default).  The KV write and decode (bf16 and
FP8 caches, single-token varlen rows) against the oracle with the same block size."""
import numpy as np
import pytest

import pagedattention_paged_kv_gb300 as pkv
from gpu_helpers import compare, gpu_step, gpu_step_fp8, oracle_step, oracle_step_fp8
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CTX = [1, 7, 8, 9, 15, 16, 17, 31, 33, 63, 64, 65, 100, 257, 1000, 2047]


@pytest.mark.parametrize("bs", [8, 32, 64])
@pytest.mark.parametrize("Hq,Hkv,d", [(64, 8, 128), (8, 2, 64)])
def test_decode_block_sizes(bs, Hq, Hkv, d):
    b = W.make_batch(f"bs{bs}", context_lens=CTX, q_lens=np.ones(len(CTX), np.int64), num_heads=Hq,
                     num_kv_heads=Hkv, head_dim=d, seed=100 + bs + d, block_size=bs, pool_fill="nan")
    out, kc, vc, err = gpu_step(b)
    ref, rkc, rvc = oracle_step(b)
    assert err == 0
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc)
    compare(out, ref)


@pytest.mark.parametrize("bs", [8, 32, 64])
def test_fp8_decode_block_sizes(bs):
    b = W.make_batch(f"bs{bs}", context_lens=CTX, q_lens=np.ones(len(CTX), np.int64), num_heads=64,
                     num_kv_heads=8, head_dim=128, seed=200 + bs, block_size=bs, pool_fill="nan")
    b = W.to_fp8_pool(b)
    out, kc, vc, err = gpu_step_fp8(b)
    ref, rkc, rvc = oracle_step_fp8(b)
    assert err == 0
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc)
    compare(out, ref)


@pytest.mark.parametrize("bs", [8, 64])
def test_gqa_decode_full_size_block_sizes(bs):
    b = W.gqa_decode(block_size=bs)
    rows = np.zeros(b.q.shape[0], np.uint8)
    rows[np.r_[0:6, 60:66, 122:128]] = 1
    out, kc, vc, err = gpu_step(b)
    ref, rkc, rvc = oracle_step(b, row_mask=rows)
    assert err == 0
    assert np.array_equal(kc, rkc) and np.array_equal(vc, rvc)
    compare(out, ref, np.nonzero(rows)[0])


def test_varlen_decode_rows_with_block_32_and_prefill_rows_refused():
    import torch
    b = W.make_batch("v32", context_lens=[40, 90, 300], q_lens=[1, 1, 1], num_heads=16, num_kv_heads=4,
                     head_dim=128, seed=9, block_size=32, varlen=True)
    out, kc, vc, err = gpu_step(b)
    ref, _, _ = oracle_step(b)
    assert err == 0
    compare(out, ref)
    b2 = W.make_batch("v32p", context_lens=[40, 90], q_lens=[4, 1], num_heads=16, num_kv_heads=4,
                      head_dim=128, seed=10, block_size=32, varlen=True)
    with pytest.raises(pkv.PagedKVError) as e:
        gpu_step(b2)
    assert e.value.status == -2
