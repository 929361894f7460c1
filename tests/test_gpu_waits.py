"""Bounded pipeline waits (failure detection without a GPU fault).

Every mbarrier wait in the attention kernels gives up after a limit, flags
PKV_DEVERR_TIMEOUT and lets its CTA return after the copies it already issued have
landed, so a stalled pipeline never hangs the GPU.  Here the limit is set to 1 ns:
consumers that find their K/V stage not yet loaded, and a producer that finds no stage
free, give up at once.  The launch must return with the timeout flag set, leave the pool
untouched, and the next launch with the default limit must match the oracle.
"""
import numpy as np
import pytest

from gpu_helpers import bf16_bits_to_f64, bf16_to_np, compare, oracle_step, torch_bf16
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_decode_wait_that_runs_out_flags_timeout_and_returns():
    import torch
    import pagedattention_paged_kv_gb300 as pkv
    b = W.gqa_decode(seed=71, num_seqs=64)
    slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos)
    kc, vc = torch_bf16(b.k_cache), torch_bf16(b.v_cache)
    pkv.reshape_and_cache(kc, vc, torch_bf16(b.k_new), torch_bf16(b.v_new), torch.from_numpy(slots).cuda())
    q = torch_bf16(b.q)
    bt = torch.from_numpy(b.block_tables).cuda()
    cl = torch.from_numpy(b.context_lens).cuda()
    assert pkv.get_device_error() == 0
    k_before, v_before = bf16_to_np(kc), bf16_to_np(vc)
    out = torch.empty_like(q)
    flags = []
    try:
        pkv.set_wait_limit_ns(1)
        for _ in range(5):  # each launch has thousands of waits that find their stage not ready
            pkv.paged_attention_decode(out, q, kc, vc, bt, cl, b.scale)
            flags.append(pkv.get_device_error())  # synchronizes: the launch has returned
            if flags[-1] & pkv.DEVERR_TIMEOUT:
                break
    finally:
        pkv.set_wait_limit_ns(0)
    assert flags[-1] & pkv.DEVERR_TIMEOUT, f"no wait ran out: flags {flags}"
    assert all(f & ~pkv.DEVERR_TIMEOUT == 0 for f in flags), flags
    assert np.array_equal(bf16_to_np(kc), k_before) and np.array_equal(bf16_to_np(vc), v_before)
    # the context is still usable and the default limit gives the oracle's result
    out = torch.full_like(q, float("nan"))
    pkv.paged_attention_decode(out, q, kc, vc, bt, cl, b.scale)
    assert pkv.get_device_error() == 0
    ref, _, _ = oracle_step(b)
    compare(bf16_bits_to_f64(bf16_to_np(out)), ref)
