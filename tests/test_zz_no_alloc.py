"""The allocation-free decode entry point (pkv_paged_attention_decode_static).

It serves callers that may not allocate device memory where they run attention (a
plugin inside a runtime that reserved all device memory up front, or a latency-critical
loop that cannot let cudaMalloc/cudaFree synchronize the device) and cannot pass a
workspace either.  It must give what the workspace-taking decode call gives.  This file
is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import bf16_to_np, torch_bf16
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _static_fn():
    import pagedattention_paged_kv_gb300 as pkv
    fn = pkv.lib().pkv_paged_attention_decode_static
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32, vp]
    fn.restype = i32
    return fn


def test_static_scratch_decode_matches_workspace_decode():
    import torch
    import pagedattention_paged_kv_gb300 as pkv
    fn = _static_fn()
    stream = torch.cuda.current_stream().cuda_stream
    # Two calls in a row on different batches: the second sees the first call's
    # leftovers in the shared scratch and must not depend on them.
    for seed, num_seqs in ((61, 128), (62, 37)):
        b = W.gqa_decode(seed=seed, num_seqs=num_seqs)
        slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos)
        kc, vc = torch_bf16(b.k_cache), torch_bf16(b.v_cache)
        q = torch_bf16(b.q)
        bt = torch.from_numpy(b.block_tables).cuda()
        cl = torch.from_numpy(b.context_lens).cuda()
        pkv.reshape_and_cache(kc, vc, torch_bf16(b.k_new), torch_bf16(b.v_new),
                              torch.from_numpy(slots).cuda())
        ref = torch.empty_like(q)
        pkv.paged_attention_decode(ref, q, kc, vc, bt, cl, b.scale)
        got = torch.full_like(q, float("nan"))
        st = fn(got.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                cl.data_ptr(), b.num_seqs, b.max_blocks_per_seq, b.num_heads, b.num_kv_heads,
                b.head_dim, b.block_size, b.num_blocks, b.scale, pkv.DTYPE_BF16, stream)
        assert st == 0, pkv.lib().pkv_status_string(st)
        assert pkv.get_device_error() == 0
        # Same plan, same kernels, same reduction order: only where the scratch lives
        # differs, so the outputs must be the same bits (a tolerance would hide a part
        # read from the previous call's leftovers).
        assert np.array_equal(bf16_to_np(got), bf16_to_np(ref)), "static-scratch decode differs"


def test_static_scratch_refuses_sizes_beyond_its_limit():
    import torch
    import pagedattention_paged_kv_gb300 as pkv
    fn = _static_fn()
    # 128 query heads over 8 KV heads (group 16) needs about 20 MB of scratch on 152 SMs.
    S, Hq, Hkv, d = 4, 128, 8, 128
    need = pkv.workspace_size(pkv.OP_DECODE, S, S, Hq, Hkv, d)
    if need <= 16 * 1024 * 1024:
        pytest.skip("this GPU's scratch need for the probe sizes fits the limit")
    q = torch.zeros(S, Hq, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, Hkv, d, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(S, 1, dtype=torch.int32, device="cuda")
    cl = torch.ones(S, dtype=torch.int32, device="cuda")
    out = torch.full((S, Hq, d), 1.5, dtype=torch.bfloat16, device="cuda")  # sentinel
    st = fn(out.data_ptr(), q.data_ptr(), kc.data_ptr(), kc.data_ptr(), bt.data_ptr(), cl.data_ptr(),
            S, 1, Hq, Hkv, d, 16, 4, 0.1, pkv.DTYPE_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == -7
    # refused before any launch: the output keeps its sentinel and no kernel flagged anything
    assert pkv.get_device_error() == 0
    assert bool((out == 1.5).all())
