"""A decode step (KV write + attention) captured as a CUDA graph and replayed gives the
same bytes as the eager calls, and the oracle's result."""
import numpy as np
import pytest

import pagedattention_paged_kv_gb300 as pkv
from gpu_helpers import bf16_bits_to_f64, bf16_to_np, compare, oracle_step, torch_bf16
from pagedattention_paged_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("varlen", [False, True])
def test_captured_step_matches_eager_and_oracle(varlen):
    import torch
    from pagedattention_paged_kv_gb300.graph import CapturedStep
    if varlen:
        b = W.make_batch("g", context_lens=[40, 300, 700], q_lens=[24, 1, 1], num_heads=64, num_kv_heads=8,
                         head_dim=128, seed=71, varlen=True)
    else:
        b = W.make_batch("g", context_lens=[1, 50, 600, 2000], q_lens=[1, 1, 1, 1], num_heads=64,
                         num_kv_heads=8, head_dim=128, seed=72)
    slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)
    kc, vc = torch_bf16(b.k_cache), torch_bf16(b.v_cache)
    q, k, v = torch_bf16(b.q), torch_bf16(b.k_new), torch_bf16(b.v_new)
    sm = torch.from_numpy(slots).cuda()
    bt = torch.from_numpy(b.block_tables).cuda()
    cl = torch.from_numpy(b.context_lens).cuda()
    qsl = torch.from_numpy(b.query_start_loc).cuda() if varlen else None
    out = torch.zeros_like(q)
    T = q.shape[0]
    ws = torch.empty(pkv.workspace_size(pkv.OP_VARLEN if varlen else pkv.OP_DECODE, b.num_seqs, T, 64, 8, 128),
                     dtype=torch.uint8, device="cuda")

    def step():
        pkv.reshape_and_cache(kc, vc, k, v, sm)
        if varlen:
            pkv.paged_attention_varlen(out, q, qsl, kc, vc, bt, cl, b.scale, max_q_len=int(b.q_lens.max()),
                                       workspace=ws)
        else:
            pkv.paged_attention_decode(out, q, kc, vc, bt, cl, b.scale, workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    cap = CapturedStep(step)
    torch.cuda.synchronize()
    out.zero_()
    torch.cuda.synchronize()
    cap.replay()
    cap.synchronize()
    assert torch.equal(out, eager)
    # a replay must really run the kernels: change an input and see the output move
    q.mul_(2)
    torch.cuda.synchronize()
    cap.replay()
    cap.synchronize()
    assert not torch.equal(out, eager)
    q.div_(2)
    torch.cuda.synchronize()
    cap.replay()
    cap.synchronize()
    assert torch.equal(out, eager)
    assert pkv.get_device_error() == 0
    ref, _, _ = oracle_step(b)
    compare(bf16_bits_to_f64(bf16_to_np(out)), ref)
