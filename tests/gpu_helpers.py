"""Shared pieces of the GPU parity tests: run one step through the C ABI and the
same step through the oracle, then compare."""
from __future__ import annotations

import numpy as np

import oracle
import pagedattention_paged_kv_gb300 as pkv
from pagedattention_paged_kv_gb300.workloads import PagedBatch

# Tolerance for bf16 outputs against the fp64 oracle: an element passes when
# |gpu - ref| <= ATOL + RTOL * |ref| (max-abs 1e-2, max-rel 2e-2).
ATOL = 1e-2
RTOL = 2e-2


def torch_bf16(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_np(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gpu_step(b: PagedBatch, workspace=None, causal=None):
    """Slot mapping (host), KV write and attention through the library.
    Returns (out fp64 [total_q, Hq, d], k_cache bits, v_cache bits, device error flags)."""
    import torch
    slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)
    kc, vc = torch_bf16(b.k_cache), torch_bf16(b.v_cache)
    k, v, q = torch_bf16(b.k_new), torch_bf16(b.v_new), torch_bf16(b.q)
    sm = torch.from_numpy(slots).cuda()
    bt = torch.from_numpy(b.block_tables).cuda()
    cl = torch.from_numpy(b.context_lens).cuda()
    out = torch.full_like(q, float("nan"))
    pkv.reshape_and_cache(kc, vc, k, v, sm)
    if b.query_start_loc is None:
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, b.scale, workspace=workspace)
    else:
        qsl = torch.from_numpy(b.query_start_loc).cuda()
        pkv.paged_attention_varlen(out, q, qsl, kc, vc, bt, cl, b.scale,
                                   causal=b.causal if causal is None else causal,
                                   max_q_len=int(b.q_lens.max()), workspace=workspace)
    err = pkv.get_device_error()
    return bf16_bits_to_f64(bf16_to_np(out)), bf16_to_np(kc), bf16_to_np(vc), err


def oracle_step(b: PagedBatch, row_mask=None, causal=None):
    """The same step through the oracle: its own slot mapping, KV write and attention."""
    orc = oracle.load()
    slots = orc.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    orc.reshape_and_cache(kc, vc, b.k_new, b.v_new, slots)
    out = orc.paged_attention(b.q, kc, vc, b.block_tables, b.context_lens, b.scale,
                              query_start_loc=b.query_start_loc,
                              causal=b.causal if causal is None else causal, row_mask=row_mask)
    return out, kc, vc


# |ref| at and above which the relative term of the tolerance is the larger one
# (RTOL * |ref| >= ATOL): only there is max-rel the figure the 2e-2 bound speaks of.
REL_GOVERNS = ATOL / RTOL


class Agreement(tuple):
    """(max_abs, max_rel) of a comparison, plus .max_rel_governed: the largest relative
    error over the elements with |ref| >= REL_GOVERNS (0.5), where the relative bound is
    the binding one, and .n_governed, how many such elements there were.  max_rel itself
    is taken over |ref| >= 1e-3, where small references make it large without any
    element being near its bound."""

    def __new__(cls, max_abs, max_rel, max_rel_governed, n_governed):
        t = super().__new__(cls, (max_abs, max_rel))
        t.max_rel_governed = max_rel_governed
        t.n_governed = n_governed
        return t


def compare(gpu: np.ndarray, ref: np.ndarray, rows=None):
    """Element-wise tolerance check; returns Agreement (max_abs, max_rel) over the rows
    compared."""
    if rows is not None:
        gpu, ref = gpu[rows], ref[rows]
    assert np.all(np.isfinite(ref)), "oracle rows missing"
    diff = np.abs(gpu - ref)
    bad = ~(diff <= ATOL + RTOL * np.abs(ref))
    big = np.abs(ref) >= 1e-3
    gov = np.abs(ref) >= REL_GOVERNS
    max_abs = float(diff.max()) if diff.size else 0.0
    max_rel = float((diff[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    max_rel_gov = float((diff[gov] / np.abs(ref[gov])).max()) if gov.any() else 0.0
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance (max_abs {max_abs:.3g}, "
                             f"max_rel {max_rel:.3g}, max_rel where |ref| >= {REL_GOVERNS} "
                             f"{max_rel_gov:.3g}); first {idx.tolist()} "
                             f"gpu {gpu[tuple(idx[0])]:.6g} ref {ref[tuple(idx[0])]:.6g}")
    return Agreement(max_abs, max_rel, max_rel_gov, int(gov.sum()))


def torch_u8(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def gpu_step_fp8(b: PagedBatch, workspace=None):
    """FP8 pool (b from workloads.to_fp8_pool): slot mapping, the quantising KV write
    and attention (decode, or varlen when b has query_start_loc) through the library.  Returns (out fp64, k_cache codes, v_cache codes,
    device error flags)."""
    import torch
    ks, vs = b.meta["k_scale"], b.meta["v_scale"]
    slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)
    kc, vc = torch_u8(b.k_cache), torch_u8(b.v_cache)
    k, v, q = torch_bf16(b.k_new), torch_bf16(b.v_new), torch_bf16(b.q)
    sm = torch.from_numpy(slots).cuda()
    bt = torch.from_numpy(b.block_tables).cuda()
    cl = torch.from_numpy(b.context_lens).cuda()
    out = torch.full_like(q, float("nan"))
    pkv.reshape_and_cache_fp8(kc, vc, k, v, sm, ks, vs)
    if b.query_start_loc is None:
        pkv.paged_attention_decode_fp8(out, q, kc, vc, bt, cl, b.scale, ks, vs, workspace=workspace)
    else:
        qsl = torch.from_numpy(b.query_start_loc).cuda()
        pkv.paged_attention_varlen(out, q, qsl, kc, vc, bt, cl, b.scale, causal=b.causal,
                                   max_q_len=int(b.q_lens.max()), workspace=workspace,
                                   k_scale=ks, v_scale=vs)
    err = pkv.get_device_error()
    return bf16_bits_to_f64(bf16_to_np(out)), kc.cpu().numpy(), vc.cpu().numpy(), err


def oracle_step_fp8(b: PagedBatch, row_mask=None):
    """The same FP8 step through the oracle."""
    orc = oracle.load()
    ks, vs = b.meta["k_scale"], b.meta["v_scale"]
    slots = orc.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    orc.reshape_and_cache_fp8(kc, vc, b.k_new, b.v_new, slots, ks, vs)
    out = orc.paged_attention_fp8(b.q, kc, vc, ks, vs, b.block_tables, b.context_lens, b.scale,
                                  query_start_loc=b.query_start_loc, causal=b.causal, row_mask=row_mask)
    return out, kc, vc
