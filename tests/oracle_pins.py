"""Pins for the oracle: facts fixed by the pages or by mathematics, each checked
against the oracle without re-typing its own code path.

Every ``pin_*`` takes an oracle instance and raises AssertionError when the
oracle disagrees.  ``test_oracle_pins.py`` runs them on the oracle;
``test_oracle_mutants.py`` runs them on deliberately broken copies of it and
requires each copy to fail at least one pin.

Sources:
  [OCP8]   OCP 8-bit Floating Point Specification (OFP8), format E4M3 -- the element
           type of the FP8 cache (the pages' headline model runs in FP8).
  [LPNH]   "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn), §2.2 BlockManager
           (pool layout), §2.3 PagedAttention Kernel (arguments and semantics).
  [LESSON] "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış Prefill"
           (aiengineeringfromscratch.com, Phase 17 - 04), "PagedAttention as a virtual
           memory system" (block table), "Chunked prefill protects the TTFT tail".
"""
from __future__ import annotations

import math

import numpy as np
import torch

from pagedattention_paged_kv_gb300.workloads import bf16_bits, bf16_to_f32, normal_bf16

SENTINEL = 0x7FC0  # a bf16 NaN pattern; any slot that should stay untouched keeps it


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------------------
# a1 slot mapping and a2 KV write
# ---------------------------------------------------------------------------

def pin_slot_mapping_worked_example(orc):
    """[LESSON] block table: logical position p lives in logical block p // 16 at
    offset p % 16, and the table names that block's physical id.  A sequence whose
    table is [7, 2, 9]: position 0 -> block 7 slot 0 (= 112), 15 -> 127,
    16 -> block 2 slot 0 (= 32), 20 -> 36, 47 -> block 9 slot 15 (= 159).
    A second sequence [3]: position 5 -> 53.  A padding token maps to -1."""
    tables = np.array([[7, 2, 9], [3, -1, -1]], dtype=np.int32)
    seq = np.array([0, 0, 0, 0, 0, 1, -1], dtype=np.int32)
    pos = np.array([0, 15, 16, 20, 47, 5, 0], dtype=np.int32)
    got = orc.slot_mapping(tables, seq, pos, 16)
    assert got.tolist() == [112, 127, 32, 36, 159, 53, -1], got.tolist()


def pin_reshape_and_cache_worked_example(orc):
    """[LPNH] §2.2 layout [num_blocks, block_size, num_kv_heads, head_dim] with
    3 blocks of 2 slots, 2 heads, head_dim 2.  Token rows are numbered so that
    every element is distinct; slots 5, 0, -1 (skip), 2 put token 0 at block 2
    offset 1, token 1 at block 0 offset 0, token 3 at block 1 offset 0.  K and V
    go to their own caches; every other element keeps the sentinel."""
    k = np.arange(16, dtype=np.uint16).reshape(4, 2, 2) + 100
    v = np.arange(16, dtype=np.uint16).reshape(4, 2, 2) + 200
    kc = np.full((3, 2, 2, 2), SENTINEL, dtype=np.uint16)
    vc = np.full((3, 2, 2, 2), SENTINEL, dtype=np.uint16)
    orc.reshape_and_cache(kc, vc, k, v, np.array([5, 0, -1, 2], dtype=np.int64))
    ek = np.full((3, 2, 2, 2), SENTINEL, dtype=np.uint16)
    ev = np.full((3, 2, 2, 2), SENTINEL, dtype=np.uint16)
    ek[2, 1] = [[100, 101], [102, 103]]
    ek[0, 0] = [[104, 105], [106, 107]]
    ek[1, 0] = [[112, 113], [114, 115]]
    ev[2, 1] = [[200, 201], [202, 203]]
    ev[0, 0] = [[204, 205], [206, 207]]
    ev[1, 0] = [[212, 213], [214, 215]]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def pin_reshape_and_cache_round_trip(orc):
    """Writing rows to distinct slots and reading the pool back as a flat
    [num_blocks * block_size, heads, dim] array at those slots returns the rows;
    all other slots are unchanged; a slot past the pool is refused."""
    rng = _rng(11)
    NB, bs, H, d = 9, 4, 3, 8
    T = 20
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = -1
    k = normal_bf16(rng, (T, H, d))
    v = normal_bf16(rng, (T, H, d))
    kc = normal_bf16(rng, (NB, bs, H, d))
    vc = normal_bf16(rng, (NB, bs, H, d))
    k0, v0 = kc.copy(), vc.copy()
    orc.reshape_and_cache(kc, vc, k, v, slots)
    flat_k, flat_v = kc.reshape(NB * bs, H, d), vc.reshape(NB * bs, H, d)
    keep = slots >= 0
    assert np.array_equal(flat_k[slots[keep]], k[keep])
    assert np.array_equal(flat_v[slots[keep]], v[keep])
    untouched = np.ones(NB * bs, bool)
    untouched[slots[keep]] = False
    assert np.array_equal(flat_k[untouched], k0.reshape(NB * bs, H, d)[untouched])
    assert np.array_equal(flat_v[untouched], v0.reshape(NB * bs, H, d)[untouched])
    try:
        orc.reshape_and_cache(kc, vc, k[:1], v[:1], np.array([NB * bs], dtype=np.int64))
    except ValueError:
        pass
    else:
        raise AssertionError("slot past the pool was accepted")


# ---------------------------------------------------------------------------
# Helpers that build a paged pool from contiguous per-sequence K/V.  The scatter
# is written with numpy block slicing, not with the oracle's element indexing.
# ---------------------------------------------------------------------------

def _paged_from_contiguous(rng, ctx, H_kv, d, bs, extra_blocks=3, nan_pool=True):
    nblk = [-(-int(c) // bs) for c in ctx]
    NB = sum(nblk) + extra_blocks
    MB = max(1, max(nblk))
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((len(ctx), MB), -1, dtype=np.int32)
    fill = SENTINEL if nan_pool else 0
    kc = np.full((NB, bs, H_kv, d), fill, dtype=np.uint16)
    vc = np.full((NB, bs, H_kv, d), fill, dtype=np.uint16)
    Ks, Vs = [], []
    at = 0
    for s, c in enumerate(ctx):
        K = normal_bf16(rng, (int(c), H_kv, d))
        V = normal_bf16(rng, (int(c), H_kv, d))
        Ks.append(K)
        Vs.append(V)
        for i in range(nblk[s]):
            b = perm[at]
            at += 1
            tables[s, i] = b
            rows = K[i * bs:(i + 1) * bs]
            kc[b, :rows.shape[0]] = rows
            vc[b, :rows.shape[0]] = V[i * bs:(i + 1) * bs]
    return kc, vc, tables, Ks, Vs


def _sdpa_rows(q_bits, K_bits, V_bits, scale, q_len, ctx, Hq, Hkv):
    """torch SDPA in fp64 over a contiguous cache (GQA by repeating KV heads).
    The query rows are the last q_len positions of a ctx-long causal prompt: they
    are placed at the bottom of a full [ctx]-row query (other rows zero) and the
    matching rows of the is_causal result are returned."""
    g = Hq // Hkv
    Q = torch.zeros(ctx, Hq, q_bits.shape[-1], dtype=torch.float64)
    Q[ctx - q_len:] = torch.from_numpy(bf16_to_f32(q_bits).astype(np.float64))
    K = torch.from_numpy(bf16_to_f32(K_bits).astype(np.float64)).repeat_interleave(g, dim=1)
    V = torch.from_numpy(bf16_to_f32(V_bits).astype(np.float64)).repeat_interleave(g, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(
        Q.transpose(0, 1), K.transpose(0, 1), V.transpose(0, 1), is_causal=True, scale=scale)
    return o.transpose(0, 1)[ctx - q_len:].numpy()


# ---------------------------------------------------------------------------
# a3-a8 attention
# ---------------------------------------------------------------------------

def pin_paged_equals_contiguous_decode(orc):
    """Decode ([LPNH] §2.3): one query row per sequence at its last position.
    The oracle over a permuted paged pool (unused slots NaN) equals torch's
    scaled_dot_product_attention in fp64 over each sequence's contiguous K/V."""
    rng = _rng(21)
    ctx = [1, 15, 16, 17, 33, 64, 100]
    Hq, Hkv, d, bs = 8, 2, 16, 16
    kc, vc, tables, Ks, Vs = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    q = normal_bf16(rng, (len(ctx), Hq, d))
    scale = 1.0 / math.sqrt(d)
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), scale)
    for s, c in enumerate(ctx):
        ref = _sdpa_rows(q[s:s + 1], Ks[s], Vs[s], scale, 1, c, Hq, Hkv)
        assert np.allclose(out[s:s + 1], ref, rtol=0, atol=1e-12), (s, np.abs(out[s] - ref).max())


def pin_paged_equals_contiguous_chunks(orc):
    """Chunked prefill ([LESSON] "Chunked prefill"): a chunk of q_len rows at the
    end of a ctx-long context is causal over its prefix plus itself, so its rows
    equal the same rows of one causal attention over the whole prompt (torch SDPA
    with is_causal=True, fp64).  Mixed with single-row decodes in one varlen call."""
    rng = _rng(22)
    ctx = [40, 7, 33, 18]
    q_lens = [24, 1, 33, 5]           # 33 = a whole prompt; 1 = a decode row
    Hq, Hkv, d, bs = 4, 1, 8, 16
    kc, vc, tables, Ks, Vs = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = normal_bf16(rng, (int(qsl[-1]), Hq, d))
    scale = 0.3
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), scale,
                              query_start_loc=qsl, causal=True)
    for s, (c, n) in enumerate(zip(ctx, q_lens)):
        ref = _sdpa_rows(q[qsl[s]:qsl[s + 1]], Ks[s], Vs[s], scale, n, c, Hq, Hkv)
        assert np.allclose(out[qsl[s]:qsl[s + 1]], ref, rtol=0, atol=1e-12), s


def pin_non_causal_varlen(orc):
    """With causal off every query row of a sequence sees all context_len keys:
    the rows equal SDPA without a mask."""
    rng = _rng(23)
    ctx, q_lens = [20, 9], [6, 3]
    Hq, Hkv, d, bs = 2, 2, 8, 16
    kc, vc, tables, Ks, Vs = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = normal_bf16(rng, (int(qsl[-1]), Hq, d))
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), 0.5,
                              query_start_loc=qsl, causal=False)
    for s in range(2):
        Q = torch.from_numpy(bf16_to_f32(q[qsl[s]:qsl[s + 1]]).astype(np.float64)).transpose(0, 1)
        K = torch.from_numpy(bf16_to_f32(Ks[s]).astype(np.float64)).transpose(0, 1)
        V = torch.from_numpy(bf16_to_f32(Vs[s]).astype(np.float64)).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=0.5).transpose(0, 1)
        assert np.allclose(out[qsl[s]:qsl[s + 1]], ref.numpy(), rtol=0, atol=1e-12)


def pin_block_permutation_invariance(orc):
    """Physical block ids carry no meaning: moving every block to another slot of
    the pool and rewriting the table leaves the output bit-for-bit unchanged."""
    rng = _rng(31)
    ctx = np.array([50, 3, 77], np.int32)
    Hq, Hkv, d, bs = 4, 2, 8, 16
    kc, vc, tables, _, _ = _paged_from_contiguous(rng, ctx, Hkv, d, bs, extra_blocks=5)
    q = normal_bf16(rng, (3, Hq, d))
    a = orc.paged_attention(q, kc, vc, tables, ctx, 0.25)
    NB = kc.shape[0]
    perm = rng.permutation(NB)             # new home of old block b is perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    b = orc.paged_attention(q, kc2, vc2, tables2, ctx, 0.25)
    assert np.array_equal(a, b)


def pin_single_key_returns_v(orc):
    """context_len = 1: the softmax has one weight, equal to 1, so the output is
    that V row exactly (for every query head of the group)."""
    rng = _rng(41)
    Hq, Hkv, d, bs = 6, 3, 8, 16
    kc, vc, tables, Ks, Vs = _paged_from_contiguous(rng, [1, 1], Hkv, d, bs)
    q = normal_bf16(rng, (2, Hq, d))
    out = orc.paged_attention(q, kc, vc, tables, np.array([1, 1], np.int32), 0.7)
    for s in range(2):
        expect = np.repeat(bf16_to_f32(Vs[s][0]).astype(np.float64), Hq // Hkv, axis=0)
        assert np.array_equal(out[s], expect)


def pin_constant_values(orc):
    """All V rows equal to one vector c: the output is c whatever the scores."""
    rng = _rng(42)
    Hq, Hkv, d, bs = 2, 1, 8, 16
    ctx = [37]
    kc, vc, tables, Ks, _ = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    c = normal_bf16(rng, (d,))
    for b in tables[0][tables[0] >= 0]:
        vc[b] = c
    q = normal_bf16(rng, (1, Hq, d))
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), 1.0)
    assert np.allclose(out[0], bf16_to_f32(c)[None, :], rtol=1e-14, atol=1e-14)


def pin_zero_query_is_mean(orc):
    """q = 0: every score is 0, the weights are uniform and the output is the
    mean of the V rows the query may see."""
    rng = _rng(43)
    Hq, Hkv, d, bs = 2, 2, 8, 16
    ctx = [29, 16]
    kc, vc, tables, _, Vs = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    q = np.zeros((2, Hq, d), np.uint16)
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), 0.5)
    for s in range(2):
        mean = bf16_to_f32(Vs[s]).astype(np.float64).mean(axis=0)
        assert np.allclose(out[s], mean, rtol=0, atol=1e-14)


def pin_dominant_key(orc):
    """A key aligned with the query and scaled far above the rest takes all the
    weight (the others get e^-(>700)): the output is that key's V row."""
    rng = _rng(44)
    Hq, Hkv, d, bs = 1, 1, 4, 16
    ctx = [21]
    kc, vc, tables, Ks, Vs = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    q = bf16_bits(np.array([[[1.0, 1.0, 1.0, 1.0]]], np.float32))
    hot = 13
    b, o = tables[0, hot // bs], hot % bs
    kc[b, o, 0] = bf16_bits(np.full(4, 256.0, np.float32))
    for i in range(ctx[0]):
        if i != hot:
            bb, oo = tables[0, i // bs], i % bs
            kc[bb, oo, 0] = bf16_bits(np.full(4, -1.0, np.float32))
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), 1.0)
    assert np.allclose(out[0, 0], bf16_to_f32(Vs[0][hot, 0]), rtol=0, atol=1e-12)


def pin_gqa_equals_replicated_mha(orc):
    """Grouped heads: 8 query heads over 2 KV heads give the same result as 8
    query heads over 8 KV heads where KV head h holds a copy of grouped head
    h // 4."""
    rng = _rng(51)
    Hq, Hkv, d, bs = 8, 2, 8, 16
    ctx = np.array([30, 5], np.int32)
    kc, vc, tables, _, _ = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    q = normal_bf16(rng, (2, Hq, d))
    a = orc.paged_attention(q, kc, vc, tables, ctx, 0.35)
    kc8 = np.repeat(kc, Hq // Hkv, axis=2)
    vc8 = np.repeat(vc, Hq // Hkv, axis=2)
    b = orc.paged_attention(q, kc8, vc8, tables, ctx, 0.35)
    assert np.array_equal(a, b)


def pin_brute_force_high_precision(orc):
    """Tiny cases against softmax attention evaluated with 40-digit arithmetic
    (mpmath), keys and values read straight from the contiguous arrays."""
    import mpmath
    mpmath.mp.dps = 40
    rng = _rng(61)
    Hq, Hkv, d, bs = 2, 1, 3, 4
    ctx = [1, 6, 11]
    q_lens = [1, 3, 11]
    kc, vc, tables, Ks, Vs = _paged_from_contiguous(rng, ctx, Hkv, d, bs)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = normal_bf16(rng, (int(qsl[-1]), Hq, d))
    scale = 0.61
    out = orc.paged_attention(q, kc, vc, tables, np.array(ctx, np.int32), scale,
                              query_start_loc=qsl, causal=True)
    qf, worst = bf16_to_f32(q), 0.0
    for s in range(3):
        Kf, Vf = bf16_to_f32(Ks[s]), bf16_to_f32(Vs[s])
        for j in range(q_lens[s]):
            r = qsl[s] + j
            visible = ctx[s] - q_lens[s] + j + 1
            for h in range(Hq):
                zs = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(qf[r, h, e])) *
                                                      mpmath.mpf(float(Kf[i, 0, e]))
                                                      for e in range(d)) for i in range(visible)]
                ws = [mpmath.exp(z) for z in zs]
                tot = mpmath.fsum(ws)
                for e in range(d):
                    ref = mpmath.fsum(w * mpmath.mpf(float(Vf[i, 0, e])) for i, w in enumerate(ws)) / tot
                    worst = max(worst, abs(float(ref) - out[r, h, e]))
    assert worst < 1e-13, worst


def pin_empty_context(orc):
    """context_len = 0 (an idle slot in the batch): the output row is zero."""
    rng = _rng(71)
    Hq, Hkv, d, bs = 2, 1, 8, 16
    kc, vc, tables, _, _ = _paged_from_contiguous(rng, [0, 9], Hkv, d, bs)
    q = normal_bf16(rng, (2, Hq, d))
    out = orc.paged_attention(q, kc, vc, tables, np.array([0, 9], np.int32), 0.5)
    assert np.array_equal(out[0], np.zeros((Hq, d)))
    assert np.all(np.isfinite(out[1]))


def pin_rejects_bad_metadata(orc):
    """A block id outside the pool or a query longer than its context is refused."""
    rng = _rng(72)
    Hq, Hkv, d, bs = 2, 1, 8, 16
    kc, vc, tables, _, _ = _paged_from_contiguous(rng, [20], Hkv, d, bs)
    q = normal_bf16(rng, (1, Hq, d))
    bad = tables.copy()
    bad[0, 1] = kc.shape[0]
    for args in ((bad, np.array([20], np.int32), None),
                 (tables, np.array([20], np.int32), np.array([0, 21], np.int32))):
        try:
            qq = q if args[2] is None else normal_bf16(rng, (21, Hq, d))
            orc.paged_attention(qq, kc, vc, args[0], args[1], 0.5, query_start_loc=args[2])
        except ValueError:
            continue
        raise AssertionError("bad metadata accepted")


def pin_chunking_is_invisible(orc):
    """[LESSON] "Chunked prefill": cutting a prompt into consecutive chunks (each
    causal over everything before it) gives every row the same output as one
    causal pass over the whole prompt."""
    rng = _rng(81)
    Hq, Hkv, d, bs = 4, 2, 8, 16
    L = 45
    kc, vc, tables, _, _ = _paged_from_contiguous(rng, [L], Hkv, d, bs)
    q = normal_bf16(rng, (L, Hq, d))
    whole = orc.paged_attention(q, kc, vc, tables, np.array([L], np.int32), 0.4,
                                query_start_loc=np.array([0, L], np.int32))
    rows = []
    for lo, hi in ((0, 16), (16, 32), (32, 45)):
        o = orc.paged_attention(q[lo:hi], kc, vc, tables, np.array([hi], np.int32), 0.4,
                                query_start_loc=np.array([0, hi - lo], np.int32))
        rows.append(o)
    assert np.array_equal(np.concatenate(rows), whole)


# ---------------------------------------------------------------------------
# Shared prefix blocks and copy-on-write ([LPNH] §4.3)
# ---------------------------------------------------------------------------

def pin_copy_blocks_worked_example(orc):
    """A block copy makes block dst equal to block src in both caches and leaves every
    other block, and the source, as they were."""
    rng = _rng(95)
    NB, bs, Hkv, d = 5, 16, 2, 8
    kc = normal_bf16(rng, (NB, bs, Hkv, d))
    vc = normal_bf16(rng, (NB, bs, Hkv, d))
    k0, v0 = kc.copy(), vc.copy()
    orc.copy_blocks(kc, vc, np.array([[3, 0], [1, 4]], np.int32))
    assert np.array_equal(kc[0], k0[3]) and np.array_equal(vc[0], v0[3])
    assert np.array_equal(kc[4], k0[1]) and np.array_equal(vc[4], v0[1])
    for b in (1, 2, 3):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
    try:
        orc.copy_blocks(kc, vc, np.array([[0, NB]], np.int32))
        raise AssertionError("a block id past the pool must be refused")
    except ValueError:
        pass


def pin_shared_prefix_blocks_are_invisible(orc):
    """[LPNH] §4.3: sequences that share a prompt prefix may point at the same read-only
    blocks.  Their outputs equal those of sequences holding private copies of the
    prefix, and the rows a sequence writes after the shared prefix stay its own."""
    rng = _rng(96)
    Hq, Hkv, d, bs = 8, 2, 16, 16
    prefix_blocks = 3
    ctx = [3 * bs + 5, 3 * bs + 16, 3 * bs + 1]
    NB = 16
    kc = normal_bf16(rng, (NB, bs, Hkv, d))
    vc = normal_bf16(rng, (NB, bs, Hkv, d))
    shared = np.array([2, 9, 5], np.int32)
    own = [np.array([11], np.int32), np.array([0], np.int32), np.array([7], np.int32)]
    tables_shared = np.stack([np.concatenate([shared, own[s]]) for s in range(3)])
    # private copies of the prefix for each sequence
    priv = [np.array([1, 3, 4], np.int32), np.array([6, 8, 10], np.int32), np.array([12, 13, 14], np.int32)]
    kp, vp = kc.copy(), vc.copy()
    for s in range(3):
        for i in range(prefix_blocks):
            kp[priv[s][i]] = kc[shared[i]]
            vp[priv[s][i]] = vc[shared[i]]
    tables_priv = np.stack([np.concatenate([priv[s], own[s]]) for s in range(3)])
    q = normal_bf16(rng, (3, Hq, d))
    cl = np.array(ctx, np.int32)
    a = orc.paged_attention(q, kc, vc, tables_shared, cl, 0.3)
    b = orc.paged_attention(q, kp, vp, tables_priv, cl, 0.3)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# FP8 cache (OCP 8-bit floating point, E4M3): the format's definition and
# torch's float8_e4m3fn type (a library implementation of the same format)
# ---------------------------------------------------------------------------

def _torch_e4m3_values(codes):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def pin_e4m3_codes_fixed_by_the_format(orc):
    """Values the E4M3 definition fixes: bias 7, three mantissa bits, subnormals
    m * 2^-9 at exponent 0, largest finite 448, NaN at S.1111.111, no infinities."""
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0,
             0xFE: -448.0}
    for c, v in known.items():
        assert orc.e4m3_decode(c) == v, (hex(c), orc.e4m3_decode(c), v)
    assert math.copysign(1.0, orc.e4m3_decode(0x80)) == -1.0 and orc.e4m3_decode(0x80) == 0.0
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))


def pin_e4m3_decode_matches_torch(orc):
    """Every finite code decodes to torch's float8_e4m3fn value."""
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    ref = _torch_e4m3_values(codes)
    got = np.array([orc.e4m3_decode(c) for c in codes])
    assert np.array_equal(got, ref)


def pin_e4m3_encode_round_to_nearest_even(orc):
    """Encoding: exact values keep their code; a value halfway between two
    neighbouring codes takes the even one; magnitudes past 448 saturate; other
    in-range values agree with torch's float8_e4m3fn cast."""
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c, hex(c)
    for c in range(0, 0x7E):
        lo, hi = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        mid = (lo + hi) / 2  # exact in float32 (at most 5 significant bits)
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == want, (hex(c), mid)
        assert orc.e4m3_encode(-mid) == want | 0x80
    for y in (448.5, 460.0, 480.0, 1e6, 3.0e38):
        assert orc.e4m3_encode(y) == 0x7E and orc.e4m3_encode(-y) == 0xFE
    rng = _rng(91)
    ys = (rng.standard_normal(4000) * np.exp2(rng.uniform(-12, 8, 4000))).astype(np.float32)
    ys = ys[np.abs(ys) <= 448]
    ref = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(y)) for y in ys], dtype=np.uint8)
    assert np.array_equal(got, ref), int(np.count_nonzero(got != ref))


def pin_fp8_write_places_and_quantises(orc):
    """FP8 KV write: the same slots as the bf16 write; with a power-of-two scale,
    a value that is exactly (e4m3 value x scale) is stored as that code, and an
    N(0,1) value x is stored as torch's e4m3 cast of x / scale (exact division)."""
    rng = _rng(92)
    NB, bs, Hkv, d = 6, 16, 2, 8
    T = 9
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = -1  # padding token
    codes_k = rng.integers(0, 0x7E, size=(T, Hkv, d)) | (rng.integers(0, 2, size=(T, Hkv, d)) << 7)
    k_scale, v_scale = 2.0 ** -6, 2.0 ** -5
    kx = np.array([orc.e4m3_decode(int(c)) for c in codes_k.ravel()]).reshape(codes_k.shape) * k_scale
    k = bf16_bits(kx.astype(np.float32))
    assert np.array_equal(bf16_to_f32(k).astype(np.float64), kx)  # exactly representable
    v = normal_bf16(rng, (T, Hkv, d))
    kc = np.full((NB, bs, Hkv, d), 0x7F, np.uint8)
    vc = np.full((NB, bs, Hkv, d), 0x7F, np.uint8)
    orc.reshape_and_cache_fp8(kc, vc, k, v, slots, k_scale, v_scale)
    v_ref = torch.from_numpy(bf16_to_f32(v) / np.float32(v_scale)).to(torch.float8_e4m3fn)
    v_ref = v_ref.view(torch.uint8).numpy()
    for t in range(T):
        if slots[t] < 0:
            continue
        b, o = divmod(int(slots[t]), bs)
        assert np.array_equal(kc[b, o], codes_k[t].astype(np.uint8)), t
        assert np.array_equal(vc[b, o], v_ref[t]), t
    written = np.zeros((NB, bs), bool)
    for t in range(T):
        if slots[t] >= 0:
            written[divmod(int(slots[t]), bs)] = True
    assert np.all(kc[~written] == 0x7F) and np.all(vc[~written] == 0x7F)


def pin_fp8_attention_equals_dequantised_bf16(orc):
    """Attention over an e4m3 pool equals attention over the bf16 pool holding the
    dequantised values (code value x scale, exact in bf16 for power-of-two scales),
    which the bf16 pins tie to torch's SDPA.  Unused slots hold the NaN code."""
    rng = _rng(93)
    ctx = [1, 16, 17, 40, 70]
    Hq, Hkv, d, bs = 8, 2, 16, 16
    nblk = [-(-c // bs) for c in ctx]
    NB = sum(nblk) + 2
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((len(ctx), max(nblk)), -1, np.int32)
    at = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[at:at + n]
        at += n
    kc = np.full((NB, bs, Hkv, d), 0x7F, np.uint8)
    vc = np.full((NB, bs, Hkv, d), 0x7F, np.uint8)
    for s, c in enumerate(ctx):
        for i in range(nblk[s]):
            n = min(bs, c - i * bs)
            kc[tables[s, i], :n] = rng.integers(0, 0x7E, size=(n, Hkv, d)) | (rng.integers(0, 2, size=(n, Hkv, d)) << 7)
            vc[tables[s, i], :n] = rng.integers(0, 0x7E, size=(n, Hkv, d)) | (rng.integers(0, 2, size=(n, Hkv, d)) << 7)
    k_scale, v_scale = 2.0 ** -7, 2.0 ** -4
    lut = np.array([orc.e4m3_decode(c) for c in range(256)])
    kb = bf16_bits((lut[kc] * k_scale).astype(np.float32))
    vb = bf16_bits((lut[vc] * v_scale).astype(np.float32))
    q = normal_bf16(rng, (len(ctx), Hq, d))
    cl = np.array(ctx, np.int32)
    got = orc.paged_attention_fp8(q, kc, vc, k_scale, v_scale, tables, cl, 0.25)
    ref = orc.paged_attention(q, kb, vb, tables, cl, 0.25)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, ref), np.abs(got - ref).max()
    # the same pools under varlen rows (prompt chunks at the end of each context, causal and
    # not, single-token rows among them): still bit-identical to the dequantised bf16 oracle
    q_lens = np.array([1, 5, 17, 1, 33], np.int64)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    qv = normal_bf16(rng, (int(qsl[-1]), Hq, d))
    for causal in (True, False):
        got = orc.paged_attention_fp8(qv, kc, vc, k_scale, v_scale, tables, cl, 0.25, query_start_loc=qsl,
                                      causal=causal)
        ref = orc.paged_attention(qv, kb, vb, tables, cl, 0.25, query_start_loc=qsl, causal=causal)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, ref), np.abs(got - ref).max()


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
