"""Seeded synthetic inputs for paged-KV attention.

This module only draws numbers and lays them out; it holds none of the
method's arithmetic (no slot mapping, no gather, no attention).  Both the
CUDA path and the fp64 oracle take their inputs from here.

The shapes follow the workloads the pages describe:

* vLLM Serving Internals lesson (aiengineeringfromscratch.com, Phase 17 - 04),
  "Numbers you should remember": Llama 3.3 70B at 128 concurrent requests;
  "PagedAttention as a virtual memory system": 16-token blocks, ~1500-token
  mean use against an 8192-token cap; "Chunked prefill": 512-token slices of a
  32k prompt; "Exercises": request lengths with mean 1500 and std 600.
* "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn), §2.2 BlockManager:
  the pool is ``[num_blocks, block_size, num_heads, head_dim]`` for K and V.

Values are bf16, the round-to-nearest-even of float32 N(0,1) draws, held as
``uint16`` bit patterns.  Every generator takes an explicit seed and uses
numpy's PCG64, so any machine reproduces the same bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even.

    Inputs are finite N(0,1) draws, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exact."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) bf16 bit patterns of the given shape, drawn in fixed-size chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))
    return out.reshape(shape)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class PagedBatch:
    """One attention step over a block-paged KV pool (host arrays).

    ``q`` has one row per query token; ``query_start_loc`` gives each
    sequence's rows (``None`` means one row per sequence, i.e. decode).
    ``k_new``/``v_new`` are the rows this step writes into the pool;
    ``new_token_seq``/``new_token_pos`` say which sequence and absolute
    position each of them belongs to.  ``context_lens`` already counts them.
    """

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    causal: bool
    q: np.ndarray                  # uint16 [total_q, Hq, d]
    k_new: np.ndarray              # uint16 [T, Hkv, d]
    v_new: np.ndarray              # uint16 [T, Hkv, d]
    new_token_seq: np.ndarray      # int32 [T]
    new_token_pos: np.ndarray      # int32 [T]
    k_cache: np.ndarray            # uint16 [NB, bs, Hkv, d]
    v_cache: np.ndarray            # uint16 [NB, bs, Hkv, d]
    block_tables: np.ndarray       # int32 [S, MB], unused entries -1
    context_lens: np.ndarray       # int32 [S]
    query_start_loc: np.ndarray | None = None  # int32 [S+1]
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def q_lens(self) -> np.ndarray:
        if self.query_start_loc is None:
            return np.ones(self.num_seqs, dtype=np.int32)
        return np.diff(self.query_start_loc).astype(np.int32)


def _assign_blocks(rng, nblk: np.ndarray, num_blocks: int, mb: int) -> np.ndarray:
    """Give sequence s the next nblk[s] entries of a seeded permutation of the pool."""
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((len(nblk), mb), -1, dtype=np.int32)
    at = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[at:at + n]
        at += n
    return tables


def make_batch(name: str, *, context_lens, q_lens, num_heads: int, num_kv_heads: int,
               head_dim: int, seed: int, num_blocks: int | None = None, headroom: float = 0.10,
               max_blocks_per_seq: int | None = None, block_size: int = BLOCK_SIZE,
               causal: bool = True, varlen: bool | None = None, pool_fill: str = "normal",
               rng: np.random.Generator | None = None) -> PagedBatch:
    """Lay out one step: pool, block tables, queries and the new K/V rows.

    Each sequence's last ``q_lens[s]`` positions are this step's new tokens
    (written into the pool by the KV-write step); the rest of its context is
    already in the pool.  ``pool_fill`` is ``"normal"`` (N(0,1) bf16 in every
    slot) or ``"nan"`` (bf16 NaN in every slot, so a read of a slot outside the
    context shows up); slots inside a context always hold N(0,1) values.
    """
    rng = rng if rng is not None else np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(context_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    S = len(ctx)
    assert ql.shape == (S,) and np.all(ql <= ctx) and np.all(ql >= 0)
    bs = block_size
    nblk = np.array([_ceil_div(int(c), bs) for c in ctx], dtype=np.int64)
    need = int(nblk.sum())
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil((1.0 + headroom) * need)))
    assert num_blocks >= need
    mb = max_blocks_per_seq if max_blocks_per_seq is not None else max(1, int(nblk.max(initial=1)))
    tables = _assign_blocks(rng, nblk, num_blocks, mb)
    Hq, Hkv, d = num_heads, num_kv_heads, head_dim
    total_q = int(ql.sum())
    q = normal_bf16(rng, (total_q, Hq, d))
    k_new = normal_bf16(rng, (total_q, Hkv, d))
    v_new = normal_bf16(rng, (total_q, Hkv, d))
    if pool_fill == "normal":
        k_cache = normal_bf16(rng, (num_blocks, bs, Hkv, d))
        v_cache = normal_bf16(rng, (num_blocks, bs, Hkv, d))
    elif pool_fill == "nan":
        k_cache = np.full((num_blocks, bs, Hkv, d), 0x7FC0, dtype=np.uint16)
        v_cache = np.full((num_blocks, bs, Hkv, d), 0x7FC0, dtype=np.uint16)
        # Fill the context slots with N(0,1) through the tables (input layout only).
        for s in range(S):
            for i in range(int(nblk[s])):
                n = min(bs, int(ctx[s]) - i * bs)
                b = tables[s, i]
                k_cache[b, :n] = normal_bf16(rng, (n, Hkv, d))
                v_cache[b, :n] = normal_bf16(rng, (n, Hkv, d))
    else:
        raise ValueError(pool_fill)
    seq_of = np.repeat(np.arange(S, dtype=np.int32), ql)
    pos_of = np.concatenate([np.arange(int(c) - int(n), int(c), dtype=np.int32)
                             for c, n in zip(ctx, ql)]) if total_q else np.zeros(0, np.int32)
    if varlen is None:
        varlen = not bool(np.all(ql == 1))
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32) if varlen else None
    return PagedBatch(name=name, num_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=bs,
                      num_blocks=num_blocks, scale=1.0 / math.sqrt(d), causal=causal, q=q,
                      k_new=k_new, v_new=v_new, new_token_seq=seq_of, new_token_pos=pos_of,
                      k_cache=k_cache, v_cache=v_cache, block_tables=tables,
                      context_lens=ctx.astype(np.int32), query_start_loc=qsl,
                      meta={"seed": seed})


def select_seqs(b: PagedBatch, seqs) -> PagedBatch:
    """The same step restricted to sequences `seqs` (same pool; their block-table rows,
    context lengths, query rows and new K/V rows, renumbered 0..len(seqs)-1)."""
    import dataclasses
    seqs = np.asarray(seqs, dtype=np.int64)
    ql = b.q_lens
    qsl = b.query_start_loc if b.query_start_loc is not None else np.arange(b.num_seqs + 1)
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs]) if len(seqs) else np.zeros(0, np.int64)
    new_of_old = np.full(b.num_seqs, -1, np.int64)
    new_of_old[seqs] = np.arange(len(seqs))
    keep = np.isin(b.new_token_seq, seqs)
    new_qsl = None
    if b.query_start_loc is not None:
        new_qsl = np.concatenate([[0], np.cumsum(ql[seqs])]).astype(np.int32)
    return dataclasses.replace(
        b, q=np.ascontiguousarray(b.q[rows]), k_new=np.ascontiguousarray(b.k_new[keep]),
        v_new=np.ascontiguousarray(b.v_new[keep]),
        new_token_seq=new_of_old[b.new_token_seq[keep]].astype(np.int32),
        new_token_pos=np.ascontiguousarray(b.new_token_pos[keep]),
        block_tables=np.ascontiguousarray(b.block_tables[seqs]),
        context_lens=np.ascontiguousarray(b.context_lens[seqs]), query_start_loc=new_qsl,
        meta={**b.meta, "selected_seqs": len(seqs)})


# ---------------------------------------------------------------------------
# FP8 pool: the same step with the pool held as e4m3 codes.
# ---------------------------------------------------------------------------

# K and V scale of the FP8 workloads: a power of two, so x / scale is exact, and
# N(0,1) values times 64 stay far inside the e4m3 range (+-448).
FP8_SCALE = 2.0 ** -6


def to_fp8_pool(b: PagedBatch, k_scale: float = FP8_SCALE, v_scale: float = FP8_SCALE,
                chunk_blocks: int = 2048) -> PagedBatch:
    """The same step with an FP8 pool: each pool byte is torch's float8_e4m3fn cast
    (a library conversion) of the bf16 pool value divided by the scale; NaN slots
    become the NaN code.  The new K/V rows stay bf16 (the KV write quantises them)."""
    import dataclasses

    import torch

    def cast(pool, scale):
        out = np.empty(pool.shape, dtype=np.uint8)
        for i in range(0, pool.shape[0], chunk_blocks):
            f = bf16_to_f32(pool[i:i + chunk_blocks]) / np.float32(scale)
            out[i:i + chunk_blocks] = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return out

    return dataclasses.replace(b, name=b.name + "_fp8", k_cache=cast(b.k_cache, k_scale),
                               v_cache=cast(b.v_cache, v_scale),
                               meta={**b.meta, "kv_dtype": "fp8_e4m3", "k_scale": float(k_scale),
                                     "v_scale": float(v_scale)})


# ---------------------------------------------------------------------------
# The five workloads.  Seeds are (workload index) * 1000 + 1.
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = 1001, **kw) -> PagedBatch:
    """4 sequences, context lengths uniform in [1,100], 4 q heads = 4 KV heads,
    head_dim 64, pool of 64 blocks assigned by a seeded permutation."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(1, 101, size=4)
    return make_batch("tiny_decode", context_lens=ctx, q_lens=np.ones(4, np.int64), num_heads=4,
                      num_kv_heads=4, head_dim=64, seed=seed, num_blocks=64, rng=rng, **kw)


def gqa_decode(seed: int = 2001, num_seqs: int = 128, ctx_lo: int = 500, ctx_hi: int = 2500,
               **kw) -> PagedBatch:
    """Llama-3.3-70B-shaped decode step of one layer: 128 sequences, 64 q heads,
    8 KV heads, head_dim 128, contexts uniform in [500,2500], 10% pool headroom."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=num_seqs)
    return make_batch("gqa_decode", context_lens=ctx, q_lens=np.ones(num_seqs, np.int64),
                      num_heads=64, num_kv_heads=8, head_dim=128, seed=seed, rng=rng, **kw)


def skewed_decode(seed: int = 3001, long_ctx: int = 32768, **kw) -> PagedBatch:
    """64 sequences: 60 with contexts uniform in [256,2048] and 4 at 32768
    (placed at seeded positions); 64 q heads, 8 KV heads, head_dim 128."""
    rng = np.random.Generator(np.random.PCG64(seed))
    short = rng.integers(256, 2049, size=60)
    ctx = np.concatenate([short, np.full(4, long_ctx)])
    ctx = ctx[rng.permutation(64)]
    mb = _ceil_div(long_ctx, BLOCK_SIZE)
    return make_batch("skewed_decode", context_lens=ctx, q_lens=np.ones(64, np.int64),
                      num_heads=64, num_kv_heads=8, head_dim=128, seed=seed, rng=rng,
                      max_blocks_per_seq=mb, **kw)


def mixed_varlen(seed: int = 4001, chunk_start: int = 16384, chunk_len: int = 512,
                 num_decodes: int = 127, **kw) -> PagedBatch:
    """One varlen step: a 512-token chunk at positions 16384-16895 of a 32k prompt
    (causal over its paged prefix plus itself) and 127 single-token decodes with
    contexts uniform in [500,2500]; 64 q heads, 8 KV heads, head_dim 128."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dec = rng.integers(500, 2501, size=num_decodes)
    ctx = np.concatenate([[chunk_start + chunk_len], dec])
    ql = np.concatenate([[chunk_len], np.ones(num_decodes, np.int64)])
    return make_batch("mixed_varlen", context_lens=ctx, q_lens=ql, num_heads=64, num_kv_heads=8,
                      head_dim=128, seed=seed, rng=rng, varlen=True, **kw)


# ---------------------------------------------------------------------------
# Continuous-batching trace: the request stream and per-iteration values.
# ---------------------------------------------------------------------------

@dataclass
class Request:
    req_id: int
    arrival: int        # iteration index at which it joins the waiting queue
    prompt_len: int
    output_len: int
    tokens: np.ndarray | None = None  # prompt token ids (shared-prefix workloads only)


def request_stream(seed: int = 5001, iterations: int = 300, rate: float = 4.0,
                   mean_prompt: float = 1500.0, std_prompt: float = 600.0, max_prompt: int = 8192,
                   out_lo: int = 16, out_hi: int = 512) -> list[Request]:
    """Poisson(rate) arrivals per iteration; log-normal prompt lengths with the
    given mean and std (rounded, clamped to [1, max_prompt]); output lengths
    uniform in [out_lo, out_hi]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sigma2 = math.log1p((std_prompt / mean_prompt) ** 2)
    mu = math.log(mean_prompt) - sigma2 / 2.0
    reqs: list[Request] = []
    for it in range(iterations):
        n = int(rng.poisson(rate))
        for _ in range(n):
            p = int(round(float(rng.lognormal(mu, math.sqrt(sigma2)))))
            p = min(max(p, 1), max_prompt)
            o = int(rng.integers(out_lo, out_hi + 1))
            reqs.append(Request(len(reqs), it, p, o))
    return reqs


def request_stream_shared_prefix(seed: int = 6001, iterations: int = 120, rate: float = 2.0,
                                 num_prefixes: int = 3, vocab: int = 32000) -> list:
    """Requests that share system prompts ("vLLM推理引擎架构PagedAttention机制与高吞吐推理"
    (lpnh.cn) §4.3): num_prefixes system prompts of seeded lengths in [200, 1200] tokens;
    each request = one of them + its own suffix of 1..400 tokens; token ids uniform in
    [0, vocab).  Poisson(rate) arrivals per iteration, outputs uniform in [8, 64].
    Each Request carries .tokens (int64 prompt ids)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    prefixes = [rng.integers(0, vocab, size=int(n)) for n in rng.integers(200, 1201, size=num_prefixes)]
    reqs = []
    rid = 0
    for it in range(iterations):
        for _ in range(int(rng.poisson(rate))):
            p = prefixes[int(rng.integers(0, num_prefixes))]
            suffix = rng.integers(0, vocab, size=int(rng.integers(1, 401)))
            tokens = np.concatenate([p, suffix]).astype(np.int64)
            reqs.append(Request(rid, it, len(tokens), int(rng.integers(8, 65)), tokens))
            rid += 1
    return reqs


def iteration_values(seed: int, iteration: int, total_q: int, num_heads: int, num_kv_heads: int,
                     head_dim: int):
    """Fresh N(0,1) bf16 q, k_new, v_new for one trace iteration."""
    rng = np.random.Generator(np.random.PCG64([seed, iteration]))
    q = normal_bf16(rng, (total_q, num_heads, head_dim))
    k = normal_bf16(rng, (total_q, num_kv_heads, head_dim))
    v = normal_bf16(rng, (total_q, num_kv_heads, head_dim))
    return q, k, v


def length_sample(seed: int, n: int, mean: float, std: float) -> np.ndarray:
    """n request lengths, normal(mean, std) rounded and clamped to >= 1 (the
    fragmentation exercise's trace)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.maximum(1, np.rint(rng.normal(mean, std, size=n))).astype(np.int64)
