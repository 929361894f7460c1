"""Benchmark of the paged-KV attention hot path on GB300.

Default workload (the headline): one decode step of one Llama-3.3-70B-shaped layer
over 128 sequences -- 64 query heads, 8 KV heads, head_dim 128, 16-token blocks,
contexts uniform in [500, 2500], blocks scattered by a random permutation of a pool
with 10% headroom.  A step is the whole hot path over one batch: the slot mapping of
the step's new tokens (host), the KV write (reshape_and_cache) and decode attention
(split contexts + log-sum-exp merge).

Prints ONE JSON line (rank 0).  `value` is HBM GB/s over the step's algorithmic bytes
(every context K/V row once, queries, outputs, new rows, block-table entries) with
inputs resident in HBM and larger than L2, timed with CUDA events per step and L2
flushed between steps by reading a 256 MB buffer (so the step starts with an L2 that
holds none of its data and no dirty lines of the flush to write back; `--flush write`
writes the buffer instead);
`e2e` is the same metric with the step's inputs copied from pinned host memory (one
packed copy) and the output copied back inside the timed region.  `--impl reference`
times the fp64 CPU oracle on the same workload instead.  `--config` selects one of
the other workloads (reported, not the headline).  Under torchrun every rank runs its
own replica (the path has no exchange step); value sums the ranks' bytes over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn: HBM GB/s (% of GB300 peak), seq-steps/s at 128 seqs"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20  # > 126 MB of L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--config", default="gqa_decode",
                   choices=["gqa_decode", "tiny_decode", "skewed_decode", "mixed_varlen", "cb_trace",
                            "gqa_decode_fp8", "mixed_varlen_fp8"])
    p.add_argument("--seed", type=int, default=None)
    p.add_argument("--block-size", type=int, default=16,
                   help="tokens per pool block for the decode workloads (8, 16, 32, 64)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--eager-step", action="store_true",
                   help="time the device step as eager library calls instead of replaying it from CUDA "
                        "graphs (the default replays the captured launches, so no host work can fall "
                        "between a step's events)")
    p.add_argument("--flush", choices=["read", "write", "none"], default="read",
                   help="between timed steps: read a 256 MB buffer (evicts the previous step's lines and "
                        "leaves L2 clean), write one (evicts them but leaves ~126 MB of dirty lines that "
                        "the step itself then writes back), or nothing (the inputs are larger than L2)")
    p.add_argument("--e2e-copy", choices=["sm", "engine"], default="sm",
                   help="e2e host<->device transfers: the library's SM copies (pkv.copy_to_device / "
                        "copy_to_host, pinned host memory read and written by the SMs) or torch's copy-engine copies")
    p.add_argument("--part", choices=["all", "chunk", "decodes"], default="all",
                   help="varlen workloads: time the step on its prefill chunks only or its decode rows "
                        "only (the same batch restricted to those sequences)")
    p.add_argument("--no-split", action="store_true",
                   help="decode rows without the split-K: every (sequence, KV-head tile) item whole in one CTA")
    p.add_argument("--separate-kv-write", action="store_true",
                   help="decode workloads: run the KV write as its own launch instead of fused into decode")
    return p.parse_args()


WORKLOADS = {
    "gqa_decode": ("gqa_decode_128seq_llama70b_layer", 2001,
                   {"num_seqs": 128, "num_heads": 64, "num_kv_heads": 8, "head_dim": 128,
                    "block_size": 16, "context_lens": "uniform[500,2500]", "pool_headroom": 0.1}),
    "gqa_decode_fp8": ("gqa_decode_128seq_llama70b_layer_fp8_e4m3_kv", 2001,
                       {"num_seqs": 128, "num_heads": 64, "num_kv_heads": 8, "head_dim": 128,
                        "block_size": 16, "context_lens": "uniform[500,2500]", "pool_headroom": 0.1,
                        "kv_dtype": "fp8_e4m3", "k_scale": 2.0 ** -6, "v_scale": 2.0 ** -6}),
    "tiny_decode": ("tiny_decode_4seq", 1001,
                    {"num_seqs": 4, "num_heads": 4, "num_kv_heads": 4, "head_dim": 64,
                     "block_size": 16, "context_lens": "uniform[1,100]", "num_blocks": 64}),
    "skewed_decode": ("skewed_decode_60short_4x32k", 3001,
                      {"num_seqs": 64, "num_heads": 64, "num_kv_heads": 8, "head_dim": 128,
                       "block_size": 16, "context_lens": "60 x uniform[256,2048] + 4 x 32768"}),
    "mixed_varlen": ("mixed_varlen_512chunk_at_16384_plus_127_decodes", 4001,
                     {"num_seqs": 128, "num_heads": 64, "num_kv_heads": 8, "head_dim": 128,
                      "block_size": 16, "chunk": "512 tokens at positions 16384-16895",
                      "decodes": "127 x context uniform[500,2500]"}),
    "mixed_varlen_fp8": ("mixed_varlen_512chunk_at_16384_plus_127_decodes_fp8_e4m3_kv", 4001,
                         {"num_seqs": 128, "num_heads": 64, "num_kv_heads": 8, "head_dim": 128,
                          "block_size": 16, "chunk": "512 tokens at positions 16384-16895",
                          "decodes": "127 x context uniform[500,2500]", "kv_dtype": "fp8_e4m3",
                          "k_scale": 2.0 ** -6, "v_scale": 2.0 ** -6}),
}


def make_batch(config, seed, block_size=16):
    from pagedattention_paged_kv_gb300 import workloads as W
    if block_size != 16:
        if config not in ("gqa_decode", "gqa_decode_fp8", "skewed_decode"):
            raise SystemExit("--block-size applies to the decode workloads only")
        if config == "gqa_decode_fp8":
            return W.to_fp8_pool(W.gqa_decode(seed=seed, block_size=block_size))
        return {"gqa_decode": W.gqa_decode, "skewed_decode": W.skewed_decode}[config](
            seed=seed, block_size=block_size)
    if config == "gqa_decode_fp8":
        return W.to_fp8_pool(W.gqa_decode(seed=seed))
    if config == "mixed_varlen_fp8":
        return W.to_fp8_pool(W.mixed_varlen(seed=seed))
    return {"gqa_decode": W.gqa_decode, "tiny_decode": W.tiny_decode,
            "skewed_decode": W.skewed_decode, "mixed_varlen": W.mixed_varlen}[config](seed=seed)


def is_fp8(b):
    return b.meta.get("kv_dtype") == "fp8_e4m3"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kv_bytes(b):
    elem = 1 if is_fp8(b) else 2
    return int(b.context_lens.astype(np.int64).sum()) * b.num_kv_heads * b.head_dim * elem * 2


def algorithmic_bytes(b):
    """(step bytes, attention-call bytes): every context row of K and V once, the
    queries and outputs once, the new K/V rows read and written once, block-table
    entries, context lengths and slots read once."""
    nblk = int(((b.context_lens.astype(np.int64) + b.block_size - 1) // b.block_size).sum())
    attn = kv_bytes(b) + 2 * b.q.size * 2 + nblk * 4 + b.num_seqs * 4
    if b.query_start_loc is not None:
        attn += (b.num_seqs + 1) * 4
    elem = 1 if is_fp8(b) else 2
    new = 2 * b.k_new.size * 2 + 2 * b.k_new.size * elem + b.k_new.shape[0] * 8  # read bf16, write cache
    return attn + new, attn


def slot_waste(b):
    """Share of the sequences' block slots that hold no token ([LPNH] §4.1: the cost of
    larger blocks)."""
    ctx = b.context_lens.astype(np.int64)
    slots = ((ctx + b.block_size - 1) // b.block_size * b.block_size).sum()
    return float((slots - ctx.sum()) / max(1, slots))


def chunk_flops(context_lens, q_lens, head_dim, num_heads):
    """Causal attention FLOPs of the multi-token rows: 4 * d * Hq per visible
    (query, key) pair (QK^T and PV, 2 FLOPs per multiply-add)."""
    pairs = 0
    for ctx, ql in zip(context_lens, q_lens):
        ctx, ql = int(ctx), int(ql)
        if ql < 2:
            continue
        first = ctx - ql + 1  # keys seen by the chunk's first row
        pairs += ql * first + ql * (ql - 1) // 2
    return 4 * head_dim * num_heads * pairs


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)  # let the sampler start before the timed loop
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def spread(ms):
    """mean, p10, p50 and p90 of per-step times given in ms, in us."""
    a = np.asarray(ms, dtype=np.float64) * 1e3
    return {"mean": float(a.mean()), "p10": float(np.percentile(a, 10)), "p50": float(np.percentile(a, 50)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "pagedattention_paged_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


DECODE_SOURCES = ("api.cu", "paged_decode.cu", "paged_decode.cuh", "decode_cta.cuh", "attn_block.cuh",
                  "bf16t_block.cuh", "fp8_block.cuh", "kv_quant.cuh", "pkv_common.cuh", "pkv_split.cuh", "merge.cuh")


VARLEN_SOURCES = ("api.cu", "paged_varlen.cu", "paged_varlen.cuh", "prefill_cta.cuh", "paged_prefill.cu",
                  "paged_prefill.cuh", "decode_cta.cuh", "paged_decode.cuh", "tcgen05.cuh", "fp32x2.cuh",
                  "attn_block.cuh", "bf16t_block.cuh", "fp8_block.cuh", "kv_quant.cuh", "pkv_common.cuh",
                  "pkv_split.cuh", "merge.cuh")


def recorded_traffic(name, sources, config):
    """dram bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source and on this bench configuration (else None)."""
    path = os.path.join(ROOT, "profiles", f"{name}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_sha") != kernel_source_sha(sources) or d.get("bench_config") != config:
        return None
    return d


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return rank, world, local, dist
    return rank, world, local, None


def max_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_step_time(b, seqs, threads=None):
    """Times the oracle (as it stands) on the step restricted to `seqs` (all heads),
    KV write of every new token included, on `threads` host threads (all cores if None).
    Returns (seconds, byte share of the sample, threads used)."""
    import oracle
    orc = oracle.load()
    all_threads = orc.num_threads()
    if threads is not None:
        orc.set_num_threads(threads)
    try:
        return _oracle_step_time(orc, b, seqs)
    finally:
        if threads is not None:
            orc.set_num_threads(all_threads)


def _oracle_step_time(orc, b, seqs):
    mask = np.zeros(b.q.shape[0], np.uint8)
    qsl = b.query_start_loc if b.query_start_loc is not None else np.arange(b.num_seqs + 1)
    for s in seqs:
        mask[qsl[s]:qsl[s + 1]] = 1
    share = float(b.context_lens[seqs].astype(np.int64).sum()) / float(b.context_lens.astype(np.int64).sum())
    kc, vc = b.k_cache.copy(), b.v_cache.copy()
    t0 = time.perf_counter()
    slots = orc.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)
    if is_fp8(b):
        ks, vs = b.meta["k_scale"], b.meta["v_scale"]
        orc.reshape_and_cache_fp8(kc, vc, b.k_new, b.v_new, slots, ks, vs)
        orc.paged_attention_fp8(b.q, kc, vc, ks, vs, b.block_tables, b.context_lens, b.scale,
                                query_start_loc=b.query_start_loc, causal=b.causal, row_mask=mask)
    else:
        orc.reshape_and_cache(kc, vc, b.k_new, b.v_new, slots)
        orc.paged_attention(b.q, kc, vc, b.block_tables, b.context_lens, b.scale,
                            query_start_loc=b.query_start_loc, causal=b.causal, row_mask=mask)
    return time.perf_counter() - t0, share, orc.num_threads()


def sample_seqs(b, n):
    return np.arange(min(n, b.num_seqs))


def run_reference(args, rank):
    if rank != 0:
        return
    seed = args.seed if args.seed is not None else WORKLOADS[args.config][1]
    b = make_batch(args.config, seed, args.block_size)
    total, _ = algorithmic_bytes(b)
    seqs = sample_seqs(b, 16)
    warmup = min(args.warmup, 1)   # the oracle has no caches to warm; one untimed run
    for _ in range(warmup):
        oracle_step_time(b, seqs)
    steps = min(args.steps, 5)     # bounded: each step is a sample of the workload
    times = []
    for _ in range(steps):
        dt, share, cores = oracle_step_time(b, seqs)
        times.append(dt)
    dt = sum(times) / len(times)
    value = total * share / dt / 1e9
    name, _, cfg = WORKLOADS[args.config]
    sample = (f"sequences {seqs[0]}..{seqs[-1]} of {b.num_seqs} (all heads, KV write of every new "
              f"token) per step; bytes scaled by their share of the total context")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, **cfg, "seed": seed,
                   "reference_arm_bounds": {"steps_requested": args.steps, "steps_run": steps,
                                            "steps_cap": 5, "warmup_requested": args.warmup,
                                            "warmup_run": warmup, "warmup_cap": 1,
                                            "sequences_per_step": len(seqs)}},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

class Packed:
    """One pinned host buffer and one device buffer with the same layout, holding a
    step's inputs (q, new K/V rows, slots, block tables, context lengths, and
    query_start_loc for varlen), so that one copy moves them all."""

    def __init__(self, arrays: dict, device):
        import torch
        self.offsets, off = {}, 0
        for k, a in arrays.items():
            self.offsets[k] = (off, a.nbytes, a.dtype, a.shape)
            off = (off + a.nbytes + 255) // 256 * 256
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=device)
        hv = self.host.numpy()
        for k, a in arrays.items():
            o, n, _, _ = self.offsets[k]
            hv[o:o + n] = np.frombuffer(np.ascontiguousarray(a).tobytes(), dtype=np.uint8)

    def host_view(self, k):
        o, n, dt, shape = self.offsets[k]
        return self.host.numpy()[o:o + n].view(dt).reshape(shape)

    def dev_view(self, k, torch_dtype):
        o, n, dt, shape = self.offsets[k]
        return self.dev[o:o + n].view(torch_dtype).view(shape)


def run_trace(args, rank, world, local, dist):
    """The continuous-batching trace: 300 scheduler iterations.  Each iteration's host part
    (scheduling, slot mapping, metadata and value copies to the device) runs first and is
    timed on the host; then a 1 GB read evicts L2 and keeps the GPU busy while the host
    enqueues the iteration's launches (block copies, KV write, one varlen attention call),
    and CUDA events around those launches give the device time.  Reports the mean device
    time per iteration (value) and, separately, the host time."""
    import torch
    from pagedattention_paged_kv_gb300 import workloads as W
    from pagedattention_paged_kv_gb300.engine import PagedKVEngine
    from pagedattention_paged_kv_gb300.scheduler import Sequence
    torch.cuda.set_device(local)
    seed = (args.seed if args.seed is not None else 5001) + rank
    NB, Hq, Hkv, d, iters = 65536, 64, 8, 128, 300
    eng = PagedKVEngine(NB, Hq, Hkv, d, max_num_seqs=128, chunk_size=512, device=f"cuda:{local}")
    by_iter = {}
    for r in W.request_stream(seed=seed, iterations=iters):
        by_iter.setdefault(r.arrival, []).append(r)
    stream = torch.cuda.current_stream()
    flush_rd = torch.ones((1 << 30) // 8, dtype=torch.int64, device=f"cuda:{local}")
    sink = torch.empty((), dtype=torch.int64, device=f"cuda:{local}")
    times, host_prep, host_enq, kvb, flops, seq_steps, tokens, launches = [], [], [], 0, 0, 0, 0, 0
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for e0, e1 in evs:
        e0.record(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for it in range(iters):
            t0 = time.perf_counter()
            for r in by_iter.get(it, []):
                eng.add(Sequence(r.req_id, r.prompt_len, r.output_len, r.arrival))
            batch = eng.schedule()
            if batch.num_seqs:
                q, k, v = W.iteration_values(seed, it, batch.num_tokens, Hq, Hkv, d)
                prep = eng.prepare(batch, q, k, v)
                torch.cuda.synchronize()
                t1 = time.perf_counter()
                host_prep.append(t1 - t0)
                torch.sum(flush_rd, dim=0, out=sink)
                e0, e1 = evs[it]
                e0.record(stream)
                t2 = time.perf_counter()
                eng.launch(prep)
                host_enq.append(time.perf_counter() - t2)
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
                ql = np.diff(batch.query_start_loc)
                kvb += int(batch.context_lens[ql == 1].astype(np.int64).sum()) * Hkv * d * 4
                flops += chunk_flops(batch.context_lens, ql, d, Hq)
                seq_steps += int((ql == 1).sum())
                launches += eng.launches(batch)
                tokens += batch.num_tokens
            eng.complete(batch)
    total_ms = max_over_ranks(sum(times), dist)
    if rank != 0:
        return
    frag = eng.sched.fragmentation_report()
    print(json.dumps({
        "metric": "continuous-batching trace: device time per iteration", "value": total_ms / len(times) * 1e3,
        "unit": "us/iteration", "higher_is_better": False, "n_gpus": world, "steps": len(times), "warmup": 0,
        "ms_per_step": total_ms / len(times), "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded request stream and N(0,1) bf16 values)",
        "config": {"workload": "cb_trace_300_iterations", "arrivals": "Poisson(4) per iteration",
                   "prompt": "log-normal mean 1500 std 600, cap 8192", "output": "uniform[16,512]",
                   "max_running": 128, "chunk": 512, "num_blocks": NB, "num_heads": Hq, "num_kv_heads": Hkv,
                   "head_dim": d, "seed": seed,
                   "l2": "a 1 GB read before each iteration's launches (evicts L2; the host enqueues meanwhile)"},
        "device_time": "CUDA events around the iteration's library launches only (block copies, KV write, "
                       "attention); scheduling, slot mapping and the metadata copies run before, on the host",
        "iteration_us": spread(times), "host_prepare_us": spread(host_prep),
        "host_enqueue_us": spread(host_enq),
        "total_ms": total_ms, "decode_kv_gbs": kvb / (total_ms * 1e-3) / 1e9,
        "chunk_tflops_over_total_time": flops / (total_ms * 1e-3) / 1e12,
        "decode_seq_steps_per_s": seq_steps / (total_ms * 1e-3), "tokens": tokens,
        "p50_us": float(np.percentile(times, 50)) * 1e3, "p99_us": float(np.percentile(times, 99)) * 1e3,
        "preemptions": eng.sched.total_preemptions, "finished": len(eng.sched.done),
        "fragmentation": frag,
        "gpu_launches": launches, "clocks": clk.summary(),
    }), flush=True)


def main():
    args = parse()
    rank, world, local, dist = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.config == "cb_trace":
        run_trace(args, rank, world, local, dist)
        return
    import torch
    import pagedattention_paged_kv_gb300 as pkv

    name, default_seed, cfg = WORKLOADS[args.config]
    seed = (args.seed if args.seed is not None else default_seed) + rank
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    b = make_batch(args.config, seed, args.block_size)
    if args.part != "all":
        if b.query_start_loc is None:
            raise SystemExit("--part applies to the varlen workloads")
        from pagedattention_paged_kv_gb300 import workloads as W
        ql = b.q_lens
        b = W.select_seqs(b, np.nonzero(ql >= 2 if args.part == "chunk" else ql == 1)[0])
        name = f"{name} ({args.part} only)"
    if args.no_split:
        pkv.set_decode_split(False)
        name = f"{name} (split-K off)"
    varlen = b.query_start_loc is not None
    total_bytes, attn_bytes = algorithmic_bytes(b)
    S, Hq, d = b.num_seqs, b.num_heads, b.head_dim
    T = b.q.shape[0]
    slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)

    # KV pool: resident state of the serving engine.
    fp8 = is_fp8(b)
    if fp8:
        kc = torch.from_numpy(b.k_cache).to(dev)
        vc = torch.from_numpy(b.v_cache).to(dev)
        ks, vs = b.meta["k_scale"], b.meta["v_scale"]
    else:
        kc = torch.from_numpy(b.k_cache.view(np.int16)).to(dev).view(torch.bfloat16)
        vc = torch.from_numpy(b.v_cache.view(np.int16)).to(dev).view(torch.bfloat16)
    arrays = {"q": b.q, "k": b.k_new, "v": b.v_new, "slots": slots, "tables": b.block_tables,
              "ctx": b.context_lens}
    if varlen:
        arrays["qsl"] = b.query_start_loc
    io = Packed(arrays, dev)
    io.dev.copy_(io.host)
    q = io.dev_view("q", torch.bfloat16)
    k_new, v_new = io.dev_view("k", torch.bfloat16), io.dev_view("v", torch.bfloat16)
    sm = io.dev_view("slots", torch.int64)
    bt, cl = io.dev_view("tables", torch.int32), io.dev_view("ctx", torch.int32)
    qsl = io.dev_view("qsl", torch.int32) if varlen else None
    max_q_len = int(b.q_lens.max())
    out = torch.empty_like(q)
    op = pkv.OP_VARLEN if varlen else pkv.OP_DECODE
    ws = torch.empty(pkv.workspace_size(op, S, T, Hq, b.num_kv_heads, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def l2_flush(i):
        if args.flush == "write":
            flush.fill_(i & 0xFF)              # evict the previous step's lines from L2 (leaves them dirty)
        elif args.flush == "read":
            torch.sum(flush_rd, dim=0, out=flush_sink)  # evict them, leaving clean lines
    stream = torch.cuda.current_stream()

    def attention(o=out, qq=q, qs=qsl, tables=bt, lens=cl):
        if varlen:
            kw = {"k_scale": ks, "v_scale": vs} if fp8 else {}
            pkv.paged_attention_varlen(o, qq, qs, kc, vc, tables, lens, b.scale, causal=b.causal,
                                       max_q_len=max_q_len, workspace=ws, **kw)
        elif fused:
            kw = {"k_scale": ks, "v_scale": vs} if fp8 else {}
            pkv.paged_attention_decode_kvwrite(o, qq, k_new, v_new, kc, vc, tables, lens, b.scale, workspace=ws, **kw)
        elif fp8:
            pkv.paged_attention_decode_fp8(o, qq, kc, vc, tables, lens, b.scale, ks, vs, workspace=ws)
        else:
            pkv.paged_attention_decode(o, qq, kc, vc, tables, lens, b.scale, workspace=ws)

    # decode steps run the KV write inside the decode launch (one new row per sequence)
    fused = not varlen and not args.separate_kv_write and b.k_new.shape[0] == S \
        and np.array_equal(b.new_token_seq, np.arange(S)) and np.array_equal(b.new_token_pos, b.context_lens - 1)

    def kv_write():
        if fused:
            return
        if fp8:
            pkv.reshape_and_cache_fp8(kc, vc, k_new, v_new, sm, ks, vs)
        else:
            pkv.reshape_and_cache(kc, vc, k_new, v_new, sm)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        kv_write()
        if ev is not None:
            ev[1].record(stream)
        attention()
        if ev is not None:
            ev[2].record(stream)

    # Timed steps run on one stream: flush, event, KV write, event, attention, event.  By
    # default the KV write and the attention call are each replayed from a CUDA graph
    # captured once (the same launches as the eager calls), and every event object is
    # created before the loop, so no host work (argument marshalling, descriptor
    # encoding, lazy event creation) can sit between a step's events while the GPU idles.
    ts = torch.cuda.Stream()
    ts.wait_stream(stream)
    with torch.cuda.stream(ts):
        for _ in range(2):  # set-up calls (per-device state, a check of the device flags)
            step()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    kv_graph = attn_graph = None
    if not args.eager_step:
        from pagedattention_paged_kv_gb300.graph import CapturedStep
        kv_graph = None if fused else CapturedStep(kv_write, stream=ts)
        attn_graph = CapturedStep(attention, stream=ts)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for e3 in events:       # create the CUDA events now, outside the timed region
        for e in e3:
            e.record(ts)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    def run_step():
        if kv_graph is not None:
            kv_graph.replay()
        elif args.eager_step:
            kv_write()

    def run_attention():
        if attn_graph is not None:
            attn_graph.replay()
        else:
            attention()

    warmup = max(3, args.warmup)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(ts):
            # the warm-up steps run right before the timed ones (after the clock sampler has
            # started), so the GPU does not sit idle between them
            for i in range(warmup):
                l2_flush(i)
                run_step()
                run_attention()
            for i in range(args.steps):
                l2_flush(i)
                events[i][0].record(ts)
                run_step()
                events[i][1].record(ts)
                run_attention()
                events[i][2].record(ts)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[2]) for e in events]
    attn_ms = [e[1].elapsed_time(e[2]) for e in events]
    kv_ms = [e[0].elapsed_time(e[1]) for e in events]
    t_step = max_over_ranks(sum(step_ms) / len(step_ms), dist)
    t_attn = sum(attn_ms) / len(attn_ms)
    hbm_peak, tc_peak, peak_kind = measured_peaks()
    value = total_bytes * world / (t_step * 1e-3) / 1e9

    # ---- end to end through the public API: inputs from pinned host memory ----
    e2e = None
    if not args.no_e2e:
        hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
        h_slots = io.host_view("slots")

        def device_part():
            if args.e2e_copy == "sm":
                pkv.copy_to_device(io.dev, io.host)
            else:
                io.dev.copy_(io.host, non_blocking=True)
            kv_write()
            attention()
            if args.e2e_copy == "sm":
                pkv.copy_to_host(hout, out)
            else:
                hout.copy_(out, non_blocking=True)

        def host_slots():
            # the fused decode step derives the new token's slot on the device
            if not fused:
                h_slots[:] = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, b.block_size)

        def eager_step():
            host_slots()
            device_part()
            stream.synchronize()

        # the same step with its launches captured once as a CUDA graph (package helper)
        graph_note = None
        try:
            from pagedattention_paged_kv_gb300.graph import CapturedStep
            cap = CapturedStep(device_part)

            def graph_step():
                host_slots()
                cap.replay()
                cap.synchronize()
        except Exception as exc:  # capture not available: report the eager path only
            graph_step, graph_note = None, f"graph capture failed: {type(exc).__name__}"

        def time_e2e(step_fn):
            for _ in range(5):
                step_fn()
            n = min(args.steps, 500)
            times = []
            for i in range(n):
                l2_flush(i)
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                step_fn()
                times.append(time.perf_counter() - t0)
            return max_over_ranks(sum(times) / len(times), dist), n

        t_eager, n_e2e = time_e2e(eager_step)
        t_graph = time_e2e(graph_step)[0] if graph_step is not None else None
        if t_graph is not None:
            # the replayed graph wrote the outputs: check them against the eager step's
            eager_step()
            ref_out = hout.clone()
            hout.zero_()
            graph_step()
            assert torch.equal(hout, ref_out), "graph replay differs from the eager step"
        t_e2e = t_graph if t_graph is not None else t_eager
        e2e = {"value": total_bytes * world / t_e2e / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": io.nbytes, "d2h_bytes_per_step": hout.numel() * 2,
               "ms_per_step": t_e2e * 1e3, "steps": n_e2e,
               "launch": "cuda_graph (pagedattention_paged_kv_gb300.graph.CapturedStep)" if t_graph else "eager",
               "copies": "SM copy kernels over pinned host memory (pkv.copy_to_device / copy_to_host)"
                         if args.e2e_copy == "sm" else "copy engines (torch Tensor.copy_)",
               "eager_ms_per_step": t_eager * 1e3}
        if graph_note:
            e2e["note"] = graph_note

    # ---- varlen only: the chunk alone and the decodes alone ----
    parts = None
    if varlen and args.part == "all":
        parts = varlen_parts(b, pkv, torch, dev, kc, vc, l2_flush, hbm_peak, tc_peak, args.config)

    if rank != 0:
        return
    # The skewed workload's split-K ablation: the same attention call with every (sequence,
    # KV-head tile) item computed whole by one CTA (no partial items, no merge work), timed
    # the same way (graph replay, L2 flushed, events created before the loop).
    ablation = None
    if args.config == "skewed_decode":
        pkv.set_decode_split(False)
        try:
            with torch.cuda.stream(ts):
                for _ in range(2):
                    attention()
            torch.cuda.synchronize()
            assert pkv.get_device_error() == 0
            abl_graph = None
            if not args.eager_step:
                from pagedattention_paged_kv_gb300.graph import CapturedStep
                abl_graph = CapturedStep(attention, stream=ts)
            n_abl = min(args.steps, 50)
            abl_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_abl)]
            for e2 in abl_ev:
                for e in e2:
                    e.record(ts)
            torch.cuda.synchronize()
            with torch.cuda.stream(ts):
                for i in range(warmup + n_abl):
                    l2_flush(i)
                    if i >= warmup:
                        abl_ev[i - warmup][0].record(ts)
                    if abl_graph is not None:
                        abl_graph.replay()
                    else:
                        attention()
                    if i >= warmup:
                        abl_ev[i - warmup][1].record(ts)
            torch.cuda.synchronize()
            assert pkv.get_device_error() == 0
        finally:
            pkv.set_decode_split(True)
        abl_ms = [e[0].elapsed_time(e[1]) for e in abl_ev]
        t_abl = sum(abl_ms) / len(abl_ms)
        ablation = {"what": "split-K off: every (sequence, KV-head tile) item computed whole by one CTA, "
                            "no merge work", "attention_us": 1e3 * t_abl, "timing": spread(abl_ms),
                    "gb_s": attn_bytes / (t_abl * 1e-3) / 1e9, "time_vs_split": t_abl / t_attn}
    launches_per_step = (0 if fused else 1) + (2 if not varlen else pkv.attention_launches(max_q_len))
    line = {
        "metric": METRIC if args.config == "gqa_decode" else f"{name}: HBM GB/s of the step",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 kv / f16 mma / f32 acc" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16, random block permutation" +
                ("; pool = e4m3 codes of x / scale)" if fp8 else ")"),
        "config": {"workload": name, **cfg, "seed": seed, "block_size": b.block_size,
                   "slot_waste": slot_waste(b),
                   "sum_context": int(b.context_lens.astype(np.int64).sum()), "num_blocks": b.num_blocks,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (126 MB) and " + {
                       "write": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB write)",
                       "read": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB read: clean eviction)",
                       "none": "not flushed"}[args.flush] + "; KV pool "
                         f"2 x {b.k_cache.nbytes / 1e6:.0f} MB"},
        "pct_of_peak": 100.0 * value / world / hbm_peak,
        "seq_steps_per_s": S * world / (t_step * 1e-3),
        "algorithmic_bytes_per_step": total_bytes,
        "kv_write_us": 1e3 * sum(kv_ms) / len(kv_ms),
        "kv_write": "fused into the decode launch" if fused else "separate launch",
        "attention_us": 1e3 * t_attn,
        "timing": {"method": ("eager library calls" if args.eager_step else
                              "each timed step replays the captured KV-write and attention graphs") +
                             " on one stream between CUDA events created before the loop",
                   "step_us": spread(step_ms), "attention_us": spread(attn_ms)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if ablation is not None:
        line["split_ablation"] = ablation
    if varlen and args.part == "chunk":
        fl = chunk_flops(b.context_lens, b.q_lens, d, Hq)
        tf = fl / (t_attn * 1e-3) / 1e12
        traffic = recorded_traffic("chunk_fp8" if fp8 else "chunk", VARLEN_SOURCES, args.config)
        line["roofline"] = {"bound": "tensor", "kernel": "paged_varlen_kernel (prefill CTAs; + merges, timed together)",
                            "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": tf / tc_peak,
                            "peak_source": "measured bf16_tflops (burst cuBLAS)",
                            "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                            "algorithmic_flops": fl}
    elif not varlen or args.part == "decodes":
        traffic = recorded_traffic("decode_fp8" if fp8 else "decode", DECODE_SOURCES, args.config)
        if varlen:
            traffic = None  # recorded for the decode-step launch, not for this batch
        achieved = attn_bytes / (t_attn * 1e-3) / 1e9
        line["roofline"] = {
            "bound": "hbm", "kernel": "paged_decode_kernel (+ merge_parts_kernel, timed together)",
            "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
            "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
            "algorithmic_bytes": attn_bytes}
    elif parts is not None:
        line.update(parts)
        overlap_figures(line)
    if not args.no_cpu_baseline:
        dt, share, cores = oracle_step_time(b, sample_seqs(b, 32))
        line["cpu_baseline"] = {
            "value": total_bytes * share / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {min(32, b.num_seqs)} of {b.num_seqs} sequences (all heads, KV write of "
                      f"every new token), one step, bytes scaled by their share of the total context"}
        if args.config in ("tiny_decode", "gqa_decode"):
            n1 = min(8, b.num_seqs)
            dt1, share1, c1 = oracle_step_time(b, sample_seqs(b, n1), threads=1)
            line["cpu_baseline"]["single_thread"] = {
                "value": total_bytes * share1 / dt1 / 1e9, "unit": "GB/s", "cores": c1,
                "sample": f"first {n1} of {b.num_seqs} sequences, one step, one host thread"}
    print(json.dumps(line), flush=True)


def varlen_parts(b, pkv, torch, dev, kc, vc, l2_flush, hbm_peak, tc_peak, config):
    """Times the chunk rows alone and the decode rows alone (same pool, same call)."""
    res = {}
    fp8 = is_fp8(b)
    ql = b.q_lens
    groups = {"chunk": np.nonzero(ql >= 2)[0], "decodes": np.nonzero(ql == 1)[0]}
    for key, seqs in groups.items():
        if len(seqs) == 0:
            continue
        rows = np.concatenate([np.arange(b.query_start_loc[s], b.query_start_loc[s + 1]) for s in seqs])
        qq = torch.from_numpy(b.q[rows].view(np.int16)).to(dev).view(torch.bfloat16)
        qsl = torch.from_numpy(np.concatenate([[0], np.cumsum(ql[seqs])]).astype(np.int32)).to(dev)
        tables = torch.from_numpy(np.ascontiguousarray(b.block_tables[seqs])).to(dev)
        lens = torch.from_numpy(np.ascontiguousarray(b.context_lens[seqs])).to(dev)
        o = torch.empty_like(qq)
        ws = torch.empty(pkv.workspace_size(pkv.OP_VARLEN, len(seqs), qq.shape[0], b.num_heads,
                                            b.num_kv_heads, b.head_dim), dtype=torch.uint8, device=dev)
        mq = int(ql[seqs].max())
        kw = {"k_scale": b.meta["k_scale"], "v_scale": b.meta["v_scale"]} if fp8 else {}

        def call():
            pkv.paged_attention_varlen(o, qq, qsl, kc, vc, tables, lens, b.scale, causal=b.causal,
                                       max_q_len=mq, workspace=ws, **kw)
        for _ in range(5):
            call()
        ts = []
        for i in range(50):
            l2_flush(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        t = float(np.median(ts))
        if key == "chunk":
            fl = chunk_flops(b.context_lens[seqs], ql[seqs], b.head_dim, b.num_heads)
            tf = fl / (t * 1e-3) / 1e12
            res["chunk_us"] = t * 1e3
            res["chunk_tflops"] = tf
            traffic = recorded_traffic("chunk_fp8" if fp8 else "chunk", VARLEN_SOURCES, config)
            res["roofline"] = {"bound": "tensor",
                               "kernel": "paged_varlen_kernel on a chunk-only batch (its prefill CTAs; "
                                         "+ merges, timed together)",
                               "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": tf / tc_peak,
                               "peak_source": "measured bf16_tflops (burst cuBLAS)" + (
                                   " x 1: the fp16 MMAs of the FP8 cache run at the bf16 dense rate"
                                   if fp8 else ""),
                               "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                               "algorithmic_flops": fl}
        else:
            byts = int(b.context_lens[seqs].astype(np.int64).sum()) * b.num_kv_heads * b.head_dim * (2 if fp8 else 4)
            res["decodes_us"] = t * 1e3
            res["decodes_gbs"] = byts / (t * 1e-3) / 1e9
    return res


def overlap_figures(line):
    """How the mixed step compares with its parts run alone: the step's attention call
    over the longer part (1.0 = the shorter part fully hidden) and over their sum."""
    if "chunk_us" in line and "decodes_us" in line:
        a = line["attention_us"]
        line["attention_over_max_of_parts"] = a / max(line["chunk_us"], line["decodes_us"])
        line["attention_over_sum_of_parts"] = a / (line["chunk_us"] + line["decodes_us"])


if __name__ == "__main__":
    main()
