"""Benchmark: one paged-KV attention step of the 128-sequence Llama-3.3-70B-shaped
GQA decode (one layer), on GB300.

A step is the whole hot path over one batch: the slot mapping of the step's new
tokens, the KV write (reshape_and_cache) and decode attention (split-K + merge).

Prints ONE JSON line (rank 0).  `value` is HBM GB/s of the device-timed step over
its algorithmic bytes (KV rows read, queries, outputs, new K/V rows, block-table
entries), with inputs resident in HBM; `e2e` is the same metric through the public
API with the step's inputs copied from pinned host memory and the output copied
back inside the timed region.  `--impl reference` times the fp64 CPU oracle on the
same workload instead.  With --gpus N under torchrun every rank runs its own
replica (the path has no exchange step), and value sums all ranks' bytes over the
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


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--seed", type=int, default=2001)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(b):
    """Bytes the step must move at minimum: every context row of K and V once, the
    queries and outputs once, the new K/V rows read and written once, and the block
    table entries and context lengths read once."""
    Hkv, d, Hq = b.num_kv_heads, b.head_dim, b.num_heads
    kv = int(b.context_lens.astype(np.int64).sum()) * Hkv * d * 2 * 2
    qo = 2 * b.q.size * 2
    new = 2 * 2 * b.k_new.size * 2
    nblk = int(((b.context_lens.astype(np.int64) + 15) // 16).sum())
    meta = nblk * 4 + b.num_seqs * 4 + b.k_new.shape[0] * 8
    attn = kv + qo + nblk * 4 + b.num_seqs * 4
    return kv + qo + new + meta, attn


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed loop runs."""

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
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("paged_decode.cu", "paged_decode.cuh", "pkv_common.cuh", "pkv_split.cuh"):
        with open(os.path.join(ROOT, "pagedattention_paged_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram bytes per decode launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_sha") != kernel_source_sha():
        return None
    return d


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return rank, world, local, pg


def run_reference(args, rank, world, pg):
    """Reference arm: the fp64 oracle on the host cores, one bounded sample per step."""
    import oracle
    from pagedattention_paged_kv_gb300 import workloads as W
    if rank != 0:
        return
    b = W.gqa_decode(seed=args.seed)
    orc = oracle.load()
    total_bytes, _ = algorithmic_bytes(b)
    sample = 16  # sequences per step (all heads)
    sub = np.arange(sample)
    mask = np.zeros(b.num_seqs, np.uint8)
    mask[sub] = 1
    frac = float(b.context_lens[sub].astype(np.int64).sum()) / float(b.context_lens.astype(np.int64).sum())

    def step():
        slots = orc.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, 16)
        kc, vc = b.k_cache, b.v_cache
        orc.reshape_and_cache(kc, vc, b.k_new, b.v_new, slots)
        orc.paged_attention(b.q, kc, vc, b.block_tables, b.context_lens, b.scale, row_mask=mask)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = total_bytes * frac / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "gqa_decode_128seq_llama70b_layer", "num_seqs": 128,
                       "num_heads": 64, "num_kv_heads": 8, "head_dim": 128, "block_size": 16,
                       "context_lens": "uniform[500,2500] seed 2001"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": orc.num_threads(),
                             "kind": "oracle",
                             "sample": f"{sample} of {b.num_seqs} sequences (all heads) per step, "
                                       f"bytes scaled by their share of the context"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(b, seconds_budget=20.0):
    """Times the oracle (as it stands) on a bounded sample of the workload."""
    import oracle
    orc = oracle.load()
    total_bytes, _ = algorithmic_bytes(b)
    sample = 32
    mask = np.zeros(b.num_seqs, np.uint8)
    mask[:sample] = 1
    frac = float(b.context_lens[:sample].astype(np.int64).sum()) / float(b.context_lens.astype(np.int64).sum())
    t0 = time.perf_counter()
    reps = 0
    while True:
        slots = orc.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, 16)
        kc, vc = b.k_cache.copy(), b.v_cache.copy()
        t1 = time.perf_counter()
        orc.reshape_and_cache(kc, vc, b.k_new, b.v_new, slots)
        orc.paged_attention(b.q, kc, vc, b.block_tables, b.context_lens, b.scale, row_mask=mask)
        reps += 1
        el = time.perf_counter() - t0
        if el > seconds_budget / 4 or reps >= 3:
            break
    dt = time.perf_counter() - t1
    return {"value": total_bytes * frac / dt / 1e9, "unit": "GB/s", "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"first {sample} of {b.num_seqs} sequences (all heads, KV write of all tokens), "
                      f"bytes scaled by their share of the total context"}


def main():
    args = parse()
    rank, world, local, pg = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world, pg)
        return
    import torch
    import pagedattention_paged_kv_gb300 as pkv
    from pagedattention_paged_kv_gb300 import workloads as W
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from gpu_helpers import torch_bf16

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    b = W.gqa_decode(seed=args.seed + rank)
    total_bytes, attn_bytes = algorithmic_bytes(b)
    S, Hq, d = b.q.shape
    slots = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, 16)

    kc = torch_bf16(b.k_cache, dev)
    vc = torch_bf16(b.v_cache, dev)
    q = torch_bf16(b.q, dev)
    k_new = torch_bf16(b.k_new, dev)
    v_new = torch_bf16(b.v_new, dev)
    sm = torch.from_numpy(slots).to(dev)
    bt = torch.from_numpy(b.block_tables).to(dev)
    cl = torch.from_numpy(b.context_lens).to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.workspace_size(pkv.OP_DECODE, S, S, Hq, b.num_kv_heads, d), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > L2 (126 MB)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        pkv.reshape_and_cache(kc, vc, k_new, v_new, sm)
        if ev is not None:
            ev[1].record(stream)
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, b.scale, workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    assert pkv.get_device_error() == 0
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)              # evict the previous step's lines from L2
            step(events[i])
        torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[2]) for e in events]
    attn_ms = [e[1].elapsed_time(e[2]) for e in events]
    kv_ms = [e[0].elapsed_time(e[1]) for e in events]
    t_step = sum(step_ms) / len(step_ms)
    if pg is not None:
        import torch.distributed as dist
        tt = torch.tensor([t_step], dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_step = float(tt.item())
    t_attn = sum(attn_ms) / len(attn_ms)
    value = total_bytes * world / (t_step * 1e-3) / 1e9
    peak, peak_kind = peaks()

    # ---- end to end through the public API, host buffers ----
    hq = torch.from_numpy(b.q.view(np.int16)).pin_memory()
    hk = torch.from_numpy(b.k_new.view(np.int16)).pin_memory()
    hv = torch.from_numpy(b.v_new.view(np.int16)).pin_memory()
    hbt = torch.from_numpy(b.block_tables).pin_memory()
    hcl = torch.from_numpy(b.context_lens).pin_memory()
    hout = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    hsm = torch.empty(len(slots), dtype=torch.int64).pin_memory()
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2 + hbt.numel() * 4 + hcl.numel() * 4 + hsm.numel() * 8
    d2h = hout.numel() * 2

    def e2e_step():
        hsm.numpy()[:] = pkv.slot_mapping(b.block_tables, b.new_token_seq, b.new_token_pos, 16)
        q.view(torch.int16).copy_(hq, non_blocking=True)
        k_new.view(torch.int16).copy_(hk, non_blocking=True)
        v_new.view(torch.int16).copy_(hv, non_blocking=True)
        bt.copy_(hbt, non_blocking=True)
        cl.copy_(hcl, non_blocking=True)
        sm.copy_(hsm, non_blocking=True)
        pkv.reshape_and_cache(kc, vc, k_new, v_new, sm)
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, b.scale, workspace=ws)
        hout.copy_(out.view(torch.int16), non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    e2e_times = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    t_e2e = sum(e2e_times) / len(e2e_times)
    if pg is not None:
        import torch.distributed as dist
        tt = torch.tensor([t_e2e], dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_e2e = float(tt.item())

    if rank != 0:
        return
    traffic = recorded_traffic()
    achieved = attn_bytes / (t_attn * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, random block permutation)",
        "config": {"workload": "gqa_decode_128seq_llama70b_layer", "num_seqs": S, "num_heads": Hq,
                   "num_kv_heads": b.num_kv_heads, "head_dim": d, "block_size": 16,
                   "context_lens": f"uniform[500,2500] seed {args.seed}",
                   "sum_context": int(b.context_lens.astype(np.int64).sum()),
                   "num_blocks": b.num_blocks, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (512 MB write); KV pool 2x"
                         f"{b.k_cache.nbytes / 1e6:.0f} MB > L2"},
        "pct_of_peak": 100.0 * value / world / peak,
        "seq_steps_per_s": S * world / (t_step * 1e-3),
        "algorithmic_bytes_per_step": total_bytes,
        "kv_write_us": 1e3 * sum(kv_ms) / len(kv_ms),
        "attention_us": 1e3 * t_attn,
        "e2e": {"value": total_bytes * world / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3},
        "gpu_launches": 3 * args.steps,
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel + paged_decode_merge_kernel",
                     "achieved": achieved, "peak": peak, "peak_kind": f"{peak_kind} (hbm_gbs burst)",
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                     "algorithmic_bytes": attn_bytes},
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
