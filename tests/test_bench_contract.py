"""CPU tests of bench.py's contract: the reference arm's JSON line (single process and
under torchrun with two gloo ranks, where rank 0 alone prints), the max-over-ranks timing
over a world-size-2 gloo group, and the closed forms the bench's work counts use."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny_decode",
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] >= 1 and d["warmup"] >= 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny_decode_4seq"


def test_reference_arm_under_two_ranks_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--config", "tiny_decode", "--gpus", "2", "--steps", "1",
           "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def _max_worker(rank, world, port, out_path):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    b = _bench()
    r, w, _, dist = b.dist_setup()
    assert (r, w) == (rank, world) and dist is not None
    dist.barrier()
    m = b.max_over_ranks(10.0 + 5.0 * rank, dist)
    dist.barrier()
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(repr(m))
    dist.destroy_process_group()


def test_max_over_ranks_over_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    out = str(tmp_path / "max")
    mp.start_processes(_max_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert [float(open(f"{out}.{r}").read()) for r in range(2)] == [15.0, 15.0]


def test_chunk_flops_counts_visible_pairs():
    b = _bench()
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(20):
        ql = int(rng.integers(2, 40))
        ctx = ql + int(rng.integers(0, 100))
        pairs = sum(ctx - ql + j + 1 for j in range(ql))  # row j sees keys 0 .. ctx - ql + j
        assert b.chunk_flops([ctx, 7], [ql, 1], 128, 64) == 4 * 128 * 64 * pairs


def test_algorithmic_bytes_of_a_decode_step():
    b = _bench()
    from pagedattention_paged_kv_gb300 import workloads as W
    batch = W.tiny_decode()
    total, attn = b.algorithmic_bytes(batch)
    ctx = batch.context_lens.astype(np.int64)
    kv = int(ctx.sum()) * batch.num_kv_heads * batch.head_dim * 2 * 2
    blocks = int(((ctx + 15) // 16).sum())
    assert attn == kv + 2 * batch.q.size * 2 + blocks * 4 + batch.num_seqs * 4
    new = batch.k_new.size
    assert total == attn + 2 * new * 2 + 2 * new * 2 + batch.k_new.shape[0] * 8


def test_recorded_traffic_needs_matching_source_and_config(tmp_path, monkeypatch):
    b = _bench()
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "pagedattention_paged_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    rec = {"bench_config": "gqa_decode", "dram_bytes_per_launch": 123, "source_sha": b.kernel_source_sha(["k.cu"])}
    (tmp_path / "profiles" / "x_traffic.json").write_text(json.dumps(rec))
    assert b.recorded_traffic("x", ["k.cu"], "gqa_decode")["dram_bytes_per_launch"] == 123
    assert b.recorded_traffic("x", ["k.cu"], "skewed_decode") is None
    (csrc / "k.cu").write_text("kernel v2")
    assert b.recorded_traffic("x", ["k.cu"], "gqa_decode") is None
