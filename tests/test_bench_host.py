"""Host-side checks of the benchmark's measurement arithmetic: the algorithmic
bytes and flops the roofline fractions divide by, recounted by brute force
from their definitions, and the gate that attaches the recorded DRAM traffic
only to the kernel sources it was captured from.  No GPU."""
import os
import sys
import time

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from varlen_flashattention_causal_gb300 import workloads as W  # noqa: E402


def _visible_pairs(q_len, kv_len):
    """(query, key) pairs a causal, bottom-right-aligned request attends to,
    counted one by one."""
    ctx = kv_len - q_len
    return sum(1 for i in range(q_len) for j in range(kv_len) if j <= ctx + i)


@pytest.mark.parametrize("q_lens,kv_lens", [([6, 4, 17, 33], [6, 4, 17, 33]),
                                             ([1, 5, 9], [40, 5, 30]),
                                             ([3], [3])])
def test_prefill_flops_counts_visible_pairs(q_lens, kv_lens):
    b = W.make_batch(q_lens, kv_lens, 8, 2, 64, 16, seed=3)
    pairs = sum(_visible_pairs(q, k) for q, k in zip(q_lens, kv_lens))
    # Q K^T and P V: 2 flops per multiply-add, D of each per pair and head
    assert bench.prefill_flops(b) == 4 * b.D * b.Hq * pairs


def test_decode_bytes_counts_each_cached_row_once_per_kv_head():
    b = W.make_batch([1, 1, 1], [17, 40, 3], 8, 2, 64, 16, seed=4)
    kv = 0
    for L in b.kv_lens:
        for _tok in range(L):
            kv += b.Hkv * b.D * 2 * 2          # K and V rows of every KV head, bf16
    qo = 2 * b.T * b.Hq * b.D * 2              # q read, out written
    pages = sum(-(-L // b.bs) for L in b.kv_lens)
    assert bench.decode_bytes(b) == kv + qo + pages * 4 + b.B * 4
    # e4m3 caches: one byte per cached value
    assert bench.decode_bytes(b, elem=1) == kv // 2 + qo + pages * 4 + b.B * 4


def test_traffic_gate_follows_the_kernel_sources(monkeypatch):
    t = dict(bench.DECODE_TRAFFIC)
    # recorded bytes are returned only while the sources hash as recorded
    monkeypatch.setattr(bench, "DECODE_TRAFFIC", dict(t, sha256=bench.source_hash(t["sources"])))
    assert bench.decode_traffic() == t["bytes"]
    monkeypatch.setattr(bench, "DECODE_TRAFFIC", dict(t, sha256="0" * 64))
    assert bench.decode_traffic() is None
    monkeypatch.setattr(bench, "DECODE_TRAFFIC", dict(t, bytes=None))
    assert bench.decode_traffic() is None


def test_recorded_traffic_is_close_to_the_algorithmic_bytes():
    """The recorded DRAM traffic of the decode split kernel stays within a few
    percent above the algorithmic bytes (K/V read once per KV head); a value
    far above would mean re-reads, far below a capture of another launch."""
    b = W.decode_llama8b(device="cpu", gen_kv=False)
    alg = bench.decode_bytes(b)
    rec = bench.DECODE_TRAFFIC["bytes"]
    assert 0.99 * alg <= rec <= 1.05 * alg


# ------------------------------------------- several ranks (gloo, CPU)

def _gloo_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        # each rank's own time; the line reports the slowest
        slowest = bench.max_over_ranks(1.5 + rank, ws)

        class Args:
            steps, warmup = 1, 3
        t0 = time.perf_counter()
        ref = bench.run_reference(Args()) if rank != 0 else None     # non-zero ranks return at once
        q.put((rank, ws, r, local, slowest, ref, time.perf_counter() - t0))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_and_only_rank0_works():
    """world_size 2 over gloo: both ranks read their place from the
    environment, agree on the slowest rank's time, and the reference arm does
    no work on rank 1."""
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[:4] for o in out] == [(0, 2, 0, 0), (1, 2, 1, 1)]
    assert all(o[4] == 2.5 for o in out)
    assert out[1][5] is None and out[1][6] < 5.0


def test_reference_arm_prints_one_contract_line(capsys, monkeypatch):
    """bench.py --impl reference on one process: exactly one JSON line with
    the benchmark contract's keys, the device arm's metric, unit and
    workload, a cpu_baseline describing this run, and an e2e object with no
    host<->device bytes (the oracle runs on the host)."""
    import json
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)

    class Args:
        steps, warmup = 1, 3
    bench.run_reference(Args(), budget_s=2.0)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "cpu_baseline", "e2e"} <= set(d)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert (d["n_gpus"], d["steps"], d["warmup"], d["higher_is_better"]) == (1, 1, 3, True)
    assert d["config"]["workload"] == bench.DECODE_WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_prefill_sample_rows_and_their_pairs():
    """The prefill CPU baseline's sample: per_request distinct rows of each
    request (all rows of a shorter one), and its unmasked-pair count
    recounted key by key."""
    b = W.make_batch([5, 40, 1], [9, 60, 30], 8, 2, 64, 16, seed=5)
    per_req = bench.prefill_sample_rows(b, 16, seed=1)
    cu = b.cu_seqlens_q.tolist()
    assert [len(r) for r in per_req] == [5, 16, 1]
    for r, rows in enumerate(per_req):
        assert len(set(rows)) == len(rows) and all(cu[r] <= t < cu[r + 1] for t in rows)
    rows = sorted(t for rr in per_req for t in rr)
    want = 0
    for t in rows:
        r = [i for i in range(b.B) if cu[i] <= t < cu[i + 1]][0]
        i, ctx = t - cu[r], b.kv_lens[r] - b.q_lens[r]
        want += sum(1 for j in range(b.kv_lens[r]) if j <= ctx + i)
    assert bench.rows_pairs(b, rows) == want
    # all rows of the batch: the prefill flop count's pairs
    all_rows = list(range(b.T))
    assert 4 * b.D * b.Hq * bench.rows_pairs(b, all_rows) == bench.prefill_flops(b)
