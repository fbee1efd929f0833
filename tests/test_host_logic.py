"""Host logic that needs no GPU: page allocation, the bench's rank
aggregation over two gloo ranks, and the oracle reference arm of bench.py."""

import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ------------------------------------------------------------ page pool
def test_page_pool_allocates_at_block_boundaries_and_reports_oom(golden_dir):
    from mqa_decode_attention_gb300.pages import PagePool

    ex = json.load(open(os.path.join(golden_dir, "paged_example.json")))
    pool = PagePool(num_pages=300, page_size=ex["page_size"])
    # make the free list hand out the example's physical blocks in order
    pool.free.clear()
    pool.free.extend(ex["block_table"] + [0, 1])
    pool.add_sequence(7)
    last = pool.reserve(7, ex["length"])
    assert last == ex["length"] - 1
    assert pool.blocks[7] == ex["block_table"]
    for t, page, off in ex["slots"]:
        assert pool.slot(7, t) == (page, off)
    t = pool.table([7], max_pages=4)
    assert t.tolist() == [ex["block_table"] + [-1]]
    assert pool.seq_lens([7]).tolist() == [42]
    # two blocks left: 32 more tokens fit, the 33rd needs a third block
    pool.add_sequence(8)
    pool.reserve(8, 32)
    with pytest.raises(RuntimeError, match="out of KV pages"):
        pool.reserve(8, 1)
    pool.release(7)
    assert len(pool.free) == 3
    pool.reserve(8, 1)


# ------------------------------------------------------ ranks over gloo
def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    slowest = bench.max_over_ranks(10.0 + rank, world)
    gbs = bench.throughput_gbs(world, 1_000_000, slowest)
    out[rank] = (slowest, gbs)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    manager = mp.Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    slowest, gbs = out[0]
    assert slowest == 11.0  # max over ranks
    assert abs(gbs - 2 * 1_000_000 / 11e-3 / 1e9) < 1e-12


# ------------------------------------------------- reference arm (oracle)
def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["higher_is_better"] is True and d["steps"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
