"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own replica;
max-over-ranks time, whole-job throughput, rank 0 alone reports.  No data-path
collective exists (sequences are independent); only the timing is reduced."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    secs = 1.0 + rank            # rank 1 is the slower replica
    mx = d.max(secs)
    tot = d.sum(100.0)
    thr = bench.aggregate(100.0 * world, mx)
    d.barrier()
    d.close()
    q.put((rank, mx, tot, thr))


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_max_time_and_aggregate(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, tot, thr in res:
        assert mx == 2.0               # the slowest rank's time, seen by every rank
        assert tot == 200.0
        assert thr == 100.0            # 2 ranks x 100 units / 2 s


def test_single_process_dist_is_a_no_op():
    import bench
    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", "1"))
    if d.world == 1:
        assert d.max(3.5) == 3.5 and d.sum(2.0) == 2.0
    assert bench.aggregate(10.0, 2.0) == 5.0


def test_algorithmic_bytes_match_cache_count():
    """Bytes the bench counts per layer are the GVA cache scalars x 2 bytes
    (N_GVA = T (G d_h + d_r), GVA analysis page 缓存账本)."""
    import bench
    import oracle
    from gva_inputs import workload
    w = workload("350m")
    assert bench.algorithmic_bytes(w, [4096] * 8) == 8 * oracle.n_gva(4096, 4, 64, 16) * 2
    assert bench.algorithmic_bytes(w, [4096] * 8) == 17825792
    assert bench.gqa_bytes(w, [4096] * 8) == 8 * oracle.n_gqa(4096, 4, 64) * 2
    wl = workload("long")
    assert bench.algorithmic_bytes(wl, [131072] * 2) == 545259520


def test_prefill_work_counts_by_brute_force():
    """The prefill line's algorithmic work: every row of history and chunk read once, and
    H (2 d_h + d_r) multiply-adds for each (query, visible token) pair, counted here by
    enumerating the causal pairs."""
    import bench
    from gva_inputs import workload
    w = workload("350m")
    L0, n = [4080, 0, 17], 16
    nbytes, flops = bench.prefill_work(w, L0, n)
    assert nbytes == sum(l0 + n for l0 in L0) * (w.G * w.d_h + w.d_r) * 2
    pairs = sum(1 for l0 in L0 for i in range(n) for j in range(l0 + n) if j <= l0 + i)
    assert flops == 2 * w.H * (2 * w.d_h + w.d_r) * pairs


def test_prefill_launch_counts():
    """Launches per prefill call the bench claims: three on the tcgen05 path when the
    kernel merges its ranges itself (the 350M chunk), four when the ranges' (max, sum)
    exceed its P buffers (a 148-range split of one group), five on the view paths."""
    import bench
    from gva_inputs import workload
    w = workload("350m")
    assert bench._prefill_chain(w, 16, "auto", 148)[1] == 3
    assert bench._prefill_chain(w, 16, "mma", 148)[1] == 5
    assert bench._prefill_chain(workload("350m", B=1, H=4, G=1), 16, "auto", 148)[1] == 4
    assert bench._prefill_chain(workload("long"), 16, "auto", 148)[1] == 3    # 64 rows, d_h 128
    assert bench._prefill_chain(workload("350m", H=64), 16, "auto", 148)[1] == 5   # 256 rows
