"""The multi-rank path of bench.py on CPU (gloo, world size 2).

The path shards over independent (batch, kv head) units, so ranks run
replicas and only the timing is reduced: max of the step time over ranks,
sum of the units processed.  This checks that reduction and that the
reference arm runs on rank 0 alone.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist()
    assert d.pg is not None and d.backend == "gloo"
    m = d.max(1.0 + rank)
    s = d.sum(10.0 * (rank + 1))
    d.barrier()
    d.close()
    q.put((rank, m, s))


def test_gloo_two_ranks_reduce_timing():
    if torch.cuda.is_available():
        pytest.skip("CPU-only check of the gloo path")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def _ref_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import contextlib
    import io

    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
                         "--workload", "0", "--cpu-seconds", "0.5"])
    q.put((rank, rc, buf.getvalue()))


def test_reference_arm_prints_on_rank0_only():
    if torch.cuda.is_available():
        pytest.skip("CPU-only check of the gloo path")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    res = dict((r, (rc, out)) for r, rc, out in (q.get(timeout=10) for _ in range(2)))
    assert res[0][0] == 0 and res[1][0] == 0
    assert '"impl": "reference"' in res[0][1]
    assert res[1][1] == ""
