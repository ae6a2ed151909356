"""The N>1 bench path on CPU: world-size-2 gloo process groups check the
max-over-ranks timing rule, the whole-job sum, and that only rank 0 reports."""
import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    m = bench.max_over_ranks(1.5 * (rank + 1), world)
    s = bench.sum_over_ranks(256.0, world)
    bench.barrier(world)
    # reference arm: rank 0 alone prints one JSON line; the other ranks do nothing
    # a sample of 3 layer-tokens that takes 0.3 s per step
    bench.reference_sample = lambda w: ((lambda: 0.3), 3, "fake sample", 1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.main.__globals__["argparse"].Namespace(warmup=0, steps=2), world, rank)
    q.put((rank, m, s, buf.getvalue()))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, s0, out0), (r1, m1, s1, out1) = res
    assert m0 == m1 == 3.0           # the slowest rank's time
    assert s0 == s1 == 512.0         # units processed by all ranks
    line = json.loads(out0.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] == round(3 / (28 * 0.3), 4)          # 3 layer-tokens in 0.3 s, 28 layers per token
    assert line["ms_per_step"] == 300.0                        # the measured time of a step's sample
    assert out1 == ""
