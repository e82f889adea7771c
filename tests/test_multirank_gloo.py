"""The benchmark's multi-rank timing logic on CPU ranks (gloo, world size 2).

The decode path shards by independent (sequence, KV head) rows with no
collective, so N GPUs run N independent replicas; the only cross-rank step is
the barrier and the max-over-ranks reduction of the per-step time, which is
checked here without a GPU.  A rank that fails before the collective is
detected by the other through a short process-group timeout.
"""
import datetime
import os
import socket
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out_q, fail_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    try:
        if rank == fail_rank:
            raise RuntimeError("injected failure before the collective")
        dist.barrier()
        out_q.put((rank, "ok", bench.max_over_ranks(values[rank], world)))
    except Exception as e:  # noqa: BLE001 - reported to the parent
        out_q.put((rank, "error", type(e).__name__))
    finally:
        if rank != fail_rank:
            try:
                dist.destroy_process_group()
            except Exception:  # noqa: BLE001
                pass


def _run(world, values, fail_rank=-1):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, values, q, fail_rank))
             for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, status, val = q.get(timeout=120)
        res[r] = (status, val)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    return res


def test_max_over_ranks_two_ranks():
    assert _run(2, [1.25, 3.5]) == {0: ("ok", 3.5), 1: ("ok", 3.5)}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0


def test_failed_rank_is_detected_by_the_other():
    res = _run(2, [1.0, 2.0], fail_rank=1)
    assert res[1] == ("error", "RuntimeError")
    assert res[0][0] == "error"      # the survivor's collective ends with an error
