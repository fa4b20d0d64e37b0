"""Host logic of bench.py's multi-rank path (replicas, no data-path
collective): two gloo ranks on CPU check the barrier and the max-over-ranks
reduction of the step time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    q.put((rank, bench.max_over_ranks(w, 10.0 + rank)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_single_rank_is_identity(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    w, r, l = bench.dist_setup()
    assert (w, r, l) == (1, 0, 0)
    assert bench.max_over_ranks(1, 3.5) == 3.5


def test_traffic_records_match_the_gemm_source():
    """The DRAM-traffic records the bench reports beside its roofline were
    taken on the current GEMM source, for the library's default token block
    (a change to the kernel, or to the default block, needs a new capture)."""
    import bench
    from megatron_transformer_layer_fwd_gb300 import mgb
    src = os.path.join(bench.ROOT, "megatron_transformer_layer_fwd_gb300", "csrc", "gemm_tc.cu")
    rec = bench.traffic_record(src, f"gemm_tc_ce_logits_tb{mgb.CE_DEFAULT_TOKEN_BLOCK}")
    assert rec is not None and rec > 0
