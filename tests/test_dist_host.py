"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2).

The path shards with no data collective: every rank runs its own independent batch (distinct
seeds, same shapes), and the only cross-rank operations are the barrier and the MAX reduction of
the timed milliseconds, which this test exercises.
"""

import multiprocessing as mp
import os
import socket


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from relu_linear_attention_gb300 import synthetic as syn

    r, w, local = bench.dist_env()
    local_ms = 10.0 + 5.0 * rank
    bench.barrier()
    m = bench.max_over_ranks(local_ms)
    seed = bench.rank_seed(1, rank)
    q, _, _ = syn.qkv(seed, (1, 8, 2, 16), "bf16")
    out_q.put((rank, r, w, local, m, seed, q.tobytes()))
    dist.destroy_process_group()


def test_two_gloo_ranks_share_only_timing():
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out_q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out_q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, env_r0, w0, l0, m0, s0, q0), (r1, env_r1, w1, l1, m1, s1, q1) = res
    assert (env_r0, env_r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    assert m0 == m1 == 15.0          # max over ranks of 10 ms and 15 ms
    assert s0 != s1 and q0 != q1     # independent batches per rank (weak scaling)
    # whole-job throughput: units of all ranks over the slowest rank's time
    units_per_rank = 4 * 4096
    assert 2 * units_per_rank / (m0 * 1e-3) == 2 * 4 * 4096 / 0.015
