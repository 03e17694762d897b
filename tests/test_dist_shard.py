"""The exchange step of one sequence split across ranks, on CPU: two gloo ranks (world size 2).

Each rank holds one shard (consecutive tokens) of the same sequences. It computes its shard's
state increment (here with the fp64 oracle, standing in for rapt_prefill_state, which needs a GPU)
and exchanges it with the binding's gather_shard_states; the L2 moments go through the binding's
allreduce_moments. Checked: the gathered increments arrive in rank order, their exclusive prefix
is the oracle's state of all tokens before the rank's shard (computed over those tokens at once,
not from the shards), their total is the whole sequence's state, and the all-reduced moments are
the whole sequence's moments.
"""

import multiprocessing as mp
import os
import socket

import numpy as np

B, LS, W, H, D = 2, 40, 2, 2, 16


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    from relu_linear_attention_gb300 import synthetic as syn

    q, k, v = syn.qkv(11, (B, W * LS, H, D), "f32")
    g = syn.rng(12)
    return q, k, v, syn.gamma_uniform(g, (H, D)), syn.gamma_uniform(g, (H, D))


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        from relu_linear_attention_gb300 import binding as R

        q, k, v, gq, gk = _inputs()
        r, w = R.shard_rank()
        sl = slice(r * LS, (r + 1) * LS)
        # this rank's shard increment (tokens at global positions r LS + t)
        _, S_r, z_r = O.rla2_prefill(q[:, sl], k[:, sl], v[:, sl], gq, gk, pos_offset=r * LS,
                                     rows=np.array([0]))
        S_parts, z_parts = R.gather_shard_states(torch.from_numpy(S_r), torch.from_numpy(z_r))
        # this rank's L2 moments [K'^T V | K'^T K'] (the definition, RLA page §2.1), all-reduced
        kf = np.maximum(k[:, sl].astype(np.float64), 0.0)
        M = np.concatenate([np.einsum("blhi,blhj->bhij", kf, v[:, sl].astype(np.float64)),
                            np.einsum("blhi,blhj->bhij", kf, kf)], axis=-1)
        M_all = R.allreduce_moments(torch.from_numpy(M)).numpy()
        out_q.put((rank, r, w, S_parts.numpy(), z_parts.numpy(), M_all))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_shard_states():
    import oracle as O

    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, W, port, out_q)) for r in range(W)]
    for p in procs:
        p.start()
    res = sorted((out_q.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v, gq, gk = _inputs()
    for rank, r, w, S_parts, z_parts, M_all in res:
        assert (r, w) == (rank, W)
        assert S_parts.shape == (W, B, H, D, D) and z_parts.shape == (W, B, H, D)
        for j in range(W):  # slot j holds rank j's shard, whichever rank gathered it
            sl = slice(j * LS, (j + 1) * LS)
            _, Sj, zj = O.rla2_prefill(q[:, sl], k[:, sl], v[:, sl], gq, gk, pos_offset=j * LS,
                                       rows=np.array([0]))
            assert np.allclose(S_parts[j], Sj, rtol=0, atol=1e-12)
            assert np.allclose(z_parts[j], zj, rtol=0, atol=1e-12)
        # the state before this rank's shard, from the whole prefix at once
        if r > 0:
            _, Sp, zp = O.rla2_prefill(q[:, :r * LS], k[:, :r * LS], v[:, :r * LS], gq, gk,
                                       rows=np.array([0]))
            assert np.allclose(S_parts[:r].sum(0), Sp, rtol=1e-12, atol=1e-10)
            assert np.allclose(z_parts[:r].sum(0), zp, rtol=1e-12, atol=1e-10)
        _, Sw, zw = O.rla2_prefill(q, k, v, gq, gk, rows=np.array([0]))
        assert np.allclose(S_parts.sum(0), Sw, rtol=1e-12, atol=1e-10)
        assert np.allclose(z_parts.sum(0), zw, rtol=1e-12, atol=1e-10)
        # all-reduced moments = the whole sequence's moments
        kf = np.maximum(k.astype(np.float64), 0.0)
        Mw = np.concatenate([np.einsum("blhi,blhj->bhij", kf, v.astype(np.float64)),
                             np.einsum("blhi,blhj->bhij", kf, kf)], axis=-1)
        assert np.allclose(M_all, Mw, rtol=1e-12, atol=1e-10)
