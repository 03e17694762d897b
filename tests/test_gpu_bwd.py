"""GPU parity of the causal RLA-2 backward (rapt_prefill_bwd / rapt_varlen_bwd) against the fp64
oracle (oracle/rla2_bwd.py), through the C ABI.

Gradients of sum dout . out w.r.t. q, k, v and the RMSNorm gains (08-rapt-algorithm.md §4.2
"backward"). Tolerance as for the forward: max per-row relative error 1e-4 for fp32 tensors and
2e-2 for bf16 tensors (fp32 arithmetic). The ReLU's derivative jumps at 0, so a row of dq (dk)
whose fp64 pre-activation has an element within 1e-5 of the row's largest magnitude is a decision
the two precisions may take differently; such rows (rare) are left out of the element-wise
comparison, and the gain gradients, which sum over every row, are compared whole. The shapes cover
one and many segments per document (segment boundaries inside and at the end of documents),
ragged last chunks, L = 1, empty and one-token documents, shared and per-head gains, and the full
size of the dense prefill workload on sampled (batch row, head) pairs.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import TOL, draw, gammas, to_dev, to_host, widen
from relu_linear_attention_gb300 import binding as R
from relu_linear_attention_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

EPS_N, BASE, EPS_D = 1e-6, 1e4, 1e-4


def _ambiguous(x, gamma, positions):
    """[n, H] rows whose pre-activation RoPE(RMSNorm(x)) has an element near 0 (relative 1e-5)."""
    n, H, d = x.shape
    bad = np.zeros((n, H), dtype=bool)
    for h in range(H):
        g = gamma[h] if np.ndim(gamma) == 2 else gamma
        y = O.rope_adjacent(O.rmsnorm(x[:, h], g, EPS_N), positions, BASE)
        bad[:, h] = np.min(np.abs(y), axis=1) < 1e-5 * np.max(np.abs(y), axis=1)
    return bad


# Largest share of rows the ReLU-decision carve-out may take: a row needs an element within
# 1e-5 of its largest magnitude, which for d <= 128 normal entries happens in well under 1 % of
# rows; a wider carve-out means the mask itself went wrong (gains or positions passed to it).
MAX_AMBIGUOUS = 0.02


def _keep(x, gamma, positions):
    """Rows compared element by element: all but the ambiguous ones, whose count is bounded."""
    bad = _ambiguous(x, gamma, positions)
    assert bad.sum() <= max(1, MAX_AMBIGUOUS * bad.size), \
        "carve-out too wide: %d of %d rows" % (bad.sum(), bad.size)
    return ~bad


def _row_err(got, ref, keep):
    assert np.isfinite(got).all()  # the rows left out of the comparison included
    return O.relative_error(got[keep], ref[keep])[0]


def _vec_err(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


DENSE_CASES = [
    # (B, L, H, d, dtype, per_head_gamma, pos_offset)
    (1, 64, 2, 16, "f32", False, 0),
    (2, 65, 2, 32, "f32", True, 5),
    (1, 200, 2, 64, "f32", False, 0),
    (1, 129, 1, 128, "f32", True, 1000),
    (2, 63, 2, 16, "bf16", False, 0),
    (1, 1, 1, 128, "bf16", False, 0),
    (2, 300, 2, 64, "bf16", True, 0),
    (1, 1000, 3, 128, "bf16", True, 7),
    (2, 384, 2, 128, "bf16", False, 3),   # whole chunks only: every tile leaves by TMA stores
    (3, 257, 5, 128, "f32", True, 0),
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: "B%dL%dH%dd%d-%s" % c[:5])
def test_prefill_bwd_matches_oracle(cuda_device, lib, case):
    B, L, H, d, dtype, per_head, off = case
    q, k, v = draw(300 + L, (B, L, H, d), dtype)
    (g,) = draw(301 + L, (B, L, H, d), dtype)[:1]
    gq, gk = gammas(302, H, d, per_head)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    dq, dk, dv, dgq, dgk = R.rapt_prefill_bwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                              to_dev(g, dtype), dev(gq), dev(gk), pos_offset=off)
    torch.cuda.synchronize()
    wq, wk, wv, wg = (widen(x, dtype) for x in (q, k, v, g))
    rq, rk, rv, rgq, rgk = O.rla2_prefill_bwd(wq, wk, wv, wg, gq, gk, EPS_N, BASE, EPS_D,
                                              pos_offset=off)
    pos = off + np.arange(L)
    for b in range(B):
        keep_q = _keep(wq[b], gq, pos)
        keep_k = _keep(wk[b], gk, pos)
        assert _row_err(to_host(dq)[b], rq[b], keep_q) <= TOL[dtype]
        assert _row_err(to_host(dk)[b], rk[b], keep_k) <= TOL[dtype]
        assert O.relative_error(to_host(dv)[b], rv[b])[0] <= TOL[dtype]
    assert _vec_err(to_host(dgq), rgq) <= TOL[dtype]
    assert _vec_err(to_host(dgk), rgk) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_varlen_bwd_matches_oracle(cuda_device, lib, dtype, d):
    lens = [1, 0, 65, 130, 3, 0, 64, 257]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H = int(cu[-1]), 2
    q, k, v = draw(310 + d, (T, H, d), dtype)
    (g,) = draw(311 + d, (T, H, d), dtype)[:1]
    gq, gk = gammas(312, H, d, d != 64)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dq, dk, dv, dgq, dgk = R.rapt_varlen_bwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                             to_dev(g, dtype), dev(cu), dev(gq), dev(gk),
                                             max_seqlen=max(lens), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    wq, wk, wv, wg = (widen(x, dtype) for x in (q, k, v, g))
    rq, rk, rv, rgq, rgk = O.rla2_varlen_bwd(wq, wk, wv, wg, cu, gq, gk, EPS_N, BASE, EPS_D)
    pos = np.concatenate([np.arange(n) for n in lens])
    keep_q = _keep(wq, gq, pos)
    keep_k = _keep(wk, gk, pos)
    assert _row_err(to_host(dq), rq, keep_q) <= TOL[dtype]
    assert _row_err(to_host(dk), rk, keep_k) <= TOL[dtype]
    assert O.relative_error(to_host(dv), rv)[0] <= TOL[dtype]
    assert _vec_err(to_host(dgq), rgq) <= TOL[dtype]
    assert _vec_err(to_host(dgk), rgk) <= TOL[dtype]


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_bwd_shared_gains_many_documents(cuda_device, lib, d):
    """Gains shared by the heads of 64 documents: the gain partials (one per document, head and
    128-token chunk) are many, so their sum runs in two stages (splits, then the splits in order);
    checked against the oracle, with every document's dq, dk, dv. The many document ends test the
    keys that few queries see, whose dk is a difference of nearly equal terms."""
    lens = [int(x) for x in np.random.default_rng(380).integers(1, 600, size=64)]
    lens[5] = 0
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H = int(cu[-1]), 4
    q, k, v = draw(381, (T, H, d), "bf16")
    (g,) = draw(382, (T, H, d), "bf16")[:1]
    gq, gk = gammas(383, H, d, False)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dq, dk, dv, dgq, dgk = R.rapt_varlen_bwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                                             to_dev(g, "bf16"), dev(cu), dev(gq), dev(gk),
                                             max_seqlen=max(lens), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    wq, wk, wv, wg = (widen(x, "bf16") for x in (q, k, v, g))
    rq, rk, rv, rgq, rgk = O.rla2_varlen_bwd(wq, wk, wv, wg, cu, gq, gk, EPS_N, BASE, EPS_D)
    pos = np.concatenate([np.arange(n) for n in lens])
    assert _row_err(to_host(dq), rq, _keep(wq, gq, pos)) <= TOL["bf16"]
    assert _row_err(to_host(dk), rk, _keep(wk, gk, pos)) <= TOL["bf16"]
    assert O.relative_error(to_host(dv), rv)[0] <= TOL["bf16"]
    assert _vec_err(to_host(dgq), rgq) <= TOL["bf16"]
    assert _vec_err(to_host(dgk), rgk) <= TOL["bf16"]


def test_prefill_bwd_full_size_sampled(cuda_device, lib):
    """The dense prefill workload (B=4, L=4096, H=16, d=128, bf16, per-head gains) in the bench's
    launch configuration; the oracle checks two whole (batch row, head) pairs. The gains' gradients
    depend on every pair, so they are checked through the one-head restriction: a second call whose
    dout is zero outside the sampled head of the sampled row gives, for that head's gain row, the
    oracle's value of that (row, head) alone."""
    w = syn.prefill_bf16(seed=1)
    B, L, H, d = w.q.shape
    (g,) = draw(320, (B, L, H, d), "bf16")[:1]
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    tq, tk, tv, tg = (to_dev(x, "bf16") for x in (w.q, w.k, w.v, g))
    dq, dk, dv, _, _ = R.rapt_prefill_bwd(tq, tk, tv, tg, dev(w.gamma_q), dev(w.gamma_k))
    torch.cuda.synchronize()
    pos = np.arange(L)
    for b, h in [(0, 0), (3, 15)]:
        qs, ks, vs, gs = (syn.bf16_bits_to_f64(x[b:b + 1, :, h:h + 1]) for x in (w.q, w.k, w.v, g))
        rq, rk, rv, _, _ = O.rla2_prefill_bwd(qs, ks, vs, gs, w.gamma_q[h:h + 1], w.gamma_k[h:h + 1],
                                              EPS_N, BASE, EPS_D)
        keep_q = _keep(qs[0], w.gamma_q[h:h + 1], pos)
        keep_k = _keep(ks[0], w.gamma_k[h:h + 1], pos)
        assert _row_err(to_host(dq[b:b + 1, :, h:h + 1])[0], rq[0], keep_q) <= TOL["bf16"]
        assert _row_err(to_host(dk[b:b + 1, :, h:h + 1])[0], rk[0], keep_k) <= TOL["bf16"]
        assert O.relative_error(to_host(dv[b:b + 1, :, h:h + 1])[0], rv[0])[0] <= TOL["bf16"]
    # gains through one (row, head): dout zero elsewhere
    b, h = 2, 9
    g1 = torch.zeros_like(tg)
    g1[b, :, h] = tg[b, :, h]
    _, _, _, dgq, dgk = R.rapt_prefill_bwd(tq, tk, tv, g1, dev(w.gamma_q), dev(w.gamma_k))
    torch.cuda.synchronize()
    qs, ks, vs, gs = (syn.bf16_bits_to_f64(x[b:b + 1, :, h:h + 1]) for x in (w.q, w.k, w.v, g))
    _, _, _, rgq, rgk = O.rla2_prefill_bwd(qs, ks, vs, gs, w.gamma_q[h:h + 1], w.gamma_k[h:h + 1],
                                           EPS_N, BASE, EPS_D)
    assert _vec_err(to_host(dgq)[h], rgq[0]) <= TOL["bf16"]
    assert _vec_err(to_host(dgk)[h], rgk[0]) <= TOL["bf16"]
    others = np.delete(to_host(dgq), h, axis=0)
    assert np.all(others == 0.0)


def test_prefill_bwd_repeats_bitwise(cuda_device, lib):
    q, k, v = draw(330, (2, 700, 3, 64), "bf16")
    (g,) = draw(331, (2, 700, 3, 64), "bf16")[:1]
    gq, gk = gammas(332, 3, 64, True)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    args = [to_dev(x, "bf16") for x in (q, k, v, g)] + [dev(gq), dev(gk)]
    first = R.rapt_prefill_bwd(*args)
    for _ in range(3):
        again = R.rapt_prefill_bwd(*args)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_bwd_side_stream_and_graph(cuda_device, lib, d):
    """The tensor-core backward forks its critical path onto a stream of its own and joins it back:
    the same bits on the default stream, on another stream, and replayed from a CUDA graph."""
    q, k, v = draw(335, (2, 700, 3, d), "bf16")
    (g,) = draw(336, (2, 700, 3, d), "bf16")[:1]
    gq, gk = gammas(337, 3, d, True)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    args = [to_dev(x, "bf16") for x in (q, k, v, g)] + [dev(gq), dev(gk)]
    first = [t.clone() for t in R.rapt_prefill_bwd(*args)]
    torch.cuda.synchronize()
    side = torch.cuda.Stream(device=cuda_device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        again = R.rapt_prefill_bwd(*args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for a, b in zip(first, again):
        assert torch.equal(a, b)
    outs = [torch.full_like(t, float("nan")) for t in first]
    ws = torch.empty(lib.rapt_prefill_bwd_workspace_size(2, 700, 3, d, 1), dtype=torch.uint8,
                     device=cuda_device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        R.rapt_prefill_bwd(*args, dq=outs[0], dk=outs[1], dv=outs[2], dgamma_q=outs[3],
                           dgamma_k=outs[4], workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(first, outs):
        assert torch.equal(a, b)


def test_prefill_bwd_from_two_threads(cuda_device, lib):
    """Two host threads, each on a stream of its own, run the tensor-core backward at once (each
    thread forks onto a side stream of its own): both give the bits of a call made alone."""
    import threading

    q, k, v = draw(338, (1, 900, 2, 128), "bf16")
    (g,) = draw(339, (1, 900, 2, 128), "bf16")[:1]
    gq, gk = gammas(340, 2, 128, False)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    args = [to_dev(x, "bf16") for x in (q, k, v, g)] + [dev(gq), dev(gk)]
    ref = [t.clone() for t in R.rapt_prefill_bwd(*args)]
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def work(slot):
        try:
            torch.cuda.set_device(cuda_device)
            stream = torch.cuda.Stream(device=cuda_device)
            with torch.cuda.stream(stream):
                outs = None
                for _ in range(3):
                    outs = R.rapt_prefill_bwd(*args)
                stream.synchronize()
            results[slot] = outs
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    for outs in results:
        assert outs is not None
        for a, b in zip(ref, outs):
            assert torch.equal(a, b)


def test_prefill_bwd_without_gains_and_empty(cuda_device, lib):
    q, k, v = draw(340, (1, 40, 2, 32), "f32")
    (g,) = draw(341, (1, 40, 2, 32), "f32")[:1]
    gq, gk = gammas(342, 2, 32, False)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    dq, dk, dv, dgq, dgk = R.rapt_prefill_bwd(to_dev(q, "f32"), to_dev(k, "f32"), to_dev(v, "f32"),
                                              to_dev(g, "f32"), dev(gq), dev(gk), need_gains=False)
    torch.cuda.synchronize()
    assert dgq is None and dgk is None
    rq, rk, rv, _, _ = O.rla2_prefill_bwd(q, k, v, g, gq, gk, EPS_N, BASE, EPS_D)
    assert O.relative_error(to_host(dv), rv)[0] <= TOL["f32"]
    # L = 0: nothing to differentiate, the gain gradients are zero
    z = torch.zeros((2, 0, 2, 32), device=cuda_device)
    _, _, _, dgq, dgk = R.rapt_prefill_bwd(z, z, z, z, dev(gq), dev(gk))
    torch.cuda.synchronize()
    assert torch.all(dgq == 0) and torch.all(dgk == 0)


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (32, "f32")])
def test_varlen_bwd_reports_malformed_cu_seqlens(cuda_device, lib, d, dtype):
    """A decreasing cu_seqlens is reported through dev_status; the well-formed first document is
    still differentiated correctly and nothing is read or written out of bounds."""
    T, H = 300, 2
    q, k, v = draw(350 + d, (T, H, d), dtype)
    (g,) = draw(351 + d, (T, H, d), dtype)[:1]
    gq, gk = gammas(352, H, d, True)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    cu = torch.tensor([0, 200, 150, T], dtype=torch.int32, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dq, dk, dv, _, _ = R.rapt_varlen_bwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype),
                                         to_dev(g, dtype), cu, dev(gq), dev(gk), max_seqlen=T,
                                         need_gains=False, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    wq, wk, wv, wg = (widen(x, dtype)[:200] for x in (q, k, v, g))
    rq, rk, rv, _, _ = O.rla2_varlen_bwd(wq, wk, wv, wg, np.array([0, 200]), gq, gk, EPS_N, BASE,
                                         EPS_D)
    assert O.relative_error(to_host(dv)[:200], rv)[0] <= TOL[dtype]
    keep_k = _keep(wk, gk, np.arange(200))
    assert _row_err(to_host(dk)[:200], rk, keep_k) <= TOL[dtype]


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_bwd_tensor_cores_shared_gains_many_segments(cuda_device, lib, d):
    """bf16 d = 64 or 128 (the tensor-core path; at 64 the tiles carry 64 zero columns) with gains
    shared by the heads, a RoPE offset and two (batch row, head) pairs only, so that every document
    is cut into many segments."""
    B, L, H, off = 2, 900, 1, 9
    q, k, v = draw(360, (B, L, H, d), "bf16")
    (g,) = draw(361, (B, L, H, d), "bf16")[:1]
    gq, gk = gammas(362, H, d, False)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    dq, dk, dv, dgq, dgk = R.rapt_prefill_bwd(to_dev(q, "bf16"), to_dev(k, "bf16"),
                                              to_dev(v, "bf16"), to_dev(g, "bf16"), dev(gq),
                                              dev(gk), pos_offset=off)
    torch.cuda.synchronize()
    wq, wk, wv, wg = (widen(x, "bf16") for x in (q, k, v, g))
    rq, rk, rv, rgq, rgk = O.rla2_prefill_bwd(wq, wk, wv, wg, gq, gk, EPS_N, BASE, EPS_D,
                                              pos_offset=off)
    pos = off + np.arange(L)
    for b in range(B):
        assert _row_err(to_host(dq)[b], rq[b], _keep(wq[b], gq, pos)) <= TOL["bf16"]
        assert _row_err(to_host(dk)[b], rk[b], _keep(wk[b], gk, pos)) <= TOL["bf16"]
        assert O.relative_error(to_host(dv)[b], rv[b])[0] <= TOL["bf16"]
    assert _vec_err(to_host(dgq), rgq) <= TOL["bf16"]
    assert _vec_err(to_host(dgk), rgk) <= TOL["bf16"]


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_bwd_multi_block_segments_sampled(cuda_device, lib, d):
    """Tensor-core backward over 4 documents x 16 heads (64 (document, head) pairs, so the plan
    cuts documents into two segments of several blocks each): a full-length document, one whose
    second segment ends inside its first suffix block, one whose second segment ends inside its
    second block, and one shorter than a segment (no prefix or suffix blocks at all). The oracle
    checks whole (document, head) pairs; positions restart at every document."""
    lens = [4096, 3000, 4005, 1500]
    cu = syn.cu_seqlens_from_lengths(lens)
    T, H = int(cu[-1]), 16
    q, k, v = draw(370, (T, H, d), "bf16")
    (g,) = draw(371, (T, H, d), "bf16")[:1]
    gq, gk = gammas(372, H, d, True)
    dev = lambda x: torch.from_numpy(x).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    dq, dk, dv, _, _ = R.rapt_varlen_bwd(to_dev(q, "bf16"), to_dev(k, "bf16"), to_dev(v, "bf16"),
                                         to_dev(g, "bf16"), dev(cu), dev(gq), dev(gk),
                                         max_seqlen=max(lens), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for doc, h in [(1, 3), (2, 10), (3, 0), (0, 15)]:
        s, e = int(cu[doc]), int(cu[doc + 1])
        pos = np.arange(e - s)
        qs, ks, vs, gs = (widen(x[s:e, h:h + 1][None], "bf16") for x in (q, k, v, g))
        rq, rk, rv, _, _ = O.rla2_prefill_bwd(qs, ks, vs, gs, gq[h:h + 1], gk[h:h + 1], EPS_N, BASE,
                                              EPS_D)
        keep_q = _keep(qs[0], gq[h:h + 1], pos)
        keep_k = _keep(ks[0], gk[h:h + 1], pos)
        assert _row_err(to_host(dq[s:e, h:h + 1]), rq[0], keep_q) <= TOL["bf16"]
        assert _row_err(to_host(dk[s:e, h:h + 1]), rk[0], keep_k) <= TOL["bf16"]
        assert O.relative_error(to_host(dv[s:e, h:h + 1]), rv[0])[0] <= TOL["bf16"]
