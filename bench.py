"""Benchmark of the RLA-2 / RAPT hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one causal RLA-2 prefill (RMSNorm -> RoPE -> ReLU features, chunked causal linear
attention with the fp32 state, Sum-denominator epilogue, final state) over one batch of the
headline workload: B=4 sequences x L=4096 tokens, H=16 heads, d=128, bf16 in/out, per-head
RMSNorm gains ~ U(0.8, 1.2). Inputs are seeded synthetic N(0, 1) (no dataset exists for this
kernel). Rank 0 prints one JSON line; `value` is prefill tokens/s over all ranks (weak scaling:
every rank runs its own independent batch, no collective on the data path).

The same line carries, measured in the same run: the decode step (256 sequences x 32 heads,
d=128, state prefilled from 512 tokens, 64 steps), the packed varlen forward (T=65536, H=32,
d=64) and the original-RLA L2 forward (B=2, L=16384, H=16, d=128) as sub-objects; the roofline
of the dominant prefill kernel (algorithmic bytes / CUDA-event time vs the measured HBM copy
bandwidth); an end-to-end number through the public API with host buffers; SM clocks sampled
during the timed region; and the fp64 oracle timed on a bounded sample on the host cores.

`--impl reference` times the fp64 CPU oracle (the only reference implementation: the pages
publish no runnable code) on the same workload, one bounded sample per step.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RAPT causal prefill tokens/s + decode tokens/s on 1 GB300; % of TC/HBM roofline"
WORKLOAD = dict(name="rla2_causal_prefill", B=4, L=4096, H=16, d=128, dtype="bf16")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20  # > 129 MB of L2


# ----------------------------------------------------------------------------- host helpers
def headline_config(world: int) -> dict:
    """The workload dictionary both arms print (the GPU arm and the oracle reference arm)."""
    return {"workload": "rla2_causal_prefill B=4 L=4096 H=16 d=128 bf16 (fp32 state)",
            "model": "RLA-2/RAPT attention layer (no projections)",
            "global_batch": WORKLOAD["B"] * world, "seq_len": WORKLOAD["L"],
            "heads": WORKLOAD["H"], "d_head": WORKLOAD["d"],
            "parallelism": "dp%d (independent batch per GPU)" % world,
            "l2": "256 MiB write, then 256 MiB read, before every timed step, outside the CUDA events"}


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.processor() or platform.machine()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base: int, rank: int) -> int:
    """Seed of a rank's independent batch (weak scaling: rank r draws its own inputs)."""
    return int(base) + 1000 * int(rank)


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar over the process group (the identity without one)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def prefill_bytes(B, L, H, d, elem=2):
    """Algorithmic HBM bytes of one prefill: read q, k, v and write out, once each."""
    return 4 * B * L * H * d * elem


def prefill_flops(B, L, H, d):
    """Algorithmic flops per token-head: state update 2d^2, readout 2d^2, z and q.z 4d."""
    return B * L * H * (4 * d * d + 4 * d)


def decode_bytes(N, H, d, elem=2):
    """Per step: S read + write (fp32), z read + write, q, k, v read and out write."""
    return N * H * (2 * d * d * 4 + 2 * d * 4 + 4 * d * elem)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.rows = []
        self.proc = None
        self.err = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError) as e:
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"error": self.err or "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        mhz = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(mhz)}


# ----------------------------------------------------------------------------- oracle timing
def oracle_sample(budget_s: float, seed: int):
    """Times the fp64 oracle on whole (batch row, head) pairs of the headline workload until
    ``budget_s`` seconds of CPU work have passed. Returns (tokens/s, pairs, seconds, cores)."""
    import oracle as O
    from relu_linear_attention_gb300 import synthetic as syn

    w = syn.prefill_bf16(seed=seed)
    q, k, v = (syn.bf16_bits_to_f64(x) for x in (w.q, w.k, w.v))
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    done = 0
    t0 = time.perf_counter()
    while done < len(pairs) and (time.perf_counter() - t0) < budget_s:
        O.rla2_prefill(q, k, v, w.gamma_q, w.gamma_k, pairs=[pairs[done]])
        done += 1
    dt = time.perf_counter() - t0
    # one pair is L tokens of one of H heads: tokens/s = pairs * L / H / seconds
    return done * w.L / w.H / dt, done, dt, os.cpu_count()


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, one (batch row, head) pair of the
    headline workload per step, rank 0 only."""
    if rank != 0:
        return 0
    import oracle as O
    from relu_linear_attention_gb300 import synthetic as syn

    w = syn.prefill_bf16(seed=rank_seed(1, 0))
    q, k, v = (syn.bf16_bits_to_f64(x) for x in (w.q, w.k, w.v))
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    for i in range(args.warmup):
        O.rla2_prefill(q, k, v, w.gamma_q, w.gamma_k, pairs=[pairs[i % len(pairs)]])
    t0 = time.perf_counter()
    for i in range(args.steps):
        O.rla2_prefill(q, k, v, w.gamma_q, w.gamma_k, pairs=[pairs[(args.warmup + i) % len(pairs)]])
    dt = time.perf_counter() - t0
    value = args.steps * w.L / w.H / dt
    sample = "%d (batch row, head) pairs of B=4 L=4096 H=16 d=128, all rows, fp64 quadratic form" % args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(world),
        "runs_on": "host cores, fp64 numpy oracle, rank 0 only",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                         "cpu_model": host_cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU arm
def _bf(t_np, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(t_np).view(np.int16)).view(torch.bfloat16).to(device)


def _events(n):
    import torch

    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_steps(fn, steps, warmup, flush, min_warm_s=0.0, counter=None):
    """Runs ``warmup`` untimed steps (at least ``min_warm_s`` seconds), then ``steps`` steps each
    bracketed by CUDA events on the current stream with an L2 flush before it (outside the
    events). Returns the list of per-step milliseconds, and with ``counter`` (a function reading
    the library's launch counter) also the number of library launches in the timed steps."""
    import torch

    t0 = time.perf_counter()
    i = 0
    while i < warmup or (time.perf_counter() - t0) < min_warm_s:
        flush()
        fn()
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    ev0, ev1 = _events(steps), _events(steps)
    c0 = counter() if counter else 0
    for s in range(steps):
        flush()
        ev0[s].record()
        fn()
        ev1[s].record()
    launches = (counter() - c0) if counter else None
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    return (ms, launches) if counter else ms


def profile_case(args):
    """One workload's calls, ``--warmup`` + ``--steps`` times with no timing, for an ncu capture
    (``--only``): a small, single-purpose command whose launches are easy to select."""
    import torch

    from relu_linear_attention_gb300 import _build, _lib, binding as R, synthetic as syn

    _build.ensure_built()
    lib = _lib.load()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    if args.only == "prefill":
        w = syn.prefill_bf16(seed=1)
        q, k, v = (_bf(x, device) for x in (w.q, w.k, w.v))
        gq, gk = (torch.from_numpy(x).to(device) for x in (w.gamma_q, w.gamma_k))
        out = torch.empty_like(q)
        call = lambda: R.rapt_prefill_fwd(q, k, v, gq, gk, out=out)
    elif args.only == "varlen":
        wv = syn.varlen_bf16(seed=2)
        q, k, v = (_bf(x, device) for x in (wv.q, wv.k, wv.v))
        cu = torch.from_numpy(wv.cu_seqlens).to(device)
        g = torch.ones(64, dtype=torch.float32, device=device)
        out = torch.empty_like(q)
        msl = int(wv.lengths.max())
        call = lambda: R.rapt_varlen_fwd(q, k, v, cu, g, g, max_seqlen=msl, out=out)
    elif args.only == "bidir":
        w = syn.prefill_bf16(seed=1)
        q, k, v = (_bf(x, device) for x in (w.q, w.k, w.v))
        gq, gk = (torch.from_numpy(x).to(device) for x in (w.gamma_q, w.gamma_k))
        out = torch.empty_like(q)
        call = lambda: R.rapt_bidir_fwd(q, k, v, gq, gk, out=out)
    elif args.only == "backward":
        w = syn.prefill_bf16(seed=1)
        q, k, v = (_bf(x, device) for x in (w.q, w.k, w.v))
        gq, gk = (torch.from_numpy(x).to(device) for x in (w.gamma_q, w.gamma_k))
        tg = torch.empty_like(q).normal_(generator=torch.Generator(device=device).manual_seed(5))
        call = lambda: R.rapt_prefill_bwd(q, k, v, tg, gq, gk)
    elif args.only == "varlen_backward":
        wv = syn.varlen_bf16(seed=2)
        q, k, v = (_bf(x, device) for x in (wv.q, wv.k, wv.v))
        cu = torch.from_numpy(wv.cu_seqlens).to(device)
        g = torch.ones(64, dtype=torch.float32, device=device)
        tg = torch.empty_like(q).normal_(generator=torch.Generator(device=device).manual_seed(6))
        msl = int(wv.lengths.max())
        call = lambda: R.rapt_varlen_bwd(q, k, v, tg, cu, g, g, max_seqlen=msl)
    elif args.only == "linear":
        gen = torch.Generator(device=device).manual_seed(6)
        x = torch.empty((16384, 2048), dtype=torch.bfloat16, device=device).normal_(generator=gen)
        w = torch.empty((6144, 2048), dtype=torch.bfloat16, device=device).normal_(generator=gen)
        y = torch.empty((16384, 6144), dtype=torch.bfloat16, device=device)
        call = lambda: R.rapt_linear_fwd(x, w, out=y)
    elif args.only == "l2_causal":
        wl = syn.l2_bf16(seed=4)
        q, k, v = (_bf(x, device) for x in (wl.q, wl.k, wl.v))
        out = torch.empty_like(q)
        call = lambda: R.rla_l2_causal_fwd(q, k, v, eps=1e-6, out=out)
    elif args.only == "l2":
        wl = syn.l2_bf16(seed=4)
        q, k, v = (_bf(x, device) for x in (wl.q, wl.k, wl.v))
        out = torch.empty_like(q)
        call = lambda: R.rla_l2_fwd(q, k, v, eps=1e-6, out=out)
    else:
        raise SystemExit("unknown --only case %r" % args.only)
    n0 = lib.rapt_launch_counter()
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.only, "calls": args.warmup + args.steps,
                      "launches": int(lib.rapt_launch_counter() - n0)}))
    return 0


def run_gpu(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from relu_linear_attention_gb300 import _build, _lib, binding as R, synthetic as syn

    _build.ensure_built()
    lib = _lib.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    peaks, peak_src = load_peaks()
    # L2 flush before every timed step: write a buffer larger than L2, then read another one, so
    # that the timed step starts with none of its data in L2 and with no dirty flush lines left to
    # write back inside its events
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    flush_sink = torch.empty((), dtype=torch.float32, device=device)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sink)

    # ---------------- headline: dense causal prefill
    B, L, H, d = WORKLOAD["B"], WORKLOAD["L"], WORKLOAD["H"], WORKLOAD["d"]
    w = syn.prefill_bf16(seed=rank_seed(1, rank))
    q, k, v = (_bf(x, device) for x in (w.q, w.k, w.v))
    gq, gk = (torch.from_numpy(x).to(device) for x in (w.gamma_q, w.gamma_k))
    out = torch.empty_like(q)
    Sf = torch.empty((B, H, d, d), dtype=torch.float32, device=device)
    zf = torch.empty((B, H, d), dtype=torch.float32, device=device)
    step = lambda: R.rapt_prefill_fwd(q, k, v, gq, gk, out=out, S_final=Sf, z_final=zf)

    clocks = ClockSampler(local)
    barrier(device)
    torch.cuda.synchronize()
    ms, timed_launches = time_steps(step, args.steps, args.warmup, flush, min_warm_s=1.0,
                                    counter=lib.rapt_launch_counter)
    barrier(device)
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(ms), device)
    ms_step = total_ms / args.steps
    value = world * B * L / (ms_step * 1e-3)
    mean_ms = statistics.fmean(ms)
    alg_bytes = prefill_bytes(B, L, H, d)
    achieved = alg_bytes / (mean_ms * 1e-3) / 1e9

    # ---------------- end to end through the public API with pinned host buffers
    # (rapt_prefill_fwd_host: the batch rows' copies in, kernels and copies out overlap on a
    # copy-in stream, the compute stream and a copy-out stream; the device staging lives in the
    # caller's workspace)
    qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hws = torch.empty(lib.rapt_prefill_host_workspace_size(B, L, H, d, 1), dtype=torch.uint8,
                      device=device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def e2e_step():
        R.rapt_prefill_fwd_host(qh, kh, vh, gq, gk, out=oh, workspace=hws, copy_in=s_in,
                                copy_out=s_out)

    e2e_ms = time_steps(e2e_step, args.steps, args.warmup, flush)
    e2e_total = max_over_ranks(sum(e2e_ms), device)
    e2e_value = world * B * L / (e2e_total / args.steps * 1e-3)
    h2d = 3 * q.numel() * q.element_size()
    d2h = out.numel() * out.element_size()
    del qh, kh, vh, oh, hws

    # ---------------- decode: 256 x 32 heads, d=128, state from 512 prefill tokens, 64 steps
    Nd, Pd, Hd, dd, nsteps = 256, 512, 32, 128, 64
    pre = syn.decode_prefix(seed=rank_seed(3, rank))
    pq, pk, pv = (_bf(x, device) for x in (pre.q, pre.k, pre.v))
    g1 = torch.ones(dd, dtype=torch.float32, device=device)
    _, S_init, z_init = R.rapt_prefill_fwd(pq, pk, pv, g1, g1, final_state=True)
    del pq, pk, pv, pre
    toks = [syn.decode_step_tokens(seed=rank_seed(3, rank), step=t) for t in range(nsteps)]
    tq = torch.stack([_bf(t.q, device) for t in toks])
    tk = torch.stack([_bf(t.k, device) for t in toks])
    tv = torch.stack([_bf(t.v, device) for t in toks])
    tp = torch.stack([torch.from_numpy(t.positions).to(device) for t in toks])
    del toks
    dout = torch.empty((Nd, Hd, dd), dtype=torch.bfloat16, device=device)
    S, z = S_init.clone(), z_init.clone()
    for t in range(max(3, args.warmup)):  # warm-up on a scratch copy of the state
        R.rapt_decode_step(tq[t], tk[t], tv[t], tp[t], g1, g1, S, z, out=dout)
    S.copy_(S_init)
    z.copy_(z_init)
    torch.cuda.synchronize()
    barrier(device)
    e0, e1 = _events(1)[0], _events(1)[0]
    e0.record()
    for t in range(nsteps):
        R.rapt_decode_step(tq[t], tk[t], tv[t], tp[t], g1, g1, S, z, out=dout)
    e1.record()
    torch.cuda.synchronize()
    dec_ms = max_over_ranks(e0.elapsed_time(e1), device) / nsteps
    dec_bytes = decode_bytes(Nd, Hd, dd)
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    decode = {"value": world * Nd / (dec_ms * 1e-3), "unit": "tokens/s", "ms_per_step": dec_ms,
              "workload": "decode N=256 H=32 d=128 bf16, fp32 state from 512 prefill tokens, "
                          "64 consecutive steps at positions 512..575",
              "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                           "bytes_per_step": dec_bytes,
                           "traffic": read_traffic("decode", "decode_kernel")}}
    del S, z, S_init, z_init, tq, tk, tv, tp, dout

    # ---------------- packed varlen (T=65536, H=32, d=64)
    wv = syn.varlen_bf16(seed=rank_seed(2, rank))
    vq, vk, vv = (_bf(x, device) for x in (wv.q, wv.k, wv.v))
    cu = torch.from_numpy(wv.cu_seqlens).to(device)
    g64 = torch.ones(64, dtype=torch.float32, device=device)
    vo = torch.empty_like(vq)
    msl = int(wv.lengths.max())
    v_ms = time_steps(lambda: R.rapt_varlen_fwd(vq, vk, vv, cu, g64, g64, max_seqlen=msl, out=vo),
                      max(3, args.steps // 2), args.warmup, flush)
    v_mean = max_over_ranks(statistics.fmean(v_ms), device)
    v_bytes = prefill_bytes(1, wv.T, 32, 64)
    varlen = {"value": world * wv.T / (v_mean * 1e-3), "unit": "tokens/s", "ms_per_step": v_mean,
              "workload": "varlen T=65536 H=32 d=64 bf16, %d documents U[128,8192]" % len(wv.lengths),
              "roofline": {"bound": "hbm", "achieved": v_bytes / (v_mean * 1e-3) / 1e9,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": v_bytes / (v_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "traffic": read_traffic("varlen", "doc_order_kernel", "prefill_tc_kernel"),
                           "kernels": "doc_order_kernel + prefill_tc_kernel<128, true> (one call: the "
                                      "d = 64 heads two per CTA, one segment per document, longest "
                                      "first)"}}
    # its backward (dq, dk, dv, dgamma; the tensor-core passes with d = 64 products)
    vg = torch.empty_like(vq).normal_(generator=torch.Generator(device=device).manual_seed(6))
    vws = torch.empty(lib.rapt_varlen_bwd_workspace_size(wv.T, len(wv.lengths), 32, 64, msl, 1),
                      dtype=torch.uint8, device=device)
    vgr = [torch.empty_like(vq) for _ in range(3)] + [torch.empty_like(g64), torch.empty_like(g64)]
    vb_ms = time_steps(
        lambda: R.rapt_varlen_bwd(vq, vk, vv, vg, cu, g64, g64, max_seqlen=msl, dq=vgr[0], dk=vgr[1],
                                  dv=vgr[2], dgamma_q=vgr[3], dgamma_k=vgr[4], workspace=vws),
        max(3, args.steps // 4), args.warmup, flush)
    vb_mean = max_over_ranks(statistics.fmean(vb_ms), device)
    vb_bytes = 7 * wv.T * 32 * 64 * 2  # q, k, v, dout read; dq, dk, dv written (bf16)
    varlen_backward = {
        "value": world * wv.T / (vb_mean * 1e-3), "unit": "tokens/s", "ms_per_step": vb_mean,
        "workload": "varlen backward T=65536 H=32 d=64 bf16, %d documents U[128,8192] (dq, dk, dv, "
                    "dgamma_q, dgamma_k)" % len(wv.lengths),
        "roofline": {"bound": "hbm", "achieved": vb_bytes / (vb_mean * 1e-3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": vb_bytes / (vb_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "algorithmic_bytes_per_call": vb_bytes,
                     "traffic": read_traffic("varlen_backward", "bwd_tc_featmap", "doc_order_kernel",
                                             "bwd_tc_forward", "bwd_tc_reverse", "bwd_tc_features*2",
                                             "bwd_gain_kernel", "bwd_gain_final"),
                     "kernels": "bwd_tc_featmap<64> + doc_order_kernel + bwd_tc_forward<64> + "
                                "bwd_tc_reverse<64> + 2 x bwd_tc_features<64> + bwd_gain_kernel + "
                                "bwd_gain_final (one call: one segment per document, longest first; "
                                "the features of q beside the reverse pass)"}}
    del vq, vk, vv, vo, wv, vg, vws, vgr

    # ---------------- original RLA, L2 denominator (B=2, L=16384, H=16, d=128)
    wl = syn.l2_bf16(seed=rank_seed(4, rank))
    lq, lk, lv = (_bf(x, device) for x in (wl.q, wl.k, wl.v))
    lo = torch.empty_like(lq)
    ws = torch.empty(lib.rla_l2_workspace_size(2, 16384, 16, 128, 1), dtype=torch.uint8, device=device)
    l_ms = time_steps(lambda: R.rla_l2_fwd(lq, lk, lv, eps=1e-6, out=lo, workspace=ws),
                      max(3, args.steps // 2), args.warmup, flush)
    l_mean = max_over_ranks(statistics.fmean(l_ms), device)
    l_bytes = prefill_bytes(2, 16384, 16, 128)
    l_flops = 2 * 16384 * 16 * (8 * 128 * 128 + 2 * 128)
    rla_l2 = {"value": world * 2 * 16384 / (l_mean * 1e-3), "unit": "tokens/s", "ms_per_step": l_mean,
              "workload": "rla_l2 B=2 L=16384 H=16 d=128 bf16, non-causal",
              "roofline": {"bound": "hbm", "achieved": l_bytes / (l_mean * 1e-3) / 1e9,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": l_bytes / (l_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "tflops": l_flops / (l_mean * 1e-3) / 1e12,
                           "traffic": read_traffic("l2", "l2_tc_moments", "l2_tc_reduce", "l2_tc_readout"),
                           "kernels": "l2_tc_moments + l2_tc_reduce + l2_tc_readout (one call)"}}
    del lq, lk, lv, lo, ws

    # ---------------- causal original RLA (L2 denominator) on the L2 workload's shapes
    wl = syn.l2_bf16(seed=rank_seed(4, rank))
    lq, lk, lv = (_bf(x, device) for x in (wl.q, wl.k, wl.v))
    lo = torch.empty_like(lq)
    ws = torch.empty(max(1, lib.rla_l2_causal_workspace_size(2, 16384, 16, 128, 1)),
                     dtype=torch.uint8, device=device)
    c_ms, c_launch = time_steps(lambda: R.rla_l2_causal_fwd(lq, lk, lv, eps=1e-6, out=lo, workspace=ws),
                                max(3, args.steps // 4), args.warmup, flush,
                                counter=lib.rapt_launch_counter)
    c_mean = max_over_ranks(statistics.fmean(c_ms), device)
    c_flops = 2 * 16384 * 16 * (8 * 128 * 128 + 2 * 128)  # q'S, q'A q', S and A updates
    c_bytes = prefill_bytes(2, 16384, 16, 128)
    l2_causal = {"value": world * 2 * 16384 / (c_mean * 1e-3), "unit": "tokens/s",
                 "ms_per_step": c_mean,
                 "workload": "rla_l2_causal B=2 L=16384 H=16 d=128 bf16 (causal L2 denominator)",
                 "launches_per_call": c_launch / max(3, args.steps // 4),
                 "roofline": {"bound": "hbm", "achieved": c_bytes / (c_mean * 1e-3) / 1e9,
                              "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": c_bytes / (c_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
                              "algorithmic_bytes_per_call": c_bytes,
                              "algorithmic_flops_per_call": c_flops,
                              "tensor_tflops_algorithmic": c_flops / (c_mean * 1e-3) / 1e12,
                              "traffic": read_traffic("l2_causal", "l2_tc_moments", "l2c_tc_kernel"),
                              "kernels": "l2_tc_moments + l2c_tc_kernel (one call; tensor cores)"}}
    del lq, lk, lv, lo, ws, wl

    # ---------------- bidirectional RLA-2 on the headline's inputs (B=4, L=4096, H=16, d=128)
    bws = torch.empty(lib.rapt_bidir_workspace_size(B, L, H, d, 1), dtype=torch.uint8, device=device)
    b_ms, b_launch = time_steps(lambda: R.rapt_bidir_fwd(q, k, v, gq, gk, out=out, workspace=bws),
                                max(3, args.steps // 2), args.warmup, flush,
                                counter=lib.rapt_launch_counter)
    b_mean = max_over_ranks(statistics.fmean(b_ms), device)
    bidir = {"value": world * B * L / (b_mean * 1e-3), "unit": "tokens/s", "ms_per_step": b_mean,
             "workload": "rla2_bidir B=4 L=4096 H=16 d=128 bf16 (non-causal, Sum denominator), "
                         "the headline's inputs",
             "launches_per_call": b_launch / max(3, args.steps // 2),
             "roofline": {"bound": "hbm", "achieved": alg_bytes / (b_mean * 1e-3) / 1e9,
                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": alg_bytes / (b_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
                          "traffic": read_traffic("bidir", "segment_state_kernel", "bidir_readout"),
                          "kernels": "segment_state_kernel + bidir_readout (one call; the second is a programmatic dependent of the first)"}}
    del bws

    # ---------------- backward of the headline prefill (dq, dk, dv, dgamma; tensor cores, fp32 states)
    tg = torch.empty_like(q).normal_(generator=torch.Generator(device=device).manual_seed(5))
    gws = torch.empty(lib.rapt_prefill_bwd_workspace_size(B, L, H, d, 1), dtype=torch.uint8,
                      device=device)
    grads = [torch.empty_like(q) for _ in range(3)] + [torch.empty_like(gq), torch.empty_like(gk)]
    g_ms, g_launch = time_steps(
        lambda: R.rapt_prefill_bwd(q, k, v, tg, gq, gk, dq=grads[0], dk=grads[1], dv=grads[2],
                                   dgamma_q=grads[3], dgamma_k=grads[4], workspace=gws),
        max(3, args.steps // 4), args.warmup, flush, counter=lib.rapt_launch_counter)
    g_mean = max_over_ranks(statistics.fmean(g_ms), device)
    g_flops = B * L * H * (12 * d * d)  # recurrence-form backward: q'S, S g, R v, R^T k', S and R updates
    g_bytes = 7 * B * L * H * d * 2     # q, k, v, dout read; dq, dk, dv written (bf16)
    backward = {"value": world * B * L / (g_mean * 1e-3), "unit": "tokens/s", "ms_per_step": g_mean,
                "workload": "rla2_causal_prefill backward B=4 L=4096 H=16 d=128 bf16 (dq, dk, dv, "
                            "dgamma_q, dgamma_k), the headline's inputs",
                "launches_per_call": g_launch / max(3, args.steps // 4),
                "roofline": {"bound": "hbm", "achieved": g_bytes / (g_mean * 1e-3) / 1e9,
                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": g_bytes / (g_mean * 1e-3) / 1e9 / peaks["hbm_gbs"],
                             "peak_source": "measured hbm_gbs (copy bandwidth)",
                             "algorithmic_bytes_per_call": g_bytes,
                             "tensor_tflops_algorithmic": g_flops / (g_mean * 1e-3) / 1e12,
                             "traffic": read_traffic("backward", "bwd_tc_featmap",
                                                     "bwd_tc_blockstate<true>", "bwd_tc_forward",
                                                     "bwd_tc_blockstate<false>", "bwd_tc_reverse",
                                                     "bwd_tc_features*2", "bwd_gain_kernel"),
                             "kernels": "bwd_tc_featmap + bwd_tc_blockstate<true> + bwd_tc_forward + "
                                        "bwd_tc_blockstate<false> + bwd_tc_reverse + "
                                        "2 x bwd_tc_features (q beside the reverse pass, then k) + "
                                        "bwd_gain_kernel (one call; tensor cores)"}}
    del tg, gws, grads

    # ---------------- one RAPT layer around the headline attention (d_model = H d = 2048), and its
    # q | k | v projection alone (the tensor-core GEMM)
    dm = H * d
    gen = torch.Generator(device=device).manual_seed(6)
    x = torch.empty((B, L, dm), dtype=torch.bfloat16, device=device).normal_(generator=gen)
    w_qkv = torch.empty((3 * H * d, dm), dtype=torch.bfloat16, device=device).normal_(
        std=dm ** -0.5, generator=gen)
    w_o = torch.empty((dm, H * d), dtype=torch.bfloat16, device=device).normal_(
        std=(H * d) ** -0.5, generator=gen)
    y = torch.empty_like(x)
    lws = torch.empty(lib.rapt_layer_workspace_size(B, L, H, d, dm), dtype=torch.uint8,
                      device=device)
    y_ms, y_launch = time_steps(
        lambda: R.rapt_layer_fwd(x, w_qkv, w_o, gq, gk, heads=H, out=y, workspace=lws),
        max(3, args.steps // 2), args.warmup, flush, counter=lib.rapt_launch_counter)
    y_mean = max_over_ranks(statistics.fmean(y_ms), device)
    qkv_out = torch.empty((B * L, 3 * H * d), dtype=torch.bfloat16, device=device)
    x2 = x.view(B * L, dm)
    p_ms = time_steps(lambda: R.rapt_linear_fwd(x2, w_qkv, out=qkv_out), max(3, args.steps // 2),
                      args.warmup, flush)
    p_mean = max_over_ranks(statistics.fmean(p_ms), device)
    p_flops = 2.0 * B * L * dm * 3 * H * d
    layer_flops = p_flops + 2.0 * B * L * H * d * dm + B * L * H * (4 * d * d + 4 * d)
    layer = {"value": world * B * L / (y_mean * 1e-3), "unit": "tokens/s", "ms_per_step": y_mean,
             "workload": "rapt_layer B=4 L=4096 H=16 d=128 d_model=2048 bf16 (q|k|v projection, "
                         "causal RLA-2, output projection), synthetic N(0, 1/fan_in) weights",
             "launches_per_call": y_launch / max(3, args.steps // 2),
             "tflops": layer_flops / (y_mean * 1e-3) / 1e12,
             "projection": {"ms": p_mean, "workload": "y = x W^T, M=16384 N=6144 K=2048 bf16",
                            "roofline": {"bound": "tensor",
                                         "achieved": p_flops / (p_mean * 1e-3) / 1e12,
                                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                         "frac": p_flops / (p_mean * 1e-3) / 1e12 / peaks["bf16_tflops"],
                                         "peak_source": "measured bf16_tflops (cuBLAS burst)",
                                         "traffic": read_traffic("linear", "linear_tc_kernel"),
                                         "kernels": "linear_tc_kernel"}}}
    del x, w_qkv, w_o, y, lws, qkv_out, x2

    # ---------------- CPU baseline: the fp64 oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1:
        tps, pairs, secs, cores = oracle_sample(args.oracle_seconds, rank_seed(1, 0))
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "cpu_model": host_cpu_model(),
               "kind": "oracle",
               "sample": "%d of 64 (batch row, head) pairs of the headline workload, all 4096 rows "
                         "each, fp64 quadratic form, %.1f s; numpy BLAS threads = host cores"
                         % (pairs, secs)}

    traffic = read_traffic("prefill", "segment_state_kernel", "prefill_tc_kernel")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": headline_config(world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernels": "segment_state_kernel + prefill_tc_kernel (one call; the second is "
                                "a programmatic dependent of the first, so the call is timed whole)",
                     "peak_source": "%s hbm_gbs (copy bandwidth)" % peak_src,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "tensor_tflops_algorithmic": prefill_flops(B, L, H, d) / (mean_ms * 1e-3) / 1e12,
                     "tensor_peak_tflops": peaks["bf16_tflops"]},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(timed_launches),
        "clocks": clk,
        "cpu_baseline": cpu,
        "rla_l2": rla_l2, "bidir": bidir, "backward": backward, "l2_causal": l2_causal,
        "layer": layer, "varlen": varlen, "varlen_backward": varlen_backward, "decode": decode,
        # the headline numbers once more, compactly, at the end of the line
        "summary": {"prefill_tokens_per_s": value, "prefill_hbm_frac": achieved / peaks["hbm_gbs"],
                    "decode_tokens_per_s": decode["value"],
                    "decode_hbm_frac": decode["roofline"]["frac"],
                    "varlen_tokens_per_s": varlen["value"],
                    "varlen_hbm_frac": varlen["roofline"]["frac"],
                    "l2_hbm_frac": rla_l2["roofline"]["frac"],
                    "e2e_tokens_per_s": e2e_value},
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def read_traffic(case: str, *kernels: str):
    """DRAM bytes per call of workload ``case`` (a ``--only`` name), summed over ``kernels`` (the
    launches of one call; ``name*n``: n launches of that kernel per call), from the committed ncu
    summary; None unless every kernel has a row for that case taken on its source as it is now (each
    row records a hash of the source file)."""
    import hashlib

    count = {}
    for k in kernels:
        name, _, n = k.partition("*")
        count[name] = int(n) if n else 1
    kernels = tuple(count)

    table = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(table):
        return None
    found = {}
    for line in open(table):
        parts = [p.strip() for p in line.strip().strip("|").split("|")]
        if len(parts) >= 5 and parts[0] == case and parts[1] in kernels:
            src = os.path.join(ROOT, "relu_linear_attention_gb300", "csrc", parts[2])
            if not os.path.exists(src):
                return None
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            if h != parts[3]:
                return None
            found[parts[1]] = float(parts[4]) * count[parts[1]]
    return sum(found.values()) if len(found) == len(kernels) else None


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--oracle-seconds", type=float, default=15.0)
    ap.add_argument("--only", choices=["prefill", "varlen", "varlen_backward", "l2", "bidir", "backward",
                             "linear", "l2_causal"], default=None,
                    help="run one workload's calls without timing (for an ncu capture)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.only is not None:
        return profile_case(args)
    return run_gpu(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
