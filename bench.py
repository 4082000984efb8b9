"""libkda benchmark: KDA prefill tokens/s and decode seq-steps/s on one GB300.

Workloads (seeded synthetic inputs, no dataset):
  prefill  scheduler step -- 4096 tokens as 8 sequences (min 64), H=32,
           dk=dv=128, bf16 inputs, fp32 512-slot pool (slots from the top half),
           chunk 64, checkpoints every 256 tokens, fused RMSNorm-gate.
  decode   256 sequences x 1 token, H=32, dk=dv=128, bf16 inputs, fp32
           1024-slot pool, fused RMSNorm-gate.
  spec     the decode batch verifying 4 draft tokens per sequence (per-token
           states kept) followed by the commit of the accepted prefixes.
  conv     the short causal convolution (width 4, SiLU) over the scheduler
           step's q, k, v projections (12288 channels), with its cache pool.
  long     one 32768-token prompt as 8 calls of 4096 tokens carrying a bf16
           state through the pool, bf16 checkpoints every 256 tokens, no gate.
  varlen   4 sequences {37, 128, 200, 512}, H=8, d=64, bf16 inputs, fp32
           pool of 16, checkpoints every 64 (a latency-bound correctness case).
A step is one prefill call, one decode step, one verify + commit, one
convolution call and the 8 long-prompt calls; each is timed in its own loop
with CUDA events on the launching stream, the L2 flushed before every timed
prefill, convolution and long-prompt call: a 256 MiB write, then a read of a
second 256 MiB buffer, so that the flush's own dirty lines are written back
before the timer starts rather than inside the timed call (the decode step
streams 1.07 GB, far above L2).  ``value`` is prefill tokens/s of the
scheduler step; the other figures sit under ``decode``, ``spec_decode``,
``conv_prefill`` and ``longprompt``.  ``e2e`` is scheduler-step prefill
tokens/s with every step's inputs copied in from pinned host memory and its
output copied back, steps pipelined over two copy streams.
``--impl reference`` times the fp64 CPU oracle on the same workload instead.
``--gpus N`` (N > 1) runs N independent replicas, one process per GPU: launched
without torchrun, the script starts them itself under torch.distributed.run;
launched as ranks (WORLD_SIZE set), each rank is one replica.  The path has no
exchange step, so no collective touches the data; rank 0 reports the aggregate.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "KDA prefill tokens/s + decode seq-steps/s on 1 GB300; % of tensor/HBM roofline"
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank values over all ranks (identity without a
    process group).  The replicas share nothing else: no data-path collective."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput of `world` independent replicas: all units over the
    slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3) if ms_max and ms_max > 0 else float("nan")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# The CUDA sources behind each recorded traffic figure: a figure stays valid
# while these files are unchanged, whatever else in the library changes.
_COMMON_SRC = ["kda_common.cuh", "kda_internal.h"]
TRAFFIC_SOURCES = {
    "prefill": ["kda_prefill.cu", "kda_prefill_tc.cu", "kda_prefill_shared.cuh", "kda_tc.cuh"]
    + _COMMON_SRC,
    "decode": ["kda_decode.cu"] + _COMMON_SRC,
    "spec": ["kda_decode_multi.cu"] + _COMMON_SRC,
    "conv": ["kda_conv.cu", "kda_tc.cuh"] + _COMMON_SRC,
}


def kernel_source_hash(group: str) -> str:
    """sha256 over the CUDA sources of one kernel group (identifies the kernels
    a recorded ncu traffic figure belongs to)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_prefill_kda_gb300", "csrc")
    for name in sorted(TRAFFIC_SOURCES[group]):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(group: str, name: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json)
    for the current sources of the kernel group, else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(group)
    if not rec or rec.get("sources_sha256") != kernel_source_hash(group):
        return None
    v = rec.get(name)
    return None if v is None else int(v)


def prefill_algorithmic(w, d):
    """Bytes every prefill call must move, and its FLOPs (triangular-aware)."""
    T, H, dk, dv, C = w.T, w.H, w.dk, w.dv, w.chunk
    ib = 2 if w.in_dtype == torch.bfloat16 else 4
    sb = 2 if w.state_dtype == torch.bfloat16 else 4
    lens = [int(x) for x in (d["cu_seqlens"][1:] - d["cu_seqlens"][:-1]).tolist()]
    n_ck = sum(L // w.checkpoint_every for L in lens) if w.checkpoint_every else 0
    n_seq = sum(1 for L in lens if L > 0)
    b = T * H * (2 * dk + dk + dv) * ib            # q, k, g, v
    b += T * H * ib                                 # beta
    b += T * H * dv * ib                            # out
    if w.gate:
        b += T * H * dv * ib + dv * ib              # gate, norm weight
    b += 2 * n_seq * H * dk * dv * sb               # state read + write
    b += n_ck * H * dk * dv * sb                    # checkpoints
    # FLOPs per chunk-head with n rows (a multiply-add is 2): the decay-weighted
    # KK^T and QK^T (lower triangles), the triangular inverse, W = T'(K e^G)
    # and U0 = T' V (T' lower triangular), the three n x dk x dv products with
    # the state (W S, (Q e^G) S, (K e^(G_last - G))^T U), A_qk U, and the decay
    # scaling of the operands.
    fl = 0
    for L in lens:
        for c0 in range(0, L, C):
            n = min(C, L - c0)
            tri = n * (n + 1) / 2
            fl += H * (2 * 2 * tri * dk          # A_kk, A_qk
                       + n * n * n / 3           # triangular inverse
                       + 2 * tri * (dk + dv)     # W, U0
                       + 2 * n * dk * dv * 3     # W S, Q S, K^T U
                       + 2 * tri * dv            # A_qk U
                       + 4 * n * dk)             # decay scaling
    return int(b), float(fl)


def decode_algorithmic(w):
    ib = 2 if w.in_dtype == torch.bfloat16 else 4
    sb = 2 if w.state_dtype == torch.bfloat16 else 4
    b = 2 * w.N * w.H * w.dk * w.dv * sb
    b += w.N * w.H * (3 * w.dk + w.dv + 1 + w.dv) * ib  # q k g v beta out
    if w.gate:
        b += w.N * w.H * w.dv * ib + w.dv * ib
    b += w.N * 4
    fl = w.N * w.H * (7 * w.dk * w.dv)
    return int(b), float(fl)


def spec_algorithmic(w, K, num_accepted):
    """Bytes of one verification call (K tokens per sequence, per-token states
    stored) plus the commit of the accepted states."""
    ib = 2 if w.in_dtype == torch.bfloat16 else 4
    sb = 2 if w.state_dtype == torch.bfloat16 else 4
    st = w.H * w.dk * w.dv * sb
    b = w.N * st                                         # pool state read
    b += w.N * K * st                                    # per-token states written
    b += w.N * K * w.H * (3 * w.dk + w.dv + 1 + w.dv) * ib  # q k g v beta out
    if w.gate:
        b += w.N * K * w.H * w.dv * ib + w.dv * ib
    b += 2 * int((num_accepted > 0).sum()) * st          # commit: read + write
    b += w.N * 8
    return int(b)


def conv_algorithmic(w, C, Wd):
    """Bytes of one short-convolution call: x read and y written once, taps and
    bias, and each sequence's cache read and written."""
    n_seq = sum(1 for L in w.seqlens if L > 0)
    return int(2 * w.T * C * 2 + C * (Wd + 1) * 2 + 2 * n_seq * (Wd - 1) * C * 2)


def prefill_conv_algorithmic(w, d, Wd):
    """Bytes and FLOPs of one prefill call with the short convolution fused in:
    the prefill's (its q, k, v reads are the reads of the packed projection
    x), plus taps and bias, each sequence's convolution cache read and
    written, and the convolution's multiply-adds."""
    b, fl = prefill_algorithmic(w, d)
    C3 = 3 * w.H * w.dk
    lens = [int(x) for x in (d["cu_seqlens"][1:] - d["cu_seqlens"][:-1]).tolist()]
    n_seq = sum(1 for L in lens if L > 0)
    b += C3 * (Wd + 1) * 2 + 2 * n_seq * (Wd - 1) * C3 * 2
    fl += 2.0 * w.T * C3 * Wd
    return int(b), float(fl)


# ----------------------------------------------------------------- GPU arm
def run_gpu(args):
    import linear_attention_prefill_kda_gb300 as kda
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()

    # ---------------- prefill (scheduler step)
    w = W.SCHED
    d = W.make_prefill(w)
    t = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    T = w.T
    cap = T // w.checkpoint_every
    ck = torch.empty(cap, w.H, w.dk, w.dv, device=dev, dtype=w.state_dtype)
    offs = torch.empty(w.N + 1, dtype=torch.int32, device=dev)
    out = torch.empty(T, w.H, w.dv, device=dev, dtype=w.in_dtype)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    wsb = kda.kda_prefill_workspace_bytes(w.N, T, w.H, w.dk, w.dv, w.chunk)
    wspace = torch.empty(wsb, dtype=torch.uint8, device=dev) if wsb else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_read = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        # write a buffer larger than L2, then read another one: the timed call
        # finds none of its inputs in L2 and no dirty lines left to write back
        flush.fill_(float(i))
        torch.sum(flush_read)
    stream = torch.cuda.current_stream()

    def prefill_call(src=t, o=out):
        kda.kda_prefill_chunked(src["q"], src["k"], src["v"], src["g"], src["beta"],
                                t["cu_seqlens"], t["state_indices"], t["pool"], o, chunk=w.chunk,
                                checkpoints=ck, checkpoint_every=w.checkpoint_every,
                                ckpt_offsets=offs, gate=src["gate"], norm_w=t["norm_w"],
                                eps=d["eps"], scale=d["scale"], workspace=wspace,
                                dev_status=status, stream=stream)

    # ---------------- decode
    dw = W.DECODE
    if args.decode_sequences:  # a smaller case of the same shape, for single-launch captures
        dw = W.DECODE.replace(N=args.decode_sequences, num_slots=4 * args.decode_sequences)
    with_decode = args.workload in ("both", "decode")
    with_prefill = args.workload in ("both", "prefill")
    with_spec = args.workload in ("both", "spec")
    SPEC_K = 4
    if with_spec:
        sp = W.make_decode_pool(dw)
        spool = sp["pool"].to(dev)
        sidx = sp["state_indices"].to(dev)
        snw = sp["norm_w"].to(dev)
        sdraft = W.make_decode_draft(dw, SPEC_K)
        sacc_host = sdraft.pop("num_accepted")
        sdr = {k: v.to(dev) for k, v in sdraft.items()}
        sacc = sacc_host.to(dev)
        sout = torch.empty(dw.N, SPEC_K, dw.H, dw.dv, device=dev, dtype=dw.in_dtype)
        sts = torch.empty(dw.N, SPEC_K, dw.H, dw.dk, dw.dv, device=dev, dtype=dw.state_dtype)

    with_conv = args.workload in ("both", "conv")
    CONV_C, CONV_W = 3 * w.H * w.dk, 4  # q, k, v projections of the scheduler step
    if with_conv:
        cdat = W.make_conv(w.seqlens, CONV_C, CONV_W, torch.bfloat16, num_slots=w.num_slots,
                           seed=17)
        cdev = {k: v.to(dev) for k, v in cdat.items()}
        cy = torch.empty_like(cdev["x"])

    # ---------------- long prompt with bf16 state: 32768 tokens as 8 calls of
    # 4096 carrying the state through the pool, checkpoints every 256 tokens
    with_long = args.workload in ("both", "longprompt")
    lw = W.LONGPROMPT
    LSEG = 4096
    if with_long:
        ld = W.make_prefill(lw)
        lsrc = {k: ld[k].to(dev) for k in ("q", "k", "v", "g", "beta")}
        lpool0 = ld["pool"].to(dev)
        lpool = lpool0.clone()
        lidx = ld["state_indices"].to(dev)
        lcu = W.cu_from_lengths([LSEG]).to(dev)
        lout = torch.empty(lw.T, lw.H, lw.dv, device=dev, dtype=lw.in_dtype)
        lck = torch.empty(lw.T // lw.checkpoint_every, lw.H, lw.dk, lw.dv, device=dev,
                          dtype=lw.state_dtype)
        lwsb = kda.kda_prefill_workspace_bytes(1, LSEG, lw.H, lw.dk, lw.dv, lw.chunk)
        lws = torch.empty(lwsb, dtype=torch.uint8, device=dev) if lwsb else None
        lper = LSEG // lw.checkpoint_every

    def long_call(c):
        sl = slice(c * LSEG, (c + 1) * LSEG)
        kda.kda_prefill_chunked(lsrc["q"][sl], lsrc["k"][sl], lsrc["v"][sl], lsrc["g"][sl],
                                lsrc["beta"][sl], lcu, lidx, lpool, lout[sl], chunk=lw.chunk,
                                checkpoints=lck[c * lper:(c + 1) * lper],
                                checkpoint_every=lw.checkpoint_every, workspace=lws,
                                dev_status=status, stream=stream)

    # ---------------- varlen: 4 sequences {37, 128, 200, 512}, H=8, d=64, bf16,
    # fp32 pool of 16, checkpoints every 64 (the d=64 tensor-core kernels)
    with_varlen = args.workload in ("both", "varlen")
    vw = W.VARLEN
    if with_varlen:
        vd = W.make_prefill(vw)
        vt = {k: (x.to(dev) if isinstance(x, torch.Tensor) else x) for k, x in vd.items()}
        vout = torch.empty(vw.T, vw.H, vw.dv, device=dev, dtype=vw.in_dtype)
        vck = torch.empty(vw.T // vw.checkpoint_every, vw.H, vw.dk, vw.dv, device=dev,
                          dtype=vw.state_dtype)
        vwsb = kda.kda_prefill_workspace_bytes(vw.N, vw.T, vw.H, vw.dk, vw.dv, vw.chunk)
        vws = torch.empty(vwsb, dtype=torch.uint8, device=dev) if vwsb else None

    def varlen_call():
        kda.kda_prefill_chunked(vt["q"], vt["k"], vt["v"], vt["g"], vt["beta"], vt["cu_seqlens"],
                                vt["state_indices"], vt["pool"], vout, chunk=vw.chunk,
                                checkpoints=vck, checkpoint_every=vw.checkpoint_every,
                                scale=vd["scale"], workspace=vws, dev_status=status,
                                stream=stream)

    # ---------------- the scheduler step with a width-4 SiLU convolution and the
    # q/k normalisation fused into the prefill (packed projection x in, no q/k/v
    # tensors in between)
    with_fused = args.workload in ("both", "convfused")
    if with_fused:
        fd = W.make_prefill_conv(w, CONV_W)
        ft = {k: (x.to(dev) if isinstance(x, torch.Tensor) else x) for k, x in fd.items()}

    def fused_call():
        kda.kda_prefill_chunked_conv(ft["x"], ft["conv_w"], ft["conv_pool"], ft["g"], ft["beta"],
                                     ft["cu_seqlens"], ft["state_indices"], ft["pool"], out,
                                     conv_b=ft["conv_b"], conv_act="silu", chunk=w.chunk,
                                     checkpoints=ck, checkpoint_every=w.checkpoint_every,
                                     ckpt_offsets=offs, gate=ft["gate"], norm_w=ft["norm_w"],
                                     eps=fd["eps"], scale=fd["scale"], workspace=wspace,
                                     dev_status=status, stream=stream)

    def conv_call():
        if not with_conv:
            return
        kda.kda_causal_conv1d_prefill(cdev["x"], cdev["w"], cdev["cu_seqlens"],
                                      cdev["state_indices"], cdev["pool"], cy, bias=cdev["b"],
                                      act="silu", dev_status=status, stream=stream)

    def spec_call():
        if not with_spec:
            return
        kda.kda_decode_multi(sdr["q"], sdr["k"], sdr["v"], sdr["g"], sdr["beta"], sidx, spool,
                             sout, sts, gate=sdr["gate"], norm_w=snw, eps=sp["eps"],
                             dev_status=status, stream=stream)
        kda.kda_commit_accepted(sts, sacc, sidx, spool, dev_status=status, stream=stream)
    if with_decode:
        pd = W.make_decode_pool(dw)
        dpool = pd["pool"].to(dev)
        didx = pd["state_indices"].to(dev)
        dnw = pd["norm_w"].to(dev)
        dsteps = [{k: v.to(dev) for k, v in W.make_decode_step(dw, s).items()} for s in range(4)]
        dout = torch.empty(dw.N, dw.H, dw.dv, device=dev, dtype=dw.in_dtype)

    def decode_call(i):
        if not with_decode:
            return
        s = dsteps[i % len(dsteps)]
        kda.kda_decode_step(s["q"], s["k"], s["v"], s["g"], s["beta"], didx, dpool, dout,
                            gate=s["gate"], norm_w=dnw, eps=pd["eps"], dev_status=status,
                            stream=stream)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        if with_prefill:
            prefill_call()
        decode_call(0)
        spec_call()
        conv_call()
        if with_long:
            lpool.copy_(lpool0)
            for c in range(lw.T // LSEG):
                long_call(c)
        if with_varlen:
            varlen_call()
        if with_fused:
            fused_call()
    barrier()

    def gpu_lead():
        # ~0.2 ms of GPU spin ahead of a start event, so that the host's own
        # time to enqueue the timed call never shows up as GPU idle inside the
        # timed interval (the spin itself lies before the start event)
        torch.cuda._sleep(400_000)

    with ClockSampler(local) as clk:
        # prefill: per-iteration events around the call, L2 flushed before each
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        for i in range(args.steps if with_prefill else 0):
            flush_l2(i)
            gpu_lead()
            starts[i].record(stream)
            prefill_call()
            ends[i].record(stream)
        barrier()
        pre_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)] if with_prefill else [float("nan")]
        # decode: back-to-back steps (each streams 1.07 GB through HBM)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        gpu_lead()
        e0.record(stream)
        for i in range(args.steps):
            decode_call(i)
        e1.record(stream)
        barrier()
        dec_ms_total = e0.elapsed_time(e1)
        # speculative verification: K=4 draft tokens per sequence + commit
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        gpu_lead()
        e2.record(stream)
        for i in range(args.steps if with_spec else 0):
            spec_call()
        e3.record(stream)
        barrier()
        spec_ms_total = e2.elapsed_time(e3)
        # short causal convolution over the scheduler step's q, k, v projections,
        # L2 flushed before each call (the 100 MB input is about L2's size)
        cstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        cends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        for i in range(args.steps if with_conv else 0):
            flush_l2(i)
            gpu_lead()
            cstarts[i].record(stream)
            conv_call()
            cends[i].record(stream)
        barrier()
        conv_ms = (sum(a.elapsed_time(b) for a, b in zip(cstarts, cends)) / args.steps
                   if with_conv else float("nan"))
        # long prompt: each step is the 8 carried calls from the initial state;
        # every call timed on its own, the L2 flushed before it
        ncall = lw.T // LSEG
        lstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps * ncall)]
        lends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps * ncall)]
        barrier()
        for i in range(args.steps if with_long else 0):
            lpool.copy_(lpool0)
            for c in range(ncall):
                flush_l2(i)
                gpu_lead()
                lstarts[i * ncall + c].record(stream)
                long_call(c)
                lends[i * ncall + c].record(stream)
        barrier()
        long_list = [a.elapsed_time(b) for a, b in zip(lstarts, lends)] if with_long else []
        long_ms = sum(long_list) / (args.steps * ncall) if with_long else float("nan")
        # varlen (a latency-bound correctness workload): each call timed with
        # the L2 flushed before it
        vstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        vends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        for i in range(args.steps if with_varlen else 0):
            flush_l2(i)
            gpu_lead()
            vstarts[i].record(stream)
            varlen_call()
            vends[i].record(stream)
        barrier()
        var_ms = (sum(a.elapsed_time(b) for a, b in zip(vstarts, vends)) / args.steps
                  if with_varlen else float("nan"))
        # fused convolution + prefill, each call timed with the L2 flushed before it
        fstarts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        fends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        for i in range(args.steps if with_fused else 0):
            flush_l2(i)
            gpu_lead()
            fstarts[i].record(stream)
            fused_call()
            fends[i].record(stream)
        barrier()
        fused_list = [a.elapsed_time(b) for a, b in zip(fstarts, fends)] if with_fused else []
        fused_ms = sum(fused_list) / args.steps if with_fused else float("nan")
    clocks = clk.summary()
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {kda.DEV_STATUS.get(st)}")

    def spread(ms):  # min / median / max of the per-call times of one rank (diagnostic)
        v = sorted(x for x in ms if x == x)
        return [round(v[0], 4), round(v[len(v) // 2], 4), round(v[-1], 4)] if v else None

    pre_ms_mean = sum(pre_ms) / len(pre_ms)
    dec_ms = dec_ms_total / args.steps
    spec_ms = spec_ms_total / args.steps if with_spec else float("nan")
    pre_ms_mean, dec_ms, spec_ms, conv_ms, long_ms, var_ms, fused_ms = max_over_ranks(
        [pre_ms_mean, dec_ms, spec_ms, conv_ms, long_ms, var_ms, fused_ms], dev)

    # ---------------- e2e through the public API with host buffers
    # Every step copies its inputs in from pinned host memory and its output
    # back, all inside the timed region.  Steps are pipelined the way a serving
    # loop runs them: step i+1's inputs are copied in (copy stream) while step i
    # computes, and step i's output is copied out (a second copy stream), with
    # the staging inputs and outputs double-buffered.
    names = ["q", "k", "v", "g", "beta", "gate"]
    host = {k: d[k].pin_memory() for k in names}
    staged = [{k: torch.empty_like(t[k]) for k in names} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    outs_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = outs_host[0].numel() * outs_host[0].element_size()
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_steps(n, start):
        cin.wait_event(start)
        cout.wait_event(start)
        for i in range(n):
            bf = i % 2
            if i >= 2:
                cin.wait_event(comp_done[bf])   # step i-2 has read these inputs
                stream.wait_event(out_done[bf])  # step i-2's output has left
            with torch.cuda.stream(cin):
                for k in names:
                    staged[bf][k].copy_(host[k], non_blocking=True)
            in_done[bf].record(cin)
            stream.wait_event(in_done[bf])
            prefill_call(staged[bf], outs[bf])
            comp_done[bf].record(stream)
            cout.wait_event(comp_done[bf])
            with torch.cuda.stream(cout):
                outs_host[bf].copy_(outs[bf], non_blocking=True)
            out_done[bf].record(cout)
        stream.wait_event(out_done[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(out_done[n % 2])

    if with_prefill:
        w0 = torch.cuda.Event()
        w0.record(stream)
        e2e_steps(2, w0)
    barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if with_prefill:
        gpu_lead()
    x0.record(stream)
    if with_prefill:
        e2e_steps(args.steps, x0)
    x1.record(stream)
    barrier()
    e2e_ms = x0.elapsed_time(x1) / args.steps
    (e2e_ms,) = max_over_ranks([e2e_ms], dev)

    pre_bytes, pre_flops = prefill_algorithmic(w, d)
    dec_bytes, dec_flops = decode_algorithmic(dw)
    def rate(num, ms):  # per second; NaN when that part was not timed
        return num / (ms * 1e-3) if ms and ms > 0 and ms == ms else float("nan")

    if not with_decode:
        dec_ms = float("nan")
    if not with_prefill:
        e2e_ms = float("nan")
    pre_gbs = rate(pre_bytes, pre_ms_mean) / 1e9
    dec_gbs = rate(dec_bytes, dec_ms) / 1e9
    pre_tflops = rate(pre_flops, pre_ms_mean) / 1e12
    spec_bytes = spec_algorithmic(dw, SPEC_K, sacc_host) if with_spec else 0
    spec_gbs = rate(spec_bytes, spec_ms) / 1e9
    conv_bytes = conv_algorithmic(w, CONV_C, CONV_W) if with_conv else 0
    lw_seg = lw.replace(seqlens=(LSEG,))
    long_bytes, long_flops = prefill_algorithmic(lw_seg, {"cu_seqlens": W.cu_from_lengths([LSEG])})
    long_gbs = rate(long_bytes, long_ms) / 1e9
    conv_gbs = rate(conv_bytes, conv_ms) / 1e9
    fused_bytes, fused_flops = prefill_conv_algorithmic(w, d, CONV_W)
    fused_gbs = rate(fused_bytes, fused_ms) / 1e9
    tokens_s = replica_rate(T, ws, pre_ms_mean)
    seqsteps_s = replica_rate(dw.N, ws, dec_ms)
    result = {
        "metric": METRIC,
        "value": round(tokens_s, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(sum(x for x in (pre_ms_mean, dec_ms) if x == x), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in / f32 accumulate",
        "data": "synthetic (seeded; distributions of the workload definitions)",
        "config": {"workload": w.name, "prefill_tokens": T, "sequences": list(w.seqlens),
                   "H": w.H, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                   "checkpoint_every": w.checkpoint_every, "state_dtype": "f32",
                   "fused_norm_gate": True, "decode_workload": dw.name, "decode_sequences": dw.N,
                   "l2": "flushed before each timed prefill call (256 MiB write, then a 256 MiB "
                         "read of another buffer, so no dirty lines are written back in the timed "
                         "call); decode "
                         "streams 1.07 GB per step (> L2)",
                   "parallelism": f"replicas x{ws}"},
        "prefill_ms": round(pre_ms_mean, 4),
        "prefill_ms_spread": spread(pre_ms),
        "roofline": {"bound": "hbm", "achieved": round(pre_gbs, 1), "peak": pk["hbm"],
                     "unit": "GB/s", "frac": round(pre_gbs / pk["hbm"], 4),
                     "traffic": recorded_traffic("prefill", "prefill_call_dram_bytes"),
                     "peak_source": pk["source"],
                     "algorithmic_bytes": pre_bytes, "algorithmic_flops": pre_flops,
                     "achieved_tflops": round(pre_tflops, 2),
                     "tensor_frac_of_bf16_peak": round(pre_tflops / pk["bf16"], 4)},
        "decode": {"value": round(seqsteps_s, 1), "unit": "seq-steps/s",
                   "ms_per_step": round(dec_ms, 4),
                   "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": pk["hbm"],
                                "unit": "GB/s", "frac": round(dec_gbs / pk["hbm"], 4),
                                "traffic": recorded_traffic("decode", "decode_step_dram_bytes"),
                                "algorithmic_bytes": dec_bytes}},
        "spec_decode": {"value": round(replica_rate(dw.N * SPEC_K, ws, spec_ms), 1),
                        "unit": "draft tokens verified/s", "draft_tokens": SPEC_K,
                        "ms_per_step": round(spec_ms, 4),
                        "roofline": {"bound": "hbm", "achieved": round(spec_gbs, 1),
                                     "peak": pk["hbm"], "unit": "GB/s",
                                     "frac": round(spec_gbs / pk["hbm"], 4),
                                     "traffic": recorded_traffic("spec", "spec_step_dram_bytes"),
                                     "algorithmic_bytes": spec_bytes}},
        "conv_prefill": {"value": round(replica_rate(T, ws, conv_ms), 1), "unit": "tokens/s",
                         "channels": CONV_C, "width": CONV_W, "ms_per_call": round(conv_ms, 4),
                         "roofline": {"bound": "hbm", "achieved": round(conv_gbs, 1),
                                      "peak": pk["hbm"], "unit": "GB/s",
                                      "frac": round(conv_gbs / pk["hbm"], 4),
                                      "traffic": recorded_traffic("conv", "conv_call_dram_bytes"),
                                      "algorithmic_bytes": conv_bytes}},
        "longprompt": {"workload": lw.name, "value": round(replica_rate(LSEG, ws, long_ms), 1),
                       "unit": "tokens/s", "calls": lw.T // LSEG, "tokens_per_call": LSEG,
                       "ms_per_call": round(long_ms, 4), "ms_spread": spread(long_list), "state_dtype": "bf16",
                       "checkpoint_every": lw.checkpoint_every,
                       "roofline": {"bound": "hbm", "achieved": round(long_gbs, 1),
                                    "peak": pk["hbm"], "unit": "GB/s",
                                    "frac": round(long_gbs / pk["hbm"], 4),
                                    "traffic": recorded_traffic("prefill",
                                                                "longprompt_call_dram_bytes"),
                                    "algorithmic_bytes": long_bytes,
                                    "algorithmic_flops": long_flops,
                                    "achieved_tflops": round(rate(long_flops, long_ms) / 1e12, 2)}},
        "varlen": {"workload": vw.name, "value": round(replica_rate(vw.T, ws, var_ms), 1),
                   "unit": "tokens/s", "ms_per_call": round(var_ms, 4),
                   "path": kda.kda_prefill_path(vw.dk, vw.dv, vw.chunk, vw.in_dtype)},
        "conv_fused_prefill": {
            "workload": w.name + "_conv4_silu", "value": round(replica_rate(T, ws, fused_ms), 1),
            "unit": "tokens/s", "ms_per_call": round(fused_ms, 4), "ms_spread": spread(fused_list),
            "separate_ms": round(conv_ms + pre_ms_mean, 4),
            "separate": "the convolution kernel and the prefill timed above, one after the other "
                        "(the q/k normalisation between them, which the library has no separate "
                        "kernel for, is not counted)",
            "roofline": {"bound": "hbm", "achieved": round(fused_gbs, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(fused_gbs / pk["hbm"], 4),
                         "traffic": recorded_traffic("prefill", "conv_fused_call_dram_bytes"),
                         "algorithmic_bytes": fused_bytes, "algorithmic_flops": fused_flops}},
        "e2e": {"value": round(replica_rate(T, ws, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "step i+1's inputs copied in while step i computes and its output "
                             "is copied out (two copy streams, double-buffered staging)"},
        "gpu_launches": args.steps * (prefill_launches(kda, w) * with_prefill + with_decode
                                      + 2 * with_spec + with_conv
                                      + (lw.T // LSEG) * prefill_launches(kda, lw) * with_long
                                      + prefill_launches(kda, vw) * with_varlen
                                      + 2 * with_fused),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, d, budget_s=args.cpu_seconds)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


def prefill_launches(kda, w) -> int:
    """Kernels one prefill call launches."""
    return int(kda.prefill_launches(w.dk, w.dv, w.chunk, w.in_dtype, w.gate))


# ----------------------------------------------------------------- CPU oracle
def _compact(d):
    """The workload with its pool reduced to the slots it touches (the oracle
    widens the pool to fp64; untouched slots do not enter the arithmetic)."""
    idx = d["state_indices"].long()
    dd = dict(d)
    dd["pool"] = d["pool"][idx].clone()
    dd["state_indices"] = torch.arange(len(idx), dtype=torch.int32)
    return dd


def _oracle_prefill_once(w, dd, nthreads=0):
    import oracle
    return oracle.prefill(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["cu_seqlens"],
                          dd["state_indices"], dd["pool"], checkpoint_every=w.checkpoint_every,
                          gate=dd["gate"], norm_w=dd["norm_w"], eps=dd["eps"], scale=dd["scale"],
                          nthreads=nthreads)


def cpu_baseline(w, d, budget_s=15.0):
    import oracle
    dd = _compact(d)
    cores = oracle.max_threads()
    n, t_total = 0, 0.0
    while t_total < budget_s and n < 50:
        t0 = time.perf_counter()
        _oracle_prefill_once(w, dd)
        t_total += time.perf_counter() - t0
        n += 1
    # the same oracle on one thread, one call
    t0 = time.perf_counter()
    _oracle_prefill_once(w, dd, nthreads=1)
    t_one = time.perf_counter() - t0
    return {"value": round(n * w.T / t_total, 1), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "one_thread": {"value": round(w.T / t_one, 1), "unit": "tokens/s",
                           "sample": f"1 full call, {t_one:.1f} s"},
            "sample": f"{n} full calls of {w.name} (fp64 C oracle, OpenMP over (sequence, head), "
                      f"pool reduced to the 8 touched slots), {t_total:.1f} s on "
                      f"{os.cpu_count()} host cores"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    w = W.SCHED
    d = W.make_prefill(w)
    dd = _compact(d)
    for _ in range(args.warmup):
        _oracle_prefill_once(w, dd)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_prefill_once(w, dd)
        times.append(time.perf_counter() - t0)
    mean = sum(times) / len(times)
    val = w.T / mean
    cores = oracle.max_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "prefill_tokens": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "chunk": w.chunk, "checkpoint_every": w.checkpoint_every},
        "cpu_baseline": {"value": round(val, 1), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step one full {w.name} call (fp64 C oracle, pool reduced "
                                   f"to the touched slots)"},
        "e2e": {"value": round(val, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _nan_to_none(x):
    if isinstance(x, float) and x != x:
        return None
    if isinstance(x, dict):
        return {k: _nan_to_none(v) for k, v in x.items()}
    if isinstance(x, list):
        return [_nan_to_none(v) for v in x]
    return x


def spawn_replicas(n: int, argv) -> int:
    """Run this script as ``n`` replica processes (one per GPU, ranks 0..n-1)
    under torch.distributed.run on this node and return its exit status.  Each
    replica runs the whole workload on its own GPU; rank 0 prints the line."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *argv]
    return subprocess.run(cmd, cwd=ROOT).returncode


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libkda", "reference"], default="libkda")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["both", "prefill", "decode", "spec", "conv",
                                           "longprompt", "varlen", "convfused"],
                    default="both",
                    help="time every part (default) or one of them (for profiling runs)")
    ap.add_argument("--decode-sequences", type=int, default=0,
                    help="sequences of the decode and verification workloads (default: the workload's "
                         "256), with a pool of four slots per sequence: a smaller case of the same "
                         "kernels for single-launch profiler captures")
    raw = list(sys.argv[1:] if argv is None else argv)
    args = ap.parse_args(raw)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not launched as ranks yet: start one replica per GPU ourselves
        sys.exit(spawn_replicas(args.gpus, raw))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but launched with WORLD_SIZE={world}")
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(_nan_to_none(res)), flush=True)


if __name__ == "__main__":
    main()
