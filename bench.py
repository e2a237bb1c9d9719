"""Benchmark: KDA prefill Mtok/s and decode tok/s on GB300, with roofline fractions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step of the headline is one kda_chunk_fwd over the single-sequence prefill
workload (B=1, H=96, T=8192, dk=dv=128, bf16 inputs, fp32 state carried in and
out, chunk 64).  Inputs are resident in HBM before timing and are larger than
L2, so no flush is needed between steps.  The same run times the decode
workload (256 sequences x 96 heads, 64 consecutive kda_decode_step calls) and
reports it under "decode".  Under torchrun every rank runs its own replica
(weak scaling; the only collective is the max-reduction of the timings).
--impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill Mtok/s & decode tok/s (H=96,d=128); % of GB300 roofline"
PREFILL = "prefill_T8192_H96_d128_bf16"
DECODE = "decode_256seq_H96_d128_64steps"
VARLEN = "varlen_32seq_H96_d128_bf16"
PREFILL_1M = "prefill_T1M_H32_d128_bf16"
FALLBACK_HBM_GBS = 6800.0
STATE_BYTES = 128 * 128 * 4


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
# Chunkwise prefill flops per (token, head) at chunk 64, d = 128, triangles
# counted exactly: 3 (C-1) d [A, W, U0] + 2 (C+1) d [P, P U] + C^2 / 3 [T]
# + 6 d^2 [W S0, Qtil S0, Kbar^T U] + d^2 / C [decay].
PREFILL_FLOP_PER_TOKEN_HEAD = 140757


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor-core rate for a kernel timed inside a long step."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured bf16_tflops_sustained"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def prefill_bytes(T, H, dk, dv, elt=2, n_states=1, states_read=None, states_written=None):
    """Algorithmic bytes: read q, k, g (dk each), v (dv), beta once, write out
    (dv) once, plus 64 KiB per fp32 state read or written (by default one of
    each per head: n_states sequences with an initial and a final state)."""
    per_token_head = elt * (3 * dk + dv + 1 + dv)
    r = n_states * H if states_read is None else states_read
    w = n_states * H if states_written is None else states_written
    return T * H * per_token_head + (r + w) * dk * dv * 4


def tensor_block(T, H, kern_ms, hbm_peak):
    """The chunkwise prefill's flops against the tensor-core peak, and the
    share of that peak the HBM roof allows (flop per byte x HBM peak)."""
    peak, src = tensor_peak()
    flops = PREFILL_FLOP_PER_TOKEN_HEAD * T * H
    achieved = flops / (kern_ms * 1e-3) / 1e12
    per_byte = PREFILL_FLOP_PER_TOKEN_HEAD / prefill_bytes(1, 1, 128, 128, n_states=0)
    return {"bound": "hbm (intensity below the ridge)", "achieved": achieved, "peak": peak,
            "peak_source": src, "unit": "TFLOP/s", "frac": achieved / peak,
            "flop_per_token_head": PREFILL_FLOP_PER_TOKEN_HEAD,
            "ceiling_frac_at_hbm_peak": per_byte * hbm_peak / 1e3 / peak,
            "goal_frac": 0.5}


def decode_bytes(N, H, dk, dv, elt=2):
    return N * H * (2 * dk * dv * 4 + elt * (3 * dk + dv + 1 + dv))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 1 <= r[0] <= t1 + 1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, a in enumerate(r[3]) if a == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


def kernel_traffic(kernel_file, profile_name):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (its sha256 is recorded in the summary)."""
    src = os.path.join(ROOT, "hybrid_linear_attention_02_gb300", "csrc", kernel_file)
    prof = os.path.join(ROOT, "profiles", profile_name)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        text = open(prof).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != sha:
        return None
    return float(m_tr.group(1))


def reduce_max(x, device="cpu"):
    """Max of a float over all ranks of the default process group (1 rank: x)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank, max_ms):
    """Whole-job units per second: every rank did the same work in <= max_ms."""
    return world * units_per_rank / (max_ms * 1e-3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    """The fp64 CPU oracle timed on the host cores on a bounded sample."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import torch

    import oracle
    from hybrid_linear_attention_02_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL]
    sample_T = 1024
    d = inputs.make_prefill(w, seed=0, device="cpu", seq_len=sample_T)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.prefill(*x, d["init_state"], d["cu_seqlens"])
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    value = sample_T / per_step / 1e6
    cores = oracle.prefill.last_threads
    sample = f"all {w.heads} heads x first {sample_T} tokens of the workload per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Mtok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL, "B": 1, "H": w.heads, "T": w.seq_len, "dk": w.dk,
                   "dv": w.dv, "chunk": w.chunk},
        "cpu_baseline": {"value": value, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "Mtok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_gpu(args):
    import torch

    import hybrid_linear_attention_02_gb300 as kda
    from hybrid_linear_attention_02_gb300 import inputs
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max(x, dev)

    hbm_peak, peak_src = peaks()
    stream = torch.cuda.current_stream()

    if args.only == "decode":
        run_decode_only(args, dev)
        return
    if args.only == "headline":
        run_headline_only(args, dev)
        return
    if args.only == "prologue":
        run_prologue_only(args, dev)
        return
    # ---------------- prefill (headline) ----------------
    w = inputs.WORKLOADS[PREFILL]
    d = inputs.make_prefill(w, seed=rank, device=dev)
    T, H = w.seq_len, w.heads
    out = torch.empty((T, H, w.dv), dtype=w.torch_dtype, device=dev)
    fin = torch.empty((1, H, w.dk, w.dv), dtype=torch.float32, device=dev)
    args_pf = [d[n] for n in ("q", "k", "v", "g", "beta")]

    def prefill_step():
        kda.chunk_fwd(*args_pf, d["init_state"], None, chunk=w.chunk, out=out,
                      final_state=fin)

    for _ in range(max(args.warmup, 3)):
        prefill_step()
    barrier()
    sampler = ClockSampler(local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        prefill_step()
        ev[i][1].record(stream)
    end.record(stream)
    barrier()
    wall1 = time.time()
    clocks = sampler.stop(wall0, wall1)
    ms_total = max_over_ranks(start.elapsed_time(end))
    ms_step = ms_total / args.steps
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    value = job_throughput(world, T, ms_step) / 1e6
    alg_bytes = prefill_bytes(T, H, w.dk, w.dv)
    achieved = alg_bytes / (kern_ms * 1e-3) / 1e9
    algo = kda.algorithm(1, T, H, w.dk, w.dv, w.torch_dtype, w.chunk)
    tc = algo.startswith("tcgen05")
    kname, kfile, kprof = {
        "tcgen05_split": ("kda_chunk_split (chunk_prep_kernel + chunk_state_kernel)",
                          "kda_chunk_split.cu", "chunk_split_prefill_T8192_H96.md"),
        "tcgen05": ("kda_chunk_tc", "kda_chunk_tc.cu", "chunk_fwd_prefill_T8192_H96.md"),
    }.get(algo, ("kda_recurrent", "kda_recurrent.cu", "chunk_fwd_prefill_T8192_H96.md"))
    # Kernels per call, from the library's own window schedule (at this size
    # the split form's two front-loaded windows: two preparations, two state
    # passes).
    launches = kda.launch_count(1, T, H, w.dk, w.dv, w.torch_dtype, w.chunk)
    traffic = kernel_traffic(kfile, kprof)

    # ---------------- e2e through the public API with host buffers ----------------
    # Every step copies its inputs from pinned host memory and reads its result
    # back; steps are pipelined as a serving loop would run them: step i + 1's
    # inputs go up on two copy streams (into the other of two device buffer
    # sets) while step i computes and its result comes down.
    host_in = [x.cpu().pin_memory() for x in args_pf + [d["init_state"]]]
    dev_in = [[torch.empty_like(x) for x in args_pf + [d["init_state"]]] for _ in range(2)]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = host_out.numel() * host_out.element_size() + host_fin.numel() * host_fin.element_size()
    copy_streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    ev_in = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]   # [buffer][copy stream]
    ev_free = [torch.cuda.Event() for _ in range(2)]                     # buffer's kernel done

    def e2e_upload(i):
        b = i % 2
        for c, cs in enumerate(copy_streams):
            cs.wait_event(ev_free[b])
            with torch.cuda.stream(cs):
                for t in range(c, len(host_in), 2):
                    dev_in[b][t].copy_(host_in[t], non_blocking=True)
            ev_in[b][c].record(cs)

    def e2e_step(i, last):
        b = i % 2
        for c in range(2):
            stream.wait_event(ev_in[b][c])
        if not last:
            e2e_upload(i + 1)
        kda.chunk_fwd(*dev_in[b][:5], dev_in[b][5], None, chunk=w.chunk, out=out, final_state=fin)
        ev_free[b].record(stream)
        host_out.copy_(out, non_blocking=True)
        host_fin.copy_(fin, non_blocking=True)

    for c in range(2):
        ev_free[c].record(stream)
    e2e_upload(0)
    for i in range(3):
        e2e_step(i, False)
    torch.cuda.synchronize()
    barrier()
    e2e_steps = max(1, min(args.steps, 20))
    start.record(stream)
    for c in range(2):
        ev_free[c].record(stream)
    e2e_upload(0)
    for i in range(e2e_steps):
        e2e_step(i, i + 1 == e2e_steps)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(start.elapsed_time(end)) / e2e_steps
    e2e_value = job_throughput(world, T, e2e_ms) / 1e6
    del host_in, dev_in, host_out, host_fin

    # ------- prefill that also writes prefix-cache checkpoints every 512 tokens -------
    ck_int = 512
    ck_offs = torch.tensor(kda.checkpoint_offsets([T], ck_int), dtype=torch.int32, device=dev)
    ck_buf = torch.empty((T // ck_int, H, w.dk, w.dv), dtype=torch.float32, device=dev)

    def ckpt_step():
        kda.chunk_fwd(*args_pf, d["init_state"], None, chunk=w.chunk, out=out, final_state=fin,
                      ckpt_interval=ck_int, ckpt_offsets=ck_offs, checkpoints=ck_buf)

    for _ in range(3):
        ckpt_step()
    barrier()
    ck_steps = max(1, min(args.steps, 20))
    start.record(stream)
    for _ in range(ck_steps):
        ckpt_step()
    end.record(stream)
    barrier()
    ck_ms = max_over_ranks(start.elapsed_time(end)) / ck_steps
    ck_bytes = alg_bytes + ck_buf.numel() * 4
    ckpt = {"interval": ck_int, "value": job_throughput(world, T, ck_ms) / 1e6,
            "unit": "Mtok/s", "ms_per_step": ck_ms, "steps": ck_steps,
            "overhead_vs_plain": ck_ms / ms_step - 1.0,
            "algorithmic_bytes_per_launch": ck_bytes,
            "achieved_gbs": ck_bytes / (ck_ms * 1e-3) / 1e9,
            "frac": ck_bytes / (ck_ms * 1e-3) / 1e9 / hbm_peak}
    del ck_buf, ck_offs

    # ------- prefill with the output epilogue (head-wise RMSNorm + sigmoid gate) -------
    gate = inputs.make_output_gate(T, H, w.dv, w.torch_dtype, seed=rank, device=dev)

    def gated_step():
        kda.chunk_fwd(*args_pf, d["init_state"], None, chunk=w.chunk, out=out, final_state=fin,
                      gate=gate)

    for _ in range(3):
        gated_step()
    barrier()
    start.record(stream)
    for _ in range(ck_steps):
        gated_step()
    end.record(stream)
    barrier()
    g_ms = max_over_ranks(start.elapsed_time(end)) / ck_steps
    g_bytes = alg_bytes + T * H * w.dv * 2 + w.dv * 4
    gated = {"value": job_throughput(world, T, g_ms) / 1e6, "unit": "Mtok/s",
             "ms_per_step": g_ms, "steps": ck_steps, "overhead_vs_plain": g_ms / ms_step - 1.0,
             "algorithmic_bytes_per_launch": g_bytes,
             "achieved_gbs": g_bytes / (g_ms * 1e-3) / 1e9,
             "frac": g_bytes / (g_ms * 1e-3) / 1e9 / hbm_peak,
             "epilogue": "out = o / sqrt(mean(o^2) + 1e-6) * w * sigmoid(z), z [T, H, dv]"}
    del gate

    # ------- single-GPU KCP: 4 segments per sequence, and the transitions alone -------
    kcp_seg = 4
    dk_ = kda._dims(1, T, H, w.dk, w.dv, w.torch_dtype)
    kws = torch.empty(int(kda.load().kda_chunk_fwd_kcp_workspace_size(ctypes.byref(dk_), kcp_seg)),
                      dtype=torch.uint8, device=dev)

    def kcp_step():
        kda.chunk_fwd_kcp(*args_pf, d["init_state"], segments=kcp_seg, out=out,
                          final_state=fin, workspace=kws)

    tws = torch.empty(int(kda.load().kda_chunk_transition_workspace_size(ctypes.byref(dk_))),
                      dtype=torch.uint8, device=dev)

    def trans_step():
        kda.chunk_transition(*args_pf, None, workspace=tws)

    legs = {}
    for name, fn in (("kcp_prefill", kcp_step), ("transition", trans_step)):
        for _ in range(3):
            fn()
        barrier()
        start.record(stream)
        for _ in range(ck_steps):
            fn()
        end.record(stream)
        barrier()
        legs[name] = max_over_ranks(start.elapsed_time(end)) / ck_steps
    kcp = {"segments": kcp_seg, "value": job_throughput(world, T, legs["kcp_prefill"]) / 1e6,
           "unit": "Mtok/s", "ms_per_step": legs["kcp_prefill"], "steps": ck_steps,
           "overhead_vs_plain": legs["kcp_prefill"] / ms_step - 1.0,
           "transition_ms": legs["transition"],
           "transition_mtok_s": job_throughput(world, T, legs["transition"]) / 1e6}
    del kws, tws

    # ------- input prologue (ShortConv, Swish, L2 norm; scaled-sigmoid decay) -------
    px = inputs.make_prologue_inputs(T, H, w.dk, w.torch_dtype, seed=rank, device=dev)
    pq, pk, pg = (torch.empty_like(px[0]) for _ in range(3))

    def prologue_step():
        kda.prologue(*px, None, q=pq, k=pk, g=pg)

    for _ in range(3):
        prologue_step()
    barrier()
    start.record(stream)
    for _ in range(ck_steps):
        prologue_step()
    end.record(stream)
    barrier()
    p_ms = max_over_ranks(start.elapsed_time(end)) / ck_steps
    p_bytes = 6 * T * H * w.dk * 2 + 2 * H * w.dk * 4 * 4 + H * 4
    prologue = {"value": job_throughput(world, T, p_ms) / 1e6, "unit": "Mtok/s",
                "ms_per_step": p_ms, "steps": ck_steps, "algorithmic_bytes_per_launch": p_bytes,
                "achieved_gbs": p_bytes / (p_ms * 1e-3) / 1e9,
                "frac": p_bytes / (p_ms * 1e-3) / 1e9 / hbm_peak, "bound": "hbm",
                "traffic": kernel_traffic("kda_prologue.cu", "prologue_T8192_H96.md")}
    del d, args_pf, out, fin, px, pq, pk, pg
    torch.cuda.empty_cache()
    # ------- the packed varlen and the million-token prefill workloads -------
    big = {}
    if args.only == "all" and not args.no_big_prefill:
        for key, wname, steps in (("varlen", VARLEN, min(args.steps, 10)),
                                  ("prefill_1m", PREFILL_1M, min(args.steps, 5))):
            big[key] = run_prefill_leg(wname, max(1, steps), dev, rank, world, start, end,
                                       stream, barrier, max_over_ranks, hbm_peak)
            torch.cuda.empty_cache()
    decode = None
    if args.only != "prefill":
        decode = run_decode_leg(args, dev, rank, world, start, end, stream, barrier,
                                max_over_ranks, hbm_peak)
    # ---------------- CPU baseline (oracle, rank 0, N=1 only) ----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only != "prefill":
        import oracle
        ws = inputs.WORKLOADS[PREFILL]
        dc = inputs.make_prefill(ws, seed=0, device="cpu")
        t0 = time.perf_counter()
        oracle.prefill(*(dc[n] for n in ("q", "k", "v", "g", "beta")), dc["init_state"],
                       dc["cu_seqlens"])
        dt = time.perf_counter() - t0
        cpu = {"value": ws.seq_len / dt / 1e6, "unit": "Mtok/s",
               "cores": oracle.prefill.last_threads, "kind": "oracle",
               "sample": f"the whole workload once (1 x {ws.seq_len} tokens x {ws.heads} heads),"
                         f" fp64, {dt:.1f} s wall"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "Mtok/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if tc else "f32", "data": "synthetic",
            "config": {"workload": PREFILL, "B": 1, "H": H, "T": T, "dk": w.dk, "dv": w.dv,
                       "chunk": w.chunk, "init_state": "N(0,0.02) fp32",
                       "l2": f"inputs ({alg_bytes / 1e9:.2f} GB) larger than L2 (129 MB); "
                             "no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                         "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic,
                         "kernel": kname,
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "kernel_ms": kern_ms},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "Mtok/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * launches,
            "clocks": clocks,
            "prefill_checkpoints": ckpt,
            "prefill_gated": gated,
            "kcp": kcp,
            "prologue": prologue,
            "tensor": tensor_block(T, H, kern_ms, hbm_peak),
            "varlen": big.get("varlen"),
            "prefill_1m": big.get("prefill_1m"),
            "decode": decode,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_prefill_leg(wname, steps, dev, rank, world, start, end, stream, barrier,
                    max_over_ranks, hbm_peak):
    """One kda_chunk_fwd per step over a whole workload (inputs resident in
    HBM, far larger than L2), timed with CUDA events on the launching stream."""
    import torch

    import hybrid_linear_attention_02_gb300 as kda
    from hybrid_linear_attention_02_gb300 import inputs
    w = inputs.WORKLOADS[wname]
    d = inputs.make_prefill(w, seed=rank, device=dev)
    T, H = d["q"].shape[:2]
    N = d["cu_seqlens"].numel() - 1
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    cu = d["cu_seqlens"] if w.varlen is not None else None
    out = torch.empty((T, H, w.dv), dtype=w.torch_dtype, device=dev)
    fin = torch.empty((N, H, w.dk, w.dv), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, kda.workspace_size(N, T, H, w.dk, w.dv, w.torch_dtype, w.chunk)),
                     dtype=torch.uint8, device=dev)

    def step():
        kda.chunk_fwd(*x, d["init_state"], cu, chunk=w.chunk, n_seqs=N, out=out,
                      final_state=fin, workspace=ws)

    for _ in range(3):
        step()
    barrier()
    start.record(stream)
    for _ in range(steps):
        step()
    end.record(stream)
    barrier()
    ms = max_over_ranks(start.elapsed_time(end)) / steps
    n_init = N * H if d["init_state"] is not None else 0
    alg = prefill_bytes(T, H, w.dk, w.dv, states_read=n_init, states_written=N * H)
    gbs = alg / (ms * 1e-3) / 1e9
    algo = kda.algorithm(N, T, H, w.dk, w.dv, w.torch_dtype, w.chunk)
    res = {"workload": wname, "n_seqs": N, "tokens": T, "heads": H,
           "value": job_throughput(world, T, ms) / 1e6, "unit": "Mtok/s",
           "ms_per_step": ms, "steps": steps, "algorithm": algo,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                        "frac": gbs / hbm_peak, "algorithmic_bytes_per_launch": alg,
                        "traffic": None,
                        "kernel": "kda_chunk_split" if algo == "tcgen05_split" else
                                  "kda_chunk_tc"},
           "tensor": tensor_block(T, H, ms, hbm_peak)}
    del d, x, out, fin, ws
    return res


def run_decode_leg(args, dev, rank, world, start, end, stream, barrier, max_over_ranks,
                   hbm_peak):
    """The decode workload: 64 consecutive steps over resident states."""
    import torch

    import hybrid_linear_attention_02_gb300 as kda
    from hybrid_linear_attention_02_gb300 import inputs
    wd = inputs.WORKLOADS[DECODE]
    N, Hd = wd.n_seqs, wd.heads
    state = inputs.make_decode_state(wd, seed=rank, device=dev)
    toks = [inputs.make_decode_tokens(wd, s, seed=rank, device=dev)
            for s in range(wd.decode_steps)]
    dout = torch.empty((N, Hd, wd.dv), dtype=wd.torch_dtype, device=dev)
    for s in range(3):
        kda.decode_step(*toks[s], state, out=dout)
    barrier()
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(wd.decode_steps)]
    start.record(stream)
    for s in range(wd.decode_steps):
        dev_ev[s][0].record(stream)
        kda.decode_step(*toks[s], state, out=dout)
        dev_ev[s][1].record(stream)
    end.record(stream)
    barrier()
    dec_ms = max_over_ranks(start.elapsed_time(end)) / wd.decode_steps
    dec_kern_ms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
    dec_bytes = decode_bytes(N, Hd, wd.dk, wd.dv)
    dec_gbs = dec_bytes / (dec_kern_ms * 1e-3) / 1e9
    dec_traffic = kernel_traffic("kda_recurrent.cu", "decode_step_64x96.md")

    return {"workload": DECODE, "value": job_throughput(world, N, dec_ms),
            "unit": "tok/s", "ms_per_step": dec_ms, "steps": wd.decode_steps,
            "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": dec_gbs / hbm_peak,
                         "algorithmic_bytes_per_launch": dec_bytes,
                         "kernel": "kda_recurrent (one token)",
                         "traffic": dec_traffic,
                         "kernel_ms": dec_kern_ms},
            "gpu_launches": wd.decode_steps}


def run_headline_only(args, dev):
    """Profiling aid: W + K calls of the headline prefill and nothing else."""
    import torch

    import hybrid_linear_attention_02_gb300 as kda
    from hybrid_linear_attention_02_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL]
    d = inputs.make_prefill(w, seed=0, device=dev)
    x = [d[n] for n in ("q", "k", "v", "g", "beta")]
    out = torch.empty((w.seq_len, w.heads, w.dv), dtype=w.torch_dtype, device=dev)
    fin = torch.empty((1, w.heads, w.dk, w.dv), dtype=torch.float32, device=dev)
    for _ in range(args.warmup + args.steps):
        kda.chunk_fwd(*x, d["init_state"], None, chunk=w.chunk, out=out, final_state=fin)
    torch.cuda.synchronize()


def run_prologue_only(args, dev):
    """Profiling aid: W + K calls of the input prologue on the headline's shape
    (8192 tokens x 96 heads) and nothing else."""
    import torch

    import hybrid_linear_attention_02_gb300 as kda
    from hybrid_linear_attention_02_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL]
    px = inputs.make_prologue_inputs(w.seq_len, w.heads, w.dk, w.torch_dtype, seed=0,
                                     device=dev)
    pq, pk, pg = (torch.empty_like(px[0]) for _ in range(3))
    for _ in range(args.warmup + args.steps):
        kda.prologue(*px, None, q=pq, k=pk, g=pg)
    torch.cuda.synchronize()


def run_decode_only(args, dev):
    """Profiling aid: the decode kernel alone on N sequences x 96 heads."""
    import torch

    import hybrid_linear_attention_02_gb300 as kda
    from hybrid_linear_attention_02_gb300 import inputs
    wd = inputs.WORKLOADS[DECODE]
    N = args.decode_seqs or wd.n_seqs
    state = inputs.make_decode_state(wd, seed=0, device=dev, n_seqs=N)
    toks = [inputs.make_decode_tokens(wd, s, seed=0, device=dev, n_seqs=N)
            for s in range(args.warmup + args.steps)]
    for t in toks:
        kda.decode_step(*t, state)
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-big-prefill", action="store_true",
                    help="skip the varlen and million-token prefill legs")
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode", "headline", "prologue"],
                    help="profiling aid: run one part only (no JSON line unless 'all')")
    ap.add_argument("--decode-seqs", type=int, default=None,
                    help="profiling aid: fewer decode sequences (small ncu case)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
