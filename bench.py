"""Benchmark of the SpargeAttention2 hot path on GB300.

One step = the whole hot path on one batch of synthetic input: block mask
(pool + pooled map + hybrid Top-k/Top-p selection + CSC lists), block-sparse
attention forward, and backward (dQ, dK, dV).  Default workload: the
Wan2.1-1.3B 480p attention shape, B=1, H=12, N=32760 (21x30x52 latents),
d=128, 128x64 blocks, k=5% with Top-p off (p=0, the fixed-K point): exactly
26 of 512 kv-blocks per row, 94.92% sparsity.  The hybrid rule at the
workload's p=0.9 is timed too ("hybrid"; near-uniform pooled rows keep most
blocks there), and so is the full step of the local-attention variant of the
shape at its own rule k=5%, p=0.9, where the hybrid rule reaches about 93%
sparsity ("hybrid_local").

Prints one JSON line (rank 0).  ``value`` = kept-FLOP TFLOP/s of fwd+bwd
(algorithmic FLOPs 4*d and 10*d per kept valid query x key pair) divided by
the device time of the whole step, mask included.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep     # mask-only and fwd timings over the k x p sweep

Under torchrun (N > 1) every rank runs the same per-GPU workload (heads are
independent; weak scaling, no data-path collective); the step time is the
max over ranks.  ``--impl reference`` times the CPU oracle (a bounded sample
of the same workload per step) on the host cores; there is no other
reference implementation of this method.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("sparse attn fwd+bwd ms & kept-FLOP TFLOP/s at 95% sparsity; "
          "% of BF16/HBM roofline")
KERNELS_PER_STEP = 9  # pool, logits, select, csc, fwd, plan, delta, dkdv, dq
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes per call of each entry point (dram__bytes_read.sum + dram__bytes_write.sum
# summed over its kernels) from one ncu capture of the default workload (480p, 128 x 64
# blocks, k = 5 %, p = 0) with the current kernels; reported as roofline.traffic on that workload only.
NCU_TRAFFIC_BYTES = {("wan480", 12, 64, 0.05, 0.0): {"bwd": 1520.7e6, "fwd": 344.0e6, "mask": 216.4e6}}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, group_backend_ready: bool):
    """Max over ranks (identity on one process)."""
    if not group_backend_ready:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, group_backend_ready: bool):
    if not group_backend_ready:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(local_ms: float, local_flops: float, steps: int, distributed: bool):
    """Whole-job throughput: FLOPs of all ranks / the slowest rank's time."""
    t_ms = reduce_max(local_ms, distributed)
    flops = reduce_sum(local_flops, distributed)
    return t_ms, flops * steps / (t_ms * 1e-3) / 1e12


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_index], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, parts))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [p for ts, p in rows if t0 - 1.0 <= ts <= t1 + 1.0] or [p for _, p in rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(p[2]) for p in inside if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for p in inside if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[6 + i] == "Active"})
        pw = [float(p[4]) for p in inside if p[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons,
                "samples": len(inside),
                "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- workload math
def kept_pairs(mask_bool, n, bq, bk):
    """Sum over kept (q-block, kv-block) tiles of valid-query x valid-key counts."""
    import torch
    mq, mk = mask_bool.shape[-2], mask_bool.shape[-1]
    rq = torch.full((mq,), bq, dtype=torch.float64, device=mask_bool.device)
    rq[-1] = n - (mq - 1) * bq
    rk = torch.full((mk,), bk, dtype=torch.float64, device=mask_bool.device)
    rk[-1] = n - (mk - 1) * bk
    return float((mask_bool.double() * rq[:, None] * rk[None, :]).sum().item())


def unpack_bits(bitmask, mk):
    import torch
    w = bitmask.to(torch.int64) & 0xFFFFFFFF
    bits = (w[..., :, None] >> torch.arange(32, device=w.device)) & 1
    return bits.reshape(*w.shape[:-1], -1)[..., :mk].bool()


# ----------------------------------------------------------------------------- CPU oracle sample
def oracle_sample(host, wl, h, qblocks, k_frac, p):
    """Runs the CPU oracle on a bounded sample of the workload: pooled map of
    head h (all kv-blocks, the sampled q-blocks), hybrid selection of those
    rows, and block-gather fwd + bwd (fp32) of those q-blocks.  Returns
    (seconds, kept fwd+bwd FLOPs of the sample)."""
    import numpy as np
    import oracle as O
    q, k, v, do = host
    n, d = wl.N, wl.d
    mq, mk = O.num_blocks(n, wl.block_q), O.num_blocks(n, wl.block_kv)
    i0, i1 = qblocks[0], qblocks[-1] + 1
    t0 = time.perf_counter()
    kbar = O.pool_blocks(k[h][None, None], wl.block_kv)
    qbar = O.pool_blocks(q[h, i0 * wl.block_q:min(n, i1 * wl.block_q)][None, None], wl.block_q)
    prob = O.row_softmax(O.pooled_logits(qbar, kbar, 1.0 / math.sqrt(d)))
    rows = O.hybrid_mask_from_prob(prob.astype(np.float32), k_frac, p)
    mask = np.zeros((1, 1, mq, mk), dtype=bool)
    mask[0, 0, i0:i1] = rows[0, 0]
    qs, ks, vs, dos = (x[h][None, None] for x in (q, k, v, do))
    O.sparse_attention_blocks(qs, ks, vs, mask, wl.block_q, wl.block_kv, dtype=np.float32,
                              qblocks=list(qblocks))
    O.sparse_attention_blocks_bwd(qs, ks, vs, dos, mask, wl.block_q, wl.block_kv,
                                  dtype=np.float32, qblocks=list(qblocks))
    dt = time.perf_counter() - t0
    rq = np.array([min(wl.block_q, n - i * wl.block_q) for i in range(i0, i1)], dtype=np.float64)
    rk = np.array([min(wl.block_kv, n - j * wl.block_kv) for j in range(mk)], dtype=np.float64)
    pairs = float((rows[0, 0] * rq[:, None] * rk[None, :]).sum())
    return dt, 14.0 * d * pairs


def host_inputs(tensors, heads):
    import numpy as np
    return tuple(t[0, :heads].float().cpu().numpy().astype(np.float32) for t in tensors)


def cpu_baseline(host, wl, k_frac, p, seconds: float):
    """Times the oracle as it stands for about `seconds` of CPU work."""
    mq = -(-wl.N // wl.block_q)
    total_t = total_f = 0.0
    h = i = 0
    nblk = 4
    while total_t < seconds:
        qb = [(i + x) % mq for x in range(nblk)]
        qb = sorted(set(qb))
        if qb[-1] - qb[0] + 1 != len(qb):
            qb = list(range(qb[0], mq))
        dt, fl = oracle_sample(host, wl, h % host[0].shape[0], qb, k_frac, p)
        total_t += dt
        total_f += fl
        i += nblk
        h += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": (f"{total_t:.1f} s of the NumPy oracle on the host: per sample, head pooling "
                       f"+ pooled map + hybrid selection + fp32 block-gather fwd+bwd of {nblk} "
                       f"q-blocks of one {wl.name} head (BLAS threads: library default)"),
            "seconds": round(total_t, 2)}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, wl, k_frac, p):
    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    import torch
    from block_sparse_attention_sparge_gb300 import synth
    tens = synth.video_inputs(wl, device="cpu", heads=2)
    host = host_inputs(tens, 2)
    mq = -(-wl.N // wl.block_q)
    # calibrate the sample so (steps + warmup) samples take about 90 s
    dt1, _ = oracle_sample(host, wl, 0, [0], k_frac, p)
    per_step = 90.0 / max(1, args.steps + args.warmup)
    nblk = int(max(1, min(16, per_step / max(dt1, 1e-3))))
    times, flops = [], []
    for s in range(args.warmup + args.steps):
        i0 = (s * nblk) % max(1, mq - nblk)
        dt, fl = oracle_sample(host, wl, s % 2, list(range(i0, i0 + nblk)), k_frac, p)
        if s >= args.warmup:
            times.append(dt)
            flops.append(fl)
    tot_t, tot_f = sum(times), sum(flops)
    value = tot_f / tot_t / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(wl, k_frac, p),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {nblk} q-block(s) of one head (pool, map, select, "
                                   f"fwd, bwd), NumPy fp32 block-gather oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    return 0


def mask_rule(wl, k_frac, p):
    mk = -(-wl.N // wl.block_kv)
    kk = max(1, min(mk, math.ceil(k_frac * mk - 1e-4)))
    if p <= 0.0:
        return (f"fixed-K Top-k (p = 0, Top-p off): {kk} of {mk} kv-blocks per row, "
                f"{1 - kk / mk:.2%} sparsity")
    return f"hybrid Top-k + Top-p: k = {k_frac:g} (K = {kk} of {mk}), p = {p:g}"


def workload_config(wl, k_frac, p):
    """The workload as both arms name it (the measured mask sparsity is a
    top-level key of the library's line, so the two configs compare equal)."""
    return {"workload": (f"{wl.name}: Wan2.1-shaped attention fwd+bwd, B={wl.B}, H={wl.H}, "
                         f"N={wl.N} ({'x'.join(map(str, wl.grid))}), d={wl.d}, "
                         f"blocks {wl.block_q}x{wl.block_kv}, k={k_frac:g}, p={p:g}"),
            "mask_rule": mask_rule(wl, k_frac, p),
            "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d, "block_q": wl.block_q,
            "block_kv": wl.block_kv, "k_frac": k_frac, "p": p, "l2": l2_note(wl)}


def l2_note(wl):
    mb = 4 * wl.B * wl.H * wl.N * wl.d * 2 / 1e6
    rel = "larger" if mb > 129.0 else "smaller"
    return f"inputs {rel} than L2 (Q, K, V, dO: {mb:.0f} MB per step vs 129 MB L2)"


# ----------------------------------------------------------------------------- our arm
def run_ours(args, wl, k_frac, p):
    import torch
    import torch.distributed as dist
    from block_sparse_attention_sparge_gb300 import binding as B
    from block_sparse_attention_sparge_gb300 import synth

    ws, rank, local = dist_info()
    distributed = ws > 1
    if distributed:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if distributed else 0)
    torch.cuda.set_device(dev)
    B.load_library()

    q, k, v, do = synth.video_inputs(wl, device=dev)
    Bn, H, N, d = q.shape
    mq, mk = -(-N // wl.block_q), -(-N // wl.block_kv)
    stream = torch.cuda.current_stream(dev)

    # persistent buffers: no allocation inside the timed loop
    mask_out = B._mask_outputs(Bn, H, mq, mk, dev, True)
    import ctypes
    shp = B.Shape(Bn, H, N, d, wl.block_q, wl.block_kv)
    nb = ctypes.c_size_t(0)
    B.load_library().sparge_mask_workspace_bytes(ctypes.byref(shp), ctypes.byref(nb))
    ws_mask = torch.empty(nb.value, dtype=torch.uint8, device=dev)
    B.load_library().sparge_attn_bwd_workspace_bytes(ctypes.byref(shp), ctypes.byref(nb))
    ws_bwd = torch.empty(nb.value, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((Bn, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(kf, pp, ev=None):
        if ev is not None:
            ev[0].record(stream)
        res = B.sparge_mask(q, k, kf, pp, out=mask_out, workspace=ws_mask, block_kv=wl.block_kv)
        if ev is not None:
            ev[1].record(stream)
        B.sparge_attn_fwd(q, k, v, res["row_idx"], res["row_cnt"], out=o, lse=lse, status=status,
                          block_kv=wl.block_kv)
        if ev is not None:
            ev[2].record(stream)
        B.sparge_attn_bwd(q, k, v, o, lse, do, res["row_idx"], res["row_cnt"], res["col_idx"],
                          res["col_cnt"], out=(dq, dk, dv), workspace=ws_bwd, status=status,
                          block_kv=wl.block_kv)
        if ev is not None:
            ev[3].record(stream)
        return res

    # work per step from the mask this rule produces
    res = step(k_frac, p)
    torch.cuda.synchronize()
    maskb = unpack_bits(mask_out["bitmask"], mk)
    pairs = kept_pairs(maskb, N, wl.block_q, wl.block_kv)
    kept_tiles = int(maskb.sum().item())
    sparsity = 1.0 - kept_tiles / float(Bn * H * mq * mk)
    fwd_flops = 4.0 * d * pairs
    bwd_flops = 10.0 * d * pairs
    step_flops = fwd_flops + bwd_flops
    mask_bytes = (2.0 * Bn * H * N * d * 2 + Bn * H * mq * ((mk + 31) // 32) * 4
                  + 2 * kept_tiles * 4 + Bn * H * (mq + mk) * 4)

    for _ in range(args.warmup):
        step(k_frac, p)
    torch.cuda.synchronize()

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[0] or "0"
    sampler = ClockSampler(gpu_index)
    time.sleep(0.3)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if distributed:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    # The timed region: K steps back to back, no event inside a step (an event
    # between two calls would stop the next call's first kernel from starting
    # its setup while the previous kernel finishes).
    start.record(stream)
    for s in range(args.steps):
        step(k_frac, p)
    stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if distributed:
        dist.barrier()
    clocks = sampler.stop(wall0, wall1)
    total_ms = start.elapsed_time(stop)
    ms_step_local = total_ms / args.steps
    # Breakdown: the same steps with CUDA events between the three calls.
    nbreak = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nbreak)]
    for s in range(nbreak):
        step(k_frac, p, evs[s])
    torch.cuda.synchronize()
    parts = {"mask": [], "fwd": [], "bwd": []}
    for e in evs:
        parts["mask"].append(e[0].elapsed_time(e[1]))
        parts["fwd"].append(e[1].elapsed_time(e[2]))
        parts["bwd"].append(e[2].elapsed_time(e[3]))
    part_ms = {kk: sum(vv) / len(vv) for kk, vv in parts.items()}
    st = B._read_status(status)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed loop")

    ms_step, value = aggregate(ms_step_local, step_flops, 1, distributed)  # all ranks

    peaks, peak_kind = load_peaks()
    # The bf16 peak that matches the run: the burst figure (a GEMM timed alone)
    # for a timed region under a second, the sustained one (a seconds-long
    # loop under the power cap) for longer runs; the other is reported beside.
    burst = float(peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained")))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    use_burst = total_ms < 1000.0
    tc_peak = burst if use_burst else sustained
    tc_other = sustained if use_burst else burst
    tc_key = "bf16_tflops" if use_burst else "bf16_tflops_sustained"
    hbm_peak = float(peaks["hbm_gbs"])
    roof = {
        "fwd": {"kernel": "sparge_attn_fwd (attn_fwd_kernel)", "bound": "tensor",
                "achieved": fwd_flops / (part_ms["fwd"] * 1e-3) / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"},
        "bwd": {"kernel": "sparge_attn_bwd (plan + delta + dK/dV + dQ kernels)", "bound": "tensor",
                "achieved": bwd_flops / (part_ms["bwd"] * 1e-3) / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"},
        "mask": {"kernel": "sparge_mask (pool + logits + select + csc kernels)", "bound": "hbm",
                 "achieved": mask_bytes / (part_ms["mask"] * 1e-3) / 1e9, "peak": hbm_peak,
                 "unit": "GB/s"},
    }
    for r in roof.values():
        r["frac"] = r["achieved"] / r["peak"]
        key = tc_key if r["bound"] == "tensor" else "hbm_gbs"
        r["peak_source"] = (f"{key} of MEASURED_PEAKS.json" if peak_kind == "measured"
                            else f"fallback {key}")
        if r["bound"] == "tensor":
            r["peak_choice"] = (f"{'burst' if use_burst else 'sustained'}: timed region "
                                f"{total_ms:.0f} ms ({'under' if use_burst else 'over'} 1 s)")
            r["frac_vs_other_peak"] = {"peak": tc_other,
                                       "frac": r["achieved"] / tc_other}
    dom = max(part_ms, key=part_ms.get)
    roofline = dict(roof[dom])
    roofline["traffic"] = NCU_TRAFFIC_BYTES.get((wl.name, wl.H, wl.block_kv, k_frac, p), {}).get(dom)
    roofline["traffic_unit"] = "bytes per call (ncu)"
    roofline["per_launch_ms"] = part_ms[dom]
    roofline["algorithmic"] = {"fwd": "4*d per kept valid (query, key) pair",
                               "bwd": "10*d per kept valid (query, key) pair",
                               "mask": "Q+K read once + bitmask, CSR/CSC and counts written"}[dom]

    # The mask alone: 50 calls back to back (Q + K = 201 MB at 480p, above the
    # L2 size), with and without the column lists the backward uses; the
    # bitmask + CSR output is the mask construction proper.
    mask_alone = None
    if not args.no_hybrid:
        mo_csr = B._mask_outputs(Bn, H, mq, mk, dev, False)
        alone = {}
        for name, mo in (("with_csc", mask_out), ("csr_only", mo_csr)):
            for _ in range(3):
                B.sparge_mask(q, k, k_frac, p, out=mo, workspace=ws_mask, block_kv=wl.block_kv)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(50):
                B.sparge_mask(q, k, k_frac, p, out=mo, workspace=ws_mask, block_kv=wl.block_kv)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 50
            nbytes = mask_bytes if name == "with_csc" else mask_bytes - kept_tiles * 4 - Bn * H * mk * 4
            alone[name] = {"ms": ms, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
                           "frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak}
        mask_alone = {"calls": 50, "note": "sparge_mask timed alone, calls back to back", **alone}

    # hybrid rule (the workload's p) on the same inputs
    hybrid = None
    if not args.no_hybrid:
        step(k_frac, wl.p)
        torch.cuda.synchronize()
        mb = unpack_bits(mask_out["bitmask"], mk)
        hp = kept_pairs(mb, N, wl.block_q, wl.block_kv)
        hs = 1.0 - float(mb.sum().item()) / float(Bn * H * mq * mk)
        nh = max(3, min(args.steps, 30))
        for _ in range(2):
            step(k_frac, wl.p)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(nh):
            step(k_frac, wl.p)
        e1.record(stream)
        torch.cuda.synchronize()
        hms = e0.elapsed_time(e1) / nh
        hybrid = {"k_frac": k_frac, "p": wl.p, "sparsity": hs, "ms_per_step": hms,
                  "tflops": 14.0 * d * hp / (hms * 1e-3) / 1e12, "steps": nh}

    # The hybrid rule where it reaches high sparsity: the local-attention
    # variant of the 480p shape (Q and K share a smooth latent field) at its
    # own rule k = 5 %, p = 0.9, whole step timed (the Top-p search included).
    local = None
    if not args.no_hybrid and wl.name == "wan480":
        lwl = dataclasses.replace(synth.WORKLOADS["wan480_local"], block_kv=wl.block_kv)
        lq, lk, lv, ldo = synth.video_inputs(lwl, device=dev)
        lo, llse = torch.empty_like(lq), torch.empty_like(lse)
        lg = tuple(torch.empty_like(lq) for _ in range(3))

        def lstep():
            r = B.sparge_mask(lq, lk, lwl.k_frac, lwl.p, out=mask_out, workspace=ws_mask, block_kv=wl.block_kv)
            B.sparge_attn_fwd(lq, lk, lv, r["row_idx"], r["row_cnt"], out=lo, lse=llse,
                              status=status, block_kv=wl.block_kv)
            B.sparge_attn_bwd(lq, lk, lv, lo, llse, ldo, r["row_idx"], r["row_cnt"],
                              r["col_idx"], r["col_cnt"], out=lg, workspace=ws_bwd,
                              status=status, block_kv=wl.block_kv)
        lstep()
        torch.cuda.synchronize()
        mb = unpack_bits(mask_out["bitmask"], mk)
        lp = kept_pairs(mb, N, wl.block_q, wl.block_kv)
        lcnt = mb.sum(-1)
        ls = 1.0 - float(mb.sum().item()) / float(Bn * H * mq * mk)
        nl = max(3, min(args.steps, 30))
        for _ in range(2):
            lstep()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(nl):
            lstep()
        e1.record(stream)
        torch.cuda.synchronize()
        lms = e0.elapsed_time(e1) / nl
        local = {"workload": f"{lwl.name}: the 480p shape with Q, K sharing a smooth latent "
                             f"field (weight {lwl.rho}, sigma {lwl.shared_sigma}), Q gain "
                             f"{lwl.q_gain}",
                 "k_frac": lwl.k_frac, "p": lwl.p, "sparsity": ls,
                 "kept_per_row": {"min": int(lcnt.min()), "median": float(lcnt.float().median()),
                                  "max": int(lcnt.max())},
                 "ms_per_step": lms, "tflops": 14.0 * d * lp / (lms * 1e-3) / 1e12, "steps": nl}
        del lq, lk, lv, ldo, lo, llse, lg
        torch.cuda.empty_cache()

    # End to end through the public API, as a user would stream batches: per step
    # the H2D copy of that step's Q, K, V, dO from pinned host memory, the step,
    # and the D2H copy of O, dQ, dK, dV into pinned host memory.  Three streams
    # pipeline consecutive steps: the H2D of step s+1 and the D2H of step s-1
    # overlap the compute of step s (device inputs and outputs are
    # double-buffered; events order every reuse).  The timed region runs from
    # before the first H2D to after the last D2H, fill and drain included.
    nsteps_e2e = 0 if args.no_e2e else max(3, min(args.steps, 20))
    h2d = 4 * q.numel() * q.element_size()
    d2h = 4 * q.numel() * q.element_size()
    e2e_ms = e2e_val = None
    if nsteps_e2e:
        hin = [t.cpu().pin_memory() for t in (q, k, v, do)]
        hout = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(4)]
        slots = [{"in": [q, k, v, do], "o": o, "lse": lse, "g": (dq, dk, dv)}]
        slots.append({"in": [torch.empty_like(t) for t in (q, k, v, do)], "o": torch.empty_like(o),
                      "lse": torch.empty_like(lse),
                      "g": tuple(torch.empty_like(t) for t in (dq, dk, dv))})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def compute(sl):
            qq, kk, vv, dd = sl["in"]
            res = B.sparge_mask(qq, kk, k_frac, p, out=mask_out, workspace=ws_mask, block_kv=wl.block_kv)
            B.sparge_attn_fwd(qq, kk, vv, res["row_idx"], res["row_cnt"], out=sl["o"],
                              lse=sl["lse"], status=status, block_kv=wl.block_kv)
            B.sparge_attn_bwd(qq, kk, vv, sl["o"], sl["lse"], dd, res["row_idx"],
                              res["row_cnt"], res["col_idx"], res["col_cnt"], out=sl["g"],
                              workspace=ws_bwd, status=status, block_kv=wl.block_kv)

        def pipelined(n, e_first=None, e_last=None):
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_cp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            for i in range(n):
                sl = slots[i % 2]
                if i >= 2:
                    s_in.wait_event(ev_cp[i - 2])  # slot inputs no longer read
                if i == 0 and e_first is not None:
                    e_first.record(s_in)
                for src, dst in zip(hin, sl["in"]):
                    with torch.cuda.stream(s_in):
                        dst.copy_(src, non_blocking=True)
                ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])  # slot outputs already read back
                compute(sl)
                ev_cp[i].record(stream)
                s_out.wait_event(ev_cp[i])
                for src, dst in zip((sl["o"],) + sl["g"], hout):
                    with torch.cuda.stream(s_out):
                        dst.copy_(src, non_blocking=True)
                ev_out[i].record(s_out)
            if e_last is not None:
                e_last.record(s_out)

        pipelined(3)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipelined(nsteps_e2e, e0, e1)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / nsteps_e2e
        e2e_ms, e2e_val = aggregate(e2e_ms, step_flops, 1, distributed)
        del slots, hin, hout

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        host = host_inputs((q, k, v, do), 2)
        cpu = cpu_baseline(host, wl, k_frac, p, args.cpu_seconds)

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded smooth Gaussian Q/K fields + sinks, N(0,1) V/dO)",
            "config": workload_config(wl, k_frac, p),
            "sparsity": sparsity,
            "breakdown_ms": part_ms,
            "dense_equiv_tflops": 14.0 * d * float(Bn * H) * N * N * ws / (ms_step * 1e-3) / 1e12,
            "roofline": roofline,
            "roofline_all": roof,
            "mask_alone": mask_alone,
            "hybrid": hybrid,
            "hybrid_local": local,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": ("pipelined over 3 streams: H2D of step s+1 and D2H of step s-1 "
                             "overlap the compute of step s; fill and drain timed")},
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(out))
    if distributed:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- sweep
SWEEP_K = (0.02, 0.05, 0.10, 0.20)
SWEEP_P = (0.7, 0.9, 0.97)


def run_sweep(args, wl):
    """Mask-only and forward timings at the 480p shape (N=32760, H=12, d=128)
    for k in {2, 5, 10, 20}%, p in {0.7, 0.9, 0.97}, on near-uniform pooled
    rows (Q, K ~ N(0, 0.05^2)) and on sink-dominated rows.  One JSON line."""
    import ctypes
    import torch
    from block_sparse_attention_sparge_gb300 import binding as B
    from block_sparse_attention_sparge_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B.load_library()
    Bn, H, N, d = 1, wl.H, wl.N, wl.d
    mq, mk = -(-N // wl.block_q), -(-N // wl.block_kv)
    mask_out = B._mask_outputs(Bn, H, mq, mk, dev, False)
    shp = B.Shape(Bn, H, N, d, wl.block_q, wl.block_kv)
    nb = ctypes.c_size_t(0)
    B.load_library().sparge_mask_workspace_bytes(ctypes.byref(shp), ctypes.byref(nb))
    ws_mask = torch.empty(nb.value, dtype=torch.uint8, device=dev)
    o = torch.empty((Bn, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bn, H, N), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, min(args.steps, 20))

    def timed(fn):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    peaks, peak_kind = load_peaks()
    tc_peak = float(peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained")))
    hbm_peak = float(peaks["hbm_gbs"])
    mask_bytes = 2.0 * Bn * H * N * d * 2
    cells = []
    for kind, gen in (("uniform", synth.uniform_inputs), ("skewed", synth.skewed_inputs)):
        q, k, v, _ = gen(wl, device=dev)
        for kf in SWEEP_K:
            for pp in SWEEP_P:
                res = B.sparge_mask(q, k, kf, pp, out=mask_out, workspace=ws_mask, block_kv=wl.block_kv)
                torch.cuda.synchronize()
                maskb = unpack_bits(mask_out["bitmask"], mk)
                pairs = kept_pairs(maskb, N, wl.block_q, wl.block_kv)
                sparsity = 1.0 - float(maskb.sum().item()) / float(Bn * H * mq * mk)
                t_mask = timed(lambda: B.sparge_mask(q, k, kf, pp, out=mask_out,
                                                     workspace=ws_mask, block_kv=wl.block_kv))
                t_fwd = timed(lambda: B.sparge_attn_fwd(q, k, v, res["row_idx"], res["row_cnt"],
                                                        out=o, lse=lse, status=status,
                                                        block_kv=wl.block_kv))
                fl = 4.0 * d * pairs
                cells.append({"rows": kind, "k_frac": kf, "p": pp, "sparsity": round(sparsity, 5),
                              "mask_ms": round(t_mask, 4),
                              "mask_frac_hbm": round(mask_bytes / (t_mask * 1e-3) / 1e9 / hbm_peak,
                                                     3),
                              "fwd_ms": round(t_fwd, 4),
                              "fwd_tflops": round(fl / (t_fwd * 1e-3) / 1e12, 1),
                              "fwd_frac_bf16": round(fl / (t_fwd * 1e-3) / 1e12 / tc_peak, 3)})
        del q, k, v
        torch.cuda.empty_cache()
    if B._read_status(status) != 0:
        raise RuntimeError("device status set during the sweep")
    print(json.dumps({
        "sweep": cells, "reps_per_cell": reps,
        "workload": (f"{wl.name} shape: B=1, H={H}, N={N}, d={d}, blocks "
                     f"{wl.block_q}x{wl.block_kv}; uniform rows Q,K~N(0,0.05^2); skewed rows: "
                     f"kv-block 0 carries K += 2 sqrt(d) u, Q += 0.5 sqrt(d) u"),
        "mask_ms": "sparge_mask with bitmask and CSR lists (no column lists)",
        "peaks": f"{peak_kind}: bf16 {tc_peak} TFLOP/s (burst), HBM {hbm_peak} GB/s"}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="wan480",
                    choices=("wan480", "wan720", "wan480_d64", "wan480_local"))
    ap.add_argument("--k-frac", type=float, default=None)
    ap.add_argument("--p", type=float, default=0.0, help="Top-p of the headline step (0 = off)")
    ap.add_argument("--block-kv", type=int, default=None, choices=(64, 128),
                    help="kv-block size (default: the workload's, 64)")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload's shape with this many heads (e.g. a smaller case "
                         "for profiler captures)")
    ap.add_argument("--no-hybrid", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sweep", action="store_true",
                    help="mask-only and fwd timings over k x p on uniform and skewed rows")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from block_sparse_attention_sparge_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.block_kv is not None:
        wl = dataclasses.replace(wl, block_kv=args.block_kv)
    if args.heads is not None:
        if args.heads < 1:
            ap.error("--heads must be >= 1")
        wl = dataclasses.replace(wl, H=args.heads)
    k_frac = wl.k_frac if args.k_frac is None else args.k_frac
    if args.impl == "reference":
        return run_reference(args, wl, k_frac, args.p)
    if args.sweep:
        return run_sweep(args, wl)
    return run_ours(args, wl, k_frac, args.p)


if __name__ == "__main__":
    sys.exit(main())
