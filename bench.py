#!/usr/bin/env python
"""Benchmark of the FP8 E4M3 packed-varlen attention hot path on GB300.

One step = the whole hot path over one batch: fa_lp_quantize (amax pass, pack passes) followed by
fa_lp_forward_varlen (the tcgen05 attention kernel), on synthetic BF16 inputs already resident in
HBM. Default workload: one segment S=30272, H=56, D=128 (MiniMax-H3 shape), Q/K/V as strided views
of one fused [T, 3, H, 128] buffer, N(0,1) BF16.

Metric: TFLOPS = 4 * sum_s L_s^2 * H * D / step time (SGLang PR #40175's FLOP convention for
non-causal attention, Speed Tests). Inputs (1.3 GB) and codes (0.65 GB) exceed the 129 MB L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--workload nvfp4_s30272_h56 times the NVFP4 path instead (K with a per-channel offset N(0, 4)),
against the dense FP4 peak. The default line also carries two sub-objects timed in the same
process by the same procedure, each with its own clock sample: "nvfp4" (nvfp4_s30272_h56) and
"sparse" (sparse_fp8_s30272_h56, block-sparse FP8 at density 0.25); --no-extra-arms skips them.

N > 1 (torchrun, one process per GPU): independent replicas of the full workload on every rank
(the path has no exchange step), max-over-ranks time, weak scaling.
--impl reference: the CPU oracle timed on the host cores over a bounded sample of the same
workload (there is no installable reference implementation of this path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "E4M3 varlen attn TFLOPS at S=30272,H=56,D=128; % of FP8 tensor peak"
METRIC_NVFP4 = "NVFP4 varlen attn TFLOPS at S=30272,H=56,D=128; % of FP4 tensor peak"
METRIC_SPARSE = ("Block-sparse E4M3 attn TFLOPS (listed 64x64 blocks) at S=30272,H=56,D=128, "
                 "density 0.25; % of FP8 tensor peak")
UNIT = "TFLOPS"
D = 128
# dense FP8 and FP4 over dense BF16 tensor rate of the part (nominal 4.5, 13.5 / 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0
FP4_OVER_BF16 = 6.0
# kernels per step: FP8 amax, pack Q/K, pack V^T, attention; NVFP4 block sums, K means, pack
# Q/K, pack V^T, qm K^T table, attention; block-sparse FP8 the FP8 quantize kernels, list merge,
# tile order, attention
KERNELS_PER_STEP = {"fp8": 4, "nvfp4": 6, "sparse": 6}
METRICS = {"fp8": METRIC, "nvfp4": METRIC_NVFP4, "sparse": METRIC_SPARSE}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum, bytes) of one attention launch from
# an ncu capture of the full-size workload (profiles/attn_traffic_s30272_h56.md), keyed by the
# workload and the SHA-256 of the kernel source at capture time (null once the kernel changed).
NCU_TRAFFIC = {
    ("fp8_s30272_h56", "b3ad149c12b4ac4340efe7ccee09fa7e91263d2f081840ce7168a8d83d44c52b"):
        2.0465e9 + 425.72e6,
    ("nvfp4_s30272_h56", "c3f77846df62152f8a18889af84af063ae7a19782cc4cdcdcdd69a12ccbcfcb0"):
        2.2708e9 + 425.24e6,
    ("sparse_fp8_s30272_h56", "eb658a222e5667e01266b4c38d660a59a787924fe699ae2e50be04b6dc2433b8"):
        1.5226e9 + 425.39e6,
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="fp8_s30272_h56")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-arms", action="store_true",
                    help="default workload only: skip the nvfp4 and sparse sub-objects")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    return ap.parse_args()


def workload(name):
    from precision_attention_diffusion_gb300 import inputs
    w = inputs.WORKLOADS[name]
    return list(w["cu"]), int(w["heads"])


def mode_of(name):
    if name.startswith("nvfp4"):
        return "nvfp4"
    return "sparse" if name.startswith("sparse") else "fp8"


def sparse_lists(name, cu, H, seed=0):
    """The block lists of a block-sparse workload (every 16th list dense)."""
    from precision_attention_diffusion_gb300 import inputs
    return inputs.block_sparse_lists(cu, H, density=inputs.WORKLOADS[name]["density"], seed=seed,
                                     dense_every=16)


def sparse_flops(cu, H, off, idx):
    """4 D x (query rows x listed keys) summed over every (head, 64-row block)."""
    import numpy as np
    rows_g, keys_s, seg_g = [], [], []
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        L = b - a
        n = -(-L // 64)
        rows_g += [min(64, L - 64 * i) for i in range(n)]
        seg_g += [s] * n
        keys_s.append(L)
    rows_g = np.asarray(rows_g, np.float64)
    G = len(rows_g)
    total = 0.0
    off = np.asarray(off, np.int64)
    idx = np.asarray(idx, np.int64)
    lens = np.asarray(keys_s)
    for j in range(H * G):
        g = j % G
        lst = idx[off[j]:off[j + 1]]
        if len(lst) == 0:
            continue
        L = lens[seg_g[g]]
        keys = 64.0 * len(lst) - (64 * (lst[-1] + 1) - L if 64 * (lst[-1] + 1) > L else 0)
        total += rows_g[g] * keys
    return 4.0 * D * total


def attn_flops(cu, H):
    return 4.0 * sum((b - a) ** 2 for a, b in zip(cu[:-1], cu[1:])) * H * D


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        bf16, bf16s, hbm, src = (float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]),
                                 float(p["hbm_gbs"]), "measured")
    except Exception:
        bf16, bf16s, hbm, src = 1900.0, 1700.0, 6800.0, "fallback"
    return dict(fp8=FP8_OVER_BF16 * bf16, fp8_sustained=FP8_OVER_BF16 * bf16s,
                fp4=FP4_OVER_BF16 * bf16, fp4_sustained=FP4_OVER_BF16 * bf16s, hbm=hbm, source=src)


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200", "-f", self.path]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        finally:
            os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        load = [x for x in sm if x > 0.5 * smax] or sm
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax,
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------------------------------------
# CPU oracle on a bounded sample of the workload (the cpu_baseline object and the reference arm)
# ------------------------------------------------------------------------------------------------
def oracle_sample(cu, H, seconds, seed=0, mode="fp8", sparse_name=None):
    """Time the oracle (as it stands, all host threads) on head 0 of the workload: quantize
    that head's full Q/K/V, then emulating attention (FP8, NVFP4 or block-sparse FP8) of R query
    rows of the longest segment. Extrapolates to the whole workload: per head, quantize once + L
    rows (a block-sparse row visits its listed keys: random rows sample the mean)."""
    import numpy as np
    import torch

    import oracle
    from precision_attention_diffusion_gb300 import inputs
    lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
    s_long = int(np.argmax(lens))
    a, b = cu[s_long], cu[s_long + 1]
    L = b - a
    T = cu[-1]
    q, k, v = inputs.qkv_separate(T, 1, seed=seed)
    bits = lambda x: x.view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    if mode == "nvfp4":
        z = oracle.nvfp4_quantize(bits(q), bits(k), bits(v), cu)
    else:
        qz = [oracle.fp8_quantize(bits(x)) for x in (q, k, v)]
    if mode == "sparse":  # head 0's lists of the workload's pattern (one head: offsets [G + 1])
        off_all, idx_all = sparse_lists(sparse_name, cu, H)
        G = (len(off_all) - 1) // H
        off0 = off_all[:G + 1].copy()
        idx0 = idx_all[:off0[-1]].copy()
    t_quant = time.perf_counter() - t0
    ncores = os.cpu_count() or 1
    g = np.random.default_rng(seed)

    def attn_rows(n):
        rows = [(int(t), 0) for t in g.integers(a, b, n)]
        t1 = time.perf_counter()
        if mode == "nvfp4":
            oracle.attn_nvfp4(z, cu, rows, 1.0 / math.sqrt(D), n_kv=64)
        elif mode == "sparse":
            oracle.attn_fp8_sparse(qz[0][0], qz[1][0], qz[2][0], qz[0][1], qz[1][1], qz[2][1], cu,
                                   off0, idx0, rows, 1.0 / math.sqrt(D), tau=8.0)
        else:
            oracle.attn_fp8(qz[0][0], qz[1][0], qz[2][0], qz[0][1], qz[1][1], qz[2][1], cu, rows,
                            1.0 / math.sqrt(D))
        return time.perf_counter() - t1

    n0 = 2 * ncores
    t_cal = attn_rows(n0)
    per_row = t_cal / n0
    budget = max(seconds - t_quant - t_cal, 0.0)
    n1 = int(budget / max(per_row, 1e-9))
    n1 = max(0, min(n1, 200000))
    t_more = attn_rows(n1) if n1 > 0 else 0.0
    R = n0 + n1
    t_attn = t_cal + t_more
    # full-workload estimate: each head quantizes once and runs every query row of every segment
    per_row = t_attn / R
    # per-row cost grows with its segment's length: scale by L_s / L_longest
    qlabel = "NVFP4" if mode == "nvfp4" else "FP8"
    alabel = {"fp8": "FP8", "nvfp4": "NVFP4", "sparse": "block-sparse FP8"}[mode]
    if mode == "sparse":
        est_s = H * (t_quant + per_row * T)
        value = sparse_flops(cu, H, off_all, idx_all) / est_s / 1e12
    else:
        est_s = H * (t_quant + per_row * sum(x * x for x in lens) / L)
        value = attn_flops(cu, H) / est_s / 1e12
    return dict(value=value, unit=UNIT, cores=ncores, kind="oracle",
                sample=(f"head 0 of {H}: {qlabel} quantize of its full Q/K/V ({T} tokens, "
                        f"{t_quant:.2f} s) + {alabel}-emulating attention of {R} random query "
                        f"rows of "
                        f"the {L}-token segment ({t_attn:.2f} s); extrapolated to all {H} heads "
                        f"and rows"),
                seconds=t_quant + t_attn, est_full_workload_s=est_s)


# ------------------------------------------------------------------------------------------------
def max_over_ranks(x: float) -> float:
    """Maximum of x over the ranks of the default process group (x itself without one). The
    tensor lives on the device for NCCL and on the host for gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    cu, H = workload(args.workload)
    per_step = max(args.cpu_seconds / 3.0, 3.0)
    mode = mode_of(args.workload)
    for _ in range(args.warmup):
        oracle_sample(cu, H, per_step / 2, mode=mode, sparse_name=args.workload)
    vals, secs = [], []
    for i in range(args.steps):
        r = oracle_sample(cu, H, per_step, seed=i, mode=mode, sparse_name=args.workload)
        vals.append(r["value"])
        secs.append(r["est_full_workload_s"])
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRICS[mode], "value": v,
        "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(secs) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"f64 ({mode.upper()}-emulating oracle)",
        "data": "synthetic", "config": config_of(args.workload, cu, H),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def link_rates(hbuf, dbuf, stream):
    """Host-device link rates on this machine (GB/s): one copy of the page-locked input buffer each
    way, timed on the device. They bound the end-to-end numbers, which move with them."""
    import torch
    res = {}
    for name, dst, src in (("h2d_gbs", dbuf, hbuf), ("d2h_gbs", hbuf, dbuf)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(src, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = src.numel() * src.element_size() / (e0.elapsed_time(e1) / 1e3) / 1e9
    return res


def config_of(name, cu, H):
    T = cu[-1]
    c = {"workload": name, "tokens": T, "heads": H, "head_dim": D,
         "segments": [b - a for a, b in zip(cu[:-1], cu[1:])],
         "qkv_layout": "strided views of one fused [T,3,H,128] BF16 buffer",
         "softmax_scale": 1 / math.sqrt(D), "causal": False,
         "l2": "inputs (1.3 GB) and codes larger than L2: no flush"}
    if mode_of(name) == "nvfp4":
        c["k_offset"] = "per-(head, channel) K offset N(0, 4), constant over tokens"
    if mode_of(name) == "sparse":
        c["block_lists"] = ("64-row query blocks x 64-key blocks; per list density 0.25 x "
                            "U[0.5, 1.5) of the key blocks, uniform without replacement, "
                            "every 16th list dense (seed 0)")
    return c


def run_arm(args, name, ws, rank, with_e2e, with_cpu):
    """One workload's device arm: W untimed steps, then K timed steps (quantize + forward on
    resident inputs) bracketed by barriers and synchronizes, with the SM clocks sampled during
    the timed region; optionally the end-to-end host-buffer leg and the CPU-oracle baseline.
    Returns the JSON line of that workload."""
    import torch

    dev = torch.cuda.current_device()
    from precision_attention_diffusion_gb300 import fa_lp

    cu, H = workload(name)
    mode = mode_of(name)
    T = cu[-1]
    flops = attn_flops(cu, H)
    if mode == "sparse":
        off_h, idx_h = sparse_lists(name, cu, H, seed=rank)
        flops = sparse_flops(cu, H, off_h, idx_h)
        d_off = torch.from_numpy(off_h).cuda()
        d_idx = torch.from_numpy(idx_h).cuda()
    g = torch.Generator(device="cuda").manual_seed(1234 + rank)
    buf = torch.randn((T, 3, H, D), generator=g, device="cuda", dtype=torch.float32)
    if mode == "nvfp4":
        from precision_attention_diffusion_gb300 import inputs
        buf[:, 1] += inputs.k_channel_offset(H, seed=rank).cuda()[None]
    buf = buf.to(torch.bfloat16)
    q, k, v = buf[:, 0], buf[:, 1], buf[:, 2]
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    plan = fa_lp.Plan(cu, H, mode=fa_lp.MODE_NVFP4 if mode == "nvfp4" else fa_lp.MODE_FP8)
    stream = torch.cuda.current_stream()

    def forward():
        if mode == "sparse":
            plan.forward_sparse(d_off, d_idx, out, stream)
        else:
            plan.forward(out, cu_dev, stream)

    def step():
        plan.quantize(q, k, v, stream)
        forward()

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if plan.last_error():
        raise RuntimeError("device wait expired during warm-up")

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    evq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    ev[0].record(stream)
    for i in range(K):
        evq[i][0].record(stream)
        plan.quantize(q, k, v, stream)
        evq[i][1].record(stream)
        evf[i][0].record(stream)
        forward()
        evf[i][1].record(stream)
    ev[1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    total_ms = ev[0].elapsed_time(ev[1])
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in evf)
    q_ms = statistics.mean(a.elapsed_time(b) for a, b in evq)
    total_ms = max_over_ranks(total_ms)
    if plan.last_error():
        raise RuntimeError("device wait expired in the timed region")
    ms_per_step = total_ms / K
    value = ws * flops / (ms_per_step / 1e3) / 1e12
    # end to end through the public call with host buffers (fa_lp_attention_host): every step
    # copies the inputs from page-locked host memory, quantizes, runs the attention and copies the
    # output back; the library overlaps the copies of one chunk of heads with the compute of the
    # next
    e2e = None
    if with_e2e and mode == "sparse":
        # block-sparse end to end through fa_lp_attention_sparse_host: every step copies Q/K/V and
        # the block lists from page-locked host memory, quantizes, runs the block-sparse forward
        # and copies the output back; head chunks overlap their copies with the compute
        hbuf = buf.cpu().pin_memory()
        hout = torch.empty((T, H, D), dtype=torch.bfloat16).pin_memory()
        hoff = torch.from_numpy(off_h).pin_memory()
        hidx = torch.from_numpy(idx_h).pin_memory()
        hq, hk, hv = hbuf[:, 0], hbuf[:, 1], hbuf[:, 2]

        def e2e_step():
            plan.attention_sparse_host(hq, hk, hv, hoff, hidx, hout, stream=stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / K)
        if plan.last_error():
            raise RuntimeError("device error in the end-to-end region")
        in_bytes = (hbuf.numel() * hbuf.element_size() + hoff.numel() * 4 + hidx.numel() * 4)
        e2e = {"value": ws * flops / (e_ms / 1e3) / 1e12, "unit": UNIT,
               "ms_per_step": e_ms, "h2d_bytes_per_step": in_bytes,
               "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "call": "fa_lp_attention_sparse_host (page-locked host buffers and lists, head "
                       "chunks of the library's choice, copies overlapping the compute)"}
        with torch.cuda.stream(stream):
            e2e["link"] = link_rates(hbuf, buf, stream)
    elif with_e2e:
        hbuf = buf.cpu().pin_memory()
        hout = torch.empty((T, H, D), dtype=torch.bfloat16).pin_memory()
        hq, hk, hv = hbuf[:, 0], hbuf[:, 1], hbuf[:, 2]

        def e2e_step():
            plan.attention_host(hq, hk, hv, hout, stream=stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / K
        if plan.last_error():
            raise RuntimeError("device wait expired in the end-to-end region")
        e_ms = max_over_ranks(e_ms)
        e2e = {"value": ws * flops / (e_ms / 1e3) / 1e12, "unit": UNIT,
               "ms_per_step": e_ms, "h2d_bytes_per_step": hbuf.numel() * hbuf.element_size(),
               "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "call": "fa_lp_attention_host (page-locked host buffers, head chunks of the "
                       "library's choice, copies overlapping the compute)"}
        with torch.cuda.stream(stream):
            e2e["link"] = link_rates(hbuf, buf, stream)

    # NVFP4: the same steps with the qm K^T table held as a ring of two head-group slots
    # (fa_lp_plan_set_table_limit): the forward builds each group's table right before its
    # attention launch; the workspace stays under 0.5 GB at S = 30272, H = 56
    ring = None
    if mode == "nvfp4":
        whole = out.clone()
        ws_whole = plan.info()["workspace_bytes"]
        limit = 64 << 20
        plan.set_table_limit(limit)
        try:
            for _ in range(2):
                step()
            torch.cuda.synchronize()
            rq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            rf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            barrier()
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            r0.record(stream)
            for i in range(K):
                rq[i][0].record(stream)
                plan.quantize(q, k, v, stream)
                rq[i][1].record(stream)
                rf[i][0].record(stream)
                forward()
                rf[i][1].record(stream)
            r1.record(stream)
            torch.cuda.synchronize()
            if plan.last_error():
                raise RuntimeError("device wait expired in the table-ring region")
            lay = plan.table_layout()
            ring = {"table_limit_bytes": limit, "heads_per_slot": lay["heads_per_slot"],
                    "slot_bytes": lay["slot_bytes"],
                    "workspace_bytes": plan.info()["workspace_bytes"],
                    "workspace_bytes_whole_table": ws_whole,
                    "ms_per_step": max_over_ranks(r0.elapsed_time(r1) / K),
                    "forward_ms": statistics.mean(a.elapsed_time(b) for a, b in rf),
                    "quantize_ms": statistics.mean(a.elapsed_time(b) for a, b in rq),
                    "output_equals_whole_table": bool(torch.equal(out, whole))}
        finally:
            plan.set_table_limit(0)
        del whole

    pk = peaks()
    achieved = flops / (fwd_ms / 1e3) / 1e12
    kname = {"nvfp4": "attn_nvfp4", "fp8": "attn_fp8", "sparse": "attn_fp8_sparse"}[mode]
    sha = file_sha(os.path.join(ROOT, "precision_attention_diffusion_gb300", "csrc", kname + ".cu"))
    traffic = NCU_TRAFFIC.get((name, sha))
    pkey = "fp4" if mode == "nvfp4" else "fp8"
    # DRAM bytes the attention launch must move: the quantized operands once, the BF16 output once
    Tp = sum(-(-(b - a) // 128) * 128 for a, b in zip(cu[:-1], cu[1:]))
    codes_bytes = (3 * Tp * H * (D // 2 + D // 16) if mode == "nvfp4" else 3 * Tp * H * D)
    ratio = FP4_OVER_BF16 if mode == "nvfp4" else FP8_OVER_BF16
    roof = {"bound": "tensor", "achieved": achieved, "peak": pk[pkey], "unit": "TFLOP/s",
            "frac": achieved / pk[pkey], "traffic": traffic,
            "kernel": kname + "_kernel", "launch_ms": fwd_ms,
            "peak_note": (f"dense {pkey.upper()} = {ratio:g} x {pk['source']} BF16 cuBLAS burst; "
                          f"frac of sustained = {achieved / pk[pkey + '_sustained']:.3f}"),
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": codes_bytes + T * H * D * 2}
    if mode == "nvfp4":
        # quantize passes: Q, K read twice (means, pack), V once; codes + scales written
        q_bytes = 5 * T * H * D * 2 + 3 * T * H * (D // 2 + D // 16)
        dtype = "nvfp4 (e2m1 + ue4m3 per 16, fp32 accumulate, bf16 in/out)"
    else:
        # quantize passes: HBM-bound; algorithmic bytes = 2 reads of Q/K/V + 1 write of the codes
        q_bytes = 2 * 3 * T * H * D * 2 + 3 * T * H * D
        dtype = "fp8_e4m3 (fp32 accumulate, bf16 in/out)"
    if mode == "sparse":
        roof["algorithmic_flops_per_launch"] = flops
        roof["launch_note"] = ("forward_ms covers the list merge (one small kernel) and the "
                               "attention kernel")
    line = {
        "metric": METRICS[mode], "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic", "config": config_of(name, cu, H),
        "forward_ms": fwd_ms, "forward_tflops": achieved, "quantize_ms": q_ms,
        "quantize_gbs": q_bytes / (q_ms / 1e3) / 1e9,
        "frac_of_fp8_peak": achieved / pk["fp8"],
        "roofline": roof, "clocks": clocks, "e2e": e2e,
        "gpu_launches": KERNELS_PER_STEP[mode] * K,
    }
    if ring is not None:
        line["table_ring"] = ring
    if with_cpu:
        line["cpu_baseline"] = oracle_sample(cu, H, args.cpu_seconds, mode=mode, sparse_name=name)
    del buf, q, k, v, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


# Sub-objects of the default line: the second hot path (NVFP4) and the block-sparse forward at the
# same shape, each timed in the same process by the same procedure with its own clock sample.
EXTRA_ARMS = (("nvfp4", "nvfp4_s30272_h56"), ("sparse", "sparse_fp8_s30272_h56"))
ARM_KEYS = ("metric", "value", "unit", "ms_per_step", "forward_ms", "forward_tflops",
            "quantize_ms", "quantize_gbs", "roofline", "clocks", "gpu_launches", "config", "dtype",
            "table_ring", "e2e")


def run_ours(args):
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)

    from precision_attention_diffusion_gb300 import build as fbuild
    fbuild.build()

    line = run_arm(args, args.workload, ws, rank, with_e2e=not args.no_e2e,
                   with_cpu=rank == 0 and ws == 1 and not args.no_cpu_baseline)
    if args.workload == "fp8_s30272_h56" and not args.no_extra_arms:
        for key, name in EXTRA_ARMS:
            sub = run_arm(args, name, ws, rank, with_e2e=not args.no_e2e, with_cpu=False)
            line[key] = {k: sub[k] for k in ARM_KEYS if k in sub}
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
