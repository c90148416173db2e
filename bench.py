"""Benchmark of the per-frame RQ-Transformer decode step on GB300.

One step = one frame of the whole hot path for every session (ring cache,
embedding sum, temporal decoder, text head, 8 depformer codebook steps, realign).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--impl native|reference]

Prints ONE JSON line (rank 0).  `value` = session-frames/s with the user tokens
already resident in HBM (rq_step_device), timed with CUDA events on the decode
stream, max over ranks; `e2e` = the same through rq_step with host buffers (the
host->device copy of the step's codes and the device->host read of its tokens inside
the timed region).  Unless --no-extra, the line also carries the other Moshi-7B
workloads measured the same way (keys batch1_mean_window: batch 1 at the 375-frame
workload's mean window; batch16; batch64: K/V pre-filled to 2900 positions), each
with its own ms_per_step, clocks, roofline and dominant kernel.  N > 1 runs N independent replicas (sessions shard across GPUs;
no collective on the data path), so scaling is weak.  The reference arm times the
CPU oracle on the host cores on the same workload.
"""
from __future__ import annotations

import argparse
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

WORKLOADS = {1: "moshi7b", 16: "moshi7b_b16", 64: "moshi7b_b64"}


def frame_bytes(c, offsets) -> dict:
    """Algorithmic bytes of one frame: every weight streamed once, the gathered
    embedding rows, the live K/V window read once and one K/V row written."""
    es, kv = c.weight_bytes, c.kv_bytes
    D, L, F, V, A = c.dim, c.layers, c.hidden, c.text_card, c.audio_card
    DD, DL, DF = c.ddim, c.dlayers, c.dhidden
    temporal = L * (3 * D * D + D * D + 2 * F * D + D * F) * es
    head = V * D * es
    dep = 8 * DL * (3 * DD * DD + DD * DD + 2 * DF * DD + DD * DF) * es
    dep_in = 8 * DD * D * es
    lin = 8 * A * DD * es
    emb = c.batch * (17 * D + 8 * DD) * es
    kv_read = sum(2 * min(o + 1, c.context) * D * kv * L for o in offsets)
    kv_write = c.batch * 2 * D * kv * L
    w = temporal + head + dep + dep_in + lin
    return {"weights": w, "temporal": temporal, "kv": kv_read + kv_write,
            "total": w + emb + kv_read + kv_write}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {
    "gemv": ("gemv_kernel.cuh", "gemv_launch.cuh", "gemv.cu", "sampling.cuh", "common.cuh",
             "kernels.h"),
    "frame": ("frame_persistent.cuh", "frame_persistent.cu", "frame_persistent_greedy.cu",
              "frame_persistent_dep.cu", "frame_persistent_band.cu", "gemv_kernel.cuh",
              "sampling.cuh", "common.cuh", "kernels.h"),
    "tc": ("tc_gemm.cu", "tc_epilogue.cuh", "tc_common.cuh", "sampling.cuh", "common.cuh",
           "kernels.h"),
    "attn": ("attn.cu", "common.cuh", "kernels.h"),
}


def source_hash(kind: str) -> str:
    h = hashlib.sha256()
    for n in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "rq_transformer_frame_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(name: str, kind: str, bytes_per_launch: float = None):
    """DRAM bytes per launch from a committed ncu summary, only if it was taken on the
    current kernel source (the summary records the source hash).  A capture of a
    smaller case is scaled by algorithmic bytes (traffic grows in proportion)."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    hsh = re.search(r"source_hash:\s*([0-9a-f]+)", txt)
    if not m or not hsh or hsh.group(1) != source_hash(kind):
        return None
    t = float(m.group(1))
    a = re.search(r"algorithmic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if bytes_per_launch is not None and a:
        t *= bytes_per_launch / float(a.group(1))
    return t


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self) -> dict:
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": mx or None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- ranks
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle arm
def oracle_frames(cfg, w, users, max_frames: int, budget_s: float):
    """Run oracle frames of session 0 until max_frames or the time budget; returns
    (frames, seconds, threads)."""
    import oracle
    orc = oracle.Oracle(cfg, w)
    st = orc.new_state()
    n, t0 = 0, time.perf_counter()
    while n < max_frames:
        orc.step(st, users[n % len(users), 0])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return n, time.perf_counter() - t0, oracle.max_threads()


def run_reference(args, cfg):
    from rq_transformer_frame_gb300 import synth
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = synth.make_weights(cfg.with_(batch=1), seed=0)
    users = synth.batch_user_tokens(cfg, args.steps + args.warmup).numpy()
    import oracle
    orc = oracle.Oracle(cfg.with_(batch=1), w)
    st = orc.new_state()
    for t in range(args.warmup):
        orc.step(st, users[t, 0])
    t0 = time.perf_counter()
    for t in range(args.steps):
        orc.step(st, users[args.warmup + t, 0])
    dt = time.perf_counter() - t0
    value = args.steps / dt  # session-frames/s of one session on the host cores
    line = {
        "impl": "reference", "metric": "frames/s", "value": value, "unit": "session-frames/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": 1,
                   "note": "oracle timed on one session of the workload"},
        "cpu_baseline": {"value": value, "unit": "session-frames/s",
                         "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": "frames %d..%d of session 0" % (args.warmup, args.warmup + args.steps)},
        "e2e": {"value": value, "unit": "session-frames/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- native arm
def time_frames(dec, d_users, d_out, d_has, first, K, stream, dev, ws, local):
    """K device-resident frames after a barrier, CUDA events on the decode stream;
    returns (seconds, max over ranks, clock samples)."""
    import torch
    dec.sync()
    barrier(ws)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for t in range(K):
            dec.step_device(d_users[first + t], d_out, d_has)
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize(dev)
    dec.sync()
    barrier(ws)
    sec = ev0.elapsed_time(ev1) / 1e3
    return max_over_ranks(sec, ws, dev), clk.summary()


def kernel_table(dec, cfg, stream, dev, hbm_peak):
    """Each linear kind and the attention launched alone over distinct layers (nothing
    L2-resident), CUDA events on the decode stream."""
    import torch
    from rq_transformer_frame_gb300 import binding
    kernels = {}
    names = {binding.RQ_OP_QKV: "qkv", binding.RQ_OP_ATTN: "attention",
             binding.RQ_OP_OUT: "out_proj", binding.RQ_OP_GATE_IN: "gate_in",
             binding.RQ_OP_GATE_OUT: "gate_out", binding.RQ_OP_HEAD: "text_head"}
    reps = 3
    for op, name in names.items():
        layers = range(cfg.layers) if op != binding.RQ_OP_HEAD else range(1)
        nb = dec.launch_op(op, 0, 0)
        dec.launch_op(op, 0, 1)  # warm
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = 0
        for _ in range(reps if op != binding.RQ_OP_HEAD else 20):
            for l in layers:
                dec.launch_op(op, l, 1)
                n += 1
        e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / n
        kernels[name] = {"us_per_launch": round(us, 2), "bytes_per_launch": nb,
                         "GB/s": round(nb / us / 1e3, 1),
                         "frac_of_measured_hbm": round(nb / us / 1e3 / hbm_peak, 4),
                         "launches_per_frame": len(layers),
                         "ms_per_frame": round(us * len(layers) / 1e3, 3)}
    return kernels


def frame_kernel_roofline(dec, cfg, stream, dev, hbm_peak, peak_kind, traffic_name):
    """The persistent whole-frame kernel at the handle's current window: launched alone
    10 times with events on the decode stream; plus the stages of the last frame."""
    import torch
    from rq_transformer_frame_gb300 import binding
    us_ops = dec.op_times()
    nb = dec.launch_op(binding.RQ_OP_FRAME, 0, 0)
    dec.launch_op(binding.RQ_OP_FRAME, 0, 2)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nrep = 10
    e0.record(stream)
    dec.launch_op(binding.RQ_OP_FRAME, 0, nrep)
    e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / nrep
    roof = {"kernel": "frame_persistent_kernel: the frame's two cooperative launches (temporal "
                      "stack, text head and input projections at 2 CTAs/SM; depformer at 1 "
                      "CTA/SM) -- every linear and attention of a frame",
            "bound": "hbm", "achieved": round(nb / us / 1e3, 1), "peak": hbm_peak,
            "unit": "GB/s", "peak_kind": peak_kind,
            "frac": round(nb / us / 1e3 / hbm_peak, 4), "us_per_launch": round(us, 1),
            "bytes_per_launch": nb,
            "traffic": profiled_traffic(traffic_name, "frame", nb) if traffic_name else None}
    stages = None
    if us_ops is not None:
        L = cfg.layers
        stages = {"temporal_ms": round(float(us_ops[:5 * L].sum()) / 1e3, 3),
                  "text_head_ms": round(float(us_ops[5 * L]) / 1e3, 3),
                  "depformer_ms": round(float(us_ops[5 * L + 1:].sum()) / 1e3, 3),
                  "ops": int(len(us_ops))}
    return roof, stages


def dominant_roofline(dec, cfg, kernels, frame_s, hbm_peak, peak_kind):
    """The kernel with the largest share of the frame (time per launch x launches)."""
    from rq_transformer_frame_gb300 import binding
    B = cfg.batch
    name = max(kernels, key=lambda k: kernels[k]["ms_per_frame"])
    dom = kernels[name]
    tensor = dec.schedule == binding.RQ_SCHEDULE_TENSOR
    if name == "attention":
        label = "attn_decode_kernel (split-K decode attention over the K/V window, one layer)"
        traffic = profiled_traffic("attn_%s.md" % cfg.name, "attn", dom["bytes_per_launch"])
    elif tensor:
        label = "tc_gemm_kernel<%d> (%s on the tcgen05 tensor cores, one layer)" % (
            (B + 15) // 16 * 16, name)
        traffic = profiled_traffic("tc_gemm_%s.md" % cfg.name, "tc", dom["bytes_per_launch"])
    else:
        label = "gemv_kernel<bf16> (%s, one layer)" % name
        traffic = profiled_traffic("gemv_moshi7b_b1.md", "gemv")
    return {"kernel": label, "bound": "hbm", "achieved": dom["GB/s"], "peak": hbm_peak,
            "unit": "GB/s", "peak_kind": peak_kind, "frac": round(dom["GB/s"] / hbm_peak, 4),
            "us_per_launch": dom["us_per_launch"], "bytes_per_launch": dom["bytes_per_launch"],
            "share_of_frame": round(dom["ms_per_frame"] / (1e3 * frame_s), 3),
            "traffic": traffic}


def make_decoder(cfg, w_dev, stream, sched, dev, prefill=0):
    """A handle of cfg on the decode stream; prefill > 0 pre-fills every session's K/V
    (synth.kv_prefill, drawn on the GPU) to that many positions."""
    import torch
    from rq_transformer_frame_gb300 import binding, synth
    with torch.cuda.stream(stream):
        dec = binding.Decoder(cfg, w_dev, stream=stream, schedule=sched)
        if prefill:
            c = cfg.with_(prefill=prefill)
            for b in range(cfg.batch):
                k, v = synth.kv_prefill(c, b, device=dev)
                dec.set_kv(b, k, v)
                del k, v
    return dec


def workload_line(cfg, w_dev, stream, dev, ws, local, K, W, prefill, hbm_peak, peak_kind):
    """One more workload measured as the headline is (device-resident codes, events
    around exactly K frames after W warm-up frames), with its own clocks and roofline."""
    import torch
    from rq_transformer_frame_gb300 import binding, synth
    B = cfg.batch
    dec = make_decoder(cfg, w_dev, stream, binding.RQ_SCHEDULE_AUTO, dev, prefill)
    users = synth.batch_user_tokens(cfg, W + K).to(dev)
    d_out = torch.zeros((B, 9), dtype=torch.int32, device=dev)
    d_has = torch.zeros(B, dtype=torch.uint8, device=dev)
    for t in range(W):
        dec.step_device(users[t], d_out, d_has)
    sec, clocks = time_frames(dec, users, d_out, d_has, W, K, stream, dev, ws, local)
    fb = [frame_bytes(cfg, [prefill + W + t] * B) for t in range(K)]
    bytes_frame = sum(f["total"] for f in fb) / K
    frame_s = sec / K
    line = {"workload": cfg.name, "batch": B, "start_offset": prefill + W,
            "frames_timed": K, "ms_per_step": 1e3 * frame_s,
            "value": ws * B / frame_s, "unit": "session-frames/s",
            "tokens_per_s": 9 * ws * B / frame_s,
            "schedule": {1: "graph", 2: "persistent", 3: "tensor"}.get(dec.schedule, "?"),
            "hbm": {"bytes_per_frame": bytes_frame,
                    "GB/s": round(bytes_frame / frame_s / 1e9, 1),
                    "frac_of_measured": round(bytes_frame / frame_s / 1e9 / hbm_peak, 4)},
            "clocks": clocks}
    if dec.schedule == binding.RQ_SCHEDULE_PERSISTENT:
        line["roofline"], line["stages"] = frame_kernel_roofline(
            dec, cfg, stream, dev, hbm_peak, peak_kind, None)
    else:
        kernels = kernel_table(dec, cfg, stream, dev, hbm_peak)
        line["roofline"] = dominant_roofline(dec, cfg, kernels, frame_s, hbm_peak, peak_kind)
        line["kernels"] = kernels
    dec.close()
    return line


def run_native(args, cfg):
    import numpy as np
    import torch

    from rq_transformer_frame_gb300 import binding, configs, synth
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    K, W, B = args.steps, args.warmup, cfg.batch
    w_host = synth.make_weights(cfg, seed=0)
    w_dev = binding.upload_weights(w_host, dev)
    stream = torch.cuda.Stream(device=dev)
    sched = {"auto": binding.RQ_SCHEDULE_AUTO, "graph": binding.RQ_SCHEDULE_GRAPH,
             "persistent": binding.RQ_SCHEDULE_PERSISTENT,
             "tensor": binding.RQ_SCHEDULE_TENSOR}[args.schedule]
    dec = make_decoder(cfg, w_dev, stream, sched, dev, cfg.prefill)
    users = synth.batch_user_tokens(cfg, W + 2 * K)
    d_users = users.to(dev)
    d_out = torch.zeros((B, 9), dtype=torch.int32, device=dev)
    d_has = torch.zeros(B, dtype=torch.uint8, device=dev)
    start0 = cfg.prefill

    # ---- warm-up, then K device-resident frames timed with events on the stream
    for t in range(W):
        dec.step_device(d_users[t], d_out, d_has)
    sec_max, clocks = time_frames(dec, d_users, d_out, d_has, W, K, stream, dev, ws, local)
    value = ws * B * K / sec_max
    offs = [[start0 + W + t] * B for t in range(K)]
    fb = [frame_bytes(cfg, o) for o in offs]
    bytes_frame = sum(f["total"] for f in fb) / K

    # ---- end to end through rq_step: host codes in, host tokens out, every step
    users_h = users.numpy()
    t0 = time.perf_counter()
    for t in range(K):
        dec.step(users_h[W + K + t])
    e2e_sec = max_over_ranks(time.perf_counter() - t0, ws, dev)
    e2e_value = ws * B * K / e2e_sec
    h2d = B * 18 * 4
    d2h = B * 18 * 4 + ((B + 3) // 4) * 4 + 4

    # ---- per-kernel timing of the GEMVs (distinct layers, so nothing is L2-resident)
    hbm_peak, peak_kind = peaks()
    kernels = kernel_table(dec, cfg, stream, dev, hbm_peak)
    dec.reset(-1)
    stages = None
    if dec.schedule == binding.RQ_SCHEDULE_PERSISTENT:
        # the frame's dominant kernel is the persistent whole-frame kernel itself
        for t in range(W):
            dec.step_device(d_users[t], d_out, d_has)
        dec.sync()
        roof, stages = frame_kernel_roofline(dec, cfg, stream, dev, hbm_peak, peak_kind,
                                             "frame_persistent_moshi7b.md")
        dec.reset(-1)
    else:
        roof = dominant_roofline(dec, cfg, kernels, sec_max / K, hbm_peak, peak_kind)
    n_launch = dec.kernels_per_frame
    sched_name = {1: "graph", 2: "persistent", 3: "tensor"}.get(dec.schedule, "?")
    dec.close()

    # ---- the other Moshi-7B workloads, each measured the same way on this GPU
    extra = {}
    if not args.no_extra and args.workload is None and args.schedule == "auto":
        KX = min(K, 20)
        # batch 1 at the mean window of the 375-frame workload (positions 0..374: 188)
        mean_pos = configs.MOSHI7B.frames // 2
        pre = max(0, mean_pos - W - KX // 2)
        todo = [("batch1_mean_window", configs.MOSHI7B, pre),
                ("batch16", configs.MOSHI7B_B16, 0),
                ("batch64", configs.MOSHI7B_B64, configs.MOSHI7B_B64.prefill)]
        for key, c, pre in todo:
            if c.name == cfg.name and pre == cfg.prefill:
                continue
            kx = min(KX, c.context - pre - W)
            extra[key] = workload_line(c, w_dev, stream, dev, ws, local, kx, W, pre,
                                       hbm_peak, peak_kind)
            torch.cuda.empty_cache()

    # ---- the oracle on this machine's host cores, on a bounded sample (rank 0, N = 1)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        c1 = cfg.with_(batch=1)
        import oracle
        orc_users = users_h
        n, s, thr = oracle_frames(c1, w_host, orc_users, 200, args.cpu_budget)
        cpu = {"value": n / s, "unit": "session-frames/s", "cores": thr, "kind": "oracle",
               "sample": "first %d frames of session 0 of %s (%.1f s)" % (n, cfg.name, s)}

    line = {
        "metric": "frames/s", "value": value, "unit": "session-frames/s", "n_gpus": ws,
        "steps": K, "warmup": W, "ms_per_step": 1e3 * sec_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": B, "frames_timed": K,
                   "start_offset": start0 + W,
                   "parallelism": "replicas" if ws > 1 else "single-gpu",
                   "l2": "not flushed: %.1f GB of weights streamed per frame >> 126 MB L2"
                         % (fb[0]["weights"] / 1e9),
                   "arith": ("bf16 weights and K/V, f32 activations and accumulation" +
                             ("; tensor-core GEMMs on two-part bf16 activation operands (16 significant bits)"
                              if sched_name == "tensor" else ""))},
        "tokens_per_s": 9 * value,
        "hbm": {"bytes_per_frame": bytes_frame, "GB/s": round(bytes_frame / (sec_max / K) / 1e9, 1),
                "frac_of_measured": round(bytes_frame / (sec_max / K) / 1e9 / hbm_peak, 4),
                "frac_of_8TBs": round(bytes_frame / (sec_max / K) / 8e12, 4)},
        "roofline": roof, "kernels": kernels, "stages": stages,
        "schedule": sched_name,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "session-frames/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K * n_launch,
        "clocks": clocks,
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--batch", type=int, default=1, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="only the headline workload (skip the other batch sizes)")
    ap.add_argument("--workload", default=None, help="override: a name from configs.CONFIGS")
    ap.add_argument("--schedule", default="auto",
                    choices=["auto", "graph", "persistent", "tensor"])
    args = ap.parse_args(argv)
    from rq_transformer_frame_gb300 import configs
    cfg = configs.CONFIGS[WORKLOADS[args.batch]]
    if args.workload:
        cfg = configs.CONFIGS[args.workload]
    if args.impl == "reference":
        return run_reference(args, cfg)
    import __graft_entry__
    __graft_entry__.build()
    return run_native(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
