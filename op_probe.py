"""Time single operations of the decode step through the C ABI (rq_launch_op).

  python op_probe.py --workload moshi7b_2layer \
      --ops gate_in,qkv --reps 3 [--frames 4] [--batch 16] [--prefill 2900] [--band q4]

Builds the decoder for the workload (seeded synthetic weights; `--batch` overrides the
session count, `--prefill n` fills every session's temporal K/V with the workload's
synthetic positions 0..n-1; `--context` shrinks the K/V window, e.g. to profile a
linear on a small device footprint; `--band q8|q4` quantizes the matrices into that weight
band, which runs under the graph schedule), runs `--frames` whole frames, then for each op launches it
once per temporal layer `--reps` times, timed with CUDA events on the decoder's stream,
and prints one JSON line per op.  Used as the command under the profiler for the kernel
summaries in profiles/.
"""
import argparse
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from rq_transformer_frame_gb300 import binding, configs, synth  # noqa: E402

OPS = {"qkv": binding.RQ_OP_QKV, "attn": binding.RQ_OP_ATTN, "out_proj": binding.RQ_OP_OUT,
       "gate_in": binding.RQ_OP_GATE_IN, "gate_out": binding.RQ_OP_GATE_OUT,
       "text_head": binding.RQ_OP_HEAD, "frame": binding.RQ_OP_FRAME}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="moshi7b_2layer")
    ap.add_argument("--ops", default="gate_in")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--frames", type=int, default=2)
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--prefill", type=int, default=-1)
    ap.add_argument("--context", type=int, default=0)
    ap.add_argument("--band", default="", choices=["", "q8", "q4"])
    a = ap.parse_args(argv)
    cfg = configs.CONFIGS[a.workload]
    if a.batch > 0:
        cfg = cfg.with_(batch=a.batch)
    if a.prefill >= 0:
        cfg = cfg.with_(prefill=a.prefill)
    if a.context > 0:
        cfg = cfg.with_(context=a.context)
    torch.cuda.set_device(0)
    w = binding.upload_weights(synth.make_weights(cfg, seed=0))
    if a.band:
        w = binding.quantize_weights(w, binding.RQ_Q8 if a.band == "q8" else binding.RQ_Q4)
        cfg = cfg.with_(weight_dtype=a.band)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dec = binding.Decoder(cfg, w, stream=stream)
        for b in range(cfg.batch if cfg.prefill else 0):
            k, v = synth.kv_prefill(cfg, b, device=torch.device("cuda", 0))
            dec.set_kv(b, k, v)
            del k, v
    users = synth.batch_user_tokens(cfg, max(a.frames, 1)).numpy()
    for t in range(a.frames):
        dec.step(users[t])
    for name in a.ops.split(","):
        op = OPS[name]
        layers = range(1) if name in ("text_head", "frame") else range(cfg.layers)
        nb = dec.launch_op(op, 0, 0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = 0
        for _ in range(a.reps):
            for l in layers:
                dec.launch_op(op, l, 1)
                n += 1
        e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / max(n, 1)
        print(json.dumps({"workload": cfg.name, "batch": cfg.batch, "prefill": cfg.prefill,
                          "schedule": dec.schedule, "op": name, "launches": n,
                          "us_per_launch": round(us, 2), "bytes_per_launch": nb,
                          "GB/s": round(nb / max(us, 1e-9) / 1e3, 1)}), flush=True)
    dec.reset(-1)
    dec.close()


if __name__ == "__main__":
    main()
