"""Seeded synthetic inputs shared by the CUDA library's callers and by the tests'
CPU oracle: random-init weights, user token streams and the pre-filled K/V.

This module holds none of the decode step's arithmetic: it only draws numbers.

Recipe:
  * every matrix and embedding table is N(0, 0.02); every RMSNorm alpha is
    1 + N(0, 0.02) (so a mis-wired alpha is visible);
  * each block of a stacked tensor (one layer, one depformer step, one table) has
    its own torch CPU generator, seeded from (seed, tensor name, block index), so
    blocks are drawn in parallel threads and the result does not depend on the
    thread count or on drawing order;
  * bf16 models round every value once to bf16 (round to nearest even); alphas are
    then kept as f32 arrays holding those bf16 values;
  * user codes are uniform in [0, user_card) from the generator seeded with
    user_seed + session; the small model replaces each code by -1 with
    probability 0.05 (a second draw from the same generator);
  * the pre-filled K/V of the batch-64 workload is N(0, 1) rounded to bf16, drawn
    per session by a torch generator on the tensor's device seeded 3 + session.
"""
from __future__ import annotations

import hashlib
import os
from concurrent.futures import ThreadPoolExecutor

import torch

from .configs import N_Q, RQConfig

# (name, kind, block shape fn, leading block dims fn) in the C-ABI layout
#   kind: "mat" = N(0, 0.02) in the weight dtype; "alpha" = 1 + N(0, 0.02), f32 storage


def weight_layout(c: RQConfig):
    """Ordered (name, kind, lead_dims, block_shape) of every weight tensor.

    The full tensor shape is lead_dims + block_shape, row-major; each block is drawn
    from its own generator."""
    D, L, F, V, A = c.dim, c.layers, c.hidden, c.text_card, c.audio_card
    DD, DL, DF = c.ddim, c.dlayers, c.dhidden
    return [
        ("emb", "mat", (16,), (A + 1, D)),
        ("text_emb", "mat", (), (V + 1, D)),
        ("norm1", "alpha", (L,), (D,)),
        ("in_proj", "mat", (L,), (3 * D, D)),
        ("out_proj", "mat", (L,), (D, D)),
        ("norm2", "alpha", (L,), (D,)),
        ("gate_in", "mat", (L,), (2 * F, D)),
        ("gate_out", "mat", (L,), (D, F)),
        ("out_norm", "alpha", (), (D,)),
        ("text_linear", "mat", (), (V, D)),
        ("dep_in", "mat", (N_Q,), (DD, D)),
        ("dep_text_emb", "mat", (), (V + 1, DD)),
        ("dep_emb", "mat", (N_Q - 1,), (A + 1, DD)),
        ("dnorm1", "alpha", (DL,), (DD,)),
        ("dnorm2", "alpha", (DL,), (DD,)),
        ("d_in_proj", "mat", (DL, N_Q), (3 * DD, DD)),
        ("d_out_proj", "mat", (DL, N_Q), (DD, DD)),
        ("d_gate_in", "mat", (DL, N_Q), (2 * DF, DD)),
        ("d_gate_out", "mat", (DL, N_Q), (DD, DF)),
        ("linears", "mat", (N_Q,), (A, DD)),
    ]


WEIGHT_NAMES = [n for n, _, _, _ in weight_layout(
    RQConfig("x", 8, 1, 1, 8, 8, 8, 8, 8, 8, 1, 1, 8, 8, "f32", "f32"))]


def _seed(seed: int, name: str, block: int) -> int:
    h = hashlib.sha256(f"rq-synth:{seed}:{name}:{block}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _draw_block(out: torch.Tensor, kind: str, bf16: bool, seed: int) -> None:
    vals = torch.randn(out.shape, generator=_gen(seed), dtype=torch.float32)
    vals.mul_(0.02)
    if kind == "alpha":
        vals.add_(1.0)
        if bf16:
            vals = vals.to(torch.bfloat16).to(torch.float32)
    out.copy_(vals)  # float32 -> bfloat16 copy rounds to nearest even


def make_weights(c: RQConfig, seed: int = 0, threads: int | None = None) -> dict:
    """All weights as contiguous CPU tensors in the C-ABI layout.

    Matrices and tables are bfloat16 (bf16 models and the bands, which quantize the bf16
    matrices) or float32; alphas float32."""
    bf16 = c.weight_dtype in ("bf16", "q8", "q4")  # the bands start from bf16 weights
    mdt = torch.bfloat16 if bf16 else torch.float32
    out, jobs = {}, []
    for name, kind, lead, block in weight_layout(c):
        dt = torch.float32 if kind == "alpha" else mdt
        t = torch.empty(tuple(lead) + tuple(block), dtype=dt)
        out[name] = t
        nblk = 1
        for d in lead:
            nblk *= d
        flat = t.view((nblk,) + tuple(block))
        for b in range(nblk):
            jobs.append((flat[b], kind, _seed(seed, name, b)))
    threads = threads or min(32, os.cpu_count() or 1)
    if threads <= 1:
        for j in jobs:
            _draw_block(j[0], j[1], bf16, j[2])
    else:
        # biggest blocks first so the pool stays busy to the end
        jobs.sort(key=lambda j: -j[0].numel())
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda j: _draw_block(j[0], j[1], bf16, j[2]), jobs))
    return out


def user_tokens(c: RQConfig, frames: int, session: int = 0) -> torch.Tensor:
    """int32 [frames][8] user-audio codes for one session."""
    g = _gen(c.user_seed + session)
    tok = torch.randint(0, c.user_card, (frames, N_Q), generator=g, dtype=torch.int64)
    if c.user_minus1 > 0:
        drop = torch.rand((frames, N_Q), generator=g) < c.user_minus1
        tok[drop] = -1
    return tok.to(torch.int32)


def batch_user_tokens(c: RQConfig, frames: int) -> torch.Tensor:
    """int32 [frames][B][8]: session b's stream is user_tokens(c, frames, b)."""
    return torch.stack([user_tokens(c, frames, b) for b in range(c.batch)], dim=1).contiguous()


def kv_prefill(c: RQConfig, session: int, device="cpu"):
    """(K, V), each [layers][prefill][dim] bfloat16, N(0,1) rounded to bf16, drawn on
    `device` by a generator seeded 3 + session (K first, then V)."""
    g = torch.Generator(device=device)
    g.manual_seed(3 + session)
    shape = (c.layers, c.prefill, c.dim)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return k, v
