"""ctypes binding of the C ABI in include/rq.h (argument marshalling only).

Every step of the decode path runs in the CUDA library (_lib/librq.so); this module
only moves pointers and sizes across the boundary.  There is no fallback: if the
library is missing, loading it raises.  PyTorch is used for device memory and
streams.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from .configs import RQConfig

LIBPATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "librq.so")

RQ_OK, RQ_ERR_ARG, RQ_ERR_TOKEN, RQ_ERR_CUDA = 0, 1, 2, 3
RQ_ERR_OOM, RQ_ERR_TIMEOUT, RQ_ERR_UNSUPPORTED, RQ_ERR_POISONED = 4, 5, 6, 7
RQ_F32, RQ_BF16 = 0, 1
RQ_OP_QKV, RQ_OP_ATTN, RQ_OP_OUT, RQ_OP_GATE_IN, RQ_OP_GATE_OUT, RQ_OP_HEAD, RQ_OP_FRAME = range(7)

WEIGHT_FIELDS = [
    "emb", "text_emb", "norm1", "in_proj", "out_proj", "norm2", "gate_in",
    "gate_out", "out_norm", "text_linear", "dep_in", "dep_text_emb", "dep_emb",
    "dnorm1", "dnorm2", "d_in_proj", "d_out_proj", "d_gate_in", "d_gate_out",
    "linears",
]

_CFG_INT_FIELDS = ["batch", "dim", "layers", "heads", "head_dim", "hidden", "context",
                   "text_card", "audio_card", "ddim", "dlayers", "dheads", "dhead_dim",
                   "dhidden", "weight_dtype", "kv_dtype"]


RQ_SCHEDULE_AUTO, RQ_SCHEDULE_GRAPH, RQ_SCHEDULE_PERSISTENT, RQ_SCHEDULE_TENSOR = 0, 1, 2, 3
RQ_PICK_GREEDY, RQ_PICK_TOPK, RQ_PICK_GUMBEL = 0, 1, 2
RQ_F32, RQ_BF16, RQ_Q8, RQ_Q4 = 0, 1, 2, 3
# stacked weight matrices (the weight bands quantize these; tables and alphas stay)
MATRIX_FIELDS = ("in_proj", "out_proj", "gate_in", "gate_out", "text_linear", "dep_in",
                 "d_in_proj", "d_out_proj", "d_gate_in", "d_gate_out", "linears")


class RqConfig(C.Structure):
    _fields_ = [(n, C.c_int32) for n in _CFG_INT_FIELDS] + \
        [("rms_eps", C.c_float), ("rope_theta", C.c_float), ("schedule", C.c_int32)]


class RqWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS]


class RQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("rq status %d: %s" % (status, msg))
        self.status = status


_LIB = None


def load() -> C.CDLL:
    """Load librq.so; raises if it has not been built (no CPU fallback exists)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIBPATH):
        raise RuntimeError("CUDA library %s is not built; run __graft_entry__.build()" % LIBPATH)
    L = C.CDLL(LIBPATH)
    P, I32 = C.c_void_p, C.c_int32
    L.rq_create.argtypes = [C.POINTER(RqConfig), C.POINTER(RqWeights), P, C.POINTER(P)]
    L.rq_destroy.argtypes = [P]
    L.rq_destroy.restype = None
    L.rq_reset.argtypes = [P, I32]
    L.rq_step.argtypes = [P, P, P, P]
    L.rq_step_forced.argtypes = [P, P, P, P, P, P]
    L.rq_step_device.argtypes = [P, P, P, P]
    L.rq_sync.argtypes = [P]
    L.rq_get_logits.argtypes = [P, P, P]
    L.rq_get_trace.argtypes = [P, P, P]
    L.rq_get_ring.argtypes = [P, P, P]
    L.rq_set_kv.argtypes = [P, I32, I32, P, P]
    L.rq_launch_op.argtypes = [P, I32, I32, I32, C.POINTER(C.c_double)]
    L.rq_set_sampling.argtypes = [P, I32, C.c_float, C.c_float, I32, I32, P]
    L.rq_get_rng.argtypes = [P, P]
    L.rq_band_row_bytes.argtypes = [I32, I32]
    L.rq_band_row_bytes.restype = C.c_size_t
    L.rq_quantize.argtypes = [I32, P, I32, C.c_int64, I32, P, P]
    L.rq_quantize.restype = C.c_int
    L.rq_prime.argtypes = [P, I32, I32, P, P]
    L.rq_replay.argtypes = [P, I32, I32, P]
    L.rq_snapshot_size.argtypes = [P, I32]
    L.rq_snapshot_size.restype = C.c_size_t
    L.rq_snapshot.argtypes = [P, I32, P, C.c_size_t]
    L.rq_restore.argtypes = [P, I32, P, C.c_size_t]
    L.rq_frame_kernel_count.argtypes = [P]
    L.rq_frame_kernel_count.restype = I32
    L.rq_schedule.argtypes = [P]
    L.rq_schedule.restype = I32
    L.rq_set_wait_limit.argtypes = [P, C.c_uint64, I32]
    L.rq_set_wait_limit.restype = C.c_int
    L.rq_get_op_times.argtypes = [P, P, I32]
    L.rq_get_op_times.restype = I32
    L.rq_last_error.argtypes = [P]
    L.rq_last_error.restype = C.c_char_p
    L.rq_status_string.argtypes = [C.c_int]
    L.rq_status_string.restype = C.c_char_p
    L.rq_abi_version.restype = I32
    L.rq_attention_workspace_size.argtypes = [I32, I32, I32, I32]
    L.rq_attention_workspace_size.restype = C.c_size_t
    L.rq_attention.argtypes = [I32, I32, I32, I32, I32, P, P, P, P, P, P, C.c_size_t, P]
    L.rq_attention.restype = C.c_int
    for f in ("rq_create", "rq_reset", "rq_step", "rq_step_forced", "rq_step_device",
              "rq_sync", "rq_get_logits", "rq_get_trace", "rq_get_ring", "rq_set_kv",
              "rq_launch_op", "rq_set_sampling", "rq_get_rng", "rq_prime", "rq_replay",
              "rq_snapshot", "rq_restore"):
        getattr(L, f).restype = C.c_int
    _LIB = L
    return L


def make_config(cfg: RQConfig, schedule: int = RQ_SCHEDULE_AUTO) -> RqConfig:
    c = RqConfig()
    for n in _CFG_INT_FIELDS:
        if n == "weight_dtype":
            v = {"bf16": RQ_BF16, "q8": RQ_Q8, "q4": RQ_Q4}.get(cfg.weight_dtype, RQ_F32)
        elif n == "kv_dtype":
            v = RQ_BF16 if cfg.kv_dtype == "bf16" else RQ_F32
        else:
            v = getattr(cfg, n)
        setattr(c, n, int(v))
    c.rms_eps = cfg.eps
    c.rope_theta = cfg.rope_theta
    c.schedule = int(schedule)
    return c


def upload_weights(host: dict, device="cuda") -> dict:
    """Copy host weight tensors (synth.make_weights) to contiguous device tensors."""
    return {k: v.to(device, non_blocking=False).contiguous() for k, v in host.items()}


def quantize(t: torch.Tensor, dtype: int, stream=None) -> torch.Tensor:
    """rq_quantize: a CUDA f32 / bf16 tensor [..., cols] into weight-band rows (uint8
    [rows * row_bytes]); cols a multiple of 32."""
    L = load()
    assert t.is_cuda and t.is_contiguous() and t.dtype in (torch.float32, torch.bfloat16)
    cols = int(t.shape[-1])
    rows = t.numel() // cols
    rb = int(L.rq_band_row_bytes(int(dtype), cols))
    if rb == 0:
        raise ValueError("cols must be a positive multiple of 32")
    out = torch.empty(rows * rb, dtype=torch.uint8, device=t.device)
    st = stream if stream is not None else torch.cuda.current_stream(t.device)
    rc = L.rq_quantize(int(dtype), t.data_ptr(), RQ_BF16 if t.dtype == torch.bfloat16 else RQ_F32,
                       rows, cols, out.data_ptr(), C.c_void_p(st.cuda_stream))
    if rc != RQ_OK:
        raise RQError(rc, "rq_quantize failed")
    return out


def quantize_weights(weights: dict, dtype: int) -> dict:
    """Device weights (bf16 / f32) with every matrix replaced by its weight-band rows."""
    return {k: (quantize(v, dtype) if k in MATRIX_FIELDS else v) for k, v in weights.items()}


def _p(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        assert t.flags["C_CONTIGUOUS"]
        return t.ctypes.data
    assert t.is_contiguous()
    return t.data_ptr()


class Decoder:
    """One rq_handle: B sessions of the per-frame decode step on the current device.

    `weights` are device tensors in the layout of include/rq.h (kept referenced for
    the handle's lifetime).  `stream` is a torch.cuda.Stream (default: the current
    stream)."""

    def __init__(self, cfg: RQConfig, weights: dict, stream=None,
                 schedule: int = RQ_SCHEDULE_AUTO):
        self.L = load()
        self.cfg = cfg
        self.weights = weights
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self._c = make_config(cfg, schedule)
        self._w = RqWeights(**{n: weights[n].data_ptr() for n in WEIGHT_FIELDS})
        h = C.c_void_p()
        st = self.L.rq_create(C.byref(self._c), C.byref(self._w),
                              C.c_void_p(self.stream.cuda_stream), C.byref(h))
        if st != RQ_OK:
            raise RQError(st, self.L.rq_last_error(None).decode())
        self.h = h
        B = cfg.batch
        self._out = np.zeros((B, 9), np.int32)
        self._own = np.zeros((B, 9), np.int32)
        self._has = np.zeros(B, np.uint8)

    def _check(self, st):
        if st != RQ_OK:
            raise RQError(st, self.L.rq_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.L.rq_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def step(self, user):
        """user [B][8] int32 -> (out [B][9], has_output [B] bool)."""
        u = np.ascontiguousarray(user, dtype=np.int32).reshape(self.cfg.batch, 8)
        self._check(self.L.rq_step(self.h, _p(u), _p(self._out), _p(self._has)))
        return self._out.copy(), self._has.astype(bool)

    def step_forced(self, user, forced):
        """-> (own [B][9], out [B][9], has_output [B])."""
        u = np.ascontiguousarray(user, dtype=np.int32).reshape(self.cfg.batch, 8)
        f = np.ascontiguousarray(forced, dtype=np.int32).reshape(self.cfg.batch, 9)
        self._check(self.L.rq_step_forced(self.h, _p(u), _p(f), _p(self._own), _p(self._out),
                                          _p(self._has)))
        return self._own.copy(), self._out.copy(), self._has.astype(bool)

    def step_device(self, d_user, d_out=None, d_has=None):
        """Enqueue a frame with device-resident int32 [B][8] input; no sync."""
        self._check(self.L.rq_step_device(self.h, _p(d_user), _p(d_out), _p(d_has)))

    def sync(self):
        self._check(self.L.rq_sync(self.h))

    def set_sampling(self, mode: int, temp: float = 0.8, temp_text: float = 0.7,
                     top_k: int = 250, top_k_text: int = 25, seeds=None):
        """Token picks (rq_set_sampling); defaults are the page's `Sampling` values.
        seeds: one per session (required unless mode is greedy)."""
        sd = None
        if seeds is not None:
            sd = np.ascontiguousarray(seeds, dtype=np.uint64)
            assert sd.shape == (self.cfg.batch,)
        self._check(self.L.rq_set_sampling(self.h, int(mode), float(temp), float(temp_text),
                                           int(top_k), int(top_k_text),
                                           None if sd is None else _p(sd)))

    def rng(self) -> np.ndarray:
        """Each session's sampler state after the last frame."""
        out = np.zeros(self.cfg.batch, np.uint64)
        self._check(self.L.rq_get_rng(self.h, _p(out)))
        return out

    def prime(self, session: int, forced, user):
        """Teacher-forced prompt steps (rq_prime): forced [n][9], user [n][8] int32."""
        f = np.ascontiguousarray(forced, dtype=np.int32).reshape(-1, 9)
        u = np.ascontiguousarray(user, dtype=np.int32).reshape(-1, 8)
        assert f.shape[0] == u.shape[0]
        self._check(self.L.rq_prime(self.h, int(session), f.shape[0], _p(f), _p(u)))

    def replay(self, session: int, x):
        """Embedding replay (rq_replay): x [n][dim] f32 (numpy or a CUDA tensor)."""
        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.float32 and x.is_contiguous()
            n = x.shape[0]
        else:
            x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, self.cfg.dim)
            n = x.shape[0]
        self._check(self.L.rq_replay(self.h, int(session), int(n), _p(x)))

    def snapshot(self, session: int) -> np.ndarray:
        """One session's ring, offset and K/V window as bytes (rq_snapshot)."""
        n = int(self.L.rq_snapshot_size(self.h, int(session)))
        buf = np.zeros(n, np.uint8)
        self._check(self.L.rq_snapshot(self.h, int(session), _p(buf), n))
        return buf

    def restore(self, session: int, snap: np.ndarray):
        snap = np.ascontiguousarray(snap, dtype=np.uint8)
        self._check(self.L.rq_restore(self.h, int(session), _p(snap), snap.size))

    def reset(self, session: int = -1):
        self._check(self.L.rq_reset(self.h, int(session)))

    def logits(self):
        c = self.cfg
        text = np.zeros((c.batch, c.text_card), np.float32)
        audio = np.zeros((c.batch, 8, c.audio_card), np.float32)
        self._check(self.L.rq_get_logits(self.h, _p(text), _p(audio)))
        return text, audio

    def trace(self):
        c = self.cfg
        emb = np.zeros((c.batch, c.dim), np.float32)
        tout = np.zeros((c.batch, c.dim), np.float32)
        self._check(self.L.rq_get_trace(self.h, _p(emb), _p(tout)))
        return emb, tout

    def ring(self):
        ring = np.zeros((self.cfg.batch, 17, 3), np.int32)
        off = np.zeros(self.cfg.batch, np.int32)
        self._check(self.L.rq_get_ring(self.h, _p(ring), _p(off)))
        return ring, off

    def set_kv(self, session: int, k, v):
        """k, v: [layers][n_pos][dim] tensors in the K/V dtype (host or device)."""
        k, v = k.contiguous(), v.contiguous()
        self._check(self.L.rq_set_kv(self.h, int(session), int(k.shape[1]), _p(k), _p(v)))

    def set_wait_limit(self, limit_ns: int, stall_op: int = -1):
        """Test hook (rq_set_wait_limit): device wait limit of the whole-frame kernel and
        an op whose grid barrier is made unreachable (-1: none)."""
        self._check(self.L.rq_set_wait_limit(self.h, int(limit_ns), int(stall_op)))

    def launch_op(self, op: int, layer: int, count: int) -> float:
        b = C.c_double(0)
        self._check(self.L.rq_launch_op(self.h, int(op), int(layer), int(count), C.byref(b)))
        return b.value

    def op_times(self):
        """Per-op microseconds of the last frame (persistent schedule), else None."""
        n = self.L.rq_get_op_times(self.h, None, 0)
        if n <= 0:
            return None
        us = np.zeros(n, np.float32)
        self.L.rq_get_op_times(self.h, _p(us), n)
        return us

    @property
    def schedule(self) -> int:
        """The schedule the handle runs (RQ_SCHEDULE_GRAPH, _PERSISTENT or _TENSOR)."""
        return int(self.L.rq_schedule(self.h))

    @property
    def kernels_per_frame(self) -> int:
        return int(self.L.rq_frame_kernel_count(self.h))


def attention(q, k, v, positions, heads: int, head_dim: int, stream=None):
    """Standalone decode attention through rq_attention (device tensors):
    q [B][H*hd] f32, k/v [B][C][H*hd] f32 or bf16, positions [B] int32 -> [B][H*hd]."""
    L = load()
    B, ctx = int(k.shape[0]), int(k.shape[1])
    out = torch.empty((B, heads * head_dim), dtype=torch.float32, device=q.device)
    nbytes = L.rq_attention_workspace_size(B, heads, head_dim, ctx)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    kvt = RQ_BF16 if k.dtype == torch.bfloat16 else RQ_F32
    rc = L.rq_attention(B, heads, head_dim, ctx, kvt, _p(q), _p(k), _p(v), _p(positions), _p(out),
                        _p(ws), nbytes, C.c_void_p(st.cuda_stream))
    if rc != RQ_OK:
        raise RQError(rc, "rq_attention")
    return out
