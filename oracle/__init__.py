"""CPU oracle of the per-frame RQ-Transformer decode step -- TEST INFRASTRUCTURE.

`rq_oracle.c` is a plain scalar f32 restatement of the definitions on
"inferencelayer 0.2.4 -- src/moshi_lm.rs"; this module is its ctypes wrapper.
Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference arm
may import it.  It imports nothing from the CUDA package and the CUDA package
imports nothing from it.

Pinned by tests/test_oracle_pins.py and tests/test_oracle_second_opinion.py.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_LIB = None

WEIGHT_FIELDS = [
    "emb", "text_emb", "norm1", "in_proj", "out_proj", "norm2", "gate_in",
    "gate_out", "out_norm", "text_linear", "dep_in", "dep_text_emb", "dep_emb",
    "dnorm1", "dnorm2", "d_in_proj", "d_out_proj", "d_gate_in", "d_gate_out",
    "linears",
]


class OrcCfg(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "dim", "layers", "heads", "head_dim", "hidden", "context", "text_card",
        "audio_card", "ddim", "dlayers", "dheads", "dhead_dim", "dhidden", "w_bf16",
        "kv_bf16")] + [("eps", C.c_float), ("rope_theta", C.c_float)]


class OrcWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS]


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = C.CDLL(path)
        P, I32, I64, F = C.c_void_p, C.c_int32, C.c_int64, C.c_float
        L.orc_gemv.argtypes = [P, I32, I32, I32, P, P]
        L.orc_rms_norm.argtypes = [P, P, I32, F, P]
        L.orc_silu.argtypes = [F]
        L.orc_silu.restype = F
        L.orc_argmax.argtypes = [P, I32]
        L.orc_argmax.restype = C.c_uint32
        L.orc_rope_row.argtypes = [P, I32, I64, I32, F]
        L.orc_attend.argtypes = [P, P, P, I32, I32, I32, P]
        L.orc_embed.argtypes = [P, I32, I32, I64, P]
        L.orc_state_new.argtypes = [C.POINTER(OrcCfg)]
        L.orc_state_new.restype = P
        L.orc_state_free.argtypes = [P]
        L.orc_state_set_kv.argtypes = [P, I32, P, P, I32]
        L.orc_state_set_kv.restype = C.c_int
        L.orc_state_get_ring.argtypes = [P, P, P]
        L.orc_temporal_step.argtypes = [C.POINTER(OrcCfg), C.POINTER(OrcWeights), P, P, P]
        L.orc_depformer_cycle.argtypes = [C.POINTER(OrcCfg), C.POINTER(OrcWeights), P,
                                          I64, P, P, P]
        L.orc_step.argtypes = [C.POINTER(OrcCfg), C.POINTER(OrcWeights), P, P, P, P, P,
                               P, P, P, P, P, P]
        L.orc_set_threads.argtypes = [I32]
        L.orc_max_threads.restype = I32
        L.orc_round_to_bf16.argtypes = [F]
        L.orc_round_to_bf16.restype = F
        U64 = C.c_uint64
        L.orc_xorshift_next.argtypes = [C.POINTER(U64)]
        L.orc_xorshift_next.restype = U64
        L.orc_xorshift_u01.argtypes = [C.POINTER(U64)]
        L.orc_xorshift_u01.restype = C.c_double
        L.orc_gumbel_pick.argtypes = [P, I32, F, C.POINTER(U64)]
        L.orc_gumbel_pick.restype = C.c_uint32
        L.orc_topk_pick.argtypes = [P, I32, F, I32, C.POINTER(U64)]
        L.orc_topk_pick.restype = C.c_uint32
        L.orc_state_set_sampling.argtypes = [P, I32, F, F, I32, I32, U64]
        L.orc_state_get_rng.argtypes = [P]
        L.orc_state_get_rng.restype = U64
        L.orc_qn_roundtrip.argtypes = [P, I32, I32, I32, I32]
        L.orc_prime_step.argtypes = [C.POINTER(OrcCfg), C.POINTER(OrcWeights), P, P, P, P]
        L.orc_replay_step.argtypes = [C.POINTER(OrcCfg), C.POINTER(OrcWeights), P, P]
        L.orc_state_clone.argtypes = [P]
        L.orc_state_clone.restype = P
        _LIB = L
    return _LIB


def _ptr(a):
    if a is None:
        return None
    if hasattr(a, "data_ptr"):  # torch tensor (bf16 tensors pass their bit patterns)
        assert a.is_contiguous() and a.device.type == "cpu"
        return a.data_ptr()
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


# ------------------------------------------------------------------ primitives

def gemv(w, x):
    """out = W x for a 2-D weight (numpy f32, or torch f32/bf16 CPU tensor)."""
    bf16 = int(hasattr(w, "dtype") and str(w.dtype) == "torch.bfloat16")
    rows, k = int(w.shape[0]), int(w.shape[1])
    x = _f32(x)
    out = np.empty(rows, np.float32)
    lib().orc_gemv(_ptr(w if hasattr(w, "data_ptr") else _f32(w)), bf16, rows, k,
                   _ptr(x), _ptr(out))
    return out


def rms_norm(x, alpha, eps=1e-8):
    x, alpha = _f32(x), _f32(alpha)
    out = np.empty_like(x)
    lib().orc_rms_norm(_ptr(x), _ptr(alpha), x.size, C.c_float(eps), _ptr(out))
    return out


def silu(x: float) -> float:
    return float(lib().orc_silu(C.c_float(x)))


def argmax(v) -> int:
    v = _f32(v)
    return int(lib().orc_argmax(_ptr(v), v.size))


def rope_row(row, pos: int, head_dim: int, theta: float = 10000.0):
    r = _f32(row).copy()
    lib().orc_rope_row(_ptr(r), r.size, int(pos), int(head_dim), C.c_float(theta))
    return r


def attend(q, ks, vs, heads: int, head_dim: int):
    q, ks, vs = _f32(q), _f32(ks), _f32(vs)
    out = np.empty(heads * head_dim, np.float32)
    lib().orc_attend(_ptr(q), _ptr(ks), _ptr(vs), int(ks.shape[0]), heads, head_dim,
                     _ptr(out))
    return out


def embed(table, tok: int, acc):
    acc = _f32(acc).copy()
    bf16 = int(hasattr(table, "dtype") and str(table.dtype) == "torch.bfloat16")
    t = table if hasattr(table, "data_ptr") else _f32(table)
    lib().orc_embed(_ptr(t), bf16, int(table.shape[1]), int(tok), _ptr(acc))
    return acc


def round_to_bf16(x: float) -> float:
    return float(lib().orc_round_to_bf16(C.c_float(x)))


def qn_roundtrip(v, bits: int, group: int = 32):
    """`qn_roundtrip`: a [rows][cols] f32 copy quantized to `bits` per value with one
    scale per `group` values of a row, and dequantized."""
    a = _f32(v).copy()
    rows, cols = a.shape
    lib().orc_qn_roundtrip(_ptr(a), rows, cols, int(bits), int(group))
    return a


# sampling ("moshi_lm.rs", `Sampling` / `pick`): modes of a session's sampler
PICK_GREEDY, PICK_TOPK, PICK_GUMBEL = 0, 1, 2


class XorShift:
    """The page's xorshift64 sampler state (`xorshift_u01`)."""

    def __init__(self, state: int):
        self.s = C.c_uint64(state)

    def next(self) -> int:
        return int(lib().orc_xorshift_next(C.byref(self.s)))

    def u01(self) -> float:
        return float(lib().orc_xorshift_u01(C.byref(self.s)))

    @property
    def state(self) -> int:
        return int(self.s.value)


def gumbel_pick(logits, temp: float, rng: XorShift) -> int:
    v = _f32(logits)
    return int(lib().orc_gumbel_pick(_ptr(v), v.size, C.c_float(temp), C.byref(rng.s)))


def topk_pick(logits, temp: float, k: int, rng: XorShift) -> int:
    v = _f32(logits)
    return int(lib().orc_topk_pick(_ptr(v), v.size, C.c_float(temp), int(k), C.byref(rng.s)))


# ------------------------------------------------------------------ model

class Oracle:
    """One model (config + host weights); sessions are `new_state()` handles."""

    def __init__(self, cfg, weights: dict):
        self.cfg = cfg
        self.weights = weights  # keep the host tensors alive
        self.c = OrcCfg(
            dim=cfg.dim, layers=cfg.layers, heads=cfg.heads, head_dim=cfg.head_dim,
            hidden=cfg.hidden, context=cfg.context, text_card=cfg.text_card,
            audio_card=cfg.audio_card, ddim=cfg.ddim, dlayers=cfg.dlayers,
            dheads=cfg.dheads, dhead_dim=cfg.dhead_dim, dhidden=cfg.dhidden,
            w_bf16=int(cfg.weight_dtype == "bf16"), kv_bf16=int(cfg.kv_dtype == "bf16"),
            eps=cfg.eps, rope_theta=cfg.rope_theta)
        self.w = OrcWeights(**{n: _ptr(weights[n]) for n in WEIGHT_FIELDS})

    def new_state(self) -> "OracleState":
        p = lib().orc_state_new(C.byref(self.c))
        if not p:
            raise MemoryError("oracle state allocation failed")
        return OracleState(p, self)

    def step(self, st: "OracleState", user, forced=None, trace: bool = False) -> dict:
        c = self.cfg
        user = np.ascontiguousarray(user, dtype=np.int32)
        assert user.shape == (8,)
        f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        own = np.zeros(9, np.int32)
        out = np.zeros(9, np.int32)
        has = np.zeros(1, np.int32)
        r = {"own": own, "out": out}
        if trace:
            r["input_tokens"] = np.zeros(17, np.int64)
            r["emb_sum"] = np.zeros(c.dim, np.float32)
            r["tout"] = np.zeros(c.dim, np.float32)
            r["text_logits"] = np.zeros(c.text_card, np.float32)
            r["audio_logits"] = np.zeros((8, c.audio_card), np.float32)
        g = lambda k: _ptr(r[k]) if k in r else None  # noqa: E731
        lib().orc_step(C.byref(self.c), C.byref(self.w), st.p, _ptr(user),
                       None if f is None else _ptr(f), _ptr(own), _ptr(out), _ptr(has),
                       g("input_tokens"), g("emb_sum"), g("tout"), g("text_logits"),
                       g("audio_logits"))
        r["has_out"] = bool(has[0])
        return r

    def prime_step(self, st: "OracleState", forced, user):
        """`step_forced`: temporal only, the ring records `forced` [9]; returns the
        embedding sum the temporal stack consumed."""
        f = np.ascontiguousarray(forced, dtype=np.int32)
        u = np.ascontiguousarray(user, dtype=np.int32)
        assert f.shape == (9,) and u.shape == (8,)
        e = np.zeros(self.cfg.dim, np.float32)
        lib().orc_prime_step(C.byref(self.c), C.byref(self.w), st.p, _ptr(f), _ptr(u), _ptr(e))
        return e

    def replay_step(self, st: "OracleState", x) -> None:
        """`advance_clock` after the temporal consumed the embedding row x [D]."""
        x = _f32(x)
        assert x.shape == (self.cfg.dim,)
        lib().orc_replay_step(C.byref(self.c), C.byref(self.w), st.p, _ptr(x))

    def temporal_step(self, st: "OracleState", x):
        x = _f32(x).copy()
        tout = np.zeros(self.cfg.dim, np.float32)
        lib().orc_temporal_step(C.byref(self.c), C.byref(self.w), st.p, _ptr(x), _ptr(tout))
        return tout

    def depformer_cycle(self, tout, text_token: int, forced=None):
        c = self.cfg
        tout = _f32(tout)
        f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        logits = np.zeros((8, c.audio_card), np.float32)
        toks = np.zeros(8, np.int32)
        lib().orc_depformer_cycle(C.byref(self.c), C.byref(self.w), _ptr(tout),
                                  int(text_token), None if f is None else _ptr(f),
                                  _ptr(logits), _ptr(toks))
        return logits, toks


class OracleState:
    def __init__(self, p, model: Oracle):
        self.p = p
        self._keep = None
        self.model = model

    def __del__(self):
        if getattr(self, "p", None):
            lib().orc_state_free(self.p)
            self.p = None

    def set_kv(self, k, v) -> None:
        """k, v: [layers][n_pos][dim] CPU tensors (bf16 or f32); offset becomes n_pos."""
        bits16 = int(str(k.dtype) == "torch.bfloat16")
        k, v = k.contiguous(), v.contiguous()
        rc = lib().orc_state_set_kv(self.p, int(k.shape[1]), _ptr(k), _ptr(v), bits16)
        if rc != 0:
            raise ValueError("n_pos exceeds the context")

    def set_sampling(self, mode: int, temp: float = 0.8, temp_text: float = 0.7,
                     top_k: int = 250, top_k_text: int = 25, seed: int = 1) -> None:
        """`MoshiLm::set_sampling` for this session (defaults: the page's `Sampling`)."""
        lib().orc_state_set_sampling(self.p, int(mode), C.c_float(temp), C.c_float(temp_text),
                                     int(top_k), int(top_k_text), C.c_uint64(seed))

    def clone(self) -> "OracleState":
        """`MoshiState::snapshot`: an independent copy."""
        p = lib().orc_state_clone(self.p)
        if not p:
            raise MemoryError("oracle state copy failed")
        return OracleState(p, self.model)

    @property
    def rng(self) -> int:
        return int(lib().orc_state_get_rng(self.p))

    def ring(self):
        ring = np.zeros((17, 3), np.int64)
        off = np.zeros(1, np.int64)
        lib().orc_state_get_ring(self.p, _ptr(ring), _ptr(off))
        return ring, int(off[0])
