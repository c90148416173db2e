"""Model shapes and workloads of the per-frame RQ-Transformer decode step.

The five workloads: a tiny f32 model, a small bf16 model, and the Moshi-7B shape at
batch 1, 16 and 64 (the last with every session's temporal K/V pre-filled to 2900
positions).  Dimensions follow "inferencelayer 0.2.4 -- src/moshi_lm.rs" (consts
DIM .. DHIDDEN, RMS_EPS, CARD, TEXT_CARD); streams, delays and the 3-slot ring are
fixed by that page's module doc and are not configurable.
"""
from dataclasses import dataclass, replace

N_STREAMS = 17
N_Q = 8


@dataclass(frozen=True)
class RQConfig:
    name: str
    dim: int
    layers: int
    heads: int
    head_dim: int
    hidden: int
    context: int
    text_card: int
    audio_card: int
    ddim: int
    dlayers: int
    dheads: int
    dhead_dim: int
    dhidden: int
    weight_dtype: str        # "f32", "bf16", or a weight band "q8" / "q4" (bf16 tables)
    kv_dtype: str            # "f32" or "bf16"
    batch: int = 1
    frames: int = 32
    eps: float = 1e-8
    rope_theta: float = 10000.0
    prefill: int = 0         # temporal K/V positions pre-filled per session
    user_card: int = 0       # user codes are drawn uniform in [0, user_card)
    user_minus1: float = 0.0  # probability that a user code is replaced by -1
    user_seed: int = 1       # seed of session 0 (session b uses user_seed + b)

    def with_(self, **kw) -> "RQConfig":
        return replace(self, **kw)

    @property
    def weight_bytes(self) -> int:
        return 2 if self.weight_dtype == "bf16" else 4

    @property
    def kv_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 4


TINY = RQConfig(
    name="tiny", dim=256, layers=2, heads=4, head_dim=64, hidden=704, context=64,
    text_card=128, audio_card=64, ddim=128, dlayers=2, dheads=4, dhead_dim=32,
    dhidden=352, weight_dtype="f32", kv_dtype="f32", batch=1, frames=32,
    user_card=64, user_seed=1)

SMALL = RQConfig(
    name="small", dim=1024, layers=8, heads=16, head_dim=64, hidden=2816, context=512,
    text_card=8000, audio_card=2048, ddim=512, dlayers=2, dheads=8, dhead_dim=64,
    dhidden=1408, weight_dtype="bf16", kv_dtype="bf16", batch=1, frames=250,
    user_card=2048, user_minus1=0.05, user_seed=1)

MOSHI7B = RQConfig(
    name="moshi7b", dim=4096, layers=32, heads=32, head_dim=128, hidden=11264,
    context=3000, text_card=32000, audio_card=2048, ddim=1024, dlayers=6, dheads=16,
    dhead_dim=64, dhidden=2816, weight_dtype="bf16", kv_dtype="bf16", batch=1,
    frames=375, user_card=2048, user_seed=1)

MOSHI7B_B16 = MOSHI7B.with_(name="moshi7b_b16", batch=16, frames=375, user_seed=1000)

MOSHI7B_B64 = MOSHI7B.with_(name="moshi7b_b64", batch=64, frames=100, prefill=2900,
                            user_seed=2000)

CONFIGS = {c.name: c for c in (TINY, SMALL, MOSHI7B, MOSHI7B_B16, MOSHI7B_B64)}

# Moshi-7B layer shapes with only 2 temporal layers: every kernel of the full model at
# its real size, in ~3 GB of device memory (used for profiler captures).
MOSHI7B_2L = MOSHI7B.with_(name="moshi7b_2layer", layers=2, frames=16)
CONFIGS[MOSHI7B_2L.name] = MOSHI7B_2L
