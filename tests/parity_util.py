"""Shared helpers of the GPU parity tests: the tolerance model and the comparison of
one frame's logits and tokens with the oracle's."""
import numpy as np

from rq_transformer_frame_gb300 import synth


def tol_of(c):
    return 1e-3 if c.weight_dtype == "f32" else 2e-2


def rel_err(got, want):
    return float(np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-30))


def margin(v):
    s = np.sort(v)
    return s[-1] - s[-2]


def check_logits_and_tokens(c, own_gpu, r, text, audio, where):
    tol = tol_of(c)
    assert rel_err(text, r["text_logits"]) <= tol, (where, rel_err(text, r["text_logits"]))
    for cb in range(8):
        e = rel_err(audio[cb], r["audio_logits"][cb])
        assert e <= tol, (where, cb, e)
    tl = r["text_logits"]
    if margin(tl) > tol * np.max(np.abs(tl)):
        assert own_gpu[0] == r["own"][0], (where, "text")
    for cb in range(8):
        lg = r["audio_logits"][cb]
        if margin(lg) > tol * np.max(np.abs(lg)):
            assert own_gpu[1 + cb] == r["own"][1 + cb], (where, cb)


_WEIGHTS = {}


def weights_of(c):
    """Seeded weights of c's shapes (batch, frames and name do not change them)."""
    key = (c.dim, c.layers, c.heads, c.head_dim, c.hidden, c.text_card, c.audio_card,
           c.ddim, c.dlayers, c.dheads, c.dhead_dim, c.dhidden, c.weight_dtype)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        _WEIGHTS[key] = synth.make_weights(c, seed=0)
    return _WEIGHTS[key]


