"""Whole-frame pin: the f32 oracle against the independent float64 restatement in
tests/ref_f64.py, over many frames, on the tiny model (f32 and a bf16 variant, runs
past the 64-position context so the window evicts) and on the small model.

The oracle runs free; the f64 restatement is forced with the oracle's own tokens,
so both follow one trajectory and every frame's logits are comparable.
"""
import numpy as np
import pytest

import oracle
from ref_f64 import Ref64
from rq_transformer_frame_gb300 import configs, synth


def _margin(v):
    s = np.sort(v)
    return s[-1] - s[-2]


def _run(c, frames, tol):
    w = synth.make_weights(c, seed=0)
    o = oracle.Oracle(c, w)
    ref = Ref64(c, w)
    so, sr = o.new_state(), ref.new_state()
    users = synth.user_tokens(c, frames).numpy()
    worst = 0.0
    for t in range(frames):
        a = o.step(so, users[t], trace=True)
        b = ref.step(sr, users[t], forced=a["own"])
        assert list(a["input_tokens"]) == list(b["input_tokens"]), t
        np.testing.assert_allclose(a["emb_sum"], b["emb_sum"], rtol=1e-6, atol=1e-7)
        for key in ("text_logits", "audio_logits", "tout"):
            scale = np.max(np.abs(b[key]))
            err = np.max(np.abs(a[key] - b[key])) / scale
            worst = max(worst, err)
            assert err <= tol, (t, key, err)
        # own tokens must agree wherever the f64 top-2 margin exceeds the tolerance
        if _margin(b["text_logits"]) > tol * np.max(np.abs(b["text_logits"])):
            assert a["own"][0] == ref.first_argmax(b["text_logits"]), t
        for cb in range(8):
            lg = b["audio_logits"][cb]
            if _margin(lg) > tol * np.max(np.abs(lg)):
                assert a["own"][1 + cb] == ref.first_argmax(lg), (t, cb)
        assert a["has_out"] == (b["out"] is not None)
        if a["has_out"]:
            assert list(a["out"]) == list(b["out"])
    return worst


def test_tiny_f32_frames_past_context():
    c = configs.TINY
    worst = _run(c, 70, 1e-4)  # context 64: frames 64..69 evict the oldest rows
    assert worst < 1e-4


def test_tiny_bf16_variant():
    c = configs.TINY.with_(name="tiny_bf16", weight_dtype="bf16", kv_dtype="bf16")
    _run(c, 12, 2e-3)  # bf16 K/V rounding of f32 vs f64 rows may differ by one ulp


@pytest.mark.slow
def test_small_bf16_frames():
    c = configs.SMALL
    _run(c, 4, 2e-3)
