"""Whole-frame pin: the f32 oracle against the independent float64 restatement in
tests/ref_f64.py, over many frames, on the tiny model (f32 and a bf16 variant, runs
past the 64-position context so the window evicts) and on the small model, and the
oracle's pre-filled start (`set_kv`, the batch-64 workload's reading of
`MoshiState::advance_clock`) against the restatement's own pre-filled state.

The oracle runs free; the f64 restatement is forced with the oracle's own tokens,
so both follow one trajectory and every frame's logits are comparable.
"""
import numpy as np
import pytest
import torch

import oracle
from ref_f64 import Ref64
from rq_transformer_frame_gb300 import configs, synth


def _margin(v):
    s = np.sort(v)
    return s[-1] - s[-2]


def _run(c, frames, tol, prefill=None):
    w = synth.make_weights(c, seed=0)
    o = oracle.Oracle(c, w)
    ref = Ref64(c, w)
    so = o.new_state()
    if prefill is None:
        sr = ref.new_state()
    else:
        k, v = prefill
        so.set_kv(k, v)
        sr = ref.prefilled_state(k.float().numpy(), v.float().numpy())
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
        ring, off = so.ring()
        assert off == sr["off"] and np.array_equal(ring, sr["ring"]), t
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


def _prefill(c, n, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(c.layers, n, c.dim, generator=g).to(dtype)
    v = torch.randn(c.layers, n, c.dim, generator=g).to(dtype)
    return k, v


def test_tiny_prefilled_start_past_context():
    """The batch-64 workload's start (offset n, ring all UNGENERATED, K/V rows 0..n-1 of
    every layer given): the oracle's `set_kv` against the f64 restatement's own
    pre-filled state.  n = 62 is 2 mod 3 like 2900, frames 0-1 read -2 from the ring
    (row 0), and from frame 2 on the 64-position window evicts the pre-filled rows
    one by one; each layer's rows differ, so a wrong layer stride or slot order shows."""
    c = configs.TINY
    worst = _run(c, 10, 1e-4, prefill=_prefill(c, 62, 3))
    assert worst < 1e-4


def test_tiny_bf16_prefilled_start():
    """The same start with bf16 K/V rows (the workload's storage)."""
    c = configs.TINY.with_(name="tiny_bf16", weight_dtype="bf16", kv_dtype="bf16")
    _run(c, 8, 2e-3, prefill=_prefill(c, 62, 4, torch.bfloat16))


def test_prefilled_rows_reach_attention():
    """A pre-filled start differs from a fresh one, and from the same rows given to the
    wrong layer, already in frame 0 (so neither the rows nor their layer are ignored)."""
    c = configs.TINY
    w = synth.make_weights(c, seed=0)
    o = oracle.Oracle(c, w)
    k, v = _prefill(c, 20, 5)
    user = synth.user_tokens(c, 1).numpy()[0]
    outs = []
    for kk, vv in ((k, v), (k.flip(0), v.flip(0))):
        st = o.new_state()
        st.set_kv(kk, vv)
        outs.append(o.step(st, user, trace=True)["text_logits"])
    st = o.new_state()
    fresh = o.step(st, user, trace=True)["text_logits"]
    assert np.max(np.abs(outs[0] - outs[1])) > 1e-3
    assert np.max(np.abs(outs[0] - fresh)) > 1e-3
