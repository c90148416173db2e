"""Parity of the CUDA decode step (through the C ABI) with the CPU oracle.

Bar: tokens, ring contents and offsets bit-exact; logits within 1e-3 * max|logit|
(f32 weights) or 2e-2 * max|logit| (bf16 weights, both sides on the same bf16
values); a token may differ only where the oracle's top-2 margin is within that
tolerance.  bf16 runs are teacher-forced with the oracle's own tokens
(rq_step_forced) so a near-tie cannot fork the two trajectories.
"""
import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding, configs, synth

from parity_util import check_logits_and_tokens, rel_err, tol_of, weights_of  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


SCHEDULES = [binding.RQ_SCHEDULE_GRAPH, binding.RQ_SCHEDULE_PERSISTENT]
SCHED_IDS = ["graph", "persistent"]
def run_free(c, frames, w=None, prefill=None, schedule=binding.RQ_SCHEDULE_AUTO):
    """Both sides run free; every token, the ring and the offset must agree."""
    w = w if w is not None else weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w), schedule=schedule)
    if schedule != binding.RQ_SCHEDULE_AUTO:
        assert dec.schedule == schedule
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    if prefill is not None:
        k, v = prefill
        st.set_kv(k, v)
        dec.set_kv(0, k.cuda(), v.cuda())
    users = synth.user_tokens(c, frames).numpy()
    for t in range(frames):
        r = orc.step(st, users[t], trace=True)
        out, has = dec.step(users[t][None])
        text, audio = dec.logits()
        emb, tout = dec.trace()
        ring, off = dec.ring()
        oring, ooff = st.ring()
        own = np.concatenate([[r["own"][0]], r["own"][1:]])
        # the ring records the step's own tokens at offset % 3: compare it whole
        assert int(off[0]) == ooff, t
        assert np.array_equal(ring[0], oring), (t, ring[0], oring)
        assert bool(has[0]) == r["has_out"], t
        if r["has_out"]:
            assert np.array_equal(out[0], r["out"]), (t, out[0], r["out"])
        np.testing.assert_array_equal(emb[0], r["emb_sum"])  # same adds, same order
        assert rel_err(tout[0], r["tout"]) <= tol_of(c), t
        check_logits_and_tokens(c, own, r, text[0], audio[0], t)
    dec.close()


def run_forced(c, frames, w=None, schedule=binding.RQ_SCHEDULE_AUTO, prefill=None):
    """The GPU is forced with the oracle's own tokens; compare own tokens + logits.
    prefill: (K, V) CPU tensors [layers][n][dim] given to both sides before frame 0."""
    w = w if w is not None else weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w), schedule=schedule)
    if schedule != binding.RQ_SCHEDULE_AUTO:
        assert dec.schedule == schedule
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    if prefill is not None:
        k, v = prefill
        st.set_kv(k, v)
        dec.set_kv(0, k.cuda(), v.cuda())
    users = synth.user_tokens(c, frames).numpy()
    for t in range(frames):
        r = orc.step(st, users[t], trace=True)
        own, out, has = dec.step_forced(users[t][None], r["own"][None])
        text, audio = dec.logits()
        assert bool(has[0]) == r["has_out"], t
        if r["has_out"]:
            assert np.array_equal(out[0], r["out"]), t
        check_logits_and_tokens(c, own[0], r, text[0], audio[0], t)
    ring, off = dec.ring()
    oring, ooff = st.ring()
    assert int(off[0]) == ooff and np.array_equal(ring[0], oring)
    dec.close()


@pytest.mark.parametrize("schedule", SCHEDULES, ids=SCHED_IDS)
def test_tiny_f32_free_run_bit_exact(schedule):
    run_free(configs.TINY, 32, schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES, ids=SCHED_IDS)
def test_tiny_f32_past_context_window(schedule):
    run_free(configs.TINY, 70, schedule=schedule)  # context 64: the window slides


@pytest.mark.parametrize("schedule", SCHEDULES, ids=SCHED_IDS)
def test_tiny_prefilled_start_and_eviction(schedule):
    c = configs.TINY
    g = torch.Generator().manual_seed(3)
    n = 62  # offset % 3 == 2 as in the batch-64 workload; frames 2.. evict
    k = torch.randn(c.layers, n, c.dim, generator=g)
    v = torch.randn(c.layers, n, c.dim, generator=g)
    run_free(c, 8, prefill=(k, v), schedule=schedule)


def test_batch1_window_crosses_to_the_per_op_frame():
    """At batch 1, windows longer than 1350 positions replay the one-kernel-per-op frame
    instead of the persistent kernel: a session pre-filled to 1345 positions crosses the
    switch in the middle of the run, and every frame must still match the oracle."""
    c = configs.TINY.with_(context=1500)
    g = torch.Generator().manual_seed(5)
    n = 1345
    k = torch.randn(c.layers, n, c.dim, generator=g)
    v = torch.randn(c.layers, n, c.dim, generator=g)
    run_free(c, 10, prefill=(k, v), schedule=binding.RQ_SCHEDULE_PERSISTENT)


@pytest.mark.parametrize("schedule", SCHEDULES, ids=SCHED_IDS)
def test_tiny_bf16_forced(schedule):
    run_forced(configs.TINY.with_(name="tiny_bf16", weight_dtype="bf16", kv_dtype="bf16"), 20,
               schedule=schedule)


@pytest.mark.parametrize("schedule", SCHEDULES, ids=SCHED_IDS)
def test_small_bf16_forced_full_run(schedule):
    run_forced(configs.SMALL, configs.SMALL.frames, schedule=schedule)


def test_auto_schedule_choice():
    c = configs.TINY
    w = binding.upload_weights(weights_of(c))
    d1 = binding.Decoder(c, w)
    assert d1.schedule == binding.RQ_SCHEDULE_PERSISTENT
    d3 = binding.Decoder(c.with_(batch=3), w)
    assert d3.schedule == binding.RQ_SCHEDULE_GRAPH
    with pytest.raises(binding.RQError):
        binding.Decoder(c.with_(batch=3), w, schedule=binding.RQ_SCHEDULE_PERSISTENT)
    d1.close()
    d3.close()


def test_batch_sessions_are_independent():
    """Session b of a batch equals an oracle run of that session alone."""
    c = configs.TINY.with_(batch=3)
    w = synth.make_weights(c, seed=0)
    dec = binding.Decoder(c, binding.upload_weights(w))
    orc = oracle.Oracle(c, w)
    sts = [orc.new_state() for _ in range(3)]
    users = synth.batch_user_tokens(c, 10).numpy()
    for t in range(10):
        rs = [orc.step(sts[b], users[t, b], trace=True) for b in range(3)]
        out, has = dec.step(users[t])
        text, audio = dec.logits()
        ring, off = dec.ring()
        for b in range(3):
            oring, ooff = sts[b].ring()
            assert np.array_equal(ring[b], oring) and off[b] == ooff, (t, b)
            if rs[b]["has_out"]:
                assert np.array_equal(out[b], rs[b]["out"]), (t, b)
            check_logits_and_tokens(c, rs[b]["own"], rs[b], text[b], audio[b], (t, b))
    dec.close()


def test_device_step_matches_host_step_bitwise():
    c = configs.TINY
    w = binding.upload_weights(synth.make_weights(c, seed=0))
    users = synth.user_tokens(c, 6)
    a = binding.Decoder(c, w)
    b = binding.Decoder(c, w)
    d_user = users.cuda()
    d_out = torch.zeros(9, dtype=torch.int32, device="cuda")
    d_has = torch.zeros(1, dtype=torch.uint8, device="cuda")
    for t in range(6):
        out, has = a.step(users[t].numpy()[None])
        b.step_device(d_user[t], d_out, d_has)
        b.sync()
        assert bool(d_has.item()) == bool(has[0])
        if has[0]:
            assert np.array_equal(d_out.cpu().numpy(), out[0])
        ta, aa = a.logits()
        tb, ab = b.logits()
        np.testing.assert_array_equal(ta, tb)
        np.testing.assert_array_equal(aa, ab)
    a.close()
    b.close()


def test_reset_one_session_restarts_it():
    c = configs.TINY.with_(batch=2)
    w = synth.make_weights(c, seed=0)
    dec = binding.Decoder(c, binding.upload_weights(w))
    users = synth.batch_user_tokens(c, 8).numpy()
    for t in range(5):
        dec.step(users[t])
    dec.reset(1)
    ring, off = dec.ring()
    assert off[1] == 0 and np.all(ring[1] == -2) and off[0] == 5
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    for t in range(3):
        r = orc.step(st, users[t, 1], trace=True)
        u = users[5 + t].copy()
        u[1] = users[t, 1]
        out, has = dec.step(u)
        text, audio = dec.logits()
        assert bool(has[1]) == r["has_out"]
        if r["has_out"]:
            assert np.array_equal(out[1], r["out"])
        check_logits_and_tokens(c, r["own"], r, text[1], audio[1], t)
    dec.close()


def test_bad_tokens_rejected_before_any_state_change():
    c = configs.TINY
    dec = binding.Decoder(c, binding.upload_weights(synth.make_weights(c, seed=0)))
    dec.step(np.zeros((1, 8), np.int32))
    before = dec.ring()
    for bad in (c.audio_card + 1, -2, 10**6):
        u = np.zeros((1, 8), np.int32)
        u[0, 3] = bad
        with pytest.raises(binding.RQError) as ei:
            dec.step(u)
        assert ei.value.status == binding.RQ_ERR_TOKEN
    f = np.zeros((1, 9), np.int32)
    f[0, 0] = c.text_card  # INITIAL is not a token a frame can generate
    with pytest.raises(binding.RQError):
        dec.step_forced(np.zeros((1, 8), np.int32), f)
    after = dec.ring()
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
    dec.step(np.full((1, 8), -1, np.int32))  # -1 and audio_card are valid codes
    dec.step(np.full((1, 8), c.audio_card, np.int32))
    dec.close()


@pytest.mark.parametrize("schedule", SCHEDULES, ids=SCHED_IDS)
def test_moshi7b_full_size_forced_frames(schedule):
    """The Moshi-7B shape at batch 1 (the benchmark's workload; AUTO runs the
    persistent schedule) against the oracle on the first frames."""
    run_forced(configs.MOSHI7B, 4, schedule=schedule)


@pytest.mark.parametrize("n_pos,frames", [(300, 4), (1345, 8)], ids=["window300", "window1345"])
def test_moshi7b_prefilled_window_forced_frames(n_pos, frames):
    """The Moshi-7B shape at batch 1 (AUTO: the persistent schedule) with the temporal
    window pre-filled by N(0,1) bf16 rows, against the oracle.  At 300 positions the
    whole-frame kernel's head_dim-128 attention runs many splits per head (16-position
    splits) and merges them in order; from 1345 the window crosses 1350 positions at
    frame 5, where the handle switches to its one-kernel-per-op frame."""
    c = configs.MOSHI7B.with_(prefill=n_pos)
    k, v = synth.kv_prefill(c, 0)
    run_forced(c, frames, prefill=(k, v))
