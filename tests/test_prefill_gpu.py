"""Prompt priming, embedding replay and session snapshots on the GPU ("moshi_lm.rs",
`MoshiLm::step_forced`, `MoshiState::advance_clock`, `MoshiState::snapshot`) against
the oracle.

Priming and replay run the temporal stack only, up to 64 positions at a time as the
columns of the tensor-core layers; their effect is the K/V window and the ring, which
the frames that follow read.  So each test primes (or replays), compares the ring and
offset bit-exactly, then runs normal frames forced with the oracle's own tokens and
compares every logit with the oracle's under the usual tolerance.  Snapshots are copies:
a restored session must continue bit-identically.
"""
import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding, configs, synth

from parity_util import rel_err, tol_of, weights_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def prompt(c, n, seed=5):
    g = torch.Generator().manual_seed(seed)
    forced = np.zeros((n, 9), np.int32)
    forced[:, 0] = torch.randint(0, c.text_card, (n,), generator=g).numpy()
    forced[:, 1:] = torch.randint(0, c.audio_card, (n, 8), generator=g).numpy()
    user = torch.randint(-1, c.audio_card + 1, (n, 8), generator=g).numpy().astype(np.int32)
    return forced, user


def follow_frames(c, dec, orc, st, frames, session=0):
    """Normal frames after the prompt, both sides forced with the oracle's tokens."""
    tol = tol_of(c)
    users = synth.user_tokens(c, frames, session=9).numpy()
    for t in range(frames):
        r = orc.step(st, users[t], trace=True)
        u = np.tile(users[t], (c.batch, 1))
        f = np.tile(r["own"], (c.batch, 1))
        own, out, has = dec.step_forced(u, f)
        text, audio = dec.logits()
        assert rel_err(text[session], r["text_logits"]) <= tol, t
        for cb in range(8):
            assert rel_err(audio[session, cb], r["audio_logits"][cb]) <= tol, (t, cb)
        ring, off = dec.ring()
        oring, ooff = st.ring()
        assert np.array_equal(ring[session], oring) and off[session] == ooff, t


@pytest.mark.parametrize("schedule", [binding.RQ_SCHEDULE_PERSISTENT, binding.RQ_SCHEDULE_GRAPH],
                         ids=["persistent", "graph"])
def test_prime_then_frames_match_oracle(schedule):
    c = configs.SMALL
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w), schedule=schedule)
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    forced, user = prompt(c, 70)  # two chunks: 64 + 6
    for t in range(70):
        orc.prime_step(st, forced[t], user[t])
    dec.prime(0, forced, user)
    ring, off = dec.ring()
    oring, ooff = st.ring()
    assert off[0] == ooff == 70 and np.array_equal(ring[0], oring)
    follow_frames(c, dec, orc, st, 4)
    dec.close()


def test_prime_across_the_window_edge():
    # context 80: a chunk may not wrap the window, so 50, then 30 up to the edge, then
    # single positions past it
    c = configs.SMALL.with_(context=80)
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    forced, user = prompt(c, 100, seed=6)
    for t in range(100):
        orc.prime_step(st, forced[t], user[t])
    dec.prime(0, forced[:50], user[:50])   # chunk of 50
    dec.prime(0, forced[50:], user[50:])   # 30 to the edge, then singles past it
    ring, off = dec.ring()
    oring, ooff = st.ring()
    assert off[0] == ooff == 100 and np.array_equal(ring[0], oring)
    follow_frames(c, dec, orc, st, 3)
    dec.close()


def test_replay_then_frames_match_oracle():
    c = configs.SMALL
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(40, c.dim, generator=g) * 0.05).numpy().astype(np.float32)
    for t in range(40):
        orc.replay_step(st, x[t])
    ring0 = dec.ring()[0][0].copy()
    dec.replay(0, torch.from_numpy(x).cuda())  # device rows
    ring, off = dec.ring()
    assert off[0] == 40 and np.array_equal(ring[0], ring0)  # the ring is not touched
    follow_frames(c, dec, orc, st, 3)
    dec.close()


def test_prime_in_a_batch_touches_only_its_session():
    c = configs.SMALL.with_(batch=16)
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    assert dec.schedule == binding.RQ_SCHEDULE_TENSOR
    forced, user = prompt(c, 20, seed=7)
    before = dec.ring()
    dec.prime(5, forced, user)
    ring, off = dec.ring()
    assert off[5] == 20 and all(off[b] == 0 for b in range(16) if b != 5)
    for b in range(16):
        if b != 5:
            assert np.array_equal(ring[b], before[0][b])
    dec.close()


def test_snapshot_restore_continues_bit_identically():
    c = configs.TINY.with_(batch=2)
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    users = synth.batch_user_tokens(c, 12).numpy()
    for t in range(5):
        dec.step(users[t])
    snap = dec.snapshot(0)
    assert snap.size == dec.L.rq_snapshot_size(dec.h, 0)
    rec = []
    for t in range(5, 9):
        dec.step(users[t])
        text, audio = dec.logits()
        rec.append((text[0].copy(), audio[0].copy(), dec.ring()[0][0].copy()))
    dec.restore(1, snap)  # session 1 takes session 0's state at frame 5
    for t in range(5, 9):
        u = users[t].copy()
        u[1] = users[t, 0]
        dec.step(u)
        text, audio = dec.logits()
        np.testing.assert_array_equal(text[1], rec[t - 5][0])
        np.testing.assert_array_equal(audio[1], rec[t - 5][1])
        assert np.array_equal(dec.ring()[0][1], rec[t - 5][2])
    bad = snap.copy()
    bad[:8] = 0
    with pytest.raises(binding.RQError):
        dec.restore(0, bad)
    dec.close()


def test_prime_rejects_bad_input_and_unsupported_models():
    c = configs.SMALL
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    forced, user = prompt(c, 4)
    bad = forced.copy()
    bad[2, 0] = c.text_card  # INITIAL is not a token a frame can generate
    with pytest.raises(binding.RQError) as ei:
        dec.prime(0, bad, user)
    assert ei.value.status == binding.RQ_ERR_TOKEN
    assert dec.ring()[1][0] == 0
    dec.close()
    t = configs.TINY  # f32 weights: the tensor-core prefill does not apply
    d2 = binding.Decoder(t, binding.upload_weights(weights_of(t)))
    f2, u2 = prompt(t, 3)
    with pytest.raises(binding.RQError) as ei:
        d2.prime(0, f2, u2)
    assert ei.value.status == binding.RQ_ERR_UNSUPPORTED
    d2.close()
