"""Token picks on the GPU ("moshi_lm.rs", `Sampling`, `pick`, `topk_sample`,
`gumbel_full_pick`, `xorshift_u01`) against the oracle's picks, in every schedule.

Each frame runs free on the GPU.  Its own tokens (the ring slot it just wrote) must be
exactly what the oracle's pick returns on the GPU's own logits from the same sampler
state; the GPU's sampler states must equal the oracle generator's after every frame.
The oracle, forced with the GPU's tokens, must reproduce the logits within the parity
tolerance, the ring and the outputs.  So the draw positions, the Gumbel scores and the
top-k selection are checked exactly, and the model arithmetic to the usual bar.
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


MODES = [binding.RQ_PICK_TOPK, binding.RQ_PICK_GUMBEL]
MODE_IDS = ["topk", "gumbel"]


def oracle_pick(mode, logits, temp, k, rng):
    if mode == binding.RQ_PICK_TOPK:
        return oracle.topk_pick(logits, temp, k, rng)
    return oracle.gumbel_pick(logits, temp, rng)


def run_sampled(c, schedule, mode, frames, check_sessions, temp=0.9, temp_text=0.6,
                top_k=5, top_k_text=3):
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w), schedule=schedule)
    assert dec.schedule == schedule
    B = c.batch
    seeds = np.array([0] + [0x9E3779B97F4A7C15 * (b + 1) % 2 ** 64 for b in range(1, B)],
                     np.uint64)  # session 0's seed 0 starts at state 1
    dec.set_sampling(mode, temp=temp, temp_text=temp_text, top_k=top_k,
                     top_k_text=top_k_text, seeds=seeds)
    rngs = [oracle.XorShift(max(int(s), 1)) for s in seeds]
    assert [int(x) for x in dec.rng()] == [r.state for r in rngs]
    orc = oracle.Oracle(c, w)
    sts = {b: orc.new_state() for b in check_sessions}
    users = synth.batch_user_tokens(c, frames).numpy()
    tol = tol_of(c)
    for t in range(frames):
        out, has = dec.step(users[t])
        text, audio = dec.logits()
        ring, off = dec.ring()
        for b in range(B):
            own = [int(ring[b, s, off[b] % 3]) for s in range(9)]
            want = [oracle_pick(mode, text[b], temp_text, top_k_text, rngs[b])]
            want += [oracle_pick(mode, audio[b, cb], temp, top_k, rngs[b]) for cb in range(8)]
            assert own == want, (t, b, own, want)
        assert [int(x) for x in dec.rng()] == [r.state for r in rngs], t
        for b in check_sessions:
            own = np.array([ring[b, s, off[b] % 3] for s in range(9)], np.int32)
            r = orc.step(sts[b], users[t, b], forced=own, trace=True)
            oring, ooff = sts[b].ring()
            assert np.array_equal(ring[b], oring) and off[b] == ooff, (t, b)
            assert bool(has[b]) == r["has_out"]
            if r["has_out"]:
                assert np.array_equal(out[b], r["out"]), (t, b)
            assert rel_err(text[b], r["text_logits"]) <= tol, (t, b)
            for cb in range(8):
                assert rel_err(audio[b, cb], r["audio_logits"][cb]) <= tol, (t, b, cb)
    dec.close()


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_sampling_graph_tiny_batch3(mode):
    c = configs.TINY.with_(batch=3)
    run_sampled(c, binding.RQ_SCHEDULE_GRAPH, mode, 8, [0, 2])


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_sampling_persistent_tiny(mode):
    run_sampled(configs.TINY, binding.RQ_SCHEDULE_PERSISTENT, mode, 8, [0])


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_sampling_persistent_small_page_defaults(mode):
    # the page's `Sampling` defaults over an 8000-token text vocabulary
    run_sampled(configs.SMALL, binding.RQ_SCHEDULE_PERSISTENT, mode, 4, [0],
                temp=0.8, temp_text=0.7, top_k=250, top_k_text=25)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_sampling_tensor_small_batch16(mode):
    c = configs.SMALL.with_(batch=16)
    run_sampled(c, binding.RQ_SCHEDULE_TENSOR, mode, 3, [0, 15],
                temp=0.8, temp_text=0.7, top_k=250, top_k_text=25)


def test_sampling_arguments_and_back_to_greedy():
    c = configs.TINY
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    one = np.array([5], np.uint64)
    for bad in (dict(mode=7, seeds=one), dict(mode=binding.RQ_PICK_TOPK, top_k=0, seeds=one),
                dict(mode=binding.RQ_PICK_TOPK, top_k=257, seeds=one),
                dict(mode=binding.RQ_PICK_GUMBEL, temp=0.0, seeds=one),
                dict(mode=binding.RQ_PICK_GUMBEL, seeds=None)):
        with pytest.raises(binding.RQError):
            dec.set_sampling(**bad)
    users = synth.user_tokens(c, 4).numpy()
    dec.set_sampling(binding.RQ_PICK_GUMBEL, seeds=one)
    dec.step(users[0][None])
    moved = int(dec.rng()[0])
    assert moved != 5
    # greedy again: states kept, tokens are the first-wins argmax of the frame's logits
    dec.set_sampling(binding.RQ_PICK_GREEDY)
    for t in range(1, 4):
        dec.step(users[t][None])
        text, audio = dec.logits()
        ring, off = dec.ring()
        own = [int(ring[0, s, off[0] % 3]) for s in range(9)]
        assert own[0] == oracle.argmax(text[0])
        assert own[1:] == [oracle.argmax(audio[0, cb]) for cb in range(8)]
    assert int(dec.rng()[0]) == moved
    dec.close()
