"""Parity of the batched tensor-core schedule (RQ_SCHEDULE_TENSOR: every linear one
tcgen05 GEMM over all sessions, bf16 operands) with the CPU oracle, session by session.

The GEMM operands are two-part bf16 expansions hi + lo of the f32 activations (16
significant bits, a relative representation error of at most 2^-17), so the plain
f32 oracle is the reference.  Same bar as the other parity tests: ring,
offsets and delayed outputs bit-exact; logits within 2e-2 * max|logit| (bf16 weights);
a token may differ only where the oracle's top-2 margin is inside that tolerance.  Teacher-forced runs force every session with a
seeded synthetic token stream on both sides, so a near-tie cannot fork a trajectory;
the free run forces the oracle with the GPU's own tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding, configs, synth

from parity_util import check_logits_and_tokens, rel_err, weights_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def forced_tokens(c, frames, seed=77):
    """int32 [frames][B][9]: text in [0, V), audio in [0, A), one generator per session."""
    out = np.zeros((frames, c.batch, 9), np.int32)
    for b in range(c.batch):
        g = torch.Generator().manual_seed(seed * 1000 + b)
        out[:, b, 0] = torch.randint(0, c.text_card, (frames,), generator=g).numpy()
        out[:, b, 1:] = torch.randint(0, c.audio_card, (frames, 8), generator=g).numpy()
    return out


def run_batch_forced(c, frames, sessions):
    """c.prefill > 0: every session starts as the batch-64 workload does -- K/V rows
    0..prefill-1 of every layer from synth.kv_prefill (drawn on the GPU), offset
    prefill, ring all UNGENERATED; the checked sessions' rows go to the oracle too."""
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w), schedule=binding.RQ_SCHEDULE_TENSOR)
    assert dec.schedule == binding.RQ_SCHEDULE_TENSOR
    orc = oracle.Oracle(c, w)
    sts = {b: orc.new_state() for b in sessions}
    if c.prefill > 0:
        for b in range(c.batch):
            k, v = synth.kv_prefill(c, b, device="cuda")
            dec.set_kv(b, k, v)
            if b in sts:
                sts[b].set_kv(k.cpu(), v.cpu())
            del k, v
        torch.cuda.synchronize()
    users = synth.batch_user_tokens(c, frames).numpy()
    forced = forced_tokens(c, frames)
    worst = 0.0
    for t in range(frames):
        rs = {b: orc.step(sts[b], users[t, b], forced=forced[t, b], trace=True)
              for b in sessions}
        own, out, has = dec.step_forced(users[t], forced[t])
        text, audio = dec.logits()
        ring, off = dec.ring()
        for b in sessions:
            r = rs[b]
            oring, ooff = sts[b].ring()
            assert int(off[b]) == ooff and np.array_equal(ring[b], oring), (t, b)
            assert bool(has[b]) == r["has_out"], (t, b)
            if r["has_out"]:
                assert np.array_equal(out[b], r["out"]), (t, b)
            check_logits_and_tokens(c, own[b], r, text[b], audio[b], (t, b))
            worst = max([worst, rel_err(text[b], r["text_logits"])] +
                        [rel_err(audio[b][k], r["audio_logits"][k]) for k in range(8)])
    dec.close()
    print(f"{c.name} B={c.batch}: worst logit error {worst:.2e} of max|logit|")
    return worst


def test_small_batch16_all_sessions_forced():
    run_batch_forced(configs.SMALL.with_(batch=16), 6, range(16))


@pytest.mark.parametrize("batch", [3, 20, 40, 64])
def test_small_padded_and_full_tiles(batch):
    """batch 3 pads the session tile to 16, 20 to 32 and 40 to 48 (the padding rows stay
    zero); 64 fills it.  From 32 sessions the K splits of a tile merge through a
    thread-block cluster's shared memory, each split finishing its own 16-session chunks
    (20: two chunks, 40: three, 64: four), at 16 through L2."""
    run_batch_forced(configs.SMALL.with_(batch=batch), 4, [0, batch // 2, batch - 1])


def first_argmax(v):
    return int(np.argmax(np.where(np.isnan(v), -np.inf, v)))


def test_small_batch16_free_run():
    """No forcing on the GPU: each argmax feeds the next depformer step and the ring.
    Each GPU token must be the first-wins argmax of the GPU's own logits (exact), and
    the oracle, forced with the GPU's tokens, must reproduce the logits, the ring and
    the delayed outputs; own tokens agree wherever the oracle's margin allows."""
    c = configs.SMALL.with_(batch=16)
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w), schedule=binding.RQ_SCHEDULE_TENSOR)
    orc = oracle.Oracle(c, w)
    sts = [orc.new_state() for _ in range(16)]
    users = synth.batch_user_tokens(c, 8).numpy()
    for t in range(8):
        out, has = dec.step(users[t])
        text, audio = dec.logits()
        ring, off = dec.ring()
        for b in range(16):
            own = ring[b][np.arange(9), int(off[b]) % 3].astype(np.int32)
            assert own[0] == first_argmax(text[b]), (t, b)
            for k in range(8):
                assert own[1 + k] == first_argmax(audio[b][k]), (t, b, k)
            r = orc.step(sts[b], users[t, b], forced=own, trace=True)
            check_logits_and_tokens(c, own, r, text[b], audio[b], (t, b))
            oring, ooff = sts[b].ring()
            assert int(off[b]) == ooff and np.array_equal(ring[b], oring), (t, b)
            assert bool(has[b]) == r["has_out"], (t, b)
            if r["has_out"]:
                assert np.array_equal(out[b], r["out"]), (t, b)
    dec.close()


def test_auto_picks_tensor_from_batch2():
    c = configs.SMALL.with_(batch=16)
    w = binding.upload_weights(weights_of(c))
    for b in (2, 4, 16):
        d = binding.Decoder(c.with_(batch=b), w)
        assert d.schedule == binding.RQ_SCHEDULE_TENSOR, b
        d.close()
    d = binding.Decoder(c.with_(batch=1), w)
    assert d.schedule == binding.RQ_SCHEDULE_PERSISTENT
    d.close()
    t = configs.TINY.with_(batch=16)  # f32 weights: the tensor schedule does not apply
    wt = binding.upload_weights(weights_of(t))
    d = binding.Decoder(t, wt)
    assert d.schedule == binding.RQ_SCHEDULE_GRAPH
    d.close()
    with pytest.raises(binding.RQError):
        binding.Decoder(t, wt, schedule=binding.RQ_SCHEDULE_TENSOR)


def test_moshi7b_batch16_forced_frames():
    """The batch-16 workload's shapes (M = 16 session tile) on the first frames."""
    run_batch_forced(configs.MOSHI7B_B16, 3, [0, 15])


def test_moshi7b_batch64_forced_frames():
    run_batch_forced(configs.MOSHI7B.with_(batch=64), 2, [0, 63])


def test_moshi7b_batch64_prefilled_workload():
    """The batch-64 workload exactly as configured: 64 sessions whose temporal K/V hold
    2900 pre-filled positions (offset 2900, ring all UNGENERATED, so frames 0-1 read
    row 0 for -2), first frames on sessions 0 and 63 against the oracle."""
    c = configs.MOSHI7B_B64
    assert c.prefill == 2900 and c.batch == 64
    run_batch_forced(c, 2, [0, 63])
