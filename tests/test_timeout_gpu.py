"""The failure path of a device-side wait that runs out (the bounded waits of the
whole-frame kernel): the frame reports RQ_ERR_TIMEOUT, the handle is poisoned until
rq_reset(h, -1), and after that reset the handle decodes like a fresh one.

The wait is made to run out without any fault: a test hook shortens the wait limit to
20 ms and makes the waits in front of one op unsatisfiable -- in the temporal launch its
grid barrier waits for one CTA more than the grid holds, in the depformer launch its
tagged words for a tag that nothing writes.  Every CTA gives up at its own bounded wait,
records the timeout in the status word, waits for its own bulk copies in flight and
returns; the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding, configs, synth

from parity_util import check_logits_and_tokens, weights_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("stall_op", [1, 7, "depformer"])
def test_wait_timeout_poisons_and_reset_recovers(stall_op):
    c = configs.TINY
    w = weights_of(c)
    dec = binding.Decoder(c, binding.upload_weights(w))
    assert dec.schedule == binding.RQ_SCHEDULE_PERSISTENT
    users = synth.user_tokens(c, 8).numpy()
    dec.step(users[0][None])
    dec.step(users[1][None])
    n_ops = len(dec.op_times())
    if stall_op == "depformer":
        stall_op = n_ops - 3  # inside the last depformer step
    with pytest.raises(binding.RQError):
        dec.set_wait_limit(20_000_000, 0)  # op 0 has no barrier in front of it
    with pytest.raises(binding.RQError):
        dec.set_wait_limit(20_000_000, n_ops)
    with pytest.raises(binding.RQError):  # the input projections beside the text head
        dec.set_wait_limit(20_000_000, 5 * c.layers + 1)
    with pytest.raises(binding.RQError):  # the depformer launch's first op waits for nothing
        dec.set_wait_limit(20_000_000, 5 * c.layers + 2)
    dec.set_wait_limit(20_000_000, stall_op)

    with pytest.raises(binding.RQError) as ei:
        dec.step(users[2][None])
    assert ei.value.status == binding.RQ_ERR_TIMEOUT
    # poisoned: every call that uses the handle's state refuses until rq_reset(h, -1)
    with pytest.raises(binding.RQError) as ei:
        dec.step(users[2][None])
    assert ei.value.status == binding.RQ_ERR_POISONED
    with pytest.raises(binding.RQError) as ei:
        dec.ring()
    assert ei.value.status == binding.RQ_ERR_POISONED
    with pytest.raises(binding.RQError) as ei:
        dec.reset(0)
    assert ei.value.status == binding.RQ_ERR_POISONED

    dec.set_wait_limit(0, -1)  # default limit, no stall
    dec.reset(-1)
    ring, off = dec.ring()
    assert int(off[0]) == 0 and np.all(ring[0] == -2)

    # the handle now decodes exactly as a fresh session: f32 tiny model, free run
    orc = oracle.Oracle(c, w)
    st = orc.new_state()
    for t in range(6):
        r = orc.step(st, users[t], trace=True)
        out, has = dec.step(users[t][None])
        text, audio = dec.logits()
        assert bool(has[0]) == r["has_out"], t
        if r["has_out"]:
            assert np.array_equal(out[0], r["out"]), t
        check_logits_and_tokens(c, r["own"], r, text[0], audio[0], t)
        ring, off = dec.ring()
        oring, ooff = st.ring()
        assert int(off[0]) == ooff and np.array_equal(ring[0], oring), t
    dec.close()


def test_wait_limit_needs_the_persistent_schedule():
    c = configs.TINY
    dec = binding.Decoder(c, binding.upload_weights(weights_of(c)),
                          schedule=binding.RQ_SCHEDULE_GRAPH)
    with pytest.raises(binding.RQError) as ei:
        dec.set_wait_limit(1000, -1)
    assert ei.value.status == binding.RQ_ERR_UNSUPPORTED
    dec.close()
