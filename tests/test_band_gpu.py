"""Weight bands on the GPU ("moshi_lm.rs", `qn_roundtrip`, the Q4_0 layout at
`q4_roundtrip`, `load_q4sim`): the device quantizer against the oracle's roundtrip, and
whole frames of band models against the Q4-roundtrip oracle (the oracle on the
quantized-and-dequantized weights in f32, as the page's `load_q4sim` does).

The GPU multiplies each stored code by its scale in f32, exactly the dequantized weight
the roundtrip oracle uses, so band frames meet the same parity bar as bf16 frames.  The
page gates a band on logits cosine and token agreement with the unquantized model; that
is reported here as a floor, not as parity.
"""
import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding, configs, synth

from parity_util import check_logits_and_tokens, weights_of

pytestmark = pytest.mark.gpu

BANDS = [(binding.RQ_Q8, 8, "q8"), (binding.RQ_Q4, 4, "q4")]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def decode_rows(raw: np.ndarray, rows: int, cols: int, bits: int) -> np.ndarray:
    """The stored band rows (include/rq.h layout) back to values q * d."""
    ng = cols // 32
    codes = cols if bits == 8 else cols // 2
    rb = codes + 4 * ng
    raw = raw.reshape(rows, rb)
    d = raw[:, codes:].copy().view(np.float32).reshape(rows, ng)
    if bits == 8:
        q = raw[:, :codes].view(np.int8).astype(np.int32).reshape(rows, ng, 32)
    else:
        b = raw[:, :codes].reshape(rows, ng, 16).astype(np.int32)
        q = np.concatenate([(b & 15) - 8, (b >> 4) - 8], axis=2)
    return (q.astype(np.float32) * d[:, :, None]).reshape(rows, cols)


@pytest.mark.parametrize("dtype,bits,name", BANDS, ids=[b[2] for b in BANDS])
def test_quantizer_matches_oracle_roundtrip(dtype, bits, name):
    g = torch.Generator().manual_seed(21)
    w = (torch.randn(70, 256, generator=g) * 0.02).to(torch.bfloat16)
    w[3, 32:64] = 0                              # a zero group: d = 0
    w[5, 0:32] = 0
    w[5, 4], w[5, 17] = -0.5, 0.5                # equal magnitudes: the first decides d
    w[7, 0:32] = torch.arange(32, dtype=torch.float32).to(torch.bfloat16) * 0.125 - 2.0
    raw = binding.quantize(w.cuda().contiguous(), dtype).cpu().numpy()
    got = decode_rows(raw, 70, 256, bits)
    want = oracle.qn_roundtrip(w.float().numpy(), bits)
    np.testing.assert_array_equal(got, want)


def band_weights_for_oracle(w_bf16: dict, bits: int) -> dict:
    """The Q4-roundtrip oracle's weights: matrices quantized and dequantized (f32),
    tables and alphas widened exactly to f32."""
    out = {}
    for k, v in w_bf16.items():
        f = v.float()
        if k in binding.MATRIX_FIELDS:
            rows = f.reshape(-1, f.shape[-1]).numpy()
            f = torch.from_numpy(oracle.qn_roundtrip(rows, bits)).reshape(f.shape)
        out[k] = f.contiguous()
    return out


SCHEDULES = [binding.RQ_SCHEDULE_GRAPH, binding.RQ_SCHEDULE_PERSISTENT]


@pytest.mark.parametrize("schedule", SCHEDULES, ids=["graph", "persistent"])
@pytest.mark.parametrize("dtype,bits,name", BANDS, ids=[b[2] for b in BANDS])
def test_band_frames_match_roundtrip_oracle(dtype, bits, name, schedule):
    c = configs.SMALL.with_(weight_dtype=name)
    w = weights_of(configs.SMALL)  # the bf16 weights the band quantizes
    dev = binding.quantize_weights(binding.upload_weights(w), dtype)
    dec = binding.Decoder(c, dev, schedule=schedule)
    assert dec.schedule == schedule
    orc = oracle.Oracle(c.with_(weight_dtype="f32"), band_weights_for_oracle(w, bits))
    st = orc.new_state()
    users = synth.user_tokens(c, 8).numpy()
    ref = oracle.Oracle(configs.SMALL, w)  # the unquantized model, for the page's gate
    st_ref = ref.new_state()
    cos, agree = [], 0
    for t in range(8):
        r = orc.step(st, users[t], trace=True)
        own, out, has = dec.step_forced(users[t][None], r["own"][None])
        text, audio = dec.logits()
        check_logits_and_tokens(c, own[0], r, text[0], audio[0], t)
        rr = ref.step(st_ref, users[t], forced=r["own"], trace=True)
        cos.append(float(np.dot(text[0], rr["text_logits"]) /
                         (np.linalg.norm(text[0]) * np.linalg.norm(rr["text_logits"]))))
        agree += int(np.argmax(text[0]) == np.argmax(rr["text_logits"]))
    print("%s: text-logit cosine to the bf16 model %.4f, argmax agreement %d/8" %
          (name, min(cos), agree))
    assert min(cos) > (0.99 if bits == 8 else 0.8)
    dec.close()


def test_band_models_refuse_the_bf16_only_schedules():
    c = configs.SMALL.with_(weight_dtype="q4")
    dev = binding.quantize_weights(binding.upload_weights(weights_of(configs.SMALL)),
                                   binding.RQ_Q4)
    with pytest.raises(binding.RQError):
        binding.Decoder(c, dev, schedule=binding.RQ_SCHEDULE_TENSOR)
    d = binding.Decoder(c, dev)  # AUTO keeps bands on one GEMV kernel per op (faster)
    assert d.schedule == binding.RQ_SCHEDULE_GRAPH
    d.close()
    d = binding.Decoder(c, dev, schedule=binding.RQ_SCHEDULE_PERSISTENT)
    assert d.schedule == binding.RQ_SCHEDULE_PERSISTENT
    d.close()
    d = binding.Decoder(c.with_(batch=2), dev)  # batch > 1: one GEMV kernel per op
    assert d.schedule == binding.RQ_SCHEDULE_GRAPH
    d.close()
    with pytest.raises(ValueError):
        binding.quantize(torch.zeros(4, 48, device="cuda"), binding.RQ_Q4)


@pytest.mark.parametrize("dtype,bits,name", BANDS, ids=[b[2] for b in BANDS])
def test_band_moshi7b_layer_shapes_persistent(dtype, bits, name):
    """The Moshi-7B layer shapes (2 temporal layers, the whole depformer and heads) as a
    weight band on the persistent kernel: gate_out's 11264-column rows run as reduction
    parts whose codes and scales are copied separately; the depformer's 1024-column rows
    give one warp per row.  Two forced frames against the roundtrip oracle."""
    base = configs.MOSHI7B_2L
    c = base.with_(weight_dtype=name)
    w = weights_of(base)
    dev = binding.quantize_weights(binding.upload_weights(w), dtype)
    dec = binding.Decoder(c, dev, schedule=binding.RQ_SCHEDULE_PERSISTENT)
    assert dec.schedule == binding.RQ_SCHEDULE_PERSISTENT
    orc = oracle.Oracle(c.with_(weight_dtype="f32"), band_weights_for_oracle(w, bits))
    st = orc.new_state()
    users = synth.user_tokens(c, 2).numpy()
    for t in range(2):
        r = orc.step(st, users[t], trace=True)
        own, out, has = dec.step_forced(users[t][None], r["own"][None])
        text, audio = dec.logits()
        check_logits_and_tokens(c, own[0], r, text[0], audio[0], t)
    dec.close()
