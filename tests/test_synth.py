"""The seeded synthetic inputs follow their stated recipe: shapes of the C-ABI layout,
N(0, 0.02) matrices and tables, 1 + N(0, 0.02) alphas, bf16 rounding for bf16 models,
user codes uniform over their card with the small model's 5% of -1, per-session streams,
and results that do not depend on the drawing threads.  CPU only."""
import torch

from rq_transformer_frame_gb300 import configs, synth


def test_weight_shapes_follow_the_abi_layout():
    c = configs.TINY
    w = synth.make_weights(c, seed=0)
    D, L, F, V, A = c.dim, c.layers, c.hidden, c.text_card, c.audio_card
    DD, DL, DF = c.ddim, c.dlayers, c.dhidden
    want = {
        "emb": (16, A + 1, D), "text_emb": (V + 1, D), "norm1": (L, D),
        "in_proj": (L, 3 * D, D), "out_proj": (L, D, D), "norm2": (L, D),
        "gate_in": (L, 2 * F, D), "gate_out": (L, D, F), "out_norm": (D,),
        "text_linear": (V, D), "dep_in": (8, DD, D), "dep_text_emb": (V + 1, DD),
        "dep_emb": (7, A + 1, DD), "dnorm1": (DL, DD), "dnorm2": (DL, DD),
        "d_in_proj": (DL, 8, 3 * DD, DD), "d_out_proj": (DL, 8, DD, DD),
        "d_gate_in": (DL, 8, 2 * DF, DD), "d_gate_out": (DL, 8, DD, DF),
        "linears": (8, A, DD),
    }
    assert set(w) == set(want)
    for k, shape in want.items():
        assert tuple(w[k].shape) == shape, k
        assert w[k].is_contiguous(), k
        assert w[k].dtype == torch.float32, k  # the tiny model is f32 throughout


def test_value_distributions():
    w = synth.make_weights(configs.SMALL, seed=0)
    m = w["gate_in"].float()
    assert m.dtype == torch.float32 and w["gate_in"].dtype == torch.bfloat16
    assert abs(float(m.mean())) < 1e-4
    assert abs(float(m.std()) - 0.02) < 2e-4
    a = w["norm1"]
    assert a.dtype == torch.float32
    assert abs(float(a.mean()) - 1.0) < 2e-3 and abs(float(a.std()) - 0.02) < 2e-3
    # bf16 models keep alphas as f32 arrays of bf16 values
    assert torch.equal(a, a.to(torch.bfloat16).float())


def test_draws_do_not_depend_on_threads():
    c = configs.TINY
    one = synth.make_weights(c, seed=3, threads=1)
    many = synth.make_weights(c, seed=3, threads=8)
    for k in one:
        assert torch.equal(one[k], many[k]), k
    other = synth.make_weights(c, seed=4, threads=1)
    assert not torch.equal(one["in_proj"], other["in_proj"])


def test_user_codes():
    t = synth.user_tokens(configs.TINY, 400)
    assert t.dtype == torch.int32 and tuple(t.shape) == (400, 8)
    assert int(t.min()) >= 0 and int(t.max()) < configs.TINY.user_card
    s = synth.user_tokens(configs.SMALL, 2000)
    minus = float((s == -1).float().mean())
    assert 0.04 < minus < 0.06  # the small model's 5% of "no code"
    kept = s[s >= 0]
    assert int(kept.max()) < configs.SMALL.user_card and int(kept.min()) >= 0
    # every card value is reachable: a uniform draw of 15 200 codes over 2048
    assert len(torch.unique(kept)) > 2000
    # Moshi-7B streams have no -1
    assert int(synth.user_tokens(configs.MOSHI7B, 200).min()) >= 0


def test_batch_streams_are_the_per_session_streams():
    c = configs.SMALL.with_(batch=3)
    b = synth.batch_user_tokens(c, 10)
    assert tuple(b.shape) == (10, 3, 8)
    for s in range(3):
        assert torch.equal(b[:, s], synth.user_tokens(c, 10, session=s))
    assert not torch.equal(b[:, 0], b[:, 1])


def test_kv_prefill_recipe():
    c = configs.TINY.with_(prefill=40)
    k, v = synth.kv_prefill(c, 2)
    assert k.dtype == torch.bfloat16 and tuple(k.shape) == (c.layers, 40, c.dim)
    assert tuple(v.shape) == tuple(k.shape)
    k2, v2 = synth.kv_prefill(c, 2)
    assert torch.equal(k, k2) and torch.equal(v, v2)
    assert not torch.equal(k, v)
    k3, _ = synth.kv_prefill(c, 3)
    assert not torch.equal(k, k3)
    assert abs(float(k.float().std()) - 1.0) < 0.05


def test_moshi7b_shape_is_the_pages():
    """The Moshi-7B workload has the page's decode shape (tests/golden/moshi7b_shape.json)."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "moshi7b_shape.json")))
    c = configs.MOSHI7B
    for k in ("dim", "layers", "heads", "head_dim", "context", "hidden", "ddim", "dlayers",
              "dheads", "dhead_dim", "dhidden", "text_card", "audio_card"):
        assert getattr(c, k) == g[k], k
    assert c.eps == g["rms_eps"]
    assert g["hidden"] == round(2 * 4.125 * g["dim"] / 3)
    assert g["dhidden"] == round(2 * 4.125 * g["ddim"] / 3)
    assert g["heads"] * g["head_dim"] == g["dim"] and g["dheads"] * g["dhead_dim"] == g["ddim"]
    assert g["ring"] == g["max_delay"] + 2 and max(g["delays"]) == g["max_delay"]
    assert len(g["delays"]) == 17
    for name in ("moshi7b_b16", "moshi7b_b64"):
        b = configs.CONFIGS[name]
        assert (b.dim, b.layers, b.hidden, b.context) == (c.dim, c.layers, c.hidden, c.context)
