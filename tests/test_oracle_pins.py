"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the definition it pins ("inferencelayer 0.2.4 -- src/moshi_lm.rs"
unless stated).  Closed forms and hand traces live in tests/golden/ with their
citations; library routines (NumPy float64, torch SDPA in float64) are used only
where they compute the textbook operation independently of the oracle.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import configs, synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _num(v):
    return float(v) if not isinstance(v, str) else float(v.replace("inf", "inf"))


PRIM = _load("primitives.json")


# ------------------------------------------------------------------ rms_norm
@pytest.mark.parametrize("case", PRIM["rms_norm"]["cases"])
def test_rms_norm_closed_forms(case):
    y = oracle.rms_norm(case["x"], case["alpha"], case["eps"])
    np.testing.assert_allclose(y, case["y"], rtol=2e-6, atol=1e-12)
    assert np.all(np.isfinite(y))


def test_rms_norm_matches_f64_definition_random():
    rng = np.random.default_rng(5)
    for n in (1, 7, 256, 4096):
        x = rng.standard_normal(n).astype(np.float32) * 0.3
        a = (1 + 0.02 * rng.standard_normal(n)).astype(np.float32)
        ref = x.astype(np.float64) * a / np.sqrt(1e-8 + np.mean(x.astype(np.float64) ** 2))
        np.testing.assert_allclose(oracle.rms_norm(x, a), ref, rtol=5e-6, atol=1e-7)


# ------------------------------------------------------------------ rope
@pytest.mark.parametrize("case", PRIM["rope"]["cases"])
def test_rope_hand_vectors(case):
    y = oracle.rope_row(case["v"], case["pos"], case["head_dim"])
    np.testing.assert_allclose(y, case["y"], rtol=1e-6, atol=2e-7)


def test_rope_frequencies_and_norms():
    """Pair i of every head turns by pos * 10000^(-2i/hd); each pair keeps its norm."""
    hd, heads = 128, 3
    rng = np.random.default_rng(1)
    v = rng.standard_normal(heads * hd).astype(np.float32)
    for pos in (1, 17, 375, 2999):
        y = oracle.rope_row(v, pos, hd).astype(np.float64).reshape(heads, hd // 2, 2)
        x = v.astype(np.float64).reshape(heads, hd // 2, 2)
        np.testing.assert_allclose(np.hypot(y[..., 0], y[..., 1]),
                                   np.hypot(x[..., 0], x[..., 1]), rtol=2e-6)
        ang = pos * 10000.0 ** (-2.0 * np.arange(hd // 2) / hd)
        # rotation angle of each pair recovered from the complex ratio y / x
        got = np.angle((y[..., 0] + 1j * y[..., 1]) / (x[..., 0] + 1j * x[..., 1]))
        want = np.angle(np.exp(1j * ang))
        d = np.angle(np.exp(1j * (got - want)))
        # f32 angle rounding: |error| <= a few ulp of pos * freq
        assert np.max(np.abs(d)) < 4e-4 * max(1.0, pos / 1000)


# ------------------------------------------------------------------ argmax / silu
@pytest.mark.parametrize("case", PRIM["argmax"]["cases"])
def test_argmax_first_wins_nan_never(case):
    v = [_num(x) for x in case["v"]]
    assert oracle.argmax(v) == case["idx"]


def test_argmax_random_ties_first_index():
    rng = np.random.default_rng(2)
    for _ in range(50):
        v = rng.integers(0, 4, size=33).astype(np.float32)
        assert oracle.argmax(v) == int(np.flatnonzero(v == v.max())[0])


@pytest.mark.parametrize("case", PRIM["silu"]["cases"])
def test_silu(case):
    assert oracle.silu(case["x"]) == pytest.approx(case["y"], rel=1e-6, abs=1e-12)


# ------------------------------------------------------------------ attention
def test_attention_single_key_is_value():
    rng = np.random.default_rng(3)
    q = rng.standard_normal(4 * 32).astype(np.float32)
    k = rng.standard_normal((1, 4 * 32)).astype(np.float32)
    v = rng.standard_normal((1, 4 * 32)).astype(np.float32)
    np.testing.assert_array_equal(oracle.attend(q, k, v, 4, 32), v[0])


def test_attention_equal_keys_mean_of_values():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(2 * 16).astype(np.float32)
    k = np.tile(rng.standard_normal((1, 32)).astype(np.float32), (5, 1))
    v = rng.standard_normal((5, 32)).astype(np.float32)
    np.testing.assert_allclose(oracle.attend(q, k, v, 2, 16), v.mean(0), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("n,heads,hd", [(1, 1, 8), (7, 4, 32), (64, 4, 64), (300, 2, 128)])
def test_attention_vs_sdpa_f64(n, heads, hd):
    rng = np.random.default_rng(n)
    q = rng.standard_normal(heads * hd).astype(np.float32)
    k = rng.standard_normal((n, heads * hd)).astype(np.float32)
    v = rng.standard_normal((n, heads * hd)).astype(np.float32)
    got = oracle.attend(q, k, v, heads, hd)
    Q = torch.tensor(q, dtype=torch.float64).view(heads, 1, hd)
    K = torch.tensor(k, dtype=torch.float64).view(n, heads, hd).transpose(0, 1)
    V = torch.tensor(v, dtype=torch.float64).view(n, heads, hd).transpose(0, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V).reshape(-1).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)


# ------------------------------------------------------------------ gemv / embed
@pytest.mark.parametrize("rows,k", [(1, 1), (5, 7), (64, 256), (300, 1408)])
def test_gemv_vs_numpy_f64(rows, k):
    rng = np.random.default_rng(rows * 31 + k)
    w = (0.02 * rng.standard_normal((rows, k))).astype(np.float32)
    x = rng.standard_normal(k).astype(np.float32)
    ref = w.astype(np.float64) @ x.astype(np.float64)
    np.testing.assert_allclose(oracle.gemv(w, x), ref, rtol=1e-5, atol=1e-6 * math.sqrt(k))


def test_gemv_bf16_weights_widened_exactly():
    g = torch.Generator().manual_seed(9)
    w = (0.02 * torch.randn(33, 520, generator=g)).to(torch.bfloat16)
    x = torch.randn(520, generator=g).numpy()
    ref = w.to(torch.float64).numpy() @ x.astype(np.float64)
    np.testing.assert_allclose(oracle.gemv(w, x), ref, rtol=1e-5, atol=1e-6 * math.sqrt(520))


def test_embed_minus_one_is_exact_zero_and_clamps():
    table = (np.arange(5 * 4, dtype=np.float32).reshape(5, 4) + 1) / 7
    acc = np.zeros(4, np.float32)
    np.testing.assert_array_equal(oracle.embed(table, -1, acc), acc)       # -1 -> nothing
    np.testing.assert_array_equal(oracle.embed(table, -2, acc), table[0])  # max(tok, 0)
    np.testing.assert_array_equal(oracle.embed(table, 3, acc), table[3])
    np.testing.assert_array_equal(oracle.embed(table, 4, acc), table[4])   # INITIAL = last row


# ------------------------------------------------------------------ whole-model pins (tiny)
@pytest.fixture(scope="module")
def tiny():
    c = configs.TINY
    w = synth.make_weights(c, seed=0)
    return c, w, oracle.Oracle(c, w)


def _symbols(c, forced_fn, user_fn, frames):
    sym = {"IT": c.text_card, "IA": c.audio_card, "UG": -2}
    for t in range(frames):
        f = forced_fn(t)
        sym["T%d" % t] = int(f[0])
        for cb in range(8):
            sym["A%d.%d" % (t, cb)] = int(f[1 + cb])
        u = user_fn(t)
        for k in range(8):
            sym["U%d.%d" % (t, k)] = int(u[k])
    return sym


def _forced(c):
    return lambda t: np.array([(3 * t + 1) % c.text_card] +
                              [(7 * cb + 5 * t + 2) % c.audio_card for cb in range(8)], np.int32)


def _user(c):
    return lambda t: np.array([(11 * t + 3 * k + 1) % c.audio_card for k in range(8)], np.int32)


def test_ring_schedule_hand_trace_fresh(tiny):
    c, w, o = tiny
    trace = _load("ring_trace.json")
    f, u = _forced(c), _user(c)
    sym = _symbols(c, f, u, 8)
    st = o.new_state()
    for row in trace["fresh"]:
        t = row["frame"]
        r = o.step(st, u(t), forced=f(t), trace=True)
        assert [int(x) for x in r["input_tokens"]] == [sym[s] for s in row["input"]], t
        if row["out"] is None:
            assert not r["has_out"]
        else:
            assert r["has_out"]
            assert [int(x) for x in r["out"]] == [sym[s] for s in row["out"]], t
    ring, off = st.ring()
    assert off == len(trace["fresh"])


def test_ring_schedule_hand_trace_prefilled(tiny):
    """Clock started at n with n % 3 == 2 and a ring still all UNGENERATED."""
    c, w, o = tiny
    trace = _load("ring_trace.json")
    f, u = _forced(c), _user(c)
    sym = _symbols(c, f, u, 8)
    st = o.new_state()
    n = 62
    assert n % 3 == 2 and n < c.context
    g = torch.Generator().manual_seed(0)
    k = torch.randn(c.layers, n, c.dim, generator=g)
    v = torch.randn(c.layers, n, c.dim, generator=g)
    st.set_kv(k, v)
    assert st.ring()[1] == n
    for row in trace["prefilled"]:
        t = row["frame"]
        r = o.step(st, u(t), forced=f(t), trace=True)
        assert [int(x) for x in r["input_tokens"]] == [sym[s] for s in row["input"]], t
        assert r["has_out"]
        assert [int(x) for x in r["out"]] == [sym[s] for s in row["out"]], t


def test_embedding_sum_frame0_is_initial_rows(tiny):
    c, w, o = tiny
    st = o.new_state()
    r = o.step(st, np.zeros(8, np.int32), trace=True)
    ref = sum(w["emb"][k][c.audio_card].double() for k in range(16)) + \
        w["text_emb"][c.text_card].double()
    np.testing.assert_allclose(r["emb_sum"], ref.numpy(), rtol=1e-6, atol=1e-7)


def test_embedding_sum_single_stream_is_that_row(tiny):
    """All streams -1 but one -> that row, bit-exactly; all -1 -> exact zero."""
    c, w, o = tiny
    st = o.new_state()
    minus = np.full(8, -1, np.int32)
    forced = np.array([-1] * 9, np.int32)
    o.step(st, minus, forced=forced)          # frame 0 (INITIAL inputs)
    o.step(st, minus, forced=forced)          # frame 1 (user d=1 streams still INITIAL)
    r = o.step(st, minus, forced=forced, trace=True)  # frame 2: every input is -1
    assert list(r["input_tokens"]) == [-1] * 17
    assert np.all(r["emb_sum"] == 0.0)
    u = minus.copy()
    u[0] = 17  # user codebook 0 has delay 0: read this very frame
    r = o.step(st, u, forced=forced, trace=True)
    assert r["input_tokens"][9] == 17 and sum(r["input_tokens"] != -1) == 1
    np.testing.assert_array_equal(r["emb_sum"], w["emb"][8][17].numpy())


def test_depformer_incremental_equals_from_scratch(tiny):
    """The per-frame K/V cycle equals recomputing steps 0..cb as one causal
    sequence (rlx_lm.rs: slice si attends to positions 0..si), for every cb."""
    from ref_f64 import Ref64
    c, w, o = tiny
    ref = Ref64(c, w)
    rng = np.random.default_rng(7)
    tout = rng.standard_normal(c.dim).astype(np.float32)
    forced = np.array([5] + list(rng.integers(0, c.audio_card, 8)), np.int32)
    logits, _ = o.depformer_cycle(tout, int(forced[0]), forced=forced)
    prevs = [int(forced[0])] + [int(x) for x in forced[1:8]]
    for cb in range(8):
        want = ref.depformer_from_scratch(tout.astype(np.float64), prevs, cb)
        scale = np.max(np.abs(want))
        assert np.max(np.abs(logits[cb] - want)) <= 1e-5 * scale, cb


def test_depformer_has_no_cross_frame_state(tiny):
    """Frame t's depformer after any history equals running it alone."""
    c, w, o = tiny
    st = o.new_state()
    u = synth.user_tokens(c, 6).numpy()
    for t in range(6):
        r = o.step(st, u[t], trace=True)
    alone_logits, alone_toks = o.depformer_cycle(r["tout"], int(r["own"][0]))
    np.testing.assert_array_equal(alone_logits, r["audio_logits"])
    np.testing.assert_array_equal(alone_toks, r["own"][1:])


def test_threads_do_not_change_bits(tiny):
    c, w, o = tiny
    outs = []
    for n in (1, 4):
        oracle.set_threads(n)
        st = o.new_state()
        r = o.step(st, np.arange(8, dtype=np.int32), trace=True)
        outs.append(r)
    oracle.set_threads(oracle.max_threads())
    for k in ("text_logits", "audio_logits", "tout"):
        np.testing.assert_array_equal(outs[0][k], outs[1][k])


# ------------------------------------------------------------------ sampling
XS = _load("xorshift64.json")


def test_xorshift_published_sequence():
    r = oracle.XorShift(XS["seed"])
    assert [r.next() for _ in range(3)] == XS["outputs"]


def test_xorshift_u01_takes_the_top_53_bits():
    r = oracle.XorShift(XS["seed"])
    for x in XS["outputs"]:
        u = r.u01()
        assert u == (x >> 11) / 2.0 ** 53 and 0.0 <= u < 1.0


def _chi2_ok(counts, probs, n):
    """Pearson chi-square against the expected frequencies, generous 1e-4 tail bound
    (df <= 7: chi2 < 30)."""
    exp = np.asarray(probs) * n
    keep = exp > 0
    stat = float((((counts - exp) ** 2)[keep] / exp[keep]).sum())
    return stat < 30.0, stat


def test_gumbel_pick_samples_softmax_of_logits_over_temp():
    # the Gumbel-max property: argmax(l/T + G) is distributed as softmax(l/T)
    logits = np.array([0.5, -1.0, 2.0, 0.0, 1.0], np.float32)
    temp = 0.8
    p = np.exp(logits.astype(np.float64) / temp)
    p /= p.sum()
    r = oracle.XorShift(12345)
    n = 60000
    counts = np.zeros(5)
    for _ in range(n):
        counts[oracle.gumbel_pick(logits, temp, r)] += 1
    ok, stat = _chi2_ok(counts, p, n)
    assert ok, (stat, counts / n, p)


def test_gumbel_pick_consumes_one_draw_per_logit():
    logits = np.zeros(37, np.float32)
    a, b = oracle.XorShift(99), oracle.XorShift(99)
    oracle.gumbel_pick(logits, 1.0, a)
    for _ in range(37):
        b.next()
    assert a.state == b.state


def test_gumbel_pick_tiny_temperature_is_argmax():
    logits = np.array([0.1, 5.0, -2.0, 4.0], np.float32)
    assert oracle.gumbel_pick(logits, 1e-6, oracle.XorShift(7)) == 1


def test_topk_pick_samples_renormalised_top_k():
    logits = np.array([0.3, 2.0, -1.0, 1.5, 1.7, -0.5, 0.9, 0.0], np.float32)
    temp, k = 0.7, 3
    top = np.argsort(-logits.astype(np.float64), kind="stable")[:k]
    p = np.zeros(8)
    p[top] = np.exp((logits[top].astype(np.float64) - logits.max()) / temp)
    p /= p.sum()
    r = oracle.XorShift(2024)
    n = 60000
    counts = np.zeros(8)
    for _ in range(n):
        counts[oracle.topk_pick(logits, temp, k, r)] += 1
    assert counts[[i for i in range(8) if i not in top]].sum() == 0
    ok, stat = _chi2_ok(counts, p, n)
    assert ok, (stat, counts / n, p)


def test_topk_pick_consumes_one_draw():
    a, b = oracle.XorShift(5), oracle.XorShift(5)
    oracle.topk_pick(np.arange(10, dtype=np.float32), 0.8, 4, a)
    b.next()
    assert a.state == b.state


def test_topk_k1_is_first_wins_argmax():
    logits = np.array([1.0, 3.0, 3.0, 2.0], np.float32)
    for seed in range(1, 20):
        assert oracle.topk_pick(logits, 0.8, 1, oracle.XorShift(seed)) == 1


def test_topk_equal_logits_walk_in_index_order():
    # two equal logits, k = 2: p = (1/2, 1/2); the draw u picks the lower index when
    # u <= 1/2 (reading: equal logits in ascending index order)
    logits = np.array([0.0, 4.0, 4.0, -3.0], np.float32)
    seen = set()
    for i in range(1, 40):
        seed = (i * 0x9E3779B97F4A7C15) & (2 ** 64 - 1)  # spread over all 64 bits
        u = oracle.XorShift(seed).u01()
        tok = oracle.topk_pick(logits, 1.0, 2, oracle.XorShift(seed))
        assert tok == (1 if u <= 0.5 else 2), (seed, u, tok)
        seen.add(tok)
    assert seen == {1, 2}


@pytest.mark.parametrize("mode,draws", [(oracle.PICK_GREEDY, lambda c: 0),
                                        (oracle.PICK_TOPK, lambda c: 9),
                                        (oracle.PICK_GUMBEL,
                                         lambda c: c.text_card + 8 * c.audio_card)])
def test_frame_draw_count_per_sampler(tiny, mode, draws):
    # `pick` runs once for the text token and once per codebook, in that order
    c, w, o = tiny
    st = o.new_state()
    st.set_sampling(mode, seed=77)
    st.set_sampling(mode, seed=77)
    ref = oracle.XorShift(77)
    o.step(st, np.arange(8, dtype=np.int32))
    for _ in range(draws(c)):
        ref.next()
    assert st.rng == (ref.state if mode != oracle.PICK_GREEDY else 77)


def test_sampled_step_tokens_follow_pick_on_its_own_logits(tiny):
    # the frame's text token is the pick over its text logits with the frame-start state
    c, w, o = tiny
    for mode in (oracle.PICK_TOPK, oracle.PICK_GUMBEL):
        st = o.new_state()
        st.set_sampling(mode, temp=0.9, temp_text=0.6, top_k=5, top_k_text=3, seed=31)
        r = o.step(st, np.arange(8, dtype=np.int32), trace=True)
        rng = oracle.XorShift(31)
        if mode == oracle.PICK_TOPK:
            tok = oracle.topk_pick(r["text_logits"], 0.6, 3, rng)
        else:
            tok = oracle.gumbel_pick(r["text_logits"], 0.6, rng)
        assert tok == r["own"][0]
        for cb in range(8):
            lg = r["audio_logits"][cb]
            t = (oracle.topk_pick(lg, 0.9, 5, rng) if mode == oracle.PICK_TOPK
                 else oracle.gumbel_pick(lg, 0.9, rng))
            assert t == r["own"][1 + cb], (mode, cb)
        assert rng.state == st.rng


# ------------------------------------------------------------------ priming, replay, snapshot
def _prime_inputs(c, t):
    f = np.array([(5 * t + 2) % c.text_card] + [(3 * cb + 7 * t + 1) % c.audio_card
                                                 for cb in range(8)], np.int32)
    return f


def test_prime_steps_leave_the_state_of_forced_full_steps(tiny):
    # `step_forced` (temporal only) and a full step forced with the same tokens differ
    # only in the outputs they discard: same ring, offset and K/V afterwards
    c, w, o = tiny
    a, b = o.new_state(), o.new_state()
    u = synth.user_tokens(c, 7).numpy()
    for t in range(6):
        f = _prime_inputs(c, t)
        r = o.step(a, u[t], forced=f, trace=True)
        e = o.prime_step(b, f, u[t])
        np.testing.assert_array_equal(e, r["emb_sum"])
    ra, oa = a.ring()
    rb, ob = b.ring()
    assert np.array_equal(ra, rb) and oa == ob == 6
    x, y = o.step(a, u[6], trace=True), o.step(b, u[6], trace=True)
    for k in ("text_logits", "audio_logits", "tout"):
        np.testing.assert_array_equal(x[k], y[k])


def test_replay_of_the_gathered_embeddings_equals_priming_kv(tiny):
    c, w, o = tiny
    a, b = o.new_state(), o.new_state()
    u = synth.user_tokens(c, 5).numpy()
    ring0, _ = b.ring()
    for t in range(5):
        e = o.prime_step(a, _prime_inputs(c, t), u[t])
        o.replay_step(b, e)
    ring1, off = b.ring()
    assert off == 5 and np.array_equal(ring0, ring1)  # advance_clock: ring untouched
    probe = np.linspace(-1, 1, c.dim).astype(np.float32)
    np.testing.assert_array_equal(o.temporal_step(a, probe), o.temporal_step(b, probe))


def test_snapshot_copy_is_independent(tiny):
    c, w, o = tiny
    a = o.new_state()
    u = synth.user_tokens(c, 8).numpy()
    for t in range(3):
        o.step(a, u[t])
    snap = a.clone()
    ra = [o.step(a, u[t], trace=True) for t in range(3, 8)]
    r0, off0 = snap.ring()
    assert off0 == 3
    rs = [o.step(snap, u[t], trace=True) for t in range(3, 8)]
    for x, y in zip(ra, rs):
        np.testing.assert_array_equal(x["own"], y["own"])
        np.testing.assert_array_equal(x["text_logits"], y["text_logits"])


# ------------------------------------------------------------------ weight bands
@pytest.mark.parametrize("bits", [4, 8])
def test_qn_roundtrip_grid_and_error_bound(bits):
    g = np.random.default_rng(3)
    v = g.normal(0, 0.02, (5, 96)).astype(np.float32)
    q = oracle.qn_roundtrip(v, bits)
    qmin = -(1 << (bits - 1))
    for r in range(5):
        for b in range(3):
            blk, out = v[r, 32 * b:32 * b + 32], q[r, 32 * b:32 * b + 32]
            mx = blk[np.argmax(np.abs(blk))]
            d = np.float32(mx / np.float32(qmin))
            # the largest-magnitude value maps to the end of the grid exactly
            assert out[np.argmax(np.abs(blk))] == np.float32(qmin) * d
            k = out / d  # every output is an integer multiple of d in [qmin, qmax]
            assert np.all(np.abs(k - np.round(k)) < 1e-3)
            assert k.min() >= qmin - 1e-3 and k.max() <= -qmin - 1 + 1e-3
            # rounding to the nearest grid point; a value beyond qmax (only possible with the
            # sign opposite to mx, |x| <= |mx|) is clamped and lands within one step
            err = np.abs(out - blk)
            clamped = np.abs(np.round(k) - (-qmin - 1)) < 1e-3
            assert np.all(err[~clamped] <= np.abs(d) * 0.5 * (1 + 1e-5) + 1e-12)
            assert np.all(err[clamped] <= np.abs(d) * (1 + 1e-5) + 1e-12)


def test_qn_roundtrip_exact_grid_values_and_zero_group():
    d = np.float32(0.125)
    ks = np.array([-8, -3, 0, 5, 7, -1, 2, -8] * 4, np.float32)
    v = (ks * d).reshape(1, 32)
    np.testing.assert_array_equal(oracle.qn_roundtrip(v, 4), v)  # already on the grid
    z = np.zeros((2, 32), np.float32)
    np.testing.assert_array_equal(oracle.qn_roundtrip(z, 4), z)  # d = 0: all zero


def test_qn_roundtrip_q4_page_scale():
    # Q4_0: "d = max / -8" with max the value of largest magnitude, ties to the first
    v = np.zeros((1, 32), np.float32)
    v[0, 3], v[0, 9], v[0, 20] = -0.5, 0.5, 0.25
    q = oracle.qn_roundtrip(v, 4)
    d = np.float32(-0.5) / np.float32(-8)  # the first of the equal magnitudes, -0.5
    assert q[0, 3] == -0.5 and q[0, 20] == np.float32(round(0.25 / d)) * d
    assert q[0, 9] == np.float32(7) * d  # +8 d is past the grid: clamped to qmax
