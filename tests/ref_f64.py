"""Second opinion for the oracle: an independent NumPy float64 restatement of the
per-frame decode step, written from "inferencelayer 0.2.4 -- src/moshi_lm.rs"
without looking at oracle/rq_oracle.c.

It is organised differently on purpose: heads are batched with reshapes and
einsum, the rotary frequencies use the theta ** (-2i / head_dim) form of
"rlx-moshi -- src/rlx_lm.rs" (`rope_tables`), the K/V window is a Python list
trimmed from the front, and the depformer can be recomputed from scratch as a
causal sequence of steps 0..cb.  Only the tests import it.
"""
from __future__ import annotations

import numpy as np

DELAYS = np.array([0, 0, 1, 1, 1, 1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 1, 1])
RING = 3  # max_delay + 2


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), returned as float64."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


class Ref64:
    def __init__(self, cfg, weights: dict):
        self.c = cfg
        self.W = {k: v.float().numpy().astype(np.float64) for k, v in weights.items()}

    # -- building blocks ---------------------------------------------------
    def rms(self, x, alpha):
        return x * alpha / np.sqrt(self.c.eps + np.mean(x * x))

    def rope(self, v, pos, head_dim):
        half = head_dim // 2
        pairs = v.reshape(-1, half, 2)
        inv_freq = self.c.rope_theta ** (-(np.arange(half) * 2.0) / head_dim)
        ang = pos * inv_freq
        re, im = pairs[..., 0], pairs[..., 1]
        out = np.stack([re * np.cos(ang) - im * np.sin(ang),
                        re * np.sin(ang) + im * np.cos(ang)], axis=-1)
        return out.reshape(v.shape)

    @staticmethod
    def attention(q, K, V, heads, head_dim, causal_row=None):
        """q [heads*hd]; K, V [n, heads*hd]."""
        n = K.shape[0]
        qh = q.reshape(heads, head_dim)
        Kh = K.reshape(n, heads, head_dim)
        Vh = V.reshape(n, heads, head_dim)
        s = np.einsum("hd,nhd->hn", qh, Kh) / np.sqrt(head_dim)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        return np.einsum("hn,nhd->hd", p, Vh).reshape(-1)

    @staticmethod
    def first_argmax(v):
        v = np.where(np.isnan(v), -np.inf, v)
        return int(np.argmax(v))  # numpy returns the first maximal index

    def ffn(self, x, alpha, w_in, w_out, hidden):
        g = w_in @ self.rms(x, alpha)
        a, b = g[:hidden], g[hidden:]
        return w_out @ (a / (1.0 + np.exp(-a)) * b)

    # -- session -------------------------------------------------------------
    def new_state(self):
        return {"ring": np.full((17, RING), -2, dtype=np.int64), "off": 0,
                "K": [[] for _ in range(self.c.layers)],
                "V": [[] for _ in range(self.c.layers)]}

    def prefilled_state(self, k, v):
        """A session that resumes at offset n with the temporal window already holding
        positions 0..n-1 of every layer: k, v [layers][n][dim] (any float dtype, taken
        as already-rotated rows).  The clock moves without generating anything, as
        `MoshiState::advance_clock` does, so the delayed-token ring stays all
        UNGENERATED (-2)."""
        st = self.new_state()
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        n = k.shape[1]
        assert k.shape == v.shape == (self.c.layers, n, self.c.dim) and n <= self.c.context
        for layer in range(self.c.layers):
            st["K"][layer] = [k[layer, p].copy() for p in range(n)]
            st["V"][layer] = [v[layer, p].copy() for p in range(n)]
        st["off"] = n
        return st

    def embed_row(self, table, tok):
        if tok == -1:
            return np.zeros(table.shape[1])
        return table[max(int(tok), 0)]

    def temporal(self, st, x):
        c, W = self.c, self.W
        pos = st["off"]
        for l in range(c.layers):
            qkv = W["in_proj"][l] @ self.rms(x, W["norm1"][l])
            q, k, v = np.split(qkv, 3)
            q = self.rope(q, pos, c.head_dim)
            k = self.rope(k, pos, c.head_dim)
            if c.kv_dtype == "bf16":
                k, v = bf16_round(k), bf16_round(v)
            st["K"][l].append(k)
            st["V"][l].append(v)
            st["K"][l] = st["K"][l][-c.context:]
            st["V"][l] = st["V"][l][-c.context:]
            o = self.attention(q, np.array(st["K"][l]), np.array(st["V"][l]),
                               c.heads, c.head_dim)
            x = x + W["out_proj"][l] @ o
            x = x + self.ffn(x, W["norm2"][l], W["gate_in"][l], W["gate_out"][l], c.hidden)
        return self.rms(x, W["out_norm"])

    def dep_input(self, tout, cb, prev):
        W = self.W
        table = W["dep_text_emb"] if cb == 0 else W["dep_emb"][cb - 1]
        return W["dep_in"][cb] @ tout + self.embed_row(table, prev)

    def depformer(self, tout, text, forced=None):
        """Incremental cycle (per-step K/V appended), own argmaxes; forced = [9]."""
        c, W = self.c, self.W
        Ks = [[] for _ in range(c.dlayers)]
        Vs = [[] for _ in range(c.dlayers)]
        prev = text if forced is None else forced[0]
        logits, toks = [], []
        for cb in range(8):
            x = self.dep_input(tout, cb, prev)
            for l in range(c.dlayers):
                qkv = W["d_in_proj"][l, cb] @ self.rms(x, W["dnorm1"][l])
                q, k, v = np.split(qkv, 3)
                Ks[l].append(k)
                Vs[l].append(v)
                o = self.attention(q, np.array(Ks[l]), np.array(Vs[l]), c.dheads, c.dhead_dim)
                x = x + W["d_out_proj"][l, cb] @ o
                x = x + self.ffn(x, W["dnorm2"][l], W["d_gate_in"][l, cb],
                                 W["d_gate_out"][l, cb], c.dhidden)
            lg = W["linears"][cb] @ x
            logits.append(lg)
            toks.append(self.first_argmax(lg))
            prev = toks[-1] if forced is None else forced[1 + cb]
        return np.array(logits), np.array(toks)

    def depformer_from_scratch(self, tout, prevs, upto):
        """Logits of step `upto`, recomputing steps 0..upto as one causal sequence:
        position j uses step-j weights and conditions on prevs[j]."""
        c, W = self.c, self.W
        n = upto + 1
        X = np.stack([self.dep_input(tout, j, prevs[j]) for j in range(n)])
        for l in range(c.dlayers):
            H = np.stack([self.rms(X[j], W["dnorm1"][l]) for j in range(n)])
            QKV = np.stack([W["d_in_proj"][l, j] @ H[j] for j in range(n)])
            Q, K, V = QKV[:, :c.ddim], QKV[:, c.ddim:2 * c.ddim], QKV[:, 2 * c.ddim:]
            O = np.stack([self.attention(Q[j], K[:j + 1], V[:j + 1], c.dheads, c.dhead_dim)
                          for j in range(n)])
            X = X + np.stack([W["d_out_proj"][l, j] @ O[j] for j in range(n)])
            X = X + np.stack([self.ffn(X[j], W["dnorm2"][l], W["d_gate_in"][l, j],
                                       W["d_gate_out"][l, j], c.dhidden) for j in range(n)])
        return W["linears"][upto] @ X[upto]

    def step(self, st, user, forced=None):
        c, W = self.c, self.W
        ring, off = st["ring"], st["off"]
        for k in range(8):
            s = 9 + k
            ring[s, (off + DELAYS[s]) % RING] = user[k]
        inp = np.where(off <= DELAYS, np.where(np.arange(17) == 0, c.text_card, c.audio_card),
                       ring[np.arange(17), off % RING])
        x = np.zeros(c.dim)
        for k in range(16):
            x = x + self.embed_row(W["emb"][k], inp[1 + k])
        x = x + self.embed_row(W["text_emb"], inp[0])
        emb_sum = x.copy()
        tout = self.temporal(st, x)
        text_logits = W["text_linear"] @ tout
        text = self.first_argmax(text_logits)
        audio_logits, audio = self.depformer(tout, text, forced)
        st["off"] = off = off + 1
        gen = np.concatenate([[text], audio]) if forced is None else np.asarray(forced)
        ring[:9, off % RING] = gen
        out = None
        if off > 1:
            out = ring[np.arange(9), (off - 1 + DELAYS[:9]) % RING].copy()
        return {"input_tokens": inp, "emb_sum": emb_sum, "tout": tout,
                "text_logits": text_logits, "audio_logits": audio_logits,
                "own": np.concatenate([[text], audio]), "out": out}
