"""Kernel-level parity of the split-K decode attention (rq_attention) with the
oracle's `attend`, at edge sizes: one key, a window still filling, a window that
has wrapped (positions past the context), the full 3000-slot Moshi context, every
supported head size, f32 and bf16 caches, mixed positions in one batch."""
import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def window_rows(cache, pos, C):
    n = min(pos + 1, C)
    return np.stack([cache[p % C] for p in range(pos + 1 - n, pos + 1)])


@pytest.mark.parametrize("B,H,hd,C,positions,dtype", [
    (1, 4, 64, 64, [0], torch.float32),          # one key: output is v exactly
    (1, 4, 64, 64, [37], torch.float32),         # window still filling, ragged last split
    (1, 4, 64, 64, [200], torch.float32),        # wrapped window (slots reused)
    (3, 2, 32, 130, [5, 129, 400], torch.float32),
    (2, 16, 64, 512, [63, 64], torch.bfloat16),
    (1, 32, 128, 3000, [2999], torch.bfloat16),  # full Moshi context
    (2, 32, 128, 3000, [3500, 1], torch.bfloat16),
])
def test_attention_matches_oracle(B, H, hd, C, positions, dtype):
    g = torch.Generator().manual_seed(B * 1000 + C)
    D = H * hd
    q = torch.randn(B, D, generator=g)
    k = torch.randn(B, C, D, generator=g).to(dtype)
    v = torch.randn(B, C, D, generator=g).to(dtype)
    pos = torch.tensor(positions, dtype=torch.int32)
    out = binding.attention(q.cuda(), k.cuda(), v.cuda(), pos.cuda(), H, hd).cpu().numpy()
    for b in range(B):
        ks = window_rows(k[b].float().numpy(), positions[b], C)
        vs = window_rows(v[b].float().numpy(), positions[b], C)
        want = oracle.attend(q[b].numpy(), ks, vs, H, hd)
        if len(ks) == 1:
            np.testing.assert_array_equal(out[b], want)
        else:
            np.testing.assert_allclose(out[b], want, rtol=1e-4, atol=2e-5)


@pytest.mark.parametrize("B", [256, 257])
def test_attention_many_sessions(B):
    """Up to 256 sessions the kernel numbers only the splits inside each window; past that
    it walks every (session, split, head) and skips the empty ones.  Both must agree with
    the oracle on windows of every length class (one key, a ragged split, full, wrapped)."""
    H, hd, C = 2, 32, 96
    g = torch.Generator().manual_seed(4242 + B)
    D = H * hd
    positions = [int(x) for x in torch.randint(0, 3 * C, (B,), generator=g)]
    positions[:4] = [0, 37, C - 1, 2 * C + 5]
    q = torch.randn(B, D, generator=g)
    k = torch.randn(B, C, D, generator=g)
    v = torch.randn(B, C, D, generator=g)
    pos = torch.tensor(positions, dtype=torch.int32)
    out = binding.attention(q.cuda(), k.cuda(), v.cuda(), pos.cuda(), H, hd).cpu().numpy()
    for b in list(range(8)) + list(range(B - 8, B)):
        ks = window_rows(k[b].numpy(), positions[b], C)
        vs = window_rows(v[b].numpy(), positions[b], C)
        want = oracle.attend(q[b].numpy(), ks, vs, H, hd)
        if len(ks) == 1:
            np.testing.assert_array_equal(out[b], want)
        else:
            np.testing.assert_allclose(out[b], want, rtol=1e-4, atol=2e-5)


def test_attention_rejects_bad_arguments():
    L = binding.load()
    assert L.rq_attention(1, 4, 48, 64, 0, 1, 1, 1, 1, 1, 1, 1 << 20, None) == binding.RQ_ERR_UNSUPPORTED
    assert L.rq_attention(0, 4, 64, 64, 0, 1, 1, 1, 1, 1, 1, 1 << 20, None) == binding.RQ_ERR_ARG
    need = L.rq_attention_workspace_size(1, 4, 64, 64)
    assert L.rq_attention(1, 4, 64, 64, 0, 1, 1, 1, 1, 1, 1, need - 1, None) == binding.RQ_ERR_ARG
