"""rq_attention_noalloc: decode attention for callers that cannot allocate device
memory (a real-time audio thread that must not stall in cudaMalloc, a plug-in with a
fixed memory budget).  Called through the C ABI, two calls in a row with different
shapes, each compared with rq_attention -- the entry point that takes a caller
workspace -- and with the CPU oracle's `attend`, within the tolerance of the attention
parity tests.  The second call splits its windows into several 64-position parts but
fewer than the first, so its merge reads partials written over the first call's
leftovers.  Oversized problems are refused before any launch.

This file is collected last so that a run stopping at the first failure has already
run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from rq_transformer_frame_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = binding.load()
    P, I32 = C.c_void_p, C.c_int32
    L.rq_attention_noalloc.argtypes = [I32, I32, I32, I32, I32, P, P, P, P, P, P]
    L.rq_attention_noalloc.restype = C.c_int
    return L


def _case(B, H, hd, ctx, positions, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    D = H * hd
    q = torch.randn(B, D, generator=g).cuda()
    k = torch.randn(B, ctx, D, generator=g).to(dtype).cuda()
    v = torch.randn(B, ctx, D, generator=g).to(dtype).cuda()
    pos = torch.tensor(positions, dtype=torch.int32).cuda()
    return q, k, v, pos


def _noalloc(L, q, k, v, pos, H, hd):
    B, ctx = k.shape[0], k.shape[1]
    out = torch.full((B, H * hd), float("nan"), device="cuda")
    kvt = binding.RQ_BF16 if k.dtype == torch.bfloat16 else binding.RQ_F32
    stream = torch.cuda.current_stream()
    rc = L.rq_attention_noalloc(B, H, hd, ctx, kvt, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                pos.data_ptr(), out.data_ptr(), C.c_void_p(stream.cuda_stream))
    return rc, out


def _oracle_attend(q, k, v, positions, H, hd):
    """The oracle's `attend` over each query's window: positions
    max(0, pos - ctx + 1) .. pos, position j in cache slot j % ctx."""
    ctx = k.shape[1]
    kk, vv, qq = k.float().cpu().numpy(), v.float().cpu().numpy(), q.cpu().numpy()
    out = []
    for b, pos in enumerate(positions):
        slots = [j % ctx for j in range(max(0, pos - ctx + 1), pos + 1)]
        out.append(oracle.attend(qq[b], kk[b][slots], vv[b][slots], H, hd))
    return np.stack(out)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    cases = [
        # Moshi temporal shape: 47 splits of the 3000-slot window for session 0
        (2, 32, 128, 3000, [2999, 17], torch.bfloat16, 1),
        # then 5 and 1 splits: the merge reads partials over the first call's leftovers
        (2, 8, 64, 512, [300, 5], torch.float32, 2),
    ]
    for B, H, hd, ctx, positions, dtype, seed in cases:
        q, k, v, pos = _case(B, H, hd, ctx, positions, dtype, seed)
        rc, got = _noalloc(lib, q, k, v, pos, H, hd)
        assert rc == binding.RQ_OK
        want = binding.attention(q, k, v, pos, H, hd)
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        np.testing.assert_allclose(got, want.cpu().numpy(), rtol=1e-4, atol=2e-5)
        np.testing.assert_allclose(got, _oracle_attend(q, k, v, positions, H, hd),
                                   rtol=1e-4, atol=2e-5)


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    B, H, hd, ctx = 64, 32, 128, 3000  # needs ~50 MB of partials, far above 4 MiB
    assert lib.rq_attention_workspace_size(B, H, hd, ctx) > (4 << 20)
    q, k, v, pos = _case(1, 1, 32, 1, [0], torch.float32, 3)  # never read
    out = torch.zeros(4, device="cuda")
    rc = lib.rq_attention_noalloc(B, H, hd, ctx, binding.RQ_BF16, q.data_ptr(), k.data_ptr(),
                                  v.data_ptr(), pos.data_ptr(), out.data_ptr(), None)
    assert rc == binding.RQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 0)
