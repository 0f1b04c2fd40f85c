"""The decode-attention entry point that allocates nothing, checked against
the workspace-based entry point (gpt2_attention) through the C ABI.

Collected last on purpose: a failure here leaves every other test already run.
It serves callers that cannot allocate device memory (a plugin given only
pointers and a stream, a process whose memory another allocator holds, a
path that must avoid cudaMalloc's synchronisation); its partial results live
in the library's own fixed 1 MiB device array."""
import ctypes as C

import numpy as np
import pytest
import torch

from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import assert_bf16_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _case(rng, B, h, t_past, t_cap):
    q = S.round_to_bf16(rng.standard_normal((B, h, 1, 64)))
    kv = np.zeros((B, 2, h, t_cap, 64), np.float32)
    kv[:, :, :, :t_past + 1] = S.round_to_bf16(rng.standard_normal((B, 2, h, t_past + 1, 64)))
    return dev(q), dev(kv)


def _call(G, q, kv, t_past, splits, out):
    B, h, _, dh = q.shape
    return G.LIB.gpt2_attention_decode_noalloc(
        C.c_void_p(q.data_ptr()), C.c_void_p(kv.data_ptr()), B, h, t_past, kv.shape[-2], dh, splits,
        C.c_void_p(out.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("B,h,t_past,splits", [(1, 4, 1000, 0), (2, 3, 300, 5), (32, 16, 1023, 0),
                                               (3, 2, 77, 1)])
def test_noalloc_matches_workspace_entry_point(G, B, h, t_past, splits):
    rng = np.random.default_rng(B * 100 + h + t_past)
    q, kv = _case(rng, B, h, t_past, t_past + 3)
    ctx = G.Context(50257, 1024, 1024, 16, 1, G.GPT2_BF16, max(B, 8), 8)
    ref = host(G.gpt2_attention(ctx, q, kv, t_past))
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    outs = []
    for _ in range(2):  # two calls in a row share the array
        out = torch.full((B, 1, h * 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(G, q, kv, t_past, splits, out) == G.GPT2_OK
        torch.cuda.synchronize()
        got = host(out)
        assert_bf16_close(got, ref, what="no-alloc decode attention")
        outs.append(got)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_noalloc_rejects_requests_beyond_its_array(G):
    rng = np.random.default_rng(1)
    q, kv = _case(rng, 32, 16, 100, 128)
    out = torch.empty((32, 1, 16 * 64), dtype=torch.bfloat16, device="cuda")
    # 32 * 16 * 64 partial results of 66 floats need 8.6 MB > 1 MiB.
    assert _call(G, q, kv, 100, 64, out) == G.GPT2_ERR_WORKSPACE
    assert _call(G, q, kv, 128, 0, out) == G.GPT2_ERR_CTX_OVERFLOW
    assert _call(G, q, kv, 100, -1, out) == G.GPT2_ERR_INVALID_ARG
    torch.cuda.synchronize()
