"""The decode-attention entry point that allocates nothing, checked through the
C ABI against the fp64 oracle and against the workspace-based entry point
(gpt2_attention).

Collected last on purpose: a failure here leaves every other test already run.
It serves callers that cannot allocate device memory (a plugin given only
pointers and a stream, a process whose memory another allocator holds, a
path that must avoid cudaMalloc's synchronisation); its partial results live
in the library's own fixed 1 MiB device array, which every call shares."""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
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
    return q, kv


def _oracle(q, kv, t_past):
    k = kv[:, 0, :, :t_past + 1].astype(np.float64)
    v = kv[:, 1, :, :t_past + 1].astype(np.float64)
    return O.merge_heads(O.causal_attention(q.astype(np.float64), k, v))


def _call(G, q, kv, t_past, splits, out):
    B, h, _, dh = q.shape
    return G.LIB.gpt2_attention_decode_noalloc(
        C.c_void_p(q.data_ptr()), C.c_void_p(kv.data_ptr()), B, h, t_past, kv.shape[-2], dh, splits,
        C.c_void_p(out.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run(G, q, kv, t_past, splits):
    B, h = q.shape[:2]
    out = torch.full((B, 1, h * 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call(G, q, kv, t_past, splits, out) == G.GPT2_OK
    torch.cuda.synchronize()
    return host(out)


@pytest.mark.parametrize("B,h,t_past,splits", [(1, 4, 1000, 0), (2, 3, 300, 5), (32, 16, 1023, 0),
                                               (3, 2, 77, 1)])
def test_noalloc_matches_oracle_and_workspace_entry_point(G, B, h, t_past, splits):
    rng = np.random.default_rng(B * 100 + h + t_past)
    qn, kvn = _case(rng, B, h, t_past, t_past + 3)
    q, kv = dev(qn), dev(kvn)
    ref = _oracle(qn, kvn, t_past)
    ctx = G.Context(50257, 1024, 1024, 16, 1, G.GPT2_BF16, max(B, 8), 8)
    ws_out = host(G.gpt2_attention(ctx, q, kv, t_past))
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    outs = []
    for _ in range(2):  # two calls in a row share the array
        got = _run(G, q, kv, t_past, splits)
        assert_bf16_close(got, ref, what="no-alloc decode attention vs oracle")
        assert_bf16_close(got, ws_out, what="no-alloc vs workspace decode attention")
        outs.append(got)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_noalloc_after_a_larger_layout(G):
    # The first call fills the shared array with many splits of many heads;
    # the second, with a different (sequence, head, split) layout, must not
    # read any of that call's leftovers.
    rng = np.random.default_rng(5)
    q1n, kv1n = _case(rng, 4, 25, 900, 904)          # 4 * 25 * 16 partials
    q2n, kv2n = _case(rng, 3, 7, 500, 512)           # 3 * 7 * 5 partials
    q1, kv1, q2, kv2 = dev(q1n), dev(kv1n), dev(q2n), dev(kv2n)
    got1 = _run(G, q1, kv1, 900, 16)
    assert_bf16_close(got1, _oracle(q1n, kv1n, 900), what="large layout")
    ref2 = _oracle(q2n, kv2n, 500)
    got2 = _run(G, q2, kv2, 500, 5)
    assert_bf16_close(got2, ref2, what="smaller layout after a larger one")
    got2b = _run(G, q2, kv2, 500, 5)
    np.testing.assert_array_equal(got2, got2b)


def test_noalloc_rejects_requests_beyond_its_array(G):
    rng = np.random.default_rng(1)
    qn, kvn = _case(rng, 32, 16, 100, 128)
    q, kv = dev(qn), dev(kvn)
    out = torch.empty((32, 1, 16 * 64), dtype=torch.bfloat16, device="cuda")
    # 32 * 16 * 64 partial results of 66 floats need 8.6 MB > 1 MiB.
    assert _call(G, q, kv, 100, 64, out) == G.GPT2_ERR_WORKSPACE
    assert _call(G, q, kv, 128, 0, out) == G.GPT2_ERR_CTX_OVERFLOW
    assert _call(G, q, kv, 100, -1, out) == G.GPT2_ERR_INVALID_ARG
    torch.cuda.synchronize()
