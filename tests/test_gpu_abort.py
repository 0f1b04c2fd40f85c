"""The failure path of the real kernels, on the GPU, without a fault.

Every wait of the tensor-core GEMM and of the prefill attention is bounded.
With the context's wait limit set to a few nanoseconds, the first wait that
is not already satisfied runs out on ordinary work: the kernel raises the
error word, drains the copies it issued, retires the MMAs it issued, frees
TMEM and returns.  The test checks that gpt2_sync_status reports the timeout
and that the same context, with the default limit back, computes correctly
(the GPU and the context stay usable).  Single-CTA and CTA-pair GEMMs, the
attention, a whole block, and the decode attention (through a context, and
through the entry point without one, whose own error word and wait limit
serve the same purpose) are covered."""
import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import assert_bf16_close, assert_gemm_f32_close, block_to_device, dev, host

pytestmark = pytest.mark.gpu

SHORT_NS = 5


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _ctx(G):
    return G.Context(50257, 1024, 768, 12, 1, G.GPT2_BF16, 8, 1024)


# (1000, 768, 768): single CTAs; (640, 768, 3072): CTA pairs (K >= 1024).
@pytest.mark.parametrize("M,N,K", [(1000, 768, 768), (640, 768, 3072)])
def test_gemm_wait_runs_out_then_context_recovers(G, M, N, K):
    rng = np.random.default_rng(M + K)
    A = S.round_to_bf16(rng.standard_normal((M, K)))
    W = S.round_to_bf16(0.05 * rng.standard_normal((N, K)))
    bias = S.round_to_bf16(0.1 * rng.standard_normal(N))
    resid = rng.standard_normal((M, N)).astype(np.float32)
    ctx = _ctx(G)
    G.gpt2_ctx_set_wait_limit(ctx, SHORT_NS)
    for _ in range(3):
        G.gpt2_linear(ctx, G.GPT2_EPI_BIAS_RESID, dev(A), dev(W), dev(bias),
                      dev(resid, torch.float32))
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_DEVICE_TIMEOUT
    G.gpt2_ctx_set_wait_limit(ctx, 0)
    out = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS_RESID, dev(A), dev(W), dev(bias),
                        dev(resid, torch.float32))
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert_gemm_f32_close(host(out), O.linear(A, W, bias) + resid, A, W, what="after the timeout")


def test_attention_wait_runs_out_then_context_recovers(G):
    rng = np.random.default_rng(11)
    B, h, T = 2, 3, 300
    q = S.round_to_bf16(rng.standard_normal((B, h, T, 64)))
    kv = S.round_to_bf16(rng.standard_normal((B, 2, h, T, 64)))
    ctx = _ctx(G)
    G.gpt2_ctx_set_wait_limit(ctx, SHORT_NS)
    for _ in range(3):
        G.gpt2_attention(ctx, dev(q), dev(kv), 0)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_DEVICE_TIMEOUT
    G.gpt2_ctx_set_wait_limit(ctx, 0)
    out = G.gpt2_attention(ctx, dev(q), dev(kv), 0)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    ref = O.merge_heads(O.causal_attention(q.astype(np.float64), kv[:, 0].astype(np.float64),
                                           kv[:, 1].astype(np.float64)))
    assert_bf16_close(host(out), ref, what="attention after the timeout")


def test_block_wait_runs_out_then_context_recovers(G):
    w = S.WORKLOADS["block_bf16_d768"]
    p = S.block_params(w, seed=4)
    x = S.block_input(w, seed=4, B=2, T=256)
    ctx = _ctx(G)
    G.gpt2_ctx_set_wait_limit(ctx, SHORT_NS)
    G.gpt2_block_forward(ctx, dev(x), block_to_device(p), 2, 256, w.d, w.n_head)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_DEVICE_TIMEOUT
    G.gpt2_ctx_set_wait_limit(ctx, 0)
    out = G.gpt2_block_forward(ctx, dev(x), block_to_device(p), 2, 256, w.d, w.n_head)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert_bf16_close(host(out), O.block_forward(x, p, w.n_head)[0], what="block after the timeout")


def _decode_case(seed, B, h, t_past):
    rng = np.random.default_rng(seed)
    q = S.round_to_bf16(rng.standard_normal((B, h, 1, 64)))
    kv = S.round_to_bf16(rng.standard_normal((B, 2, h, t_past + 1, 64)))
    ref = O.merge_heads(O.causal_attention(q.astype(np.float64), kv[:, 0].astype(np.float64),
                                           kv[:, 1].astype(np.float64)))
    return q, kv, ref


def _nan_or_right(got, ref):
    """Each (sequence, head) output row either NaN (its wait ran out) or the
    oracle's; at least one row hit by the timeout."""
    B, _, hd = got.shape
    rows = got.reshape(B, hd // 64, 64)
    want = ref.reshape(B, hd // 64, 64)
    nan_rows = np.isnan(rows).all(axis=-1)
    assert nan_rows.any()
    assert not np.isnan(rows[~nan_rows]).any()
    if (~nan_rows).any():
        assert_bf16_close(rows[~nan_rows], want[~nan_rows], what="rows that finished")


# (2, 3): split keys and the combine kernel; (32, 16): one split per (sequence, head).
@pytest.mark.parametrize("B,h", [(2, 3), (32, 16)])
def test_decode_attention_wait_runs_out_then_context_recovers(G, B, h):
    """The decode kernel's waits take the context's limit too: a timed-out
    (sequence, head) is written as NaN, the status reports the timeout, and
    the context then computes correctly."""
    q, kv, ref = _decode_case(12, B, h, 700)
    ctx = G.Context(50257, 1024, 1024, 16, 1, G.GPT2_BF16, 32, 8)
    G.gpt2_ctx_set_wait_limit(ctx, SHORT_NS)
    got = G.gpt2_attention(ctx, dev(q), dev(kv), 700)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_DEVICE_TIMEOUT
    _nan_or_right(host(got), ref)
    G.gpt2_ctx_set_wait_limit(ctx, 0)
    out = G.gpt2_attention(ctx, dev(q), dev(kv), 700)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert_bf16_close(host(out), ref, what="decode attention after the timeout")


def test_noalloc_decode_wait_runs_out_then_recovers(G):
    """The entry point without a context reports a timed-out wait through its
    own error word (gpt2_attention_decode_noalloc_status) and NaN rows, then
    computes correctly once the default limit is back."""
    q, kv, ref = _decode_case(13, 2, 3, 700)
    assert G.gpt2_attention_decode_noalloc_status() == G.GPT2_OK
    G.gpt2_attention_decode_noalloc_set_wait_limit(SHORT_NS)
    try:
        got = G.gpt2_attention_decode_noalloc(dev(q), dev(kv), 700, splits=4)
        assert G.gpt2_attention_decode_noalloc_status() == G.GPT2_ERR_DEVICE_TIMEOUT
    finally:
        G.gpt2_attention_decode_noalloc_set_wait_limit(0)
    _nan_or_right(host(got), ref)
    assert G.gpt2_attention_decode_noalloc_status() == G.GPT2_OK  # the read cleared it
    out = G.gpt2_attention_decode_noalloc(dev(q), dev(kv), 700, splits=4)
    assert G.gpt2_attention_decode_noalloc_status() == G.GPT2_OK
    assert_bf16_close(host(out), ref, what="no-alloc decode attention after the timeout")
