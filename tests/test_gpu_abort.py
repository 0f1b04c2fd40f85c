"""The failure path of the real kernels, on the GPU, without a fault.

Every wait of the tensor-core GEMM and of the prefill attention is bounded.
With the context's wait limit set to a few nanoseconds, the first wait that
is not already satisfied runs out on ordinary work: the kernel raises the
error word, drains the copies it issued, retires the MMAs it issued, frees
TMEM and returns.  The test checks that gpt2_sync_status reports the timeout
and that the same context, with the default limit back, computes correctly
(the GPU and the context stay usable).  Single-CTA and CTA-pair GEMMs, the
attention, and a whole block are covered."""
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
